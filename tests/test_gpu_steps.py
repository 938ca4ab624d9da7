"""GPU: several greedy decode steps in one launch, and speculative verify with on-device greedy acceptance.

* mk_decode_steps runs N greedy steps in ONE launch (step s embeds the greedy token of step s - 1 on the
  device): its tokens equal N single-step calls token for token and its last logits equal theirs bit for bit
  (same program, same arithmetic), on a hybrid gated-delta-net / GQA stack and on a KDA / MLA / MoE stack;
  the tokens also follow the oracle's greedy decode (up to a near-tie, after which the two may diverge).
* mk_verify_step decides how many drafts greedy decoding accepts: blocks whose first k drafts are the
  oracle's greedy continuation accept k + 1 rows and emit the oracle's bonus token; the next call then takes
  its anchor and position straight from the device output and matches the oracle."""
import copy

import numpy as np
import pytest
import torch

from synthetic import config, make_tokens, make_weights

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from decode_megakernel_04_gb300 import _build
    _build.build()


def _hybrid():
    return config("hybrid_gdn_gqa", n_layers=4, d_model=512, ffn_dim=1024, vocab=4096)


def _moe():
    import dataclasses
    return dataclasses.replace(config("moe_kda_mla"), n_layers=4, d_model=1024, n_experts=16, top_k=4,
                               expert_dim=512, vocab=4096, lin_heads=8)


def _pair(cfg, w, B, T, seed, max_ctx):
    from decode_megakernel_04_gb300 import Megakernel
    dev = torch.device("cuda")
    ctx = make_tokens(seed, "ctx", (B, T), cfg.vocab, device=dev).contiguous()
    a = Megakernel(cfg, w, max_batch=B, max_rows=8, max_ctx=max_ctx)
    b = Megakernel(cfg, w, max_batch=B, max_rows=8, max_ctx=max_ctx)
    a.prefill(ctx)
    b.prefill(ctx)
    return a, b, ctx


@pytest.mark.parametrize("model", ["hybrid", "moe"])
def test_multi_step_equals_single_steps(model):
    cfg = _hybrid() if model == "hybrid" else _moe()
    dev = torch.device("cuda")
    w = make_weights(cfg, seed=3, device=dev)
    B, T, S = 2, 29, 12
    a, b, _ = _pair(cfg, w, B, T, 3, 64)
    tok0 = make_tokens(3, "first", (B,), cfg.vocab, device=dev).contiguous()
    pos0 = torch.full((B,), T, dtype=torch.int32, device=dev)
    out = torch.full((S, B), -1, dtype=torch.int32, device=dev)
    la = torch.empty((B, cfg.vocab), device=dev)
    a.steps(tok0, pos0, S, out, la)
    assert a.status() == 0
    tok = tok0.view(B, 1).clone()
    lb = torch.empty((B, cfg.vocab), device=dev)
    single = []
    for s in range(S):
        am = torch.empty((B,), dtype=torch.int32, device=dev)
        b.step(tok, pos0 + s, lb, am)
        assert b.status() == 0
        single.append(am.clone())
        tok = am.view(B, 1).clone()
    assert torch.equal(out, torch.stack(single)), (out, torch.stack(single))
    assert torch.equal(la, lb)
    # and the launch leaves the handle where S single steps leave it: one more single step on each agrees
    nxt = out[-1].view(B, 1).contiguous()
    for h, l in ((a, la), (b, lb)):
        h.step(nxt, pos0 + S, l, None)
        assert h.status() == 0
    assert torch.equal(la, lb)
    a.close()
    b.close()


def test_multi_step_follows_the_oracle_and_host_entry_point():
    from decode_megakernel_04_gb300 import Megakernel
    from oracle import Oracle
    cfg = _hybrid()
    dev = torch.device("cuda")
    w = make_weights(cfg, seed=4, device=dev)
    B, T, S = 2, 21, 16
    ctx = make_tokens(4, "ctx", (B, T), cfg.vocab, device=dev).contiguous()
    mk = Megakernel(cfg, w, max_batch=B, max_rows=8, max_ctx=64)
    mk.prefill(ctx)
    tok0 = make_tokens(4, "first", (B,), cfg.vocab).numpy().astype(np.int32)
    pos0 = np.full(B, T, dtype=np.int32)
    out = np.zeros((S, B), dtype=np.int32)
    mk.steps_host(tok0, pos0, S, out)
    orc = Oracle(cfg, w, B, 64)
    orc.prefill(ctx.cpu().numpy())
    tok = tok0.astype(np.int64)[:, None]
    live = np.ones(B, dtype=bool)   # sequences whose tokens still agree with the oracle's greedy decode
    for s in range(S):
        ref = orc.step(tok, pos0 + s)[:, 0]
        g = ref.argmax(-1)
        top2 = np.sort(ref, axis=-1)[:, -2:]
        for b in range(B):
            if live[b] and out[s, b] != g[b]:
                assert top2[b, 1] - top2[b, 0] < 2 * TOL, (s, b, out[s, b], g[b])
                live[b] = False     # a near-tie: the kernel took the other token and continues from it
        tok = g[:, None]
    assert live.any()
    mk.close()


def test_verify_step_accepts_on_device_and_chains():
    from decode_megakernel_04_gb300 import Megakernel
    from gpu_harness import Report, compare_logits
    from oracle import Oracle, ops
    cfg = _hybrid()
    dev = torch.device("cuda")
    w = make_weights(cfg, seed=5, device=dev)
    B, T, R = 2, 33, 8
    ctx = make_tokens(5, "ctx", (B, T), cfg.vocab, device=dev).contiguous()
    mk = Megakernel(cfg, w, max_batch=B, max_rows=R, max_ctx=96)
    mk.prefill(ctx)
    orc = Oracle(cfg, w, B, 96)
    orc.prefill(ctx.cpu().numpy())
    anchor = make_tokens(5, "anchor", (B,), cfg.vocab).numpy().astype(np.int64)
    rep = Report()
    pos = np.full(B, T, dtype=np.int64)
    for rnd, ks in enumerate(((2, 5), (7, 0), (0, 3))):
        # drafts: the oracle's greedy continuation for k_b tokens, then a different token
        seq = copy.deepcopy(orc)
        greedy = np.zeros((B, R), dtype=np.int64)
        t = anchor[:, None]
        for r in range(R):
            greedy[:, r] = seq.step(t, pos + r)[:, 0].argmax(-1)
            t = greedy[:, r:r + 1]
        block = np.zeros((B, R), dtype=np.int64)
        block[:, 0] = anchor
        for b, k in enumerate(ks):
            block[b, 1:1 + k] = greedy[b, :k]
            if k < R - 1:
                block[b, 1 + k] = (greedy[b, k] + 1) % cfg.vocab
        ref = orc.step(block, pos)
        logits = torch.empty((B * R, cfg.vocab), device=dev)
        acc = torch.full((3, B), -1, dtype=torch.int32, device=dev)
        mk.verify(torch.from_numpy(block.astype(np.int32)).to(dev).contiguous(),
                  torch.from_numpy(pos.astype(np.int32)).to(dev), acc, logits)
        assert mk.status() == 0
        compare_logits(logits.cpu().numpy().reshape(B, R, -1), ref, TOL, rep, f"verify {rnd}")
        got = acc.cpu().numpy()
        want = np.array([ops.greedy_accept(ref[b], block[b]) for b in range(B)]).T   # [2, B]: a, bonus
        agree = True
        for b in range(B):
            a, bonus = want[:, b]
            assert a == ks[b] + 1 or np.diff(np.sort(ref[b], axis=-1)[:, -2:], axis=-1).min() < 2 * TOL
            if got[0, b] != a or got[1, b] != bonus:
                # only an oracle near-tie at a deciding row may change the outcome
                gaps = np.diff(np.sort(ref[b], axis=-1)[:, -2:], axis=-1)[:, 0]
                assert gaps[:min(a, R)].min() < 2 * TOL, (rnd, b, got[:, b], a, bonus)
                agree = False
            assert got[2, b] == pos[b] + got[0, b]
        if not agree:
            break   # the two runs took different (both valid) paths: nothing further to compare
        # chain on the device: the next call's anchor and positions are the verify step's output; the oracle
        # takes the same step from its own acceptance (equal to the kernel's here)
        nxt_tok = acc[1].view(B, 1).contiguous()
        nxt_pos = acc[2].contiguous()
        l1 = torch.empty((B, cfg.vocab), device=dev)
        mk.step(nxt_tok, nxt_pos, l1, None)
        assert mk.status() == 0
        anchor = want[1].astype(np.int64)
        pos = pos + want[0].astype(np.int64)
        ref1 = orc.step(anchor[:, None], pos)[:, 0]
        compare_logits(l1.cpu().numpy(), ref1, TOL, rep, f"after verify {rnd}")
        anchor = ref1.argmax(-1)
        pos = pos + 1
    assert not rep.errors, "\n".join(rep.errors[:10])
    mk.close()
