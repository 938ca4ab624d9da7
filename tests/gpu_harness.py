"""Shared driver for the GPU parity tests: runs the CUDA megakernel (through the C ABI) and the oracle
on the same seeded inputs and compares every step.

Comparison rules (floating point decides an integer here, so near-ties are handled explicitly):
  * logits: max |gpu - oracle| <= tol over every row of every step, against the exact oracle;
  * greedy tokens: equal, unless the oracle's top-1 / top-2 gap is below 2 * tol, in which case either
    token is accepted; the oracle's token is fed to both sides (teacher forcing), so one near-tie never
    makes the two runs diverge;
  * MoE routing: the top-k is compared in the pages' precision (activations, hence the cached keys, values
    and latents, stored in bf16): a second oracle with bf16-stored caches decides each row's experts, the
    kernel's own picks must equal them except at near-ties (ROUTE_TIE), and the exact oracle and the kernel
    (through its routing override) both compute with them.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import Oracle
from synthetic import make_tokens, make_weights


class Report:
    def __init__(self):
        self.max_err = 0.0
        self.steps = 0
        self.token_mismatch = 0
        self.near_ties = 0
        self.route_ties = 0
        self.routed_rows = 0
        self.compared = 0
        self.errors = []


ROUTE_TIE = 1e-4   # router scores this close at the top-k boundary may be picked either way in fp32


def check_routing(orc, log, pos0, R: int, rep, what: str):
    """Compares the experts the kernel picked itself (its routing log, by position) with the routing oracle's
    own picks of its last call, as sets per (layer, sequence, row). A difference is accepted only where the
    oracle's k-th and (k+1)-th biased scores lie within ROUTE_TIE (a near-tie that fp32 may break the other
    way). Both sides then still compute with the routing oracle's picks (the kernel through its routing
    override, the exact oracle through forced_routing), so one near-tie never makes the runs diverge."""
    if log is None:
        return
    k = orc.cfg.top_k
    lg = log.cpu().numpy()
    for layer, (idx, biased) in orc.routing.items():
        B = idx.shape[0]
        for b in range(B):
            for r in range(R):
                got = np.sort(lg[layer, b, int(pos0[b]) + r])
                want = np.sort(idx[b, r])
                rep.routed_rows += 1
                if np.array_equal(got, want):
                    continue
                s = -np.sort(-biased[b, r])
                gap = s[k - 1] - s[k] if s.shape[0] > k else np.inf
                if gap < ROUTE_TIE:
                    rep.route_ties += 1
                else:
                    rep.errors.append(f"{what}: layer {layer} seq {b} row {r}: experts {got.tolist()} vs oracle "
                                      f"{want.tolist()} (boundary gap {gap:.3g})")


def compare_logits(gpu: np.ndarray, ref: np.ndarray, tol: float, rep: Report, what: str):
    err = float(np.max(np.abs(gpu.astype(np.float64) - ref)))
    rep.compared += 1
    rep.max_err = max(rep.max_err, err)
    if not np.isfinite(err) or err > tol:
        rep.errors.append(f"{what}: max |diff| {err:.4g} > {tol}")
    g_arg = gpu.argmax(-1)
    o_sorted = np.sort(ref, axis=-1)
    gap = o_sorted[..., -1] - o_sorted[..., -2]
    o_arg = ref.argmax(-1)
    for idx in np.ndindex(o_arg.shape):
        if g_arg[idx] != o_arg[idx]:
            if gap[idx] < 2 * tol:
                rep.near_ties += 1
            else:
                rep.token_mismatch += 1
                rep.errors.append(f"{what} row {idx}: greedy {g_arg[idx]} vs oracle {o_arg[idx]} (gap {gap[idx]:.3g})")


def oracle_prefill_blocks(orc, ctx: np.ndarray, block: int):
    """The oracle's prefill of ctx [B, T] run as consecutive blocks of `block` rows, each committed by the
    next call's positions (the same step semantics as one T-row block, with bounded memory)."""
    orc.reset()
    B, T = ctx.shape
    for c0 in range(0, T, block):
        orc.step(ctx[:, c0:c0 + block], np.full(B, c0, dtype=np.int64))
    orc.commit(T - (T - 1) // block * block)


def oracle_fork(orc1, B: int):
    """A batch-B oracle whose every sequence is a copy of sequence 0 of `orc1` (caches, states, counts):
    the oracle-side counterpart of mk_fork_sequence. Plain array copies; the weights are shared."""
    o = Oracle(orc1.cfg, orc1.w, B, orc1.max_ctx)
    o.c[:] = orc1.c[0]
    o.u[:] = orc1.u[0]
    for i, (K, V) in orc1.kv.items():
        o.kv[i] = (np.repeat(K[:1], B, axis=0), np.repeat(V[:1], B, axis=0))
    for i, lat in orc1.lat.items():
        o.lat[i] = np.repeat(lat[:1], B, axis=0)
    for i, S in orc1.S.items():
        o.S[i] = np.repeat(S[:1], B, axis=0)
        o.snaps[i] = [orc1.snaps[i][0].copy() for _ in range(B)]
    return o


def attention_ring_chunks(mk, B: int, R: int, T: int) -> list:
    """For every attention op of the (B, R) program on this device: how many weight-ring chunks one
    attention instruction streams at context T (positions per chunk instruction / positions per ring
    chunk). What the long-context tests assert: the multi-chunk online-softmax loop really runs."""
    from decode_megakernel_04_gb300 import binding
    n_sm = mk.info().n_sm
    ops, _ = binding.plan(mk.desc, mk.wtab, n_sm, B, R)
    out = []
    for op in ops:
        if op["type"] == 3:      # GQA attention: K and V of P positions per 32 KB chunk
            P = 32768 // (4 * op["head_dim"])
        elif op["type"] == 6:    # MLA attention: 576-wide bf16 latents
            P = 32768 // (2 * 576)
        else:
            continue
        per_instr = -(-T // op["nchunk"])
        out.append(-(-per_instr // P))
    return out


# long-context oracle prefills (one sequence), kept for the other batch sizes of the same model and context
_PREFILLED: dict = {}


def run_case(cfg, B: int, T: int, decode_steps: int = 0, verify_accepts=(), R_verify: int = 8,
             seed: int = 0, tol: float = 2e-2, max_ctx: int | None = None, check_argmax: bool = True,
             fork: bool = False, oracle_block: int | None = None, min_ring_chunks: int = 0):
    """Prefill T context tokens per sequence, then `decode_steps` greedy single-row steps, then one
    R_verify-row verify step per entry of verify_accepts (the entry is the accepted length of that block,
    applied by the next call's positions).
    fork: one context is prefilled for sequence 0 and copied to the others (mk_fork_sequence on the GPU,
    array copies in the oracle); the steps then give every sequence its own tokens.
    oracle_block: the oracle prefills in blocks of this many rows (long contexts).
    min_ring_chunks: assert that every attention instruction streams at least this many ring chunks."""
    from decode_megakernel_04_gb300 import Megakernel

    dev = torch.device("cuda")
    w = make_weights(cfg, seed=seed, device=dev)
    rows_max = R_verify if verify_accepts else 1
    extra = decode_steps + (len(verify_accepts) + 1) * R_verify + 8
    max_ctx = max_ctx or (T + extra)
    mk = Megakernel(cfg, w, max_batch=B, max_rows=max(rows_max, 8), max_ctx=max_ctx)
    rep = Report()
    if min_ring_chunks:
        for R_ in ([1] if decode_steps or not verify_accepts else []) + ([R_verify] if verify_accepts else []):
            chunks = attention_ring_chunks(mk, B, R_, T)
            assert chunks and min(chunks) >= min_ring_chunks, f"rows {R_}: ring chunks per instruction {chunks}"
    Bc = 1 if fork else B
    ctx = make_tokens(seed, "ctx", (Bc, T), cfg.vocab, device=dev).contiguous()
    log = override = orc_r = None
    if cfg.ffn == "moe":
        log = torch.full((cfg.n_layers, B, max_ctx, cfg.top_k), -1, dtype=torch.int32, device=dev)
        mk.set_routing_log(log)
        override = torch.full((cfg.n_layers, B, max_ctx, cfg.top_k), -1, dtype=torch.int32, device=dev)
        mk.set_routing_override(override)

    def oracle_call(o, o_r, tok, pos):
        """The exact oracle's logits of one call; for MoE models the routing oracle (bf16-stored caches, the
        pages' activation precision) runs first, and its picks drive the exact oracle and the kernel."""
        if o_r is not None:
            o_r.step(tok, pos)
            forced = {i: idx for i, (idx, _) in o_r.routing.items()}
            o.forced_routing = forced
            for i, idx in forced.items():
                for b in range(idx.shape[0]):
                    override[i, b, int(pos[b]):int(pos[b]) + idx.shape[1]] = torch.from_numpy(
                        idx[b].astype(np.int32)).to(dev)
        return o.step(tok, pos)

    key = (cfg, T, seed, max_ctx, oracle_block)
    if fork and oracle_block and key in _PREFILLED:
        orc = _PREFILLED[key]
    else:
        orc = Oracle(cfg, w, Bc, max_ctx)
        if cfg.ffn == "moe":
            orc_r = Oracle(cfg, orc.w, Bc, max_ctx, cache_round="bf16")
        if oracle_block:
            oracle_prefill_blocks(orc, ctx.cpu().numpy(), oracle_block)
        else:
            orc.reset()
            if orc_r is not None:
                orc_r.reset()
            oracle_call(orc, orc_r, ctx.cpu().numpy(), np.zeros(Bc, dtype=np.int64))
            orc.commit(T)
            if orc_r is not None:
                orc_r.commit(T)
        if fork and oracle_block:
            _PREFILLED[key] = orc
    mk.prefill(ctx)
    for b in range(1, B if fork else 1):
        mk.fork(0, b)
    if orc_r is not None:
        check_routing(orc_r, log, np.zeros(Bc, dtype=np.int64), T, rep, "prefill")
    if fork:
        orc = oracle_fork(orc, B)   # copies: the cached prefill stays untouched
    pos = np.full(B, T, dtype=np.int64)
    tok = make_tokens(seed, "start", (B, 1), cfg.vocab).numpy().astype(np.int64)
    V = cfg.vocab
    for s in range(decode_steps):
        ref = oracle_call(orc, orc_r, tok, pos)[:, 0]
        logits = torch.empty((B, V), device=dev, dtype=torch.float32)
        am = torch.empty((B,), device=dev, dtype=torch.int32)
        mk.step(torch.from_numpy(tok.astype(np.int32)).to(dev), torch.from_numpy(pos.astype(np.int32)).to(dev),
                logits, am)
        st = mk.status()
        assert st == 0, f"device status {st}"
        g = logits.cpu().numpy()
        check_routing(orc_r, log, pos, 1, rep, f"decode step {s}")
        compare_logits(g, ref, tol, rep, f"decode step {s}")
        if check_argmax:
            # the kernel's own argmax must be the argmax of the logits it wrote
            assert np.array_equal(am.cpu().numpy(), g.argmax(-1)), "in-kernel argmax differs from logits argmax"
        tok = ref.argmax(-1)[:, None].astype(np.int64)
        pos = pos + 1
        rep.steps += 1
    for vi, acc in enumerate(verify_accepts):
        drafts = make_tokens(seed, f"draft{vi}", (B, R_verify - 1), cfg.vocab).numpy().astype(np.int64)
        block = np.concatenate([tok, drafts], axis=1)
        ref = oracle_call(orc, orc_r, block, pos)
        logits = torch.empty((B * R_verify, V), device=dev, dtype=torch.float32)
        am = torch.empty((B * R_verify,), device=dev, dtype=torch.int32)
        mk.step(torch.from_numpy(block.astype(np.int32)).to(dev).contiguous(),
                torch.from_numpy(pos.astype(np.int32)).to(dev), logits, am)
        st = mk.status()
        assert st == 0, f"device status {st}"
        g = logits.cpu().numpy().reshape(B, R_verify, V)
        check_routing(orc_r, log, pos, R_verify, rep, f"verify block {vi}")
        compare_logits(g, ref, tol, rep, f"verify block {vi}")
        if check_argmax:
            assert np.array_equal(am.cpu().numpy().reshape(B, R_verify), g.argmax(-1))
        # accept `acc` rows: the next anchor is the oracle's greedy token after the last accepted row
        tok = ref[:, acc - 1].argmax(-1)[:, None].astype(np.int64)
        pos = pos + acc
        rep.steps += 1
    # one more decode step to check the commit of the last verify block
    if verify_accepts:
        ref = oracle_call(orc, orc_r, tok, pos)[:, 0]
        logits = torch.empty((B, V), device=dev, dtype=torch.float32)
        mk.step(torch.from_numpy(tok.astype(np.int32)).to(dev), torch.from_numpy(pos.astype(np.int32)).to(dev),
                logits, None)
        assert mk.status() == 0
        check_routing(orc_r, log, pos, 1, rep, "decode after verify")
        compare_logits(logits.cpu().numpy(), ref, tol, rep, "decode after verify")
    mk.close()
    return rep
