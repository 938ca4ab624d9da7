"""GPU parity: the CUDA megakernel (called through the C ABI) against the oracle, element by element, on
the same seeded inputs. Logits within 2e-2 max-abs (bf16 weights, fp32 accumulation) and identical
greedy tokens except at oracle near-ties (see tests/gpu_harness.py)."""
import numpy as np
import pytest
import torch

from synthetic import config, make_tokens, make_weights

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from decode_megakernel_04_gb300 import _build
    _build.build()


def _check(rep):
    assert not rep.errors, "\n".join(rep.errors[:10])
    assert rep.token_mismatch == 0


def test_tiny_dense_greedy_16_steps():
    """The tiny dense workload as specified: batch 1, 128-token context, 16 greedy steps."""
    from gpu_harness import run_case
    rep = run_case(config("tiny_dense"), B=1, T=128, decode_steps=16, tol=TOL_BF16)
    _check(rep)


def test_tiny_dense_batch_and_verify():
    """Batch 3, ragged context (37, not a multiple of the 8-row prefill chunk), decode then 8-row verify
    blocks with accepted lengths 3, 8, 1 and 6."""
    from gpu_harness import run_case
    rep = run_case(config("tiny_dense"), B=3, T=37, decode_steps=2, verify_accepts=(3, 8, 1, 6), tol=TOL_BF16)
    _check(rep)


def test_tiny_dense_single_token_context():
    from gpu_harness import run_case
    rep = run_case(config("tiny_dense"), B=2, T=1, decode_steps=3, tol=TOL_BF16)
    _check(rep)


def test_hybrid_gdn_gqa_full_width_4_layers():
    """Full-width hybrid stack (d 5120, GQA 24/4 x 256, GDN 16 x 128, FFN 17408, vocab 151936), cut to 4
    layers (3 GDN + 1 GQA), batch 2, 61-token context, greedy decode and verify blocks."""
    from gpu_harness import run_case
    cfg = config("hybrid_gdn_gqa", n_layers=4)
    rep = run_case(cfg, B=2, T=61, decode_steps=2, verify_accepts=(3, 6), tol=TOL_BF16)
    _check(rep)


def test_hybrid_batch8_decode():
    from gpu_harness import run_case
    cfg = config("hybrid_gdn_gqa", n_layers=4)
    rep = run_case(cfg, B=8, T=20, decode_steps=2, tol=TOL_BF16)
    _check(rep)


def test_invalid_inputs_set_device_status():
    """A token outside the vocabulary and a position outside the committed window are rejected on the
    device (MK_ERR_DEVICE) without a fault; the handle keeps working afterwards."""
    from decode_megakernel_04_gb300 import Megakernel
    cfg = config("tiny_dense")
    dev = torch.device("cuda")
    w = make_weights(cfg, seed=0, device=dev)
    mk = Megakernel(cfg, w, max_batch=1, max_rows=8, max_ctx=64)
    mk.prefill(make_tokens(0, "ctx", (1, 10), cfg.vocab, device=dev))
    logits = torch.empty((1, cfg.vocab), device=dev)
    bad_tok = torch.tensor([[cfg.vocab]], dtype=torch.int32, device=dev)
    mk.step(bad_tok, torch.tensor([10], dtype=torch.int32, device=dev), logits)
    assert mk.status() == 6
    good = torch.tensor([[5]], dtype=torch.int32, device=dev)
    mk.step(good, torch.tensor([12], dtype=torch.int32, device=dev), logits)   # beyond c + u = 10
    assert mk.status() == 6
    mk.step(good, torch.tensor([10], dtype=torch.int32, device=dev), logits)
    assert mk.status() == 0
    assert torch.isfinite(logits).all()
    mk.close()


def test_host_entry_point_matches_device_entry_point():
    """mk_decode_step_host (host buffers, copies inside) returns the same greedy tokens and logits as
    mk_decode_step on an identically prepared handle."""
    from decode_megakernel_04_gb300 import Megakernel
    cfg = config("tiny_dense")
    dev = torch.device("cuda")
    w = make_weights(cfg, seed=1, device=dev)
    ctx = make_tokens(1, "ctx", (2, 16), cfg.vocab, device=dev)
    a = Megakernel(cfg, w, max_batch=2, max_rows=8, max_ctx=64)
    b = Megakernel(cfg, w, max_batch=2, max_rows=8, max_ctx=64)
    a.prefill(ctx)
    b.prefill(ctx)
    tok = np.array([[3], [9]], dtype=np.int32)
    pos = np.array([16, 16], dtype=np.int32)
    la = torch.empty((2, cfg.vocab), device=dev)
    ama = torch.empty((2,), dtype=torch.int32, device=dev)
    a.step(torch.from_numpy(tok).to(dev), torch.from_numpy(pos).to(dev), la, ama)
    assert a.status() == 0
    amb = np.zeros(2, dtype=np.int32)
    lb = np.zeros((2, cfg.vocab), dtype=np.float32)
    b.step_host(tok, pos, amb, lb)
    np.testing.assert_array_equal(ama.cpu().numpy(), amb)
    np.testing.assert_array_equal(la.cpu().numpy(), lb)
    a.close()
    b.close()


TOL_NVFP4 = 5e-2


def _check_moe(rep):
    _check(rep)
    assert rep.routed_rows > 0
    assert rep.compared >= 2, f"only {rep.compared} steps compared ({rep.route_ties} routing near-ties)"


def test_kda_decode_and_verify():
    """KDA (per-channel decay) recurrent layers at full width (64 heads x 128 / 128, d 7168) with a dense
    FFN: batch 2, ragged context, decode and verify blocks (pending-row replay of the delta rule)."""
    import dataclasses
    from gpu_harness import run_case
    cfg = dataclasses.replace(config("moe_kda_mla"), n_layers=2, mixers=("kda", "kda"), ffn="dense",
                              ffn_dim=2048, vocab=32768)
    rep = run_case(cfg, B=2, T=29, decode_steps=2, verify_accepts=(3, 6), tol=TOL_BF16)
    _check(rep)


def test_kda_mla_moe_full_width_two_layers():
    """One KDA and one MLA layer at the full widths of the MoE / KDA / MLA model (d 7168; MLA 64 heads,
    latent 512 + rope 64, q_lora 1536; experts d x 2048 bf16, 1 shared), with 16 routed experts top-4 so
    the oracle stays small; batch 2: prefill (16 rows per call: two expert passes), decode, verify."""
    import dataclasses
    from gpu_harness import run_case
    cfg = dataclasses.replace(config("moe_kda_mla"), n_layers=2, mixers=("kda", "mla"), n_experts=16, top_k=4,
                              vocab=32768)
    rep = run_case(cfg, B=2, T=37, decode_steps=2, verify_accepts=(3, 6), tol=TOL_BF16)
    _check_moe(rep)


def test_mla_moe_batch8_decode():
    """MLA + MoE at batch 8 (8-row expert GEMV groups, one head group per warp, many context chunks)."""
    import dataclasses
    from gpu_harness import run_case
    cfg = dataclasses.replace(config("moe_kda_mla"), n_layers=1, mixers=("mla",), d_model=2048, n_experts=64,
                              top_k=8, expert_dim=512, vocab=8192)
    rep = run_case(cfg, B=8, T=45, decode_steps=2, tol=TOL_BF16)
    _check_moe(rep)


def test_nvfp4_moe_256_experts():
    """NVFP4 experts (e2m1 codes, e4m3 block scales, fp32 tensor scales), 256 experts top-8 + 1 shared,
    router bias, with GQA 8/2 x 128; narrow (d 512, experts 512) so the dequantised oracle stays small."""
    from gpu_harness import run_case
    cfg = config("moe_nvfp4_gqa", n_layers=2, d_model=512, expert_dim=512, vocab=8192, n_q_heads=8,
                 n_kv_heads=2, head_dim=128)
    rep = run_case(cfg, B=2, T=33, decode_steps=2, verify_accepts=(3, 6), tol=TOL_NVFP4)
    _check_moe(rep)


def test_nvfp4_moe_full_width_one_layer():
    """One layer of the NVFP4 MoE model at full width (d 6144, GQA 48/8 x 128, experts 6144 x 2048), 32
    experts top-8, batch 1 decode."""
    from gpu_harness import run_case
    cfg = config("moe_nvfp4_gqa", n_layers=1, n_experts=32, vocab=16384)
    rep = run_case(cfg, B=1, T=12, decode_steps=3, tol=TOL_NVFP4)
    _check_moe(rep)


def test_fork_sequence():
    """One prefill of sequence 0 forked to sequences 1 and 2 equals three separate prefills of the same
    context: decode and verify steps with different tokens per sequence match the oracle (GQA + GDN)."""
    from decode_megakernel_04_gb300 import Megakernel
    from gpu_harness import Report, compare_logits
    from oracle import Oracle
    cfg = config("hybrid_gdn_gqa", n_layers=4, vocab=8192)
    dev = torch.device("cuda")
    w = make_weights(cfg, seed=1, device=dev)
    B, T, R = 3, 21, 8
    mk = Megakernel(cfg, w, max_batch=B, max_rows=R, max_ctx=64)
    orc = Oracle(cfg, w, B, 64)
    ctx = make_tokens(1, "ctx", (1, T), cfg.vocab, device=dev).contiguous()
    mk.prefill(ctx)
    mk.fork(0, 1)
    mk.fork(0, 2)
    orc.prefill(np.repeat(ctx.cpu().numpy(), B, axis=0))
    rep = Report()
    pos = np.full(B, T, dtype=np.int64)
    for s, rows in enumerate((1, R, 1)):
        tok = make_tokens(1, f"fork{s}", (B, rows), cfg.vocab).numpy().astype(np.int64)
        logits = torch.empty((B * rows, cfg.vocab), device=dev)
        mk.step(torch.from_numpy(tok.astype(np.int32)).to(dev).contiguous(),
                torch.from_numpy(pos.astype(np.int32)).to(dev), logits)
        assert mk.status() == 0
        ref = orc.step(tok, pos)
        compare_logits(logits.cpu().numpy().reshape(B, rows, -1), ref, TOL_BF16, rep, f"step {s}")
        pos = pos + (rows if rows == 1 else 5)
    mk.close()
    _check(rep)


def test_hybrid_batch4_decode():
    """Batch 4 at full width: 4 activation rows of width 5120 fill the shared-memory staging area of the
    tensor-core GEMV exactly."""
    from gpu_harness import run_case
    cfg = config("hybrid_gdn_gqa", n_layers=4)
    rep = run_case(cfg, B=4, T=20, decode_steps=2, tol=TOL_BF16)
    _check(rep)


def test_watchdog_timeout_then_recovery():
    """The kernel's wait limit set to 1 ns: the first dependency or ring wait that polls twice runs out, the
    step stops with MK_ERR_TIMEOUT in the status word (no trap, no fault, every CTA returns after its
    copies in flight land), mk_get_status reports it and resets the counters, and the same handle then runs
    a fresh prefill and a step that equal a new handle's bit for bit."""
    from decode_megakernel_04_gb300 import Megakernel
    from decode_megakernel_04_gb300.binding import MK_ERR_TIMEOUT
    cfg = config("hybrid_gdn_gqa", n_layers=4, d_model=512, ffn_dim=1024, vocab=4096)
    dev = torch.device("cuda")
    w = make_weights(cfg, seed=2, device=dev)
    ctx = make_tokens(2, "ctx", (2, 24), cfg.vocab, device=dev)
    tok = torch.tensor([[7], [9]], dtype=torch.int32, device=dev)
    pos = torch.tensor([24, 24], dtype=torch.int32, device=dev)
    mk = Megakernel(cfg, w, max_batch=2, max_rows=8, max_ctx=64)
    mk.prefill(ctx)
    assert mk.status() == 0
    mk.set_wait_limit(1)
    logits = torch.empty((2, cfg.vocab), device=dev)
    mk.step(tok, pos, logits)
    assert mk.status() == MK_ERR_TIMEOUT
    assert mk.status() == 0          # reported once, then cleared
    mk.set_wait_limit(2_000_000_000)
    mk.prefill(ctx)
    mk.step(tok, pos, logits)
    assert mk.status() == 0
    ref = Megakernel(cfg, w, max_batch=2, max_rows=8, max_ctx=64)
    ref.prefill(ctx)
    want = torch.empty_like(logits)
    ref.step(tok, pos, want)
    assert ref.status() == 0
    assert torch.equal(logits, want)
    mk.close()
    ref.close()


@pytest.mark.parametrize("B", [16, 64])
def test_hybrid_batch_above_8(B):
    """Concurrency above batch 8: 16 and 64 sequences decoding in one launch (tcgen05 GEMV tiles of 32 and 128
    TMEM columns; prefill in launches of 64 / B rows per sequence), against the oracle."""
    from gpu_harness import run_case
    cfg = config("hybrid_gdn_gqa", n_layers=4, d_model=512, ffn_dim=1024, vocab=4096)
    rep = run_case(cfg, B=B, T=12, decode_steps=2, tol=TOL_BF16)
    _check(rep)
