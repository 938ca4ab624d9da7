"""Pins for the pages' own expert format in the oracle: FP8-E4M3 gate / up with one bf16 scale per 256 rows
and MXFP4 down (Kimi K3's TPU megakernel, "How it maps onto a TPU v7", the precision paragraph).

Each test checks an oracle decoder against something other than itself: the format's closed forms, torch's
own float8 / bfloat16 types, hand-built blocks, or the re-encoding's exactness (the loader's bit-for-bit check).
"""
import numpy as np
import pytest
import torch

from oracle import Oracle, ops
from synthetic import E2M1_GRID, config, make_tokens, make_weights, quantize_mxfp4, reencode_fp8_rows

RNG = np.random.default_rng(4321)


def test_e8m0_closed_forms():
    got = ops.e8m0_value(np.array([127, 128, 126, 0, 254, 255]))
    np.testing.assert_array_equal(got[:5], [1.0, 2.0, 0.5, 2.0 ** -127, 2.0 ** 127])
    assert np.isnan(got[5])


def test_bf16_value_matches_torch():
    bits = RNG.integers(0, 1 << 16, 50_000).astype(np.int64)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite patterns only
    want = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(ops.bf16_value(bits), want)


def _hand_value(code, x):
    mag = E2M1_GRID[code & 7]
    return (-mag if code & 8 else mag) * 2.0 ** x


def test_mxfp4_hand_block():
    """One 32-input block with E8M0 = 130 (scale 8): every code decodes to its grid value times 8; the
    low nibble holds the even element."""
    codes = np.arange(32) % 16
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)[None, :]
    got = ops.mxfp4_decode(packed, np.array([[130]], dtype=np.uint8))[0]
    np.testing.assert_array_equal(got, [_hand_value(int(c), 3) for c in codes])


def test_mxfp4_encoder_rounding_rule():
    """Shared exponent floor(log2 amax) - 2; e2m1 round to nearest, ties to the even code, saturating at 6."""
    w = np.zeros((3, 32), dtype=np.float32)
    w[0, :6] = [5.0, 2.5, 1.25, 0.25, -3.5, 0.75]   # amax 5: X = 0; ties go to 4, 2, 1, 0, -4, 1
    w[1, :2] = [7.9, -0.1]                            # amax 7.9: X = 0; 7.9 saturates to 6
    q, x = quantize_mxfp4(torch.from_numpy(w))
    assert x.tolist() == [[127], [127], [0]]            # the all-zero block takes X = -127
    got = ops.mxfp4_decode(q.numpy(), x.numpy())
    np.testing.assert_array_equal(got[0, :6], [4.0, 2.0, 1.0, 0.0, -4.0, 1.0])
    np.testing.assert_array_equal(got[1, :2], [6.0, 0.0])
    assert not got[2].any()


def test_mxfp4_grid_round_trip_exact():
    """Values already on a block's grid (e2m1 x 2^X, the block's largest magnitude 4 or 6 x 2^X so that X is
    the block's own exponent) encode and decode exactly."""
    rows, K = 64, 256
    X = RNG.integers(-20, 20, (rows, K // 32))
    codes = RNG.integers(0, 16, (rows, K))
    codes[:, ::32] = RNG.choice([6, 7, 14, 15], (rows, K // 32))  # one element of magnitude 4 or 6 per block
    vals = np.array([[_hand_value(int(codes[r, k]), int(X[r, k // 32])) for k in range(K)] for r in range(rows)])
    q, x = quantize_mxfp4(torch.from_numpy(vals.astype(np.float32)))
    np.testing.assert_array_equal(x.numpy().astype(np.int64) - 127, X)
    np.testing.assert_array_equal(ops.mxfp4_decode(q.numpy(), x.numpy()), vals)


def test_fp8_reencode_is_exact_with_one_scale_per_256_rows():
    """The re-encoded gate / up decode to the MXFP4 values bit for bit; rows 0..255, 256..511 and the partial
    block 512..551 each take their own scale (their magnitudes differ by 2^6 and 2^-5)."""
    w = np.clip(RNG.standard_normal((552, 64)), -2.9, 2.9).astype(np.float32)
    w[0, 0] = w[300, 5] = w[520, 9] = 3.0  # each row block's largest magnitude: shared exponent -1 before scaling
    w[256:512] *= 64.0
    w[512:] /= 32.0
    q, x = quantize_mxfp4(torch.from_numpy(w))
    codes, sbits = reencode_fp8_rows(q, x)
    assert codes.shape == (552, 64) and sbits.shape == (3,)
    mx = ops.mxfp4_decode(q.numpy(), x.numpy())
    np.testing.assert_array_equal(ops.fp8_rows_decode(codes.numpy(), sbits.numpy()), mx)
    s = ops.bf16_value(sbits.numpy())
    assert s[1] / s[0] == 64.0 and s[2] / s[0] == 2.0 ** -5
    # every code is a finite e4m3 value, and the scale is applied per 256-row block: doubling scale 1
    # doubles exactly rows 256..511
    assert np.isfinite(ops.e4m3_value(codes.numpy())).all()
    s2 = sbits.numpy().copy()
    s2[1] = int(torch.tensor([2.0 * s[1]], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF
    d2 = ops.fp8_rows_decode(codes.numpy(), s2)
    np.testing.assert_array_equal(d2[:256], mx[:256])
    np.testing.assert_array_equal(d2[256:512], 2.0 * mx[256:512])
    np.testing.assert_array_equal(d2[512:], mx[512:])


def test_fp8_reencode_raises_when_not_exact():
    """One 256-row block whose values span more binades than e4m3 holds under one scale is refused."""
    w = np.zeros((256, 32), dtype=np.float32)
    w[0, 0] = 2.0 ** 20
    w[1, 0] = 1.5 * 2.0 ** -20
    q, x = quantize_mxfp4(torch.from_numpy(w))
    with pytest.raises(ValueError):
        reencode_fp8_rows(q, x)


def _tiny_f4(**kw):
    spec = dict(n_layers=2, d_model=64, vocab=97, n_q_heads=4, n_kv_heads=2, head_dim=16, n_experts=8, top_k=2,
                n_shared=1, expert_dim=32, expert_fmt="f4", init_std=0.2)
    spec.update(kw)
    return config("moe_nvfp4_gqa", **spec)


def test_oracle_f4_experts_decode_the_stored_bytes():
    """The oracle's f4 experts are the decoded bytes: gate / up as e4m3 x bf16 row-block scale, down as
    e2m1 x 2^(E8M0 - 127); and the re-encoded gate equals the MXFP4 encoding of the same draw."""
    cfg = _tiny_f4()
    wt = make_weights(cfg, seed=5, device="cpu")
    o = Oracle(cfg, wt, 1, 4)
    g = o.expert(0, "e", "gate", 3)
    c0, sb = int(wt["layers.0.e_gate.f8"][3, 0, 0]), int(wt["layers.0.e_gate.f8s"][3, 0])
    assert g[0, 0] == ops.e4m3_value(c0) * ops.bf16_value(sb)
    d = o.expert(0, "e", "down", 3)
    qd, xd = int(wt["layers.0.e_down.q"][3, 0, 0]), int(wt["layers.0.e_down.x"][3, 0, 0])
    assert d[0, 0] == ops.e2m1_value(qd & 15) * ops.e8m0_value(xd)
    assert g.shape == (cfg.expert_dim, cfg.d_model) and d.shape == (cfg.d_model, cfg.expert_dim)
    # the loader's claim end to end: the FP8 gate decodes to the MXFP4 encoding of the same bf16 draw
    from synthetic.workloads import _bf16
    draw = _bf16((cfg.expert_dim, cfg.d_model), 5, "layers.0.e_gate.3", cfg.init_std, "cpu").float()
    q, x = quantize_mxfp4(draw)
    np.testing.assert_array_equal(g, ops.mxfp4_decode(q.numpy(), x.numpy()))


def test_oracle_f4_moe_closed_form_one_row():
    """The f4 MoE FFN of one row equals the shared expert plus the renormalised picked experts, computed
    directly from the decoded matrices."""
    cfg = _tiny_f4(router_bias_std=0.05)
    wt = make_weights(cfg, seed=9, device="cpu")
    o = Oracle(cfg, wt, 1, 4)
    h = np.random.default_rng(3).standard_normal((1, 1, cfg.d_model))
    got = o.moe(0, h)[0, 0]
    y = h[0, 0]
    z = wt["layers.0.w_router"].float().numpy().astype(np.float64) @ y
    s = 1 / (1 + np.exp(-z))
    pick = np.argsort(-(s + wt["layers.0.router_bias"].numpy()), kind="stable")[: cfg.top_k]
    wts = cfg.route_scale * s[pick] / s[pick].sum()

    def ffn(kind, e):
        gw, uw, dw = (o.expert(0, kind, m, e) for m in ("gate", "up", "down"))
        gg = gw @ y
        return dw @ ((gg / (1 + np.exp(-gg))) * (uw @ y))

    want = ffn("s", 0) + sum(wi * ffn("e", e) for e, wi in zip(pick, wts))
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-13)


def test_oracle_f4_token_by_token_equals_prefill():
    cfg = _tiny_f4()
    w = make_weights(cfg, seed=0, device="cpu")
    B, T = 2, 7
    toks = make_tokens(0, "ctx", (B, T), cfg.vocab).numpy()
    a = Oracle(cfg, w, B, 16)
    block = a.step(toks, np.zeros(B, dtype=int))
    b = Oracle(cfg, w, B, 16)
    rows = [b.step(toks[:, t:t + 1], np.full(B, t))[:, 0] for t in range(T)]
    np.testing.assert_allclose(block, np.stack(rows, axis=1), rtol=1e-9, atol=1e-9)


def test_binding_refuses_the_f4_format():
    """The kernel has no f4 expert path yet: the binding says so instead of reading the bytes as NVFP4."""
    from decode_megakernel_04_gb300 import binding
    with pytest.raises(ValueError, match="no kernel path"):
        binding.model_desc(_tiny_f4(), 1, 1, 16)
