"""Pins for the oracle's primitive operations: library routines, closed forms, explicit forms.

Each test checks an oracle function against something other than itself: a torch routine, a
closed form, an explicit (non-recurrent) formula, or a brute-force enumeration.
"""
import numpy as np
import pytest
import torch

from oracle import ops
from synthetic import quantize_nvfp4, E2M1_GRID

RNG = np.random.default_rng(1234)


def test_bf16_round_matches_torch():
    x = RNG.standard_normal(100_000).astype(np.float32) * np.float32(3.0)
    x[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]  # exact ties: to even
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(ops.bf16_round(x), want)


def test_rmsnorm_matches_torch():
    x = RNG.standard_normal((5, 64))
    g = RNG.standard_normal(64)
    want = torch.nn.functional.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(ops.rmsnorm(x, g, 1e-6), want, rtol=1e-12, atol=1e-12)


def test_rmsnorm_constant_vector():
    c, eps = 0.37, 1e-6
    x = np.full(32, c)
    np.testing.assert_allclose(ops.rmsnorm(x, np.ones(32), eps), c / np.sqrt(c * c + eps), rtol=1e-14)


def test_silu_matches_torch():
    z = RNG.standard_normal(1000) * 4
    np.testing.assert_allclose(ops.silu(z), torch.nn.functional.silu(torch.from_numpy(z)).numpy(),
                               rtol=1e-13, atol=1e-15)


def test_rope_identity_at_zero_and_norm():
    x = RNG.standard_normal((3, 64))
    np.testing.assert_array_equal(ops.rope(x, np.zeros((3,)), 1e4), x)
    y = ops.rope(x, np.array([5.0, 100.0, 4095.0]), 1e4)
    # each rotated pair keeps its length
    np.testing.assert_allclose(y[:, :32] ** 2 + y[:, 32:] ** 2, x[:, :32] ** 2 + x[:, 32:] ** 2, rtol=1e-12)


def test_rope_complex_form():
    d, theta = 16, 1e4
    x = RNG.standard_normal(d)
    pos = 37.0
    z = x[: d // 2] + 1j * x[d // 2:]
    freqs = np.array([theta ** (-2 * i / d) for i in range(d // 2)])
    zr = z * np.exp(1j * pos * freqs)
    want = np.concatenate([zr.real, zr.imag])
    np.testing.assert_allclose(ops.rope(x, np.array(pos), theta), want, rtol=1e-12, atol=1e-12)


def test_rope_relative_position():
    q, k = RNG.standard_normal(32), RNG.standard_normal(32)
    a = ops.rope(q, np.array(10.0), 1e4) @ ops.rope(k, np.array(3.0), 1e4)
    b = ops.rope(q, np.array(110.0), 1e4) @ ops.rope(k, np.array(103.0), 1e4)
    np.testing.assert_allclose(a, b, rtol=1e-10)


@pytest.mark.parametrize("hq,hkv,p0,R", [(4, 1, 0, 1), (6, 2, 9, 3), (8, 8, 5, 8), (24, 4, 31, 8)])
def test_gqa_matches_sdpa(hq, hkv, p0, R):
    hd = 16
    T = p0 + R
    q = RNG.standard_normal((R, hq, hd))
    K = RNG.standard_normal((T, hkv, hd))
    V = RNG.standard_normal((T, hkv, hd))
    got = ops.gqa_block_attention(q, K, V, p0)
    rep = hq // hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(rep, dim=0)[None]
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(rep, dim=0)[None]
    mask = torch.from_numpy(np.arange(T)[None, :] <= (p0 + np.arange(R))[:, None])
    want = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)[0].permute(1, 0, 2)
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-10, atol=1e-12)


def test_attention_single_key_returns_v():
    q = RNG.standard_normal((1, 4, 8))
    K = RNG.standard_normal((1, 2, 8))
    V = RNG.standard_normal((1, 2, 8))
    o = ops.gqa_block_attention(q, K, V, 0)
    np.testing.assert_allclose(o[0], V[0][[0, 0, 1, 1]], rtol=1e-14)


def _explicit_delta(S0, qs, ks, vs, alphas, betas):
    """S_T = A_T..A_1 S_0 + sum_i A_T..A_{i+1} beta_i k_i v_i^T with A_j = (I - beta_j k_j k_j^T) D_j."""
    dk = S0.shape[0]
    T = len(ks)
    A = []
    for j in range(T):
        a = np.asarray(alphas[j], dtype=float)
        D = np.diag(a) if a.ndim else a * np.eye(dk)
        A.append((np.eye(dk) - betas[j] * np.outer(ks[j], ks[j])) @ D)
    outs = []
    for t in range(1, T + 1):
        P = np.eye(dk)
        for j in range(t):
            P = A[j] @ P
        S = P @ S0
        for i in range(t):
            Pi = np.eye(dk)
            for j in range(i + 1, t):
                Pi = A[j] @ Pi
            S = S + Pi @ (betas[i] * np.outer(ks[i], vs[i]))
        outs.append(S.T @ qs[t - 1])
    return S, outs


@pytest.mark.parametrize("per_channel", [False, True])
@pytest.mark.parametrize("T", [1, 2, 6])
def test_delta_rule_matches_explicit_form(per_channel, T):
    dk, dv = 4, 4
    S0 = RNG.standard_normal((dk, dv))
    qs = [ops.l2_normalize(RNG.standard_normal(dk)) for _ in range(T)]
    ks = [ops.l2_normalize(RNG.standard_normal(dk)) for _ in range(T)]
    vs = [RNG.standard_normal(dv) for _ in range(T)]
    alphas = [ops.sigmoid(RNG.standard_normal(dk if per_channel else ())) for _ in range(T)]
    betas = [float(ops.sigmoid(RNG.standard_normal())) for _ in range(T)]
    S = S0.copy()
    outs = []
    for t in range(T):
        S, o = ops.delta_rule_step(S, qs[t], ks[t], vs[t], alphas[t], betas[t])
        outs.append(o)
    S_exp, outs_exp = _explicit_delta(S0, qs, ks, vs, alphas, betas)
    np.testing.assert_allclose(S, S_exp, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(np.array(outs), np.array(outs_exp), rtol=1e-12, atol=1e-12)


def test_delta_rule_identity_and_overwrite():
    S = RNG.standard_normal((8, 6))
    q = RNG.standard_normal(8)
    k = ops.l2_normalize(RNG.standard_normal(8), eps=0.0)
    v = RNG.standard_normal(6)
    S1, o = ops.delta_rule_step(S, q, k, v, 1.0, 0.0)
    np.testing.assert_array_equal(S1, S)
    np.testing.assert_allclose(o, S.T @ q, rtol=1e-14)
    S2, _ = ops.delta_rule_step(S, q, k, v, 1.0, 1.0)
    np.testing.assert_allclose(k @ S2, v, rtol=1e-12, atol=1e-12)


def test_route_matches_stable_sort():
    for trial in range(200):
        E, k = (64, 8) if trial % 2 else (256, 8)
        z = RNG.standard_normal(E) * 2
        bias = RNG.standard_normal(E) * 0.01 if trial % 3 else np.zeros(E)
        if trial % 5 == 0:  # exact ties
            z[3] = z[40] = z[50] = z.max() + 1.0
            bias[3] = bias[40] = bias[50] = 0.0
        idx, w, biased = ops.route(z, bias, k, 2.5)
        order = np.argsort(-biased, kind="stable")[:k]
        np.testing.assert_array_equal(idx, order)
        s = 1 / (1 + np.exp(-z))
        np.testing.assert_allclose(w, 2.5 * s[order] / s[order].sum(), rtol=1e-14)
        np.testing.assert_allclose(w.sum(), 2.5, rtol=1e-14)


def test_route_tie_lowest_index():
    z = np.zeros(16)
    idx, _, _ = ops.route(z, np.zeros(16), 4, 1.0)
    np.testing.assert_array_equal(idx, [0, 1, 2, 3])


def test_e2m1_table_from_definition():
    vals = ops.e2m1_value(np.arange(16))
    np.testing.assert_array_equal(vals[:8], E2M1_GRID)
    np.testing.assert_array_equal(vals[8:], [-v for v in E2M1_GRID])


def test_e4m3_matches_torch():
    bits = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(bits).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = ops.e4m3_value(bits)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])


def test_nvfp4_grid_round_trip_exact():
    rows, K = 6, 64
    nb = K // 16
    codes = RNG.integers(0, 16, size=(rows, K))
    codes[:, ::16] = 7  # every block holds a max-magnitude element (6.0), so its scale is recovered
    # e4m3-representable block scales; one block at 448 and one all-zero block
    scale_bits = RNG.integers(0x08, 0x7E, size=(rows, nb)).astype(np.uint8)
    scale_bits[0, 0] = 0x7E  # 448
    scales = ops.e4m3_value(scale_bits)
    scales[rows - 1, nb - 1] = 0.0
    grid = np.array(E2M1_GRID + tuple(-v for v in E2M1_GRID))
    w = grid[codes] * np.repeat(scales, 16, axis=1)   # tensor scale = amax / 2688 = 1
    q, s, g = quantize_nvfp4(torch.from_numpy(w).float())
    assert float(g) == 1.0
    back = ops.nvfp4_decode(q.numpy(), s.numpy(), float(g))
    np.testing.assert_array_equal(back, w)


def test_linear_is_float64_product():
    x = RNG.standard_normal((3, 300))
    w = RNG.standard_normal((5000, 300)).astype(np.float32)
    np.testing.assert_allclose(ops.linear(x, w, block=777), x @ w.astype(np.float64).T, rtol=1e-12)


def test_nvfp4_expert_stack_matches_per_expert_encoding():
    """The stacked encoder (one tensor scale per expert) gives the same bytes as encoding each expert alone,
    including an all-zero expert."""
    from synthetic import quantize_nvfp4_experts
    w = torch.from_numpy(RNG.standard_normal((5, 7, 64)) * 0.02).float()
    w[3] = 0.0
    q, s, g = quantize_nvfp4_experts(w)
    for e in range(5):
        qe, se, ge = quantize_nvfp4(w[e])
        assert torch.equal(q[e], qe) and torch.equal(s[e], se) and float(g[e]) == float(ge)
