"""Pins for the oracle's MLA front half and its KDA decay layout.

MLA (absorbed latent attention): the oracle's layer is checked against an independent formulation in
torch (float64): RMSNorm by ``torch.nn.functional.rms_norm``, RoPE as a complex multiplication, the
unabsorbed per-head keys and values, and ``scaled_dot_product_attention`` with a causal mask. On top of
that, invariances that a plausible slip breaks: a dropped c_q or c_kv norm (the layer must not care about
the scale of W_DQ or of the latent rows of W_DKV, but must care about the scale of its rope rows), a
misplaced nope / rope split (killing the rope term from the query side or from the key side must give the
same layer), and the first-token closed form (one key: the layer returns W_O [W_UV[h] c_0]_h whatever the
query path holds).

KDA: which row of the decay projection gates which (head, key channel). A two-token closed form where one
(head, channel) keeps its state and every other channel is wiped fixes the [head, channel] row order.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import Oracle
from synthetic import config, make_weights

F64 = torch.float64


def _mla_cfg(**kw):
    spec = dict(n_layers=1, mixers=("mla",), d_model=48, vocab=61, mla_heads=3, q_lora=24, kv_lora=16,
                qk_nope=8, qk_rope=8, v_head=6, n_experts=4, top_k=2, n_shared=1, expert_dim=16, init_std=0.3)
    spec.update(kw)
    cfg = config("moe_kda_mla")
    import dataclasses
    return dataclasses.replace(cfg, **spec)


def _mla_weights(cfg, seed=0):
    """Weights as float64 numpy, with random norm gains so a gain applied in the wrong place shows."""
    w = {k: v.float().numpy().astype(np.float64) for k, v in make_weights(cfg, seed=seed, device="cpu").items()}
    rng = np.random.default_rng(seed + 100)
    for name in ("layers.0.q_norm", "layers.0.kv_norm"):
        w[name] = rng.uniform(0.5, 1.5, size=w[name].shape)
    return w


def _oracle_mla(cfg, w, h):
    """The oracle's MLA layer over one block of rows at positions 0 .. R-1 (one sequence)."""
    o = Oracle(cfg, w, 1, h.shape[0] + 4)
    return o.mla(0, h[None], np.zeros(1, dtype=np.int64))[0]


def _rope_complex(x, pos, theta):
    """RoPE written as a complex multiplication: the pair (x_i, x_{i + D/2}) is the complex number
    x_i + j x_{i + D/2}, turned by the angle pos * theta^(-2i / D)."""
    d = x.shape[-1]
    half = d // 2
    inv = theta ** (-(2.0 * torch.arange(half, dtype=F64)) / d)
    ang = pos.to(F64)[:, None] * inv[None, :]                       # [T, half]
    while ang.dim() < x.dim():
        ang = ang.unsqueeze(-2)                                     # broadcast over heads
    z = torch.complex(x[..., :half], x[..., half:]) * torch.polar(torch.ones_like(ang), ang)
    return torch.cat([z.real, z.imag], dim=-1)


def _torch_mla(cfg, w, h):
    """Unabsorbed MLA in torch: per head k = [W_UK[h]^T c_t, k_r,t], v = W_UV[h] c_t, causal SDPA."""
    H, nope, rp, lora, vh = cfg.mla_heads, cfg.qk_nope, cfg.qk_rope, cfg.kv_lora, cfg.v_head
    t = {k: torch.from_numpy(np.asarray(v, dtype=np.float64)) for k, v in w.items() if k.startswith("layers.0.")}
    x = torch.from_numpy(h)
    T = x.shape[0]
    pos = torch.arange(T)
    c_q = F.rms_norm(x @ t["layers.0.w_dq"].T, (cfg.q_lora,), weight=t["layers.0.q_norm"], eps=cfg.norm_eps)
    qf = (c_q @ t["layers.0.w_uq"].T).view(T, H, nope + rp)
    kv = x @ t["layers.0.w_dkv"].T
    c = F.rms_norm(kv[:, :lora], (lora,), weight=t["layers.0.kv_norm"], eps=cfg.norm_eps)
    k_r = _rope_complex(kv[:, lora:], pos, cfg.rope_theta)          # [T, rp], shared by the heads
    q_r = _rope_complex(qf[..., nope:], pos, cfg.rope_theta)        # [T, H, rp]
    q = torch.cat([qf[..., :nope], q_r], dim=-1).transpose(0, 1)    # [H, T, nope + rp]
    k_nope = torch.einsum("tl,hln->htn", c, t["layers.0.w_uk"])     # [H, T, nope]
    k = torch.cat([k_nope, k_r[None].expand(H, T, rp)], dim=-1)
    v = torch.einsum("tl,hvl->htv", c, t["layers.0.w_uv"])          # [H, T, vh]
    o = F.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True,
                                       scale=1.0 / math.sqrt(nope + rp))[0]
    return (o.transpose(0, 1).reshape(T, H * vh) @ t["layers.0.wo"].T).numpy()


@pytest.mark.parametrize("T", [1, 2, 7])
@pytest.mark.parametrize("seed", [0, 1])
def test_mla_matches_torch_unabsorbed(T, seed):
    cfg = _mla_cfg()
    w = _mla_weights(cfg, seed)
    h = np.random.default_rng(seed).standard_normal((T, cfg.d_model))
    np.testing.assert_allclose(_oracle_mla(cfg, w, h), _torch_mla(cfg, w, h), rtol=1e-10, atol=1e-12)


def test_mla_first_token_closed_form():
    """One key: the softmax weight is 1 whatever the scores, so the layer is W_O [W_UV[h] c_0]_h with
    c_0 = RMSNorm(y W_DKV[:kv_lora]) * kv_norm, and the query path (W_DQ, q_norm, W_UQ) has no effect."""
    cfg = _mla_cfg()
    w = _mla_weights(cfg, 3)
    y = np.random.default_rng(3).standard_normal(cfg.d_model)
    lora = cfg.kv_lora
    a = w["layers.0.w_dkv"][:lora] @ y
    c0 = a / np.sqrt(np.mean(a * a) + cfg.norm_eps) * w["layers.0.kv_norm"]
    heads = [w["layers.0.w_uv"][hh] @ c0 for hh in range(cfg.mla_heads)]
    want = w["layers.0.wo"] @ np.concatenate(heads)
    got = _oracle_mla(cfg, w, y[None])[0]
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)
    w2 = dict(w)
    rng = np.random.default_rng(4)
    for name in ("layers.0.w_dq", "layers.0.w_uq", "layers.0.q_norm"):
        w2[name] = rng.standard_normal(w[name].shape)
    np.testing.assert_allclose(_oracle_mla(cfg, w2, y[None])[0], want, rtol=1e-12, atol=1e-13)


def test_mla_norm_invariances():
    """c_q and c_kv are RMS-normalised: scaling W_DQ, or the latent rows of W_DKV, changes nothing (up to
    the epsilon); scaling the rope rows of W_DKV (not normalised) changes the layer."""
    cfg = _mla_cfg(norm_eps=1e-30)
    w = _mla_weights(cfg, 5)
    h = np.random.default_rng(5).standard_normal((6, cfg.d_model))
    base = _oracle_mla(cfg, w, h)
    lora = cfg.kv_lora
    w_q = dict(w)
    w_q["layers.0.w_dq"] = 7.0 * w["layers.0.w_dq"]
    np.testing.assert_allclose(_oracle_mla(cfg, w_q, h), base, rtol=1e-10, atol=1e-12)
    w_c = dict(w)
    w_c["layers.0.w_dkv"] = w["layers.0.w_dkv"].copy()
    w_c["layers.0.w_dkv"][:lora] *= 0.2
    np.testing.assert_allclose(_oracle_mla(cfg, w_c, h), base, rtol=1e-10, atol=1e-12)
    w_r = dict(w)
    w_r["layers.0.w_dkv"] = w["layers.0.w_dkv"].copy()
    w_r["layers.0.w_dkv"][lora:] *= 3.0
    assert np.max(np.abs(_oracle_mla(cfg, w_r, h) - base)) > 1e-3


def test_mla_rope_split_zeroing():
    """The scores are q~.c + q_r.k_r: zeroing the rope rows of every head of W_UQ (q_r = 0) or the rope
    rows of W_DKV (k_r = 0) both remove the second term and must give the same layer; zeroing the last
    rows of the nope part instead must not."""
    cfg = _mla_cfg()
    w = _mla_weights(cfg, 6)
    h = np.random.default_rng(6).standard_normal((5, cfg.d_model))
    H, nope, rp, lora = cfg.mla_heads, cfg.qk_nope, cfg.qk_rope, cfg.kv_lora
    wq0 = dict(w)
    wq0["layers.0.w_uq"] = w["layers.0.w_uq"].copy().reshape(H, nope + rp, -1)
    wq0["layers.0.w_uq"][:, nope:] = 0.0
    wq0["layers.0.w_uq"] = wq0["layers.0.w_uq"].reshape(H * (nope + rp), -1)
    wk0 = dict(w)
    wk0["layers.0.w_dkv"] = w["layers.0.w_dkv"].copy()
    wk0["layers.0.w_dkv"][lora:] = 0.0
    a, b = _oracle_mla(cfg, wq0, h), _oracle_mla(cfg, wk0, h)
    np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)
    assert np.max(np.abs(a - _oracle_mla(cfg, w, h))) > 1e-3      # the rope term is not negligible
    wn0 = dict(w)
    wn0["layers.0.w_uq"] = w["layers.0.w_uq"].copy().reshape(H, nope + rp, -1)
    wn0["layers.0.w_uq"][:, nope - rp:nope] = 0.0
    wn0["layers.0.w_uq"] = wn0["layers.0.w_uq"].reshape(H * (nope + rp), -1)
    assert np.max(np.abs(_oracle_mla(cfg, wn0, h) - b)) > 1e-3


def _kda_cfg():
    import dataclasses
    cfg = config("moe_kda_mla")
    return dataclasses.replace(cfg, n_layers=1, mixers=("kda",), d_model=32, vocab=37, lin_heads=3, lin_dk=4,
                               lin_dv=5, ffn="dense", ffn_dim=16, init_std=0.3)


@pytest.mark.parametrize("head,chan", [(0, 1), (1, 2), (2, 1)])
def test_kda_decay_row_layout_two_tokens(head, chan):
    """Decay row j gates key channel j % dk of head j // dk. The decay projection is set so that at the
    second token only (head, chan) keeps its state (alpha = sigmoid(+60) = 1) and every other channel is
    wiped (alpha = sigmoid(-60) ~ 1e-26). From a zero state, token 1 leaves S = beta_1 k1 v1^T per head; then
    head `head` sees S' = beta_1 k1[chan] e_chan v1^T, u = v2 - S'^T k2, o = S'^T q2 + beta_2 (k2 . q2) u,
    and every other head o = beta_2 (k2 . q2) v2 (k, q the L2-normalised key and query, q also / sqrt(dk))."""
    cfg = _kda_cfg()
    H, dk, dv = cfg.lin_heads, cfg.lin_dk, cfg.lin_dv
    w = {k: v.float().numpy().astype(np.float64) for k, v in make_weights(cfg, seed=8, device="cpu").items()}
    rng = np.random.default_rng(8)
    h = rng.standard_normal((1, 2, cfg.d_model))
    y2 = h[0, 1]
    sign = -np.ones(H * dk)
    sign[head * dk + chan] = 1.0
    w["layers.0.wa"] = (60.0 * sign)[:, None] * (y2 / (y2 @ y2))[None, :]
    o = Oracle(cfg, w, 1, 4)
    got = o.delta(0, "kda", h)                                   # [1, 2, d] after W_O
    p = "layers.0."
    q = (h[0] @ w[p + "wq"].T).reshape(2, H, dk)
    k = (h[0] @ w[p + "wk"].T).reshape(2, H, dk)
    v = (h[0] @ w[p + "wv"].T).reshape(2, H, dv)
    beta = 1.0 / (1.0 + np.exp(-(h[0] @ w[p + "wb"].T)))         # [2, H]
    qn = q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6) / np.sqrt(dk)
    kn = k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
    out2 = np.empty((H, dv))
    for hh in range(H):
        fresh = beta[1, hh] * (kn[1, hh] @ qn[1, hh]) * v[1, hh]
        if hh != head:
            out2[hh] = fresh
            continue
        keep = beta[0, hh] * kn[0, hh, chan]                      # S' = keep * e_chan v1^T
        u = v[1, hh] - keep * kn[1, hh, chan] * v[0, hh]
        out2[hh] = keep * qn[1, hh, chan] * v[0, hh] + beta[1, hh] * (kn[1, hh] @ qn[1, hh]) * u
    want = w[p + "wo"] @ out2.reshape(-1)
    np.testing.assert_allclose(got[0, 1], want, rtol=1e-11, atol=1e-12)
