"""Pins for the oracle's whole-step semantics on tiny models of every family.

* decode token by token equals one causal block over the same tokens (prefill);
* an R-row verify block equals R sequential single-row steps;
* partial acceptance equals having run only the accepted rows;
* absorbed MLA equals unabsorbed MLA;
* batch rows are independent;
* the block composition equals its closed form at the first token (attention over one key is v).
"""
import numpy as np
import pytest
import torch

from oracle import Oracle, ops
from synthetic import config, make_weights, make_tokens

TINY = {
    "dense": dict(name="tiny_dense"),
    "gdn_gqa": dict(name="hybrid_gdn_gqa", n_layers=4, d_model=64, vocab=97, n_q_heads=4, n_kv_heads=2,
                    head_dim=16, lin_heads=2, lin_dk=8, lin_dv=8, ffn_dim=96),
    "kda_mla_moe": dict(name="moe_kda_mla", n_layers=4, d_model=64, vocab=97, lin_heads=2, lin_dk=8,
                        lin_dv=8, mla_heads=2, q_lora=32, kv_lora=16, qk_nope=8, qk_rope=8, v_head=8,
                        n_experts=8, top_k=2, n_shared=1, expert_dim=32),
    "nvfp4_moe": dict(name="moe_nvfp4_gqa", n_layers=2, d_model=64, vocab=97, n_q_heads=4, n_kv_heads=2,
                      head_dim=16, n_experts=8, top_k=2, n_shared=1, expert_dim=32),
}


def tiny(kind, **kw):
    spec = dict(TINY[kind])
    name = spec.pop("name")
    spec.update(kw)
    # larger weights than the workloads' 0.02 so the tiny models are far from trivial
    spec.setdefault("init_std", 0.2)
    return config(name, **spec)


def _weights(cfg, seed=0):
    return make_weights(cfg, seed=seed, device="cpu")


@pytest.mark.parametrize("kind", list(TINY))
def test_token_by_token_equals_prefill(kind):
    cfg = tiny(kind)
    w = _weights(cfg)
    B, T = 2, 9
    toks = make_tokens(0, "ctx", (B, T), cfg.vocab).numpy()
    a = Oracle(cfg, w, B, 32)
    block = a.step(toks, np.zeros(B, dtype=int))   # one causal block over all T tokens
    a.commit(T)
    b = Oracle(cfg, w, B, 32)
    rows = []
    for t in range(T):
        rows.append(b.step(toks[:, t:t + 1], np.full(B, t))[:, 0])
    np.testing.assert_allclose(block, np.stack(rows, axis=1), rtol=1e-9, atol=1e-9)
    # next token after the prefix agrees too (state / caches carried the same way)
    nxt = make_tokens(0, "next", (B, 1), cfg.vocab).numpy()
    np.testing.assert_allclose(a.step(nxt, np.full(B, T)), b.step(nxt, np.full(B, T)), rtol=1e-9, atol=1e-9)


@pytest.mark.parametrize("kind", list(TINY))
@pytest.mark.parametrize("accept", [1, 3, 8])
def test_verify_block_equals_sequential_steps(kind, accept):
    cfg = tiny(kind)
    w = _weights(cfg)
    B, T0, R = 2, 5, 8
    ctx = make_tokens(0, "ctx", (B, T0), cfg.vocab).numpy()
    block = make_tokens(0, "draft", (B, R), cfg.vocab).numpy()
    after = make_tokens(0, "after", (B, 1), cfg.vocab).numpy()

    v = Oracle(cfg, w, B, 32)
    v.prefill(ctx)
    got = v.step(block, np.full(B, T0))
    got_next = v.step(after, np.full(B, T0 + accept))   # commits `accept` rows of the block

    s = Oracle(cfg, w, B, 32)
    s.prefill(ctx)
    want = []
    for r in range(R):
        want.append(s.step(block[:, r:r + 1], np.full(B, T0 + r))[:, 0])
        if r == accept - 1:
            snap = Oracle(cfg, w, B, 32)
            snap.prefill(np.concatenate([ctx, block[:, :accept]], axis=1))
    np.testing.assert_allclose(got, np.stack(want, axis=1), rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(got_next, snap.step(after, np.full(B, T0 + accept)), rtol=1e-9, atol=1e-9)


def test_position_outside_pending_window_rejected():
    cfg = tiny("gdn_gqa")
    o = Oracle(cfg, _weights(cfg), 1, 32)
    o.prefill(np.array([[1, 2, 3]]))
    o.step(np.array([[4, 5]]), np.array([3]))
    with pytest.raises(ValueError):
        o.step(np.array([[6]]), np.array([6]))     # only 2 pending rows: 3..5 is valid
    with pytest.raises(ValueError):
        o.step(np.array([[6]]), np.array([2]))     # before the committed prefix


def test_mla_absorbed_equals_unabsorbed():
    cfg = tiny("kda_mla_moe")
    w = _weights(cfg)
    B, T0, R = 2, 6, 3
    o = Oracle(cfg, w, B, 32)
    o.prefill(make_tokens(0, "ctx", (B, T0), cfg.vocab).numpy())
    rng = np.random.default_rng(7)
    h = rng.standard_normal((B, R, cfg.d_model))
    pos = np.full(B, T0)
    lat0 = o.lat[3].copy()
    a = o.mla(3, h, pos, absorbed=True)
    o.lat[3] = lat0.copy()
    b = o.mla(3, h, pos, absorbed=False)
    np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("kind", list(TINY))
def test_batch_rows_independent(kind):
    cfg = tiny(kind)
    w = _weights(cfg)
    toks = make_tokens(0, "ctx", (3, 6), cfg.vocab).numpy()
    o3 = Oracle(cfg, w, 3, 16)
    all3 = o3.step(toks, np.zeros(3, dtype=int))
    for b in range(3):
        o1 = Oracle(cfg, w, 1, 16)
        np.testing.assert_allclose(all3[b], o1.step(toks[b:b + 1], np.zeros(1, dtype=int))[0],
                                   rtol=1e-10, atol=1e-10)


def test_first_token_closed_form_dense():
    """One dense GQA layer at position 0: the only key is the token itself, so every query head h
    returns the cached v of kv head floor(h * Hkv / Hq) and the layer is a fixed chain of matrix
    products."""
    cfg = tiny("dense", n_layers=1, n_q_heads=4, n_kv_heads=2)
    w = {k: v.float().numpy().astype(np.float64) for k, v in _weights(cfg, seed=3).items()}
    tok = 17
    eps = cfg.norm_eps

    def n(x, g):
        return x / np.sqrt(np.mean(x * x) + eps) * g

    x0 = w["embed"][tok]
    v = w["layers.0.wv"] @ n(x0, w["layers.0.attn_norm"])
    hd = cfg.head_dim
    heads = [v[(h * cfg.n_kv_heads // cfg.n_q_heads) * hd:][:hd] for h in range(cfg.n_q_heads)]
    x1 = x0 + w["layers.0.wo"] @ np.concatenate(heads)
    y = n(x1, w["layers.0.ffn_norm"])
    g = w["layers.0.w_gate"] @ y
    x2 = x1 + w["layers.0.w_down"] @ ((g / (1 + np.exp(-g))) * (w["layers.0.w_up"] @ y))
    want = w["embed"] @ n(x2, w["final_norm"])
    o = Oracle(cfg, _weights(cfg, seed=3), 1, 4)
    got = o.step(np.array([[tok]]), np.array([0]))[0, 0]
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-11)


def test_first_token_closed_form_delta():
    """One gated-delta-net layer at the first token from a zero state: S = beta k_hat v^T, so the
    output of each head is beta (k_hat . q_hat) v."""
    cfg = tiny("gdn_gqa", n_layers=1)
    assert cfg.mixers == ("gdn",)
    wt = _weights(cfg, seed=5)
    w = {k: v.float().numpy().astype(np.float64) for k, v in wt.items()}
    tok = 11
    x0 = w["embed"][tok]
    y = x0 / np.sqrt(np.mean(x0 * x0) + cfg.norm_eps)
    H, dk, dv = cfg.lin_heads, cfg.lin_dk, cfg.lin_dv
    q = (w["layers.0.wq"] @ y).reshape(H, dk)
    k = (w["layers.0.wk"] @ y).reshape(H, dk)
    v = (w["layers.0.wv"] @ y).reshape(H, dv)
    beta = 1 / (1 + np.exp(-(w["layers.0.wb"] @ y)))
    qh = q / np.sqrt((q * q).sum(1, keepdims=True) + 1e-6) / np.sqrt(dk)
    kh = k / np.sqrt((k * k).sum(1, keepdims=True) + 1e-6)
    o = (beta * (kh * qh).sum(1))[:, None] * v
    x1 = x0 + w["layers.0.wo"] @ o.reshape(-1)
    y1 = x1 / np.sqrt(np.mean(x1 * x1) + cfg.norm_eps)
    g = w["layers.0.w_gate"] @ y1
    x2 = x1 + w["layers.0.w_down"] @ ((g / (1 + np.exp(-g))) * (w["layers.0.w_up"] @ y1))
    want = w["lm_head"] @ (x2 / np.sqrt(np.mean(x2 * x2) + cfg.norm_eps))
    got = Oracle(cfg, wt, 1, 4).step(np.array([[tok]]), np.array([0]))[0, 0]
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-11)


def test_moe_closed_form_one_row():
    """MoE FFN of one row written out directly: shared expert + sum of renormalised sigmoid weights
    times the picked experts; the pick is the stable sort of the biased scores."""
    cfg = tiny("nvfp4_moe", n_layers=1, router_bias_std=0.05)
    wt = _weights(cfg, seed=9)
    o = Oracle(cfg, wt, 1, 4)
    rng = np.random.default_rng(3)
    h = rng.standard_normal((1, 1, cfg.d_model))
    got = o.moe(0, h)[0, 0]
    y = h[0, 0]
    z = wt["layers.0.w_router"].float().numpy().astype(np.float64) @ y
    s = 1 / (1 + np.exp(-z))
    biased = s + wt["layers.0.router_bias"].numpy()
    pick = np.argsort(-biased, kind="stable")[: cfg.top_k]
    wts = cfg.route_scale * s[pick] / s[pick].sum()

    def ffn(kind, e):
        gw, uw, dw = (o.expert(0, kind, m, e) for m in ("gate", "up", "down"))
        g = gw @ y
        return dw @ ((g / (1 + np.exp(-g))) * (uw @ y))

    want = ffn("s", 0) + sum(wi * ffn("e", e) for e, wi in zip(pick, wts))
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-13)
    # the NVFP4 decode the oracle used is the exact e2m1 * e4m3 * fp32 product of the stored bytes
    dec = o.expert(0, "e", "gate", 1)
    q = wt["layers.0.e_gate.q"][1].numpy()
    code0 = q[0, 0] & 15
    sc = ops.e4m3_value(wt["layers.0.e_gate.s"][1].numpy()[0, 0])
    assert dec[0, 0] == ops.e2m1_value(code0) * sc * np.float64(wt["layers.0.e_gate.g"][1].item())


@pytest.mark.parametrize("kind", ["dense", "kda_mla_moe"])
def test_bf16_cache_reading_rounds_only_the_cache(kind):
    """cache_round="bf16" stores exactly the bf16 rounding of what the exact oracle stores (in the first
    cached layer, whose inputs are the same in both)."""
    cfg = tiny(kind)
    w = _weights(cfg)
    toks = make_tokens(0, "ctx", (2, 5), cfg.vocab).numpy()
    a, b = Oracle(cfg, w, 2, 16), Oracle(cfg, w, 2, 16, cache_round="bf16")
    a.step(toks, np.zeros(2, dtype=int))
    b.step(toks, np.zeros(2, dtype=int))
    first = 0 if cfg.mixers[0] == "gqa" else 3
    if cfg.mixers[first] == "gqa":
        for x, y in zip(a.kv[first], b.kv[first]):
            np.testing.assert_array_equal(ops.bf16_round(x), y)
    else:
        # layer 3 is the first MLA layer; its inputs differ only through layers 0..2, which have no cache
        np.testing.assert_array_equal(ops.bf16_round(a.lat[first][:, :5]), b.lat[first][:, :5])


def test_forced_routing_uses_given_experts():
    """forced_routing = the oracle's own picks changes nothing; a different forced set gives the MoE closed
    form over those experts with weights renormalised over their sigmoid scores, while `routing` still
    records the row's own picks."""
    cfg = tiny("nvfp4_moe", n_layers=1, router_bias_std=0.05)
    wt = _weights(cfg, seed=9)
    rng = np.random.default_rng(11)
    h = rng.standard_normal((1, 1, cfg.d_model))
    o = Oracle(cfg, wt, 1, 4)
    base = o.moe(0, h)
    own = o.routing[0][0].copy()
    o._forced = {0: own}
    np.testing.assert_array_equal(o.moe(0, h), base)
    pick = np.array([[[5, 1]]])
    assert not np.array_equal(np.sort(pick[0, 0]), np.sort(own[0, 0]))
    o._forced = {0: pick}
    got = o.moe(0, h)[0, 0]
    np.testing.assert_array_equal(o.routing[0][0], own)
    y = h[0, 0]
    z = wt["layers.0.w_router"].float().numpy().astype(np.float64) @ y
    s = 1 / (1 + np.exp(-z))
    wts = cfg.route_scale * s[[5, 1]] / s[[5, 1]].sum()

    def ffn(kind, e):
        gw, uw, dw = (o.expert(0, kind, m, e) for m in ("gate", "up", "down"))
        g = gw @ y
        return dw @ ((g / (1 + np.exp(-g))) * (uw @ y))

    want = ffn("s", 0) + wts[0] * ffn("e", 5) + wts[1] * ffn("e", 1)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("k", [0, 2, 7])
def test_greedy_accept_equals_sequential_greedy_prefix(k):
    """A verify block whose first k drafts are what sequential greedy decoding from the anchor produces, and
    whose next draft differs, accepts k + 1 rows and emits that decoding's (k + 1)-th token as the bonus."""
    import copy
    cfg = tiny("gdn_gqa")
    w = _weights(cfg)
    o = Oracle(cfg, w, 1, 32)
    o.prefill(make_tokens(0, "ctx", (1, 6), cfg.vocab).numpy())
    anchor = 5
    seq = copy.deepcopy(o)
    greedy, tok = [], anchor
    for t in range(8):
        tok = int(np.argmax(seq.step(np.array([[tok]]), np.array([6 + t]))[0, 0]))
        greedy.append(tok)
    drafts = list(greedy[:k])
    if k < 7:
        drafts.append((greedy[k] + 1) % cfg.vocab)
    drafts += [0] * (7 - len(drafts))
    block = np.array([anchor] + drafts)
    logits = o.step(block[None], np.array([6]))[0]
    a, bonus = ops.greedy_accept(logits, block)
    assert a == k + 1
    assert bonus == greedy[k]
