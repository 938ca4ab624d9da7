"""Whole-stack decode step, plain and slow: the definition the CUDA megakernel is checked against.

Block structure (pre-norm, no biases):   x += Mixer(RMSNorm(x));  x += FFN(RMSNorm(x))
then a final RMSNorm and the LM head. Layer i uses full attention (GQA or MLA) when i % 4 == 3 and
a delta-rule mixer (gated delta net or KDA) otherwise; the pages' kernel branches on
``index % 4 == 3`` per layer (Kimi K3's TPU megakernel, "How it maps onto a TPU v7").

Step semantics (what one call computes), per sequence b:
  * the sequence has c_b committed tokens and u_b pending rows left by the previous call;
  * a call with ``positions[b] = p_b`` (c_b <= p_b <= c_b + u_b) commits the first p_b - c_b pending
    rows and discards the rest: the recurrent state becomes the state after those rows and cache
    entries at positions >= p_b are dead;
  * the R new rows sit at positions p_b .. p_b + R - 1; row r attends over positions 0 .. p_b + r and
    sees the recurrent state advanced through rows 0 .. r; logits are returned for every row;
  * afterwards c_b = p_b and u_b = R.
This is how the pages' verify step works: eight rows of one sequence are checked at once and only the
accepted prefix is kept (Kimi K3's TPU megakernel, "What DSpark changes per step"). Plain decode is
R = 1 with p_b advancing by one. A prefill is one block of T rows that is then committed whole.

Parity status: every mixer, the router and the FFNs are pinned (tests/test_oracle_*.py). The block
composition is pinned by closed forms at the first token (attention over one key returns v; the delta
rule from a zero state is one rank-1 update). The MLA front half (the c_q and c_kv norms, the nope /
rope split of the up-projected query, RoPE on the query and on the rope key) is pinned against an
independent torch formulation (complex-number RoPE, scaled_dot_product_attention on the unabsorbed
heads) and by invariances that a dropped norm or a misplaced split breaks; the KDA decay layout (which
row of the decay projection gates which head and key channel) by a two-token closed form. The caches
hold exact (float64) keys, values and latents.
This module is test infrastructure: only the tests, the package's smoke check and the benchmark's CPU
baseline use it; the CUDA path never imports it.
"""
from __future__ import annotations

import numpy as np

from . import ops

F64 = np.float64


def _np(t):
    """torch tensor or array -> numpy; bf16 -> float32 (exact)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu()
            if t.dtype == torch.bfloat16:
                t = t.float()
            return t.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t)


class Oracle:
    """The decode step of one model for a batch of ``batch`` sequences.

    ``weights`` maps the names drawn by ``synthetic.make_weights`` to tensors or arrays.

    ``cache_round="bf16"`` stores the cached keys, values and MLA latents rounded to bf16 instead of exactly.
    The definition keeps them exact; this mode is the pages' statement that the reference computes with a
    bf16 trunk and bf16 activations (Kimi K3's TPU megakernel, "Is it like for like?"), used where floating
    point decides an integer: the router's top-k is compared in that precision, because bf16-stored
    activations move router scores by up to ~1e-3 and flip picks whose scores are that close.

    ``forced_routing`` (a dict layer -> expert ids [B, R, top_k], consumed by the next ``step``) makes the MoE
    layers use the given experts (weights renormalised over their own sigmoid scores) while ``routing`` still
    records each row's own picks: how the exact oracle follows the routing decided in the pages' precision."""

    def __init__(self, cfg, weights: dict, batch: int, max_ctx: int, cache_round: str | None = None):
        self.cfg = cfg
        self.B = batch
        self.max_ctx = max_ctx
        self.w = {k: _np(v) for k, v in weights.items()}
        self._dequant_cache: dict = {}
        assert cache_round in (None, "bf16")
        self.cache_round = cache_round
        self.forced_routing = None
        self._forced = None
        self.reset()

    def _store(self, x):
        """A value as the cache keeps it (exact, or bf16 in the ``cache_round`` reading)."""
        return ops.bf16_round(x) if self.cache_round == "bf16" else x

    # ------------------------------------------------------------------------------------------
    def reset(self):
        cfg, B = self.cfg, self.B
        self.c = np.zeros(B, dtype=np.int64)   # committed tokens
        self.u = np.zeros(B, dtype=np.int64)   # pending rows of the previous call
        self.kv = {}      # layer -> (K, V) [B, max_ctx, Hkv, hd]   (gqa)
        self.lat = {}     # layer -> [B, max_ctx, kv_lora + rope]    (mla)
        self.S = {}       # layer -> [B, H, dk, dv] committed state  (gdn/kda)
        self.snaps = {}   # layer -> list over b of [R, H, dk, dv] states after each pending row
        for i, kind in enumerate(cfg.mixers):
            if kind == "gqa":
                shape = (B, self.max_ctx, cfg.n_kv_heads, cfg.head_dim)
                self.kv[i] = (np.zeros(shape), np.zeros(shape))
            elif kind == "mla":
                self.lat[i] = np.zeros((B, self.max_ctx, cfg.kv_lora + cfg.qk_rope))
            else:
                self.S[i] = np.zeros((B, cfg.lin_heads, cfg.lin_dk, cfg.lin_dv))
                self.snaps[i] = [np.zeros((0, cfg.lin_heads, cfg.lin_dk, cfg.lin_dv)) for _ in range(B)]
        self.routing = {}

    # ------------------------------------------------------------------------------------------
    def W(self, name):
        return self.w[name]

    def expert(self, layer: int, kind: str, mat: str, e: int) -> np.ndarray:
        """Weight of expert ``e`` (kind "e" routed, "s" shared), matrix "gate"/"up"/"down"."""
        name = f"layers.{layer}.{kind}_{mat}"
        if self.cfg.expert_fmt == "bf16":
            return self.w[name][e]
        key = (name, e)
        if key not in self._dequant_cache:
            if self.cfg.expert_fmt == "nvfp4":
                self._dequant_cache[key] = ops.nvfp4_decode(
                    self.w[name + ".q"][e], self.w[name + ".s"][e], float(self.w[name + ".g"][e]))
            elif mat == "down":  # "f4": MXFP4 down projection
                self._dequant_cache[key] = ops.mxfp4_decode(self.w[name + ".q"][e], self.w[name + ".x"][e])
            else:  # "f4": FP8-E4M3 gate / up with one bf16 scale per 256 rows
                self._dequant_cache[key] = ops.fp8_rows_decode(self.w[name + ".f8"][e], self.w[name + ".f8s"][e])
        return self._dequant_cache[key]

    # ------------------------------------------------------------------------------------------
    def step(self, tokens, positions) -> np.ndarray:
        """One call: tokens [B, R] int, positions [B] int -> logits [B, R, V] float64."""
        cfg = self.cfg
        tokens = np.asarray(tokens, dtype=np.int64)
        positions = np.asarray(positions, dtype=np.int64)
        B, R = tokens.shape
        assert B == self.B
        for b in range(B):
            a = positions[b] - self.c[b]
            if not (0 <= a <= self.u[b]) or positions[b] + R > self.max_ctx:
                raise ValueError(f"sequence {b}: position {positions[b]} outside "
                                 f"[{self.c[b]}, {self.c[b] + self.u[b]}] or beyond the context")
            for i in self.S:
                if a > 0:
                    self.S[i][b] = self.snaps[i][b][a - 1]
            self.c[b] = positions[b]
        if np.any(tokens < 0) or np.any(tokens >= cfg.vocab):
            raise ValueError("token id out of range")

        x = self.W("embed")[tokens].astype(F64)  # [B, R, d]
        self._forced, self.forced_routing = self.forced_routing, None
        for i, kind in enumerate(cfg.mixers):
            h = ops.rmsnorm(x, self.W(f"layers.{i}.attn_norm"), cfg.norm_eps)
            x = x + self.mixer(i, kind, h, positions)
            h = ops.rmsnorm(x, self.W(f"layers.{i}.ffn_norm"), cfg.norm_eps)
            x = x + self.ffn(i, h)
        self.x_final = x
        h = ops.rmsnorm(x, self.W("final_norm"), cfg.norm_eps)
        head = self.W("embed") if cfg.tied else self.W("lm_head")
        self.u[:] = R
        return ops.linear(h, head)

    def prefill(self, tokens) -> np.ndarray:
        """Process a whole context [B, T] from an empty state as one block and commit it."""
        tokens = np.asarray(tokens)
        self.reset()
        logits = self.step(tokens, np.zeros(self.B, dtype=np.int64))
        self.commit(tokens.shape[1])
        return logits

    def commit(self, n: int):
        """Commit the first n pending rows of every sequence (no new rows)."""
        for b in range(self.B):
            assert n <= self.u[b]
            for i in self.S:
                if n > 0:
                    self.S[i][b] = self.snaps[i][b][n - 1]
                self.snaps[i][b] = self.snaps[i][b][:0]
            self.c[b] += n
            self.u[b] = 0

    # ------------------------------------------------------------------------------------------
    def mixer(self, i: int, kind: str, h: np.ndarray, positions) -> np.ndarray:
        if kind == "gqa":
            return self.gqa(i, h, positions)
        if kind in ("gdn", "kda"):
            return self.delta(i, kind, h)
        if kind == "mla":
            return self.mla(i, h, positions)
        raise ValueError(kind)

    def gqa(self, i, h, positions):
        """Grouped-query attention layer over the KV cache. The cache keeps the rotated keys and the
        values exactly (float64): the pages say nothing about cache precision, so the definition holds
        them unrounded, and a cache stored in a narrower type is an implementation choice whose
        rounding the comparison tolerance has to absorb."""
        cfg = self.cfg
        hq, hkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
        B, R, _ = h.shape
        p = f"layers.{i}."
        q = ops.linear(h, self.W(p + "wq")).reshape(B, R, hq, hd)
        k = ops.linear(h, self.W(p + "wk")).reshape(B, R, hkv, hd)
        v = ops.linear(h, self.W(p + "wv")).reshape(B, R, hkv, hd)
        K, V = self.kv[i]
        out = np.empty((B, R, hq * hd))
        for b in range(B):
            pos = positions[b] + np.arange(R)
            qb = ops.rope(q[b], pos[:, None], cfg.rope_theta)
            kb = ops.rope(k[b], pos[:, None], cfg.rope_theta)
            K[b, pos] = self._store(kb)
            V[b, pos] = self._store(v[b])
            o = ops.gqa_block_attention(qb, K[b], V[b], int(positions[b]))
            out[b] = o.reshape(R, hq * hd)
        return ops.linear(out, self.W(p + "wo"))

    def delta(self, i, kind, h):
        """Gated delta net (scalar decay per head) or KDA (decay per key channel) layer."""
        cfg = self.cfg
        H, dk, dv = cfg.lin_heads, cfg.lin_dk, cfg.lin_dv
        B, R, _ = h.shape
        p = f"layers.{i}."
        q = ops.linear(h, self.W(p + "wq")).reshape(B, R, H, dk)
        k = ops.linear(h, self.W(p + "wk")).reshape(B, R, H, dk)
        v = ops.linear(h, self.W(p + "wv")).reshape(B, R, H, dv)
        a_logit = ops.linear(h, self.W(p + "wa"))
        alpha = ops.sigmoid(a_logit).reshape(B, R, H, dk) if kind == "kda" else ops.sigmoid(a_logit)
        beta = ops.sigmoid(ops.linear(h, self.W(p + "wb")))      # [B, R, H]
        q_hat = ops.l2_normalize(q) / np.sqrt(dk)
        k_hat = ops.l2_normalize(k)
        out = np.empty((B, R, H, dv))
        for b in range(B):
            S = self.S[i][b].copy()
            snaps = np.empty((R, H, dk, dv))
            for r in range(R):
                for hh in range(H):
                    S[hh], out[b, r, hh] = ops.delta_rule_step(
                        S[hh], q_hat[b, r, hh], k_hat[b, r, hh], v[b, r, hh],
                        alpha[b, r, hh], beta[b, r, hh])
                snaps[r] = S
            self.snaps[i][b] = snaps
        return ops.linear(out.reshape(B, R, H * dv), self.W(p + "wo"))

    def mla_qkv(self, i, h, positions):
        """Shared front half of MLA: queries split into (nope, rope), the new latents appended."""
        cfg = self.cfg
        H, nope, rp, lora = cfg.mla_heads, cfg.qk_nope, cfg.qk_rope, cfg.kv_lora
        B, R, _ = h.shape
        p = f"layers.{i}."
        c_q = ops.rmsnorm(ops.linear(h, self.W(p + "w_dq")), self.W(p + "q_norm"), cfg.norm_eps)
        qf = ops.linear(c_q, self.W(p + "w_uq")).reshape(B, R, H, nope + rp)
        kv = ops.linear(h, self.W(p + "w_dkv"))
        c_kv = ops.rmsnorm(kv[..., :lora], self.W(p + "kv_norm"), cfg.norm_eps)
        lat = self.lat[i]
        q_nope = qf[..., :nope]
        q_rope = np.empty((B, R, H, rp))
        for b in range(B):
            pos = positions[b] + np.arange(R)
            q_rope[b] = ops.rope(qf[b, :, :, nope:], pos[:, None], cfg.rope_theta)
            k_r = ops.rope(kv[b, :, lora:], pos, cfg.rope_theta)
            lat[b, pos] = self._store(np.concatenate([c_kv[b], k_r], axis=-1))
        return q_nope, q_rope

    def mla(self, i, h, positions, absorbed: bool = True):
        """Multi-head latent attention over a cache of one (kv_lora + rope)-wide latent per position
        (576 = 512 + 64 in the pages' model: Kimi K3's TPU megakernel, "Why one user at a time is a
        bandwidth problem").

        Absorbed form (what the decode step computes): q~_h = W_UK[h] q_nope_h, scores
        (q~_h . c_t + q_rope_h . k_r,t) / sqrt(nope + rope), o_lat_h = sum_t p_t c_t, o_h = W_UV[h] o_lat_h.
        Unabsorbed form (``absorbed=False``, for the pin): k_h,t = [W_UK[h]^T c_t, k_r,t],
        v_h,t = W_UV[h] c_t and ordinary attention."""
        cfg = self.cfg
        H, nope, rp, lora, vh = cfg.mla_heads, cfg.qk_nope, cfg.qk_rope, cfg.kv_lora, cfg.v_head
        B, R, _ = h.shape
        p = f"layers.{i}."
        q_nope, q_rope = self.mla_qkv(i, h, positions)
        w_uk = self.W(p + "w_uk").astype(F64)   # [H, lora, nope]
        w_uv = self.W(p + "w_uv").astype(F64)   # [H, vh, lora]
        scale = 1.0 / np.sqrt(nope + rp)
        out = np.empty((B, R, H, vh))
        for b in range(B):
            p0 = int(positions[b])
            T = p0 + R
            c = self.lat[i][b, :T, :lora]
            kr = self.lat[i][b, :T, lora:]
            mask = np.arange(T)[None, :] <= (p0 + np.arange(R))[:, None]   # [R, T]
            for hh in range(H):
                if absorbed:
                    qt = q_nope[b, :, hh] @ w_uk[hh].T                    # [R, lora]
                    s = (qt @ c.T + q_rope[b, :, hh] @ kr.T) * scale       # [R, T]
                    s = np.where(mask, s, -np.inf)
                    o_lat = ops.softmax_attend(s, c)                       # [R, lora]
                    out[b, :, hh] = o_lat @ w_uv[hh].T
                else:
                    k_nope = c @ w_uk[hh]                                  # [T, nope]
                    vv = c @ w_uv[hh].T                                    # [T, vh]
                    kk = np.concatenate([k_nope, kr], axis=-1)
                    qq = np.concatenate([q_nope[b, :, hh], q_rope[b, :, hh]], axis=-1)
                    s = (qq @ kk.T) * scale
                    s = np.where(mask, s, -np.inf)
                    out[b, :, hh] = ops.softmax_attend(s, vv)
        return ops.linear(out.reshape(B, R, H * vh), self.W(p + "wo"))

    # ------------------------------------------------------------------------------------------
    def ffn(self, i, h):
        cfg = self.cfg
        p = f"layers.{i}."
        if cfg.ffn == "dense":
            return ops.swiglu(h, self.W(p + "w_gate"), self.W(p + "w_up"), self.W(p + "w_down"))
        return self.moe(i, h)

    def moe(self, i, h):
        """Router, shared expert(s) with weight 1, routed experts weighted by the router: the
        per-layer order of the pages' MoE block (Kimi K3's TPU megakernel, Figure 4 caption)."""
        cfg = self.cfg
        p = f"layers.{i}."
        B, R, d = h.shape
        z = ops.linear(h, self.W(p + "w_router"))            # [B, R, E]
        bias = self.W(p + "router_bias")
        out = np.zeros((B, R, d))
        idx_all = np.zeros((B, R, cfg.top_k), dtype=np.int64)
        biased_all = np.zeros((B, R, cfg.n_experts))
        for b in range(B):
            for r in range(R):
                y = h[b, r]
                acc = np.zeros(d)
                for s_ in range(cfg.n_shared):
                    acc += ops.swiglu(y, self.expert(i, "s", "gate", s_), self.expert(i, "s", "up", s_),
                                      self.expert(i, "s", "down", s_))
                idx, wts, biased = ops.route(z[b, r], bias, cfg.top_k, cfg.route_scale)
                idx_all[b, r] = idx
                biased_all[b, r] = biased
                if self._forced is not None and i in self._forced:
                    idx = np.asarray(self._forced[i][b, r], dtype=np.int64)
                    s_used = ops.sigmoid(z[b, r][idx])
                    wts = cfg.route_scale * s_used / np.sum(s_used)
                for e, we in zip(idx, wts):
                    acc += we * ops.swiglu(y, self.expert(i, "e", "gate", e), self.expert(i, "e", "up", e),
                                           self.expert(i, "e", "down", e))
                out[b, r] = acc
        self.routing[i] = (idx_all, biased_all)
        return out
