"""Algorithmic bytes of one decode step, for the HBM roofline.

A decode step at small batch is weight streaming: every matrix of the dense trunk is read once per step,
plus the routed experts actually selected, plus the KV / latent cache read, the new cache rows written,
the recurrent state read and written once, and the logits written (the pages' single-stream roofline:
bytes per token over HBM bandwidth, Kimi K3's TPU megakernel, "The bandwidth arithmetic").
"""
from __future__ import annotations

BF16 = 2
FP32 = 4


def floor_ms(total_bytes: float, bandwidth_gbs: float) -> float:
    """Time to move `total_bytes` at `bandwidth_gbs` (GB/s = 1e9 B/s), in ms."""
    return total_bytes / (bandwidth_gbs * 1e9) * 1e3


def expected_union(n_experts: int, top_k: int, rows: int) -> float:
    """Expected number of distinct experts when `rows` rows each pick `top_k` of `n_experts` uniformly
    and independently: E (1 - (1 - k/E)^rows)."""
    return n_experts * (1.0 - (1.0 - top_k / n_experts) ** rows)


def expert_bytes(cfg) -> int:
    """Bytes of one routed expert (gate, up, down)."""
    f, d = cfg.expert_dim, cfg.d_model
    n = 3 * f * d
    if cfg.expert_fmt == "nvfp4":
        return n // 2 + n // 16 + 3 * FP32  # e2m1 codes, e4m3 block scales, per-matrix fp32 scales
    return n * BF16


def dense_weight_bytes(cfg) -> int:
    """Bytes of every non-routed matrix read by one step (all layers, LM head; embedding rows excluded)."""
    d = cfg.d_model
    total = d * BF16  # final norm
    total += cfg.vocab * d * BF16  # LM head (a tied embedding is read in full as the head)
    for kind in cfg.mixers:
        total += 2 * d * BF16  # the two norms
        if kind == "gqa":
            hq, hkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
            total += (hq + 2 * hkv) * hd * d * BF16 + d * hq * hd * BF16
        elif kind in ("gdn", "kda"):
            h, dk, dv = cfg.lin_heads, cfg.lin_dk, cfg.lin_dv
            na = h * dk if kind == "kda" else h
            total += (2 * h * dk + h * dv + na + h) * d * BF16 + d * h * dv * BF16
        elif kind == "mla":
            h = cfg.mla_heads
            total += cfg.q_lora * d * BF16 + cfg.q_lora * BF16
            total += h * (cfg.qk_nope + cfg.qk_rope) * cfg.q_lora * BF16
            total += (cfg.kv_lora + cfg.qk_rope) * d * BF16 + cfg.kv_lora * BF16
            total += h * cfg.kv_lora * cfg.qk_nope * BF16 + h * cfg.v_head * cfg.kv_lora * BF16
            total += d * h * cfg.v_head * BF16
        if cfg.ffn == "dense":
            total += 3 * cfg.ffn_dim * d * BF16
        else:
            total += cfg.n_experts * d * BF16  # router
            total += cfg.n_shared * expert_bytes(cfg)
    return total


def step_bytes(cfg, batch: int, rows: int, prefix: list[int], expert_reads: int | None = None) -> dict:
    """Algorithmic bytes of one step of `batch` sequences x `rows` rows; prefix[b] = cached positions of
    sequence b before the step. expert_reads = routed experts read (the union per layer summed over
    layers), taken from the step's actual routing; None = the uniform-routing expectation."""
    n = batch * rows
    d = cfg.d_model
    out = {"weights": dense_weight_bytes(cfg) + n * d * BF16}
    kv_read = kv_write = state = 0
    for kind in cfg.mixers:
        if kind == "gqa":
            per_pos = 2 * cfg.n_kv_heads * cfg.head_dim * BF16
            kv_read += sum(prefix) * per_pos
            kv_write += n * per_pos
        elif kind == "mla":
            per_pos = (cfg.kv_lora + cfg.qk_rope) * BF16
            kv_read += sum(prefix) * per_pos
            kv_write += n * per_pos
        else:
            state += 2 * batch * cfg.lin_heads * cfg.lin_dk * cfg.lin_dv * FP32
    out["kv_read"] = kv_read
    out["kv_write"] = kv_write
    out["state"] = state
    if cfg.ffn == "moe":
        if expert_reads is None:
            expert_reads = expected_union(cfg.n_experts, cfg.top_k, n) * cfg.n_layers
        out["experts"] = int(expert_reads * expert_bytes(cfg))
    out["logits"] = n * cfg.vocab * FP32
    out["total"] = sum(out.values())
    return out
