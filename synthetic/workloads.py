"""Model shapes and seeded inputs for the five decode workloads.

Every tensor is drawn from its own ``torch.Generator`` whose seed is a hash of (seed, tensor name),
so any tensor can be regenerated alone and the draw does not depend on generation order.
Draws are N(0, init_std) in fp32, rounded to bf16 round-to-nearest-even by ``Tensor.to``.
Norm gains are 1. Expert weights of NVFP4 models are drawn the same way and then encoded by
``synthetic.nvfp4.quantize_nvfp4``; those of the "f4" format (the pages' own: FP8-E4M3 gate / up with a
bf16 scale per 256 rows, MXFP4 down) are encoded to MXFP4 by ``synthetic.mxfp4.quantize_mxfp4`` and the
gate / up re-encoded by ``synthetic.mxfp4.reencode_fp8_rows``.

Draws on "cuda" and on "cpu" differ for the same seed (different generators); a test that compares
the two paths generates once, on one device, and hands copies of the same tensors to both.
"""
from __future__ import annotations

import dataclasses
import hashlib
from dataclasses import dataclass, field

import torch

from .nvfp4 import quantize_nvfp4_experts
from .mxfp4 import quantize_mxfp4, reencode_fp8_rows


@dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    d_model: int
    vocab: int
    mixers: tuple  # per layer: "gqa" | "gdn" | "kda" | "mla"
    ffn: str  # "dense" | "moe"
    tied: bool = False
    norm_eps: float = 1e-6
    rope_theta: float = 1e4
    init_std: float = 0.02
    # grouped-query attention
    n_q_heads: int = 0
    n_kv_heads: int = 0
    head_dim: int = 0
    # gated delta net / Kimi delta attention
    lin_heads: int = 0
    lin_dk: int = 0
    lin_dv: int = 0
    # multi-head latent attention
    mla_heads: int = 0
    q_lora: int = 0
    kv_lora: int = 0
    qk_nope: int = 0
    qk_rope: int = 0
    v_head: int = 0
    # feed-forward
    ffn_dim: int = 0
    n_experts: int = 0
    top_k: int = 0
    n_shared: int = 0
    expert_dim: int = 0
    route_scale: float = 1.0
    router_bias_std: float = 0.0
    expert_fmt: str = "bf16"  # "bf16" | "nvfp4" | "f4" (FP8-E4M3 gate / up + MXFP4 down; oracle only)

    def with_layers(self, n_layers: int) -> "ModelConfig":
        """Same widths, fewer (or more) layers; the mixer pattern is re-derived."""
        return dataclasses.replace(self, n_layers=n_layers, mixers=_pattern(self, n_layers))


def _pattern(cfg: ModelConfig, n_layers: int) -> tuple:
    kinds = set(cfg.mixers)
    if kinds == {"gqa"}:
        return ("gqa",) * n_layers
    lin = "gdn" if "gdn" in kinds else "kda"
    full = "mla" if "mla" in kinds else "gqa"
    # layer i is a full-attention layer iff i % 4 == 3, a linear (delta-rule) layer otherwise
    return tuple(full if i % 4 == 3 else lin for i in range(n_layers))


def _mk(name, n_layers, lin=None, full="gqa", **kw) -> ModelConfig:
    if lin is None:
        mixers = (full,) * n_layers
    else:
        mixers = tuple(full if i % 4 == 3 else lin for i in range(n_layers))
    return ModelConfig(name=name, n_layers=n_layers, mixers=mixers, **kw)


CONFIGS: dict[str, ModelConfig] = {
    # 2-layer dense decoder, context 128, 16 greedy steps at batch 1
    "tiny_dense": _mk(
        "tiny_dense", 2, d_model=256, vocab=1024, ffn="dense", tied=True,
        n_q_heads=4, n_kv_heads=1, head_dim=64, ffn_dim=512),
    # 64 layers, 3 gated-delta-net : 1 GQA, bf16, context 4096 (also run as 8-row verify)
    "hybrid_gdn_gqa": _mk(
        "hybrid_gdn_gqa", 64, lin="gdn", full="gqa", d_model=5120, vocab=151936, ffn="dense",
        n_q_heads=24, n_kv_heads=4, head_dim=256, lin_heads=16, lin_dk=128, lin_dv=128,
        ffn_dim=17408),
    # 12 layers, 3 KDA : 1 MLA, MoE 64 experts top-8 + 1 shared, bf16, context 8192
    "moe_kda_mla": _mk(
        "moe_kda_mla", 12, lin="kda", full="mla", d_model=7168, vocab=163840, ffn="moe",
        lin_heads=64, lin_dk=128, lin_dv=128, mla_heads=64, q_lora=1536, kv_lora=512,
        qk_nope=128, qk_rope=64, v_head=128, n_experts=64, top_k=8, n_shared=1,
        expert_dim=2048, route_scale=2.5),
    # 16 GQA layers, MoE 256 experts top-8 + 1 shared in NVFP4, router bias, context 8192
    "moe_nvfp4_gqa": _mk(
        "moe_nvfp4_gqa", 16, d_model=6144, vocab=202048, ffn="moe", n_q_heads=48, n_kv_heads=8,
        head_dim=128, n_experts=256, top_k=8, n_shared=1, expert_dim=2048, route_scale=2.5,
        router_bias_std=0.01, expert_fmt="nvfp4"),
}


def config(name: str, n_layers: int | None = None, **overrides) -> ModelConfig:
    cfg = CONFIGS[name]
    if n_layers is not None:
        cfg = cfg.with_layers(n_layers)
    if overrides:
        cfg = dataclasses.replace(cfg, **overrides)
        if "n_layers" in overrides:
            cfg = cfg.with_layers(overrides["n_layers"])
    return cfg


def _seed(seed: int, name: str) -> int:
    h = hashlib.sha256(f"{seed}:{name}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _randn(shape, seed, name, std, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(seed, name))
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def _bf16(shape, seed, name, std, device) -> torch.Tensor:
    return _randn(shape, seed, name, std, device).to(torch.bfloat16)


def weight_names(cfg: ModelConfig) -> dict[str, tuple]:
    """Name -> shape of every bf16/fp32 tensor (NVFP4 expert tensors are listed by their
    logical [.., out, in] shape under the base name; ``make_weights`` stores them as
    ``<name>.q``/``.s``/``.g``)."""
    d = cfg.d_model
    out = {"embed": (cfg.vocab, d), "final_norm": (d,)}
    if not cfg.tied:
        out["lm_head"] = (cfg.vocab, d)
    for i, kind in enumerate(cfg.mixers):
        p = f"layers.{i}."
        out[p + "attn_norm"] = (d,)
        out[p + "ffn_norm"] = (d,)
        if kind == "gqa":
            hq, hkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
            out[p + "wq"] = (hq * hd, d)
            out[p + "wk"] = (hkv * hd, d)
            out[p + "wv"] = (hkv * hd, d)
            out[p + "wo"] = (d, hq * hd)
        elif kind in ("gdn", "kda"):
            h, dk, dv = cfg.lin_heads, cfg.lin_dk, cfg.lin_dv
            out[p + "wq"] = (h * dk, d)
            out[p + "wk"] = (h * dk, d)
            out[p + "wv"] = (h * dv, d)
            out[p + "wa"] = (h * dk, d) if kind == "kda" else (h, d)
            out[p + "wb"] = (h, d)
            out[p + "wo"] = (d, h * dv)
        elif kind == "mla":
            h = cfg.mla_heads
            out[p + "w_dq"] = (cfg.q_lora, d)
            out[p + "q_norm"] = (cfg.q_lora,)
            out[p + "w_uq"] = (h * (cfg.qk_nope + cfg.qk_rope), cfg.q_lora)
            out[p + "w_dkv"] = (cfg.kv_lora + cfg.qk_rope, d)
            out[p + "kv_norm"] = (cfg.kv_lora,)
            out[p + "w_uk"] = (h, cfg.kv_lora, cfg.qk_nope)
            out[p + "w_uv"] = (h, cfg.v_head, cfg.kv_lora)
            out[p + "wo"] = (d, h * cfg.v_head)
        else:
            raise ValueError(kind)
        if cfg.ffn == "dense":
            out[p + "w_gate"] = (cfg.ffn_dim, d)
            out[p + "w_up"] = (cfg.ffn_dim, d)
            out[p + "w_down"] = (d, cfg.ffn_dim)
        else:
            e, f = cfg.n_experts, cfg.expert_dim
            out[p + "w_router"] = (e, d)
            out[p + "router_bias"] = (e,)
            out[p + "e_gate"] = (e, f, d)
            out[p + "e_up"] = (e, f, d)
            out[p + "e_down"] = (e, d, f)
            out[p + "s_gate"] = (cfg.n_shared, f, d)
            out[p + "s_up"] = (cfg.n_shared, f, d)
            out[p + "s_down"] = (cfg.n_shared, d, f)
    return out


_ONES = ("final_norm", "attn_norm", "ffn_norm", "q_norm", "kv_norm")
_EXPERT = ("e_gate", "e_up", "e_down", "s_gate", "s_up", "s_down")


def make_weights(cfg: ModelConfig, seed: int = 0, device="cpu") -> dict[str, torch.Tensor]:
    """Draw every weight of ``cfg``. bf16 tensors keep their logical shape; NVFP4 expert
    tensors become ``<name>.q`` (uint8, two e2m1 codes per byte, element 2i in the low nibble),
    ``<name>.s`` (uint8 e4m3 bits, one per 16 inputs) and ``<name>.g`` (fp32, one per expert). In the
    "f4" format a down projection becomes ``<name>.q`` (packed e2m1 codes) and ``<name>.x`` (uint8 E8M0,
    one per 32 inputs); a gate / up projection ``<name>.f8`` (uint8 e4m3 codes, one per weight) and
    ``<name>.f8s`` (int32 holding bf16 bits, one per 256 rows)."""
    out: dict[str, torch.Tensor] = {}
    for name, shape in weight_names(cfg).items():
        leaf = name.rsplit(".", 1)[-1]
        if leaf in _ONES:
            out[name] = torch.ones(shape, dtype=torch.bfloat16, device=device)
        elif leaf == "router_bias":
            if cfg.router_bias_std > 0:
                out[name] = _randn(shape, seed, name, cfg.router_bias_std, device)
            else:
                out[name] = torch.zeros(shape, dtype=torch.float32, device=device)
        elif leaf in _EXPERT and cfg.expert_fmt == "nvfp4":
            # experts are drawn one by one (each from its own stream) and encoded 16 at a time
            qs, ss, gs = [], [], []
            for e0 in range(0, shape[0], 16):
                w = torch.stack([_bf16(shape[1:], seed, f"{name}.{e}", cfg.init_std, device).float()
                                 for e in range(e0, min(shape[0], e0 + 16))])
                q, s, g = quantize_nvfp4_experts(w)
                qs.append(q)
                ss.append(s)
                gs.append(g)
                del w
            out[name + ".q"] = torch.cat(qs)
            out[name + ".s"] = torch.cat(ss)
            out[name + ".g"] = torch.cat(gs).to(torch.float32)
        elif leaf in _EXPERT and cfg.expert_fmt == "f4":
            # MXFP4 as shipped; gate / up re-encoded to e4m3 codes with one bf16 scale per 256 rows
            enc = [quantize_mxfp4(_bf16(shape[1:], seed, f"{name}.{e}", cfg.init_std, device).float())
                   for e in range(shape[0])]
            if leaf.endswith("_down"):
                out[name + ".q"] = torch.stack([q for q, _ in enc])
                out[name + ".x"] = torch.stack([x for _, x in enc])
            else:
                f8 = [reencode_fp8_rows(q, x) for q, x in enc]
                out[name + ".f8"] = torch.stack([c for c, _ in f8])
                out[name + ".f8s"] = torch.stack([sb for _, sb in f8])
        elif leaf in _EXPERT:
            out[name] = torch.stack(
                [_bf16(shape[1:], seed, f"{name}.{e}", cfg.init_std, device) for e in range(shape[0])])
        else:
            out[name] = _bf16(shape, seed, name, cfg.init_std, device)
    return out


def make_tokens(seed: int, tag: str, shape, vocab: int, device="cpu") -> torch.Tensor:
    """Uniform token ids in [0, vocab) as int32, from the stream (seed, tag)."""
    g = torch.Generator(device=device)
    g.manual_seed(_seed(seed, "tokens:" + tag))
    return torch.randint(0, vocab, tuple(shape), generator=g, device=device, dtype=torch.int64).to(torch.int32)


@dataclass(frozen=True)
class Workload:
    """A benchmarked or parity-tested run of one model."""
    model: str
    batches: tuple
    context: int
    rows: int = 1  # query rows per sequence per step (8 for speculative verify)
    accept_lengths: tuple = ()
    steps: int = 16
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny_dense_greedy": Workload("tiny_dense", (1,), 128, steps=16),
    "hybrid_gdn_gqa_decode": Workload("hybrid_gdn_gqa", (1, 2, 4, 8), 4096),
    "hybrid_gdn_gqa_verify": Workload("hybrid_gdn_gqa", (1, 2), 4096, rows=8, accept_lengths=(3, 6)),
    "moe_kda_mla_decode": Workload("moe_kda_mla", (1, 4, 8), 8192),
    "moe_kda_mla_verify": Workload("moe_kda_mla", (1,), 8192, rows=8, accept_lengths=(3, 6)),
    "moe_nvfp4_gqa_decode": Workload("moe_nvfp4_gqa", (1, 2, 4, 8), 8192),
    "moe_nvfp4_gqa_verify": Workload("moe_nvfp4_gqa", (1,), 8192, rows=8, accept_lengths=(3, 6)),
}
