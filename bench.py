#!/usr/bin/env python
"""Decode benchmark of the GB300 whole-model megakernel.

Headline: the hybrid gated-delta-net / GQA stack (64 layers, d_model 5120, bf16, 4096-token random context)
decoding greedily at batch 1, one megakernel launch per step. The default run also times, in `results`, every
(model, batch, mode) of the plan: the hybrid stack at batch 1..64 and in 8-row verify (batch 1 and 2,
accepted lengths 6 and 3), the KDA/MLA MoE model (8192 context) and the NVFP4 MoE model (8192 context), and
`multi_step`: 16 greedy steps per launch. Prints ONE JSON line (rank 0). `value` is decode tokens/s with
every input already in HBM (CUDA events on the launch stream); `e2e` is the same through the host-buffer
C-ABI entry point (token and position copies in, greedy token out, every step). `roofline` divides the
algorithmic bytes of a step (weights + KV read + KV write + recurrent state read/write + routed experts
actually selected + logits) by the measured step time and by the measured HBM copy bandwidth (and by the
nominal 8 TB/s). `cpu_baseline` is the CPU oracle timed on a sample of the same step (an estimate: see
OracleSampler).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mk|reference] [--workload all|NAME]
                  [--batch B] [--sweep B1,B2] [--quick]
Under torchrun every rank runs an independent replica on its own GPU (the path has no exchange step);
`value` sums the tokens of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s at batch 1–8 on 1 GB300; achieved HBM GB/s vs 8 TB/s roofline"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0   # the roofline the workload's target is stated against

# DRAM bytes per launch from one ncu capture, keyed by (workload, batch) and valid only for the kernel
# sources they were taken with (the hash below); null once the sources change.
KNOWN_TRAFFIC: dict = {
    # a 4-layer full-width capture of the same kernel, scaled to 64 layers by the algorithmic bytes
    ("hybrid_gdn_gqa_decode", 1): (42.92e9, "d1a69160638aa9b1"),
}


def sources_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_megakernel_04_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--workload", default="all",
                    help="'all' (default): every model's batch / verify plan, the hybrid decode at batch 1 as the "
                         "headline; or one workload name with --batch / --sweep")
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--sweep", default="", help="single-workload runs: extra batch sizes ('' = none)")
    ap.add_argument("--quick", action="store_true", help="'all' runs: the hybrid model's batch 1..8 entries only")
    ap.add_argument("--budget-s", type=float, default=900.0, help="skip further models after this many seconds")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (diagnostic runs only)")
    ap.add_argument("--context", type=int, default=0, help="override the context length (diagnostic runs only)")
    ap.add_argument("--accept", type=int, default=6, help="accepted length per verify step (verify workloads)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class Clocks:
    """nvidia-smi samples of this GPU's SM clock and throttle reasons during the timed region."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            self.proc.wait(timeout=10)
            self.out.close()

    def summary(self) -> dict:
        mhz, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            lines = open(self.path).read().strip().splitlines()
        except OSError:
            lines = []
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            if self.uuid and parts[0] != self.uuid:
                continue
            try:
                mhz.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if self.path:
            os.unlink(self.path)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(mhz)}


def dist_setup(args):
    """One process per GPU under torchrun (NCCL); the same host logic runs over gloo on a machine without a
    GPU, which is how the multi-rank path is tested."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(ws: int, units_per_rank: float, seconds: float) -> float:
    """Units all ranks processed per second of the slowest rank (every rank runs the same replica work)."""
    return ws * units_per_rank / seconds


# ------------------------------------------------------------------------------------------------
# CPU oracle on a bounded sample of the step
# ------------------------------------------------------------------------------------------------
class OracleSampler:
    """The oracle's decode step on a bounded sample of the model, timed on the host cores: one period of the
    layer pattern (k = 4 layers: three delta-rule layers and one attention layer) at full width, every cache
    and state filled for `context` positions (random values: the step's cost does not depend on them, and no
    GPU data reaches the oracle), and the LM head over the full vocabulary. A full step is estimated as the
    time of the k layers times n_layers / k plus the head: the depth is scaled, the context and the
    vocabulary are the workload's own. MoE models keep one layer (their experts alone are tens of GB)."""

    def __init__(self, cfg, weights_cpu_fn, batch: int, rows: int, context: int):
        from oracle import Oracle
        self.cfg, self.batch, self.rows, self.context = cfg, batch, rows, context
        self.k = 1 if cfg.ffn == "moe" else (4 if cfg.n_layers >= 4 else cfg.n_layers)
        self.sub = cfg.with_layers(self.k)
        self.orc = Oracle(self.sub, weights_cpu_fn(self.sub), batch, context + 64 * rows + 64)
        rng = np.random.default_rng(0)
        for i, (K, V) in self.orc.kv.items():
            K[:, :context] = rng.standard_normal(K[:, :context].shape)
            V[:, :context] = rng.standard_normal(V[:, :context].shape)
        for i, lat in self.orc.lat.items():
            lat[:, :context] = rng.standard_normal(lat[:, :context].shape)
        for i, S in self.orc.S.items():
            S[:] = 0.01 * rng.standard_normal(S.shape)
        self.orc.c[:] = context
        self.orc.u[:] = 0
        self.rng = rng
        self.pos = np.full(batch, context)

    def step(self):
        """One timed step; returns (seconds of the sample step, estimated seconds of a full-model step)."""
        from oracle import ops
        sub = self.sub
        toks = self.rng.integers(0, sub.vocab, size=(self.batch, self.rows))
        t0 = time.perf_counter()
        self.orc.step(toks, self.pos)
        t_step = time.perf_counter() - t0
        self.pos = self.pos + (1 if self.rows == 1 else 0)
        if self.rows > 1:   # a verify block: the next sample step re-verifies at the same position
            self.orc.u[:] = self.rows
        h = ops.rmsnorm(self.orc.x_final, self.orc.W("final_norm"), sub.norm_eps)
        t0 = time.perf_counter()
        ops.linear(h, self.orc.W("embed") if sub.tied else self.orc.W("lm_head"))
        t_head = time.perf_counter() - t0
        return t_step, (t_step - t_head) * self.cfg.n_layers / self.k + t_head

    def describe(self, n_steps: int) -> str:
        return (f"estimate: oracle (numpy float64) step of {self.k} of {self.cfg.n_layers} layers at full width "
                f"with caches and states filled for {self.context} positions (random contents) plus the LM head "
                f"over the full vocabulary, batch {self.batch}, {self.rows} row(s), {n_steps} step(s); "
                f"layer time x {self.cfg.n_layers / self.k:g} for the full depth")


def sample_weights_from(w: dict, sub):
    """The tensors of `sub` (its first layers, the embedding and the LM head) copied to the host from a full
    model's weights."""
    out = {}
    for name, t in w.items():
        if name.startswith("layers.") and int(name.split(".")[1]) >= sub.n_layers:
            continue
        out[name] = t.cpu()
    return out


def oracle_sample(cfg, weights_cpu_fn, batch: int, rows: int, context: int, n_steps: int = 2):
    """Time the oracle on its sample (OracleSampler). Returns (tok/s estimate, full-step seconds estimate,
    description)."""
    smp = OracleSampler(cfg, weights_cpu_fn, batch, rows, context)
    est = statistics.median([smp.step()[1] for _ in range(n_steps)])
    return batch * rows / est, est, smp.describe(n_steps)


# ------------------------------------------------------------------------------------------------
def run_reference(args, wl, cfg):
    """The oracle as the reference arm: timed on the host cores, rank 0 only. The sample is built once; each
    warm-up and timed step is one oracle step of it. `ms_per_step` is the measured wall time of a sample
    step; `value` is the full-model rate that sample estimates (see OracleSampler)."""
    import torch
    from synthetic import make_weights
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if ws > 1 and rank != 0:
        return
    B, R = args.batch, wl.rows
    tok_per_step = B * (args.accept if R > 1 else 1)
    T = args.context or wl.context
    smp = OracleSampler(cfg, lambda sub: make_weights(sub, seed=0, device="cpu"), B, R, T)
    for _ in range(args.warmup):
        smp.step()
    runs = [smp.step() for _ in range(args.steps)]
    wall = statistics.median([r[0] for r in runs])
    est = statistics.median([r[1] for r in runs])
    desc = smp.describe(args.steps)
    val = tok_per_step / est
    cores = os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall * 1e3,
            "full_step_ms_estimate": est * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, cfg, B, args),
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    del torch


def workload_config(wl, cfg, B, args):
    desc = {
        "hybrid_gdn_gqa": "hybrid gated-delta-net/GQA stack, d_model 5120, bf16",
        "tiny_dense": "tiny dense GQA decoder, d_model 256",
        "moe_kda_mla": "KDA/MLA MoE 64e top-8, d_model 7168, bf16",
        "moe_nvfp4_gqa": "GQA MoE 256e top-8, NVFP4 experts, d_model 6144",
    }[cfg.name]
    mode = f"{wl.rows}-row verify, accepted length {args.accept}" if wl.rows > 1 else "greedy decode"
    T = args.context or wl.context
    return {"workload": f"{desc}, {cfg.n_layers} layers, {mode}, batch {B}, {T}-token context",
            "batch": B, "rows": wl.rows, "context": T, "layers": cfg.n_layers,
            "prefill": f"one {T}-token random-token prefill, forked to all {B} sequences before the timed steps",
            "l2": "inputs larger than L2 (every step streams the whole weight set, far above 129 MB)"}


# The measurements of the default run, per model: (batch, rows, accepted length); rows > 1 is a verify step
# whose positions advance by the accepted length. The first hybrid entry is the headline.
PLAN = {
    "hybrid_gdn_gqa": [(1, 1, 1), (2, 1, 1), (4, 1, 1), (8, 1, 1), (16, 1, 1), (32, 1, 1), (64, 1, 1),
                       (1, 8, 6), (1, 8, 3), (2, 8, 6), (2, 8, 3)],
    "moe_kda_mla": [(1, 1, 1), (4, 1, 1), (8, 1, 1), (1, 8, 6), (1, 8, 3)],
    "moe_nvfp4_gqa": [(1, 1, 1), (2, 1, 1), (4, 1, 1), (8, 1, 1), (1, 8, 6), (1, 8, 3)],
}
MULTI_STEPS = 16   # greedy steps per launch of the multi-step measurement


class ModelBench:
    """One model on one GPU: weights drawn once, one handle whose last sequence (the reserve) holds the
    prefilled context; every measurement first forks the reserve to its sequences, so each starts at
    exactly the workload's context."""

    def __init__(self, cfg, T, max_batch, steps_budget, dev, rank, sh):
        import torch
        from decode_megakernel_04_gb300 import Megakernel
        from synthetic import make_tokens, make_weights
        self.cfg, self.T, self.dev, self.rank, self.sh = cfg, T, dev, rank, sh
        self.w = make_weights(cfg, seed=0, device=dev)
        self.reserve = max_batch
        self.max_ctx = T + steps_budget
        self.mk = Megakernel(cfg, self.w, max_batch=max_batch + 1, max_rows=8, max_ctx=self.max_ctx,
                             device=dev.index or 0)
        ctx = make_tokens(rank, "ctx", (1, T), cfg.vocab, device=dev).contiguous()
        # prefill the reserve: a 1-sequence prefill fills sequence 0, which is then copied to the reserve
        self.mk.prefill(ctx, stream=sh)
        self.mk.fork(0, self.reserve, stream=sh)
        torch.cuda.synchronize()
        self.make_tokens = make_tokens

    def measure(self, B, R, acc, W, K, clocks_uuid, ws, routing_steps=4):
        """W warm-up and K timed steps of B sequences x R rows (positions advance by acc); returns a dict."""
        import torch
        cfg, mk, dev, sh = self.cfg, self.mk, self.dev, self.sh
        for b in range(B):
            mk.fork(self.reserve, b, stream=sh)
        steps = W + K
        adv = acc if R > 1 else 1
        toks = self.make_tokens(self.rank, f"stream{B}x{R}", (steps + 1, B, R), cfg.vocab, device=dev).contiguous()
        pos = torch.tensor([[self.T + s * adv] * B for s in range(steps)], dtype=torch.int32, device=dev)
        logits = torch.empty((B * R, cfg.vocab), dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream(dev)
        for s in range(W):
            mk.step(toks[s], pos[s], logits, toks[s + 1].view(-1) if R == 1 else None, stream=sh)
        st = mk.status(sh)
        if st != 0:
            raise RuntimeError(f"device status {st} after warm-up")
        torch.cuda.synchronize()
        barrier(ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with Clocks(clocks_uuid) as clk:
            e0.record(stream)
            for s in range(W, steps):
                mk.step(toks[s], pos[s], logits, toks[s + 1].view(-1) if R == 1 else None, stream=sh)
            e1.record(stream)
            torch.cuda.synchronize()
        barrier(ws)
        st = mk.status(sh)
        if st != 0:
            raise RuntimeError(f"device status {st}")
        ms = max_over_ranks(e0.elapsed_time(e1) / K, ws)
        expert_reads = None
        if cfg.ffn == "moe":
            expert_reads = self.routed_experts(B, R, adv, routing_steps)
        from decode_megakernel_04_gb300 import roofline
        ctx_mean = self.T + (W + K / 2.0) * adv
        acct = roofline.step_bytes(cfg, B, R, [ctx_mean] * B, expert_reads=expert_reads)
        return {"ms": ms, "clocks": clk.summary(), "bytes": acct, "expert_reads": expert_reads, "context": ctx_mean}

    def routed_experts(self, B, R, adv, n_steps):
        """Routed experts a step of this shape reads: the union of the experts its rows selected, per layer, from
        the routing log of a few more steps of the same kind (outside the timed region)."""
        import torch
        cfg, mk, dev, sh = self.cfg, self.mk, self.dev, self.sh
        for b in range(B):
            mk.fork(self.reserve, b, stream=sh)
        log = torch.full((cfg.n_layers, self.reserve + 1, self.max_ctx, cfg.top_k), -1, dtype=torch.int32,
                         device=dev)
        mk.set_routing_log(log)
        toks = self.make_tokens(self.rank, f"route{B}x{R}", (n_steps, B, R), cfg.vocab, device=dev).contiguous()
        logits = torch.empty((B * R, cfg.vocab), dtype=torch.float32, device=dev)
        unions = []
        for s in range(n_steps):
            p_s = self.T + s * adv
            mk.step(toks[s], torch.full((B,), p_s, dtype=torch.int32, device=dev), logits, None, stream=sh)
            if mk.status(sh) != 0:
                raise RuntimeError("device status in the routing-log steps")
            lg = log.cpu().numpy()
            u = 0
            for layer in range(cfg.n_layers):
                rows = [lg[layer, b, p_s + r] for b in range(B) for r in range(R)]
                u += len(np.unique(np.concatenate(rows)))
            unions.append(u)
        mk.set_routing_log(None)
        del log
        return float(np.mean(unions))

    def e2e(self, W, K, ws):
        """Decode through the host-buffer entry point (token and position copies in, greedy token out)."""
        B = 1
        mk = self.mk
        mk.fork(self.reserve, 0, stream=self.sh)
        tk = np.array([[7]], dtype=np.int32)
        am = np.zeros(B, dtype=np.int32)
        for s in range(W):
            mk.step_host(tk, np.full(B, self.T + s, dtype=np.int32), am, stream=self.sh)
            tk = am.reshape(B, 1).copy()
        barrier(ws)
        t0 = time.perf_counter()
        for s in range(W, W + K):
            mk.step_host(tk, np.full(B, self.T + s, dtype=np.int32), am, stream=self.sh)
            tk = am.reshape(B, 1).copy()
        dt = max_over_ranks((time.perf_counter() - t0) / K, ws)
        return {"value": whole_job_rate(ws, B, dt), "unit": "tokens/s", "h2d_bytes_per_step": int(4 * (B + B)),
                "d2h_bytes_per_step": int(4 * B), "ms_per_step": dt * 1e3,
                "how": "mk_decode_step_host: token and position copied in, greedy token copied out, every step"}

    def multi_step(self, W, K, ws):
        """MULTI_STEPS greedy steps per launch (mk_decode_steps), device-timed, and through the host-buffer
        entry point (one host call per MULTI_STEPS tokens)."""
        import torch
        mk, dev, sh = self.mk, self.dev, self.sh
        S = MULTI_STEPS
        mk.fork(self.reserve, 0, stream=sh)
        tok = torch.tensor([7], dtype=torch.int32, device=dev)
        out = torch.zeros((S,), dtype=torch.int32, device=dev)
        stream = torch.cuda.current_stream(dev)
        for s in range(W):
            mk.steps(tok, torch.tensor([self.T + s * S], dtype=torch.int32, device=dev), S, out, stream=sh)
        torch.cuda.synchronize()
        pos = [torch.tensor([self.T + s * S], dtype=torch.int32, device=dev) for s in range(W, W + K)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s in range(K):
            mk.steps(tok, pos[s], S, out, stream=sh)
        e1.record(stream)
        torch.cuda.synchronize()
        if mk.status(sh) != 0:
            raise RuntimeError("device status in the multi-step launches")
        ms = max_over_ranks(e0.elapsed_time(e1) / K, ws)
        mk.fork(self.reserve, 0, stream=sh)
        tk = np.array([7], dtype=np.int32)
        o = np.zeros((S, 1), dtype=np.int32)
        for s in range(W):
            mk.steps_host(tk, np.array([self.T + s * S], dtype=np.int32), S, o, stream=sh)
        t0 = time.perf_counter()
        for s in range(W, W + K):
            mk.steps_host(tk, np.array([self.T + s * S], dtype=np.int32), S, o, stream=sh)
        dt = max_over_ranks((time.perf_counter() - t0) / K, ws)
        return {"steps_per_launch": S, "ms_per_launch": ms, "tokens_per_s": whole_job_rate(ws, S, ms * 1e-3),
                "e2e_tokens_per_s": whole_job_rate(ws, S, dt), "e2e_ms_per_call": dt * 1e3, "h2d_bytes_per_call": 8,
                "d2h_bytes_per_call": 4 * S}

    def close(self):
        import torch
        self.mk.close()
        del self.w
        torch.cuda.empty_cache()


def result_entry(model, B, R, acc, m, hbm, ws):
    ms = m["ms"]
    gbs = m["bytes"]["total"] / (ms * 1e-3) / 1e9
    e = {"workload": model, "batch": B, "rows": R, "mode": "verify" if R > 1 else "decode",
         "ms_per_step": ms, "tokens_per_s": whole_job_rate(ws, B * (acc if R > 1 else 1), ms * 1e-3),
         "hbm_gbs": gbs, "frac": gbs / hbm, "frac_nominal_8tbs": gbs / NOMINAL_HBM_GBS,
         "bytes_per_step": m["bytes"]["total"], "context": m["context"], "clocks": m["clocks"]}
    if R > 1:
        e["accepted_length"] = acc
        e["verify_steps_per_s"] = 1e3 / ms
    if m["expert_reads"] is not None:
        e["routed_experts_read"] = m["expert_reads"]
    return e


def run_mk(args, wl, cfg):
    import torch
    from decode_megakernel_04_gb300 import _build
    from synthetic import config

    ws, rank, local = dist_setup(args)
    if rank == 0:
        _build.build()
    barrier(ws)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sh = torch.cuda.current_stream(dev).cuda_stream
    W, K = args.warmup, args.steps
    hbm, peak_kind = peaks()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    t_start = time.time()

    if args.workload == "all":
        plan = {m: list(v) for m, v in PLAN.items()}
        if args.quick:
            plan = {"hybrid_gdn_gqa": [e for e in PLAN["hybrid_gdn_gqa"] if e[0] <= 8]}
    else:
        R0 = wl.rows
        batches = [args.batch] + [int(x) for x in args.sweep.split(",") if x.strip() and int(x) != args.batch]
        plan = {wl.model: [(b, R0, args.accept if R0 > 1 else 1) for b in batches if b * R0 <= 64]}
    head_model = next(iter(plan))
    results, head, multi, e2e, cpu = [], None, None, None, None
    T_head = None
    for model, entries in plan.items():
        if time.time() - t_start > args.budget_s and results:
            results.append({"workload": model, "skipped": f"time budget of {args.budget_s:.0f} s reached"})
            continue
        mcfg = cfg if model == cfg.name else config(model)
        if args.layers:
            mcfg = mcfg.with_layers(args.layers)
        from synthetic.workloads import WORKLOADS
        T = args.context or {"hybrid_gdn_gqa": 4096, "tiny_dense": 128}.get(model, 8192)
        budget = (W + K) * 8 + 64 + (W + K) * MULTI_STEPS + 64
        mb = ModelBench(mcfg, T, max(e[0] for e in entries), budget, dev, rank, sh)
        for i, (B, R, acc) in enumerate(entries):
            m = mb.measure(B, R, acc, W, K if (model == head_model and i == 0) else max(5, K // 2), uuid, ws)
            results.append(result_entry(model, B, R, acc, m, hbm, ws))
            if model == head_model and i == 0:
                head = (B, R, acc, m)
                T_head = T
        if model == head_model:
            if not args.no_e2e:
                e2e = mb.e2e(W, K, ws)
                multi = mb.multi_step(W, max(5, K // 2), ws)
            if rank == 0 and not args.no_cpu:
                rate, est, desc = oracle_sample(mcfg, lambda sub: sample_weights_from(mb.w, sub), head[0], head[1], T)
                cpu = {"value": rate, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle", "sample": desc}
        mb.close()
    if rank != 0:
        return
    B, R, acc, m = head
    hcfg = cfg if head_model == cfg.name else config(head_model)
    if args.layers:
        hcfg = hcfg.with_layers(args.layers)
    ms = m["ms"]
    achieved = m["bytes"]["total"] / (ms * 1e-3) / 1e9
    key = (args.workload if args.workload != "all" else "hybrid_gdn_gqa_decode", B)
    traffic = None
    if key in KNOWN_TRAFFIC and KNOWN_TRAFFIC[key][1] == sources_hash() and not args.layers:
        traffic = KNOWN_TRAFFIC[key][0]
    hwl = WORKLOADS_BY_MODEL(head_model, R)
    line = {
        "metric": METRIC, "value": whole_job_rate(ws, B * (acc if R > 1 else 1), ms * 1e-3), "unit": "tokens/s", "n_gpus": ws,
        "steps": K, "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if hcfg.expert_fmt == "bf16" else "bf16+nvfp4", "data": "synthetic",
        "config": workload_config(hwl, hcfg, B, argparse.Namespace(accept=acc, context=T_head)),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "frac_nominal_8tbs": achieved / NOMINAL_HBM_GBS, "traffic": traffic,
                     "peak_kind": f"{peak_kind} copy bandwidth", "bytes_per_step": m["bytes"]},
        "verify_steps_per_s": (1e3 / ms) if R > 1 else None,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": K, "clocks": m["clocks"],
        "results": results, "multi_step": multi,
        "kernel": "megakernel (one persistent launch per step; mk_decode_steps: one launch per 16 steps)",
        "bench_s": time.time() - t_start,
    }
    print(json.dumps(line))


def WORKLOADS_BY_MODEL(model, R):
    from synthetic.workloads import WORKLOADS
    for name, w in WORKLOADS.items():
        if w.model == model and w.rows == R:
            return w
    return next(w for w in WORKLOADS.values() if w.model == model)


def main():
    args = parse()
    from synthetic import config
    from synthetic.workloads import WORKLOADS
    wl = WORKLOADS["hybrid_gdn_gqa_decode" if args.workload == "all" else args.workload]
    cfg = config(wl.model, n_layers=args.layers or None)
    if args.impl == "reference":
        run_reference(args, wl, cfg)
    else:
        run_mk(args, wl, cfg)


if __name__ == "__main__":
    main()
