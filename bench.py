#!/usr/bin/env python
"""Decode benchmark of the GB300 whole-model megakernel.

Default: the hybrid gated-delta-net / GQA stack (64 layers, d_model 5120, bf16, 4096-token random context)
decoding greedily at batch 1, one megakernel launch per step, plus a sweep over batch 2, 4 and 8.
Prints ONE JSON line (rank 0). `value` is decode tokens/s with every input already in HBM (CUDA events on
the launch stream); `e2e` is the same through the host-buffer C-ABI entry point (token and position copies
in, greedy tokens out, every step). `roofline` divides the algorithmic bytes of a step (weights + KV read +
KV write + recurrent state read/write + logits) by the measured step time and by the measured HBM copy
bandwidth. `cpu_baseline` is the CPU oracle timed on a bounded sample of the same step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mk|reference] [--workload NAME] [--batch B]
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
    ("hybrid_gdn_gqa_decode", 1): (42.83e9, "b39980a8e12caa51"),
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
    ap.add_argument("--workload", default="hybrid_gdn_gqa_decode")
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--sweep", default="2,4,8", help="extra batch sizes timed after the headline ('' = none)")
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
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
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
    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------------
# CPU oracle on a bounded sample of the step
# ------------------------------------------------------------------------------------------------
class OracleSampler:
    """The oracle's decode step on a bounded sample of the model, built once and timed per step: the first
    k layers at full width (k = 4: three delta-rule layers and one attention layer; 1 for MoE models, whose
    layers hold tens of GB of experts) and an LM head over the first 1/8 of the vocabulary, after a
    16-token prefill. The layer time is scaled to the full depth and the head time to the full vocabulary."""

    def __init__(self, cfg, weights_cpu_fn, batch: int, rows: int):
        from oracle import Oracle
        self.cfg, self.batch, self.rows = cfg, batch, rows
        self.k = 1 if cfg.ffn == "moe" else (4 if cfg.n_layers >= 4 else cfg.n_layers)
        self.head_frac = 8 if cfg.vocab >= 8 * 1024 else 1
        self.sub = dataclasses.replace(cfg.with_layers(self.k), vocab=cfg.vocab // self.head_frac)
        self.orc = Oracle(self.sub, weights_cpu_fn(self.sub), batch, 64 + 64 * rows)
        self.rng = np.random.default_rng(0)
        self.orc.prefill(self.rng.integers(0, self.sub.vocab, size=(batch, 16)))
        self.pos = np.full(batch, 16)

    def step(self) -> float:
        """One timed step; returns the estimated seconds of a full-model step."""
        from oracle import ops
        sub = self.sub
        toks = self.rng.integers(0, sub.vocab, size=(self.batch, self.rows))
        t0 = time.perf_counter()
        self.orc.step(toks, self.pos)
        t_step = time.perf_counter() - t0
        self.pos = self.pos + self.rows
        h = ops.rmsnorm(self.orc.x_final, self.orc.W("final_norm"), sub.norm_eps)
        t0 = time.perf_counter()
        ops.linear(h, self.orc.W("embed") if sub.tied else self.orc.W("lm_head"))
        t_head = time.perf_counter() - t0
        return (t_step - t_head) * self.cfg.n_layers / self.k + t_head * self.head_frac

    def describe(self, n_steps: int) -> str:
        return (f"oracle (numpy float64) decode step of the first {self.k} of {self.cfg.n_layers} layers at full "
                f"width plus an LM head over 1/{self.head_frac} of the vocabulary, batch {self.batch}, "
                f"{self.rows} row(s), 16-token context, {n_steps} step(s); layer time scaled to "
                f"{self.cfg.n_layers} layers, head time to the full vocabulary")


def sample_weights_from(w: dict, sub):
    """The tensors of `sub` (its first layers, embedding / LM head rows of its vocabulary) copied to the
    host from a full model's weights."""
    out = {}
    for name, t in w.items():
        if name.startswith("layers.") and int(name.split(".")[1]) >= sub.n_layers:
            continue
        if name in ("embed", "lm_head"):
            t = t[: sub.vocab]
        out[name] = t.cpu()
    return out


def oracle_sample(cfg, weights_cpu_fn, batch: int, rows: int, n_steps: int = 2):
    """Time the oracle on its bounded sample (OracleSampler). Returns (tok/s, seconds per step estimate,
    description)."""
    smp = OracleSampler(cfg, weights_cpu_fn, batch, rows)
    est = statistics.median([smp.step() for _ in range(n_steps)])
    return batch * rows / est, est, smp.describe(n_steps)


# ------------------------------------------------------------------------------------------------
def run_reference(args, wl, cfg):
    """The oracle as the reference arm: timed on the host cores, rank 0 only; the sample is built once
    and each of the warm-up + timed steps is one oracle step on it."""
    import torch
    from synthetic import make_weights
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if ws > 1 and rank != 0:
        return
    B, R = args.batch, wl.rows
    tok_per_step = B * (args.accept if R > 1 else 1)

    smp = OracleSampler(cfg, lambda sub: make_weights(sub, seed=0, device="cpu"), B, R)
    for _ in range(args.warmup):
        smp.step()
    sec = statistics.median([smp.step() for _ in range(args.steps)])
    desc = smp.describe(args.steps)
    val = tok_per_step / sec
    cores = os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
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
            "prefill": f"one {T}-token random-token prefill, forked to all {B} sequences",
            "l2": "inputs larger than L2 (every step streams the whole weight set, far above 129 MB)"}


def run_mk(args, wl, cfg):
    import torch
    from decode_megakernel_04_gb300 import Megakernel, _build, roofline
    from synthetic import make_tokens, make_weights

    ws, rank, local = dist_setup(args)
    if rank == 0:
        _build.build()
    barrier(ws)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    w = make_weights(cfg, seed=0, device=dev)
    R = wl.rows
    adv = args.accept if R > 1 else 1
    T = args.context or wl.context
    W, K = args.warmup, args.steps
    hbm, peak_kind = peaks()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass

    def measure(B, K_, with_e2e):
        max_ctx = T + (W + K_ + 2) * adv * (2 if with_e2e else 1) + 5 * adv + 2 * R + 16
        mk = Megakernel(cfg, w, max_batch=B, max_rows=8, max_ctx=max_ctx, device=local)
        # one prefill of sequence 0, forked to the others (the decode steps then diverge: every row draws
        # its own tokens); the caches and states of every sequence are separate copies in HBM
        ctx = make_tokens(rank, "ctx", (1, T), cfg.vocab, device=dev).contiguous()
        mk.prefill(ctx, stream=sh)
        for b in range(1, B):
            mk.fork(0, b, stream=sh)
        torch.cuda.synchronize()
        steps = W + K_
        toks = torch.empty((steps + 1, B, R), dtype=torch.int32, device=dev)
        toks.copy_(make_tokens(rank, "stream", (steps + 1, B, R), cfg.vocab, device=dev))
        pos = torch.tensor([[T + s * adv] * B for s in range(steps)], dtype=torch.int32, device=dev)
        logits = torch.empty((B * R, cfg.vocab), dtype=torch.float32, device=dev)
        for s in range(W):
            am = toks[s + 1].view(-1) if R == 1 else None
            mk.step(toks[s], pos[s], logits, am, stream=sh)
        if mk.status(sh) != 0:
            raise RuntimeError("device status after warm-up: " + str(mk.status(sh)))
        torch.cuda.synchronize()
        barrier(ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with Clocks(uuid) as clk:
            e0.record(stream)
            for s in range(W, steps):
                am = toks[s + 1].view(-1) if R == 1 else None
                mk.step(toks[s], pos[s], logits, am, stream=sh)
            e1.record(stream)
            torch.cuda.synchronize()
        barrier(ws)
        st = mk.status(sh)
        if st != 0:
            raise RuntimeError(f"device status {st}")
        ms = e0.elapsed_time(e1) / K_
        ms = max_over_ranks(ms, ws)
        e2e = None
        if with_e2e:
            p0 = T + steps * adv
            tk = toks[steps].cpu().numpy().astype(np.int32).reshape(B, R).copy()
            am = np.zeros(B * R, dtype=np.int32)
            for s in range(W):
                mk.step_host(tk, np.full(B, p0 + s * adv, dtype=np.int32), am, stream=sh)
                if R == 1:
                    tk = am.reshape(B, 1).copy()
            barrier(ws)
            t0 = time.perf_counter()
            for s in range(W, steps):
                mk.step_host(tk, np.full(B, p0 + s * adv, dtype=np.int32), am, stream=sh)
                if R == 1:
                    tk = am.reshape(B, 1).copy()
            dt = (time.perf_counter() - t0) / K_
            dt = max_over_ranks(dt, ws)
            e2e = {"value": ws * B * adv / dt, "unit": "tokens/s",
                   "h2d_bytes_per_step": int(4 * (B * R + B)), "d2h_bytes_per_step": int(4 * B * R),
                   "ms_per_step": dt * 1e3}
        expert_reads = None
        if cfg.ffn == "moe":
            # routed experts read per step: the union of the experts the step's rows selected, per layer,
            # from the routing log of a few more steps of the same token stream (outside the timed region)
            log = torch.full((cfg.n_layers, B, max_ctx, cfg.top_k), -1, dtype=torch.int32, device=dev)
            mk.set_routing_log(log)
            unions = []
            base = T + steps * adv * (2 if with_e2e else 1)   # past every position used above
            for s in range(4):
                p_s = base + s * adv
                mk.step(toks[(W + s) % (steps + 1)], torch.full((B,), p_s, dtype=torch.int32, device=dev), logits, None, stream=sh)
                if mk.status(sh) != 0:
                    raise RuntimeError("device status in the routing-log steps")
                lg = log.cpu().numpy()
                u = 0
                for layer in range(cfg.n_layers):
                    rows = [lg[layer, b, p_s + r] for b in range(B) for r in range(R)]
                    u += len(np.unique(np.concatenate(rows)))
                unions.append(u)
            mk.set_routing_log(None)
            expert_reads = float(np.mean(unions))
        mk.close()
        del ctx, toks, pos, logits
        return ms, clk.summary(), e2e, expert_reads

    B = args.batch
    ms, clocks, e2e, ereads = measure(B, K, not args.no_e2e)
    acct = roofline.step_bytes(cfg, B, R, [T + W * adv + K * adv // 2] * B, expert_reads=ereads)
    achieved = acct["total"] / (ms * 1e-3) / 1e9
    sweep = {}
    for sb in [int(x) for x in args.sweep.split(",") if x.strip()]:
        if sb == B or sb * R > 64:
            continue
        sms, sclk, _, sereads = measure(sb, max(5, K // 2), False)
        sacct = roofline.step_bytes(cfg, sb, R, [T + W * adv + K * adv // 4] * sb, expert_reads=sereads)
        sweep[str(sb)] = {"tokens_per_s": ws * sb * adv / (sms * 1e-3), "ms_per_step": sms,
                          "hbm_gbs": sacct["total"] / (sms * 1e-3) / 1e9,
                          "frac": sacct["total"] / (sms * 1e-3) / 1e9 / hbm,
                          "frac_nominal_8tbs": sacct["total"] / (sms * 1e-3) / 1e9 / NOMINAL_HBM_GBS}
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu:
        rate, est, desc = oracle_sample(cfg, lambda sub: sample_weights_from(w, sub), B, R)
        cpu = {"value": rate * (adv / R if R > 1 else 1), "unit": "tokens/s", "cores": os.cpu_count(),
               "kind": "oracle", "sample": desc}
    key = (args.workload, B)
    traffic = None
    if key in KNOWN_TRAFFIC and KNOWN_TRAFFIC[key][1] == sources_hash():
        traffic = KNOWN_TRAFFIC[key][0]
    line = {
        "metric": METRIC, "value": ws * B * adv / (ms * 1e-3), "unit": "tokens/s", "n_gpus": ws,
        "steps": K, "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if cfg.expert_fmt == "bf16" else "bf16+nvfp4", "data": "synthetic",
        "config": workload_config(wl, cfg, B, args),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "frac_nominal_8tbs": achieved / NOMINAL_HBM_GBS, "traffic": traffic,
                     "peak_kind": f"{peak_kind} copy bandwidth", "bytes_per_step": acct},
        "verify_steps_per_s": (1e3 / ms) if R > 1 else None,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": K, "clocks": clocks,
        "sweep": sweep, "kernel": "megakernel (one persistent launch per step)",
    }
    print(json.dumps(line))


def main():
    args = parse()
    from synthetic import config
    from synthetic.workloads import WORKLOADS
    wl = WORKLOADS[args.workload]
    cfg = config(wl.model, n_layers=args.layers or None)
    if args.impl == "reference":
        run_reference(args, wl, cfg)
    else:
        run_mk(args, wl, cfg)


if __name__ == "__main__":
    main()
