#!/usr/bin/env python
"""Benchmark of the DSpark/DFlash drafter step on one GB300 (or N replicas).

Workload (default): the MiniCPM-shaped drafter in bf16 (H 2048, m 5 taps,
d 2048, 16 heads of 128, 5 layers, F 4096, gamma 8, V 73448, Markov rank 256),
batch 1.  One step = a fresh sequence ingests L = 1024 context rows of
features [1024, 10240] (Eq 2 + Eq 3 into the per-layer K/V caches) and drafts
one block of 8 tokens over that context.  Inputs are seeded synthetic draws
(weights N(0, 0.02), norms 1, features and embedding N(0, 1)); 16 distinct
feature batches (21 MB each) are cycled, so every step streams > 1 GB of
weights, caches and features: far more than the 129 MB L2.

Prints one JSON line: draft blocks/s (= steps/s) over the whole job, context
tokens/s, the per-phase rates, the roofline of the dominant kernel class
(timed live with CUDA events on the launching stream), clocks sampled during
the timed region, the end-to-end rate through the host-buffer C-ABI calls, and
the CPU oracle's rate on a bounded sample.

--impl reference times the CPU oracle itself on the same workload (rank 0).
Multi-GPU (torchrun): every rank runs an independent replica; no collective
touches the data path (replicas only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic as syn  # noqa: E402

POOL = 16  # distinct feature batches cycled through the steps


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="minicpm_L1024")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap.parse_args()


# --------------------------------------------------------------------------- distributed (replicas)

def dist_setup(n):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 200 ms) during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 8:
                continue
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except ValueError:
                continue
            for nm, v in zip(names, r[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- work accounting

def class_work(cls: str, cfg, T: int, L: int):
    """Algorithmic bytes and flops of one timed range of a kernel class, and its bound.

    T: context rows ingested per step; L: context length at draft time.
    bf16 weights/caches (2 B), fp32 activations/logits (4 B)."""
    d, F, H, V, r, g, nL, mH = (cfg.d_draft, cfg.ff, cfg.hidden, cfg.vocab, cfg.markov_rank, cfg.gamma,
                                cfg.n_layers, cfg.feat_dim)
    if cls == "ingest_proj":
        return dict(bytes=T * mH * 2 + d * mH * 2 + T * d * 4, flops=2 * T * mH * d, bound="tensor")
    if cls == "ingest_kv":
        return dict(bytes=nL * (T * d * 2 + 2 * d * d * 2 + T * 2 * d * 2), flops=nL * 2 * T * d * 2 * d, bound="tensor")
    if cls == "out_proj":
        return dict(bytes=V * d * 2 + g * V * 4, flops=2 * g * V * d, bound="hbm")
    if cls == "attention":
        return dict(bytes=2 * (L + g) * d * 2, flops=4 * g * (L + g) * d, bound="hbm")
    if cls == "markov_argmax":
        return dict(bytes=V * r * 2 + g * V * 4, flops=2 * g * V * r, bound="hbm")
    if cls == "qkv_proj":
        return dict(bytes=3 * d * d * 2, flops=2 * g * 3 * d * d, bound="hbm")
    if cls == "o_proj":
        return dict(bytes=d * d * 2, flops=2 * g * d * d, bound="hbm")
    if cls == "gate_up_proj":
        return dict(bytes=2 * F * d * 2, flops=2 * g * 2 * F * d, bound="hbm")
    if cls == "down_proj":
        return dict(bytes=F * d * 2, flops=2 * g * F * d, bound="hbm")
    if cls == "block_build":
        return dict(bytes=d * H * 2, flops=2 * d * H, bound="hbm")
    return dict(bytes=0, flops=0, bound="hbm")


def draft_bytes_min(cfg, L):
    """Algorithmic bytes of one batch-1 draft block: every weight once (w2 once),
    the caches of all layers, the embedding row."""
    d, F, H, V, r, nL = cfg.d_draft, cfg.ff, cfg.hidden, cfg.vocab, cfg.markov_rank, cfg.n_layers
    layers = nL * (4 * d * d + 3 * F * d) * 2
    return layers + d * H * 2 + V * d * 2 + V * r * 2 + cfg.gamma * r * 2 + nL * 2 * (L + cfg.gamma) * d * 2 + H * 2


def ingest_flops(cfg, T):
    d, mH, nL = cfg.d_draft, cfg.feat_dim, cfg.n_layers
    return 2 * T * mH * d + nL * 2 * T * d * 2 * d


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), "src": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


def load_traffic(kernel_class: str, workload: str):
    """DRAM bytes per range from a committed ncu summary, if it still matches the kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    ent = table.get(f"{workload}/{kernel_class}")
    if not ent:
        return None
    import hashlib
    src = os.path.join(ROOT, ent["source"])
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    return ent["bytes_per_range"] if digest == ent.get("source_sha") else None


# --------------------------------------------------------------------------- CPU oracle timing

def time_oracle(wl, W, feats_pool, anchors, seconds: float, max_steps: int):
    import oracle
    cfg = wl.cfg
    dr = oracle.Drafter(cfg, W)
    n, t0 = 0, time.perf_counter()
    while n < max_steps:
        dr.reset(0)
        dr.ingest(feats_pool[n % len(feats_pool)])
        dr.draft(int(anchors[n % len(anchors)]))
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return n, dt


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# --------------------------------------------------------------------------- main

def main():
    args = parse()
    wl = syn.WORKLOADS[args.workload]
    cfg = wl.cfg
    assert wl.n_seqs == 1 and cfg.dtype == "bf16", "the bench drives batch-1 bf16 workloads"
    rank, world, local = dist_setup(args.gpus)
    T = wl.ctx_len
    metric = "draft blocks/s (batch 1, fresh context of 1024 rows ingested per block)"

    anchors = syn.anchors(syn.Workload(wl.name, cfg, steps=POOL))[:, 0]
    if args.impl == "reference":
        if rank != 0:
            return
        W = syn.make_weights(cfg, seed=0)
        pool = [syn.make_feats(cfg, T, seed=0, step=i) for i in range(min(POOL, 4))]
        import oracle  # noqa: F401
        n_w = max(1, args.warmup)
        time_oracle(wl, W, pool, anchors, 1e9, n_w)
        n, dt = time_oracle(wl, W, pool, anchors, 1e9, args.steps)
        v = n / dt
        line = {"impl": "reference", "metric": metric, "value": v, "unit": "blocks/s", "n_gpus": args.gpus,
                "steps": n, "warmup": n_w, "ms_per_step": 1e3 * dt / n, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": wl.name, "ctx_len": T, "gamma": cfg.gamma, "batch": 1},
                "cpu_baseline": {"value": v, "unit": "blocks/s", "cores": cpu_cores(), "kind": "oracle",
                                 "sample": f"{n} full steps (ingest {T} rows + 1 block), fp64 numpy"},
                "e2e": {"value": v, "unit": "blocks/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch

    import block_draft_model_gb300 as bdm
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    bdm.build()
    bdm.load()
    W = syn.make_weights(cfg, seed=0)
    Wd = {}
    for k, v in W.items():
        t = torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).to(dev)
        Wd[k] = t.view(torch.bfloat16) if v.dtype == np.uint16 else t
    pool_np = [syn.make_feats(cfg, T, seed=0, step=i) for i in range(POOL)]
    pool = [torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16) for x in pool_np]
    g = bdm.Drafter(hidden=cfg.hidden, n_taps=cfg.n_taps, d_draft=cfg.d_draft, n_heads=cfg.n_heads,
                    n_layers=cfg.n_layers, ff_mult=cfg.ff_mult, gamma=cfg.gamma, vocab=cfg.vocab,
                    markov_rank=cfg.markov_rank, eps=cfg.eps, dtype=bdm.BF16, max_ctx=T, weights=Wd)
    stream = torch.cuda.current_stream(dev)
    tok = torch.empty(cfg.gamma, dtype=torch.int32, device=dev)
    conf = torch.empty(cfg.gamma, dtype=torch.float32, device=dev)

    def step(i):
        g.reset(0)
        g.ingest_context(pool[i % POOL])
        g.draft(int(anchors[i % POOL]), tok, conf)

    # warm-up, with a profile of every kernel class to find the dominant one
    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    g.profile(-1)
    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    prof_all = g.profile_read()
    g.profile(0)
    dominant = max(prof_all, key=lambda k: prof_all[k][0])

    # timed region: K steps; only the dominant class carries event pairs
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    g.profile(1 << prof_all[dominant][3])
    l0 = g.launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = g.launch_count() - l0
    prof = g.profile_read()
    g.profile(0)
    ms = ev0.elapsed_time(ev1)
    ms_max = reduce_max(ms, world, dev)
    clk = clocks.stop() if rank == 0 else None

    # the dominant kernel's live timing (ranges recorded on the launching stream in the timed region)
    dms, dranges, dlaunch, _ = prof[dominant]
    peaks = load_peaks()
    work = class_work(dominant, cfg, T, T)
    per_range_s = dms / 1e3 / max(dranges, 1)
    if work["bound"] == "tensor":
        ach = work["flops"] / per_range_s / 1e12
        peak = peaks["bf16_tflops"]
        unit = "TFLOP/s"
    else:
        ach = work["bytes"] / per_range_s / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    roofline = {"kernel": dominant, "bound": work["bound"], "achieved": ach, "peak": peak, "unit": unit,
                "frac": ach / peak, "peak_src": peaks["src"], "traffic": load_traffic(dominant, wl.name),
                "algorithmic_per_launch": work["bytes"] if work["bound"] == "hbm" else work["flops"],
                "avg_range_us": per_range_s * 1e6, "launches_per_range": dlaunch / max(dranges, 1),
                "share_of_step": prof_all[dominant][0] / sum(v[0] for v in prof_all.values())}

    # phases (outside the timed region): ingest-only and draft-only rates
    def timed(fn, n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(n):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    nph = max(10, min(args.steps, 50))
    ms_ingest = timed(lambda i: (g.reset(0), g.ingest_context(pool[i % POOL])), nph)
    g.reset(0)
    g.ingest_context(pool[0])
    ms_draft = timed(lambda i: g.draft(int(anchors[i % POOL]), tok, conf), nph)
    per_class = {k: round(v[0] / 4, 4) for k, v in prof_all.items() if v[1]}

    # end to end through the host-buffer C-ABI calls (pinned host memory)
    host_pool = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in pool_np[:4]]
    tok_h = torch.empty(cfg.gamma, dtype=torch.int32).pin_memory()
    conf_h = torch.empty(cfg.gamma, dtype=torch.float32).pin_memory()
    ne2e = max(5, min(args.steps, 50))
    for i in range(2):
        g.reset(0)
        g.ingest_context_host(host_pool[i % 4])
        g.draft_host(int(anchors[i % POOL]), tok_h, conf_h)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(ne2e):
        g.reset(0)
        g.ingest_context_host(host_pool[i % 4])
        g.draft_host(int(anchors[i % POOL]), tok_h, conf_h)
    e2e_s = reduce_max(time.perf_counter() - t0, world, dev)
    assert g.check() == 0

    value = world * args.steps / (ms_max / 1e3)
    line = {"metric": metric, "value": value, "unit": "blocks/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "ctx_len": T, "gamma": cfg.gamma, "batch": 1, "d_draft": cfg.d_draft,
                       "vocab": cfg.vocab, "parallelism": f"replicas{world}" if world > 1 else "single",
                       "l2": "inputs larger than L2 (>1 GB streamed per step; 16 feature batches cycled)"},
            "ctx_tokens_per_s": value * T,
            "phases": {"ingest_ms": ms_ingest, "ingest_ctx_tokens_per_s": T / (ms_ingest / 1e3),
                       "ingest_tflops": ingest_flops(cfg, T) / (ms_ingest / 1e3) / 1e12,
                       "draft_ms": ms_draft, "draft_blocks_per_s": 1e3 / ms_draft,
                       "draft_bytes_min": draft_bytes_min(cfg, T),
                       "draft_gbs_of_bytes_min": draft_bytes_min(cfg, T) / (ms_draft / 1e3) / 1e9,
                       "per_class_ms": per_class},
            "roofline": roofline,
            "clocks": clk,
            "gpu_launches": launches,
            "e2e": {"value": world * ne2e / e2e_s, "unit": "blocks/s",
                    "h2d_bytes_per_step": int(T * cfg.feat_dim * 2), "d2h_bytes_per_step": int(cfg.gamma * 8)}}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n, dt = time_oracle(wl, W, pool_np[:4], anchors, args.cpu_seconds, 50)
        line["cpu_baseline"] = {"value": n / dt, "unit": "blocks/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": f"{n} full steps (ingest {T} rows + 1 block) of the same workload, fp64"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    g.close()


if __name__ == "__main__":
    main()
