#!/usr/bin/env python
"""Benchmark of the DSpark/DFlash drafter step on one GB300 (or N replicas).

Workload (default, --workload minicpm_L1024): the MiniCPM-shaped drafter in
bf16 (H 2048, m 5 taps, d 2048, 16 heads of 128, 5 layers, F 4096, gamma 8,
V 73448, Markov rank 256), batch 1.  One step = a fresh sequence ingests
L = 1024 context rows of features [1024, 10240] (Eq 2 + Eq 3 into the
per-layer K/V caches) and drafts one block of 8 tokens over that context.
Inputs are seeded synthetic draws (weights N(0, 0.02), norms 1, features and
embedding N(0, 1)); 16 distinct feature batches (21 MB each) are cycled, so
every step streams > 1 GB of weights, caches and features: far more than the
129 MB L2.

Other workloads (same JSON line): gemma_L32768_ingest (a fresh 32768-row
context and 16 blocks per step), gemma_L4096_stream (1-6 new rows and one
block per step over a 4096-row context), gemma_batched64 (64 ragged sequences,
1-6 new rows and one block each per step).

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
import dataclasses
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
    ap.add_argument("--temperature", type=float, default=0.0,
                    help="> 0: the Markov chain draws its tokens (top-k candidates) instead of the argmax")
    ap.add_argument("--top-k", type=int, default=0)
    ap.add_argument("--n-kv-heads", type=int, default=0,
                    help="grouped-query variant: K/V heads of the drafter (0: one per query head)")
    ap.add_argument("--qk-norm", action="store_true", help="variant: per-head RMSNorm of Q and K")
    ap.add_argument("--rope-theta", type=float, default=0.0, help="variant: rotary embedding base (0: none)")
    ap.add_argument("--oracle-single-thread", action="store_true",
                    help="(internal) time the CPU oracle on a bounded sample in this process and print it as JSON")
    ap.add_argument("--layers", choices=["auto", "per_kernel", "persistent_mma", "step_tc"], default="auto",
                    help="form of the batch-1 draft layers (dspark_set_path): auto, one kernel per projection, "
                         "every layer in one warp-MMA launch, or the whole step in one tcgen05 launch")
    ap.add_argument("--tc-phase", choices=["ingest_L32768", "batched_out_proj"],
                    help="run only this tensor-core phase (for a profiler), print its line and exit")
    ap.add_argument("--no-tc-phases", action="store_true",
                    help="skip the tensor-core phases (32768-row ingest, batched out_proj GEMM) of the default run")
    ap.add_argument("--record-traffic", nargs=6,
                    metavar=("NCU_RAW_CSV", "CLASS", "WORKLOAD", "SOURCE", "LAUNCHES_PER_RANGE", "CAPTURE"),
                    help="write the profiles/traffic.json entry of a kernel class from an ncu raw-page CSV, then exit")
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

def class_work(cls: str, cfg, T: int, L_total: int, B: int):
    """Algorithmic bytes and flops of one timed range of a kernel class, and its bound.

    T: context rows in one ingest range; L_total: context rows summed over the
    B sequences of one draft; B: sequences per draft.  bf16 weights, features
    and caches (2 B), fp32 logits (4 B).  A projection over <= 16 activation
    rows streams its weights once (HBM-bound); more rows make it a dense
    contraction (tensor-bound)."""
    d, F, H, V, r, g, nL, mH = (cfg.d_draft, cfg.ff, cfg.hidden, cfg.vocab, cfg.markov_rank, cfg.gamma,
                                cfg.n_layers, cfg.feat_dim)
    dkv = cfg.d_kv  # K/V width (d without grouped-query attention)
    rows = B * g
    gemm_bound = "hbm" if rows <= 16 else "tensor"
    if cls == "ingest_proj":
        return dict(bytes=T * mH * 2 + d * mH * 2 + T * d * 4, flops=2 * T * mH * d,
                    bound="tensor" if T > 16 else "hbm")
    if cls == "ingest_kv":
        return dict(bytes=nL * (T * d * 2 + 2 * dkv * d * 2 + T * 2 * dkv * 2), flops=nL * 2 * T * d * 2 * dkv,
                    bound="tensor" if T > 16 else "hbm")
    if cls == "out_proj":
        return dict(bytes=V * d * 2 + rows * V * 4, flops=2 * rows * V * d, bound=gemm_bound)
    if cls == "attention":
        return dict(bytes=2 * (L_total + rows) * dkv * 2, flops=4 * g * (L_total + rows) * d, bound="hbm")
    if cls == "markov_argmax":
        return dict(bytes=V * r * 2 + rows * V * 4, flops=2 * rows * V * r, bound="hbm")
    if cls == "qkv_proj":
        return dict(bytes=(d + 2 * dkv) * d * 2, flops=2 * rows * (d + 2 * dkv) * d, bound=gemm_bound)
    if cls == "o_proj":
        return dict(bytes=d * d * 2, flops=2 * rows * d * d, bound=gemm_bound)
    if cls == "gate_up_proj":
        return dict(bytes=2 * F * d * 2, flops=2 * rows * 2 * F * d, bound=gemm_bound)
    if cls == "down_proj":
        return dict(bytes=F * d * 2, flops=2 * rows * F * d, bound=gemm_bound)
    if cls == "draft_layers":  # every layer of a batch-1 draft in one launch
        return dict(bytes=nL * ((2 * d * d + 2 * dkv * d + 3 * F * d) * 2 + 2 * (L_total + rows) * dkv * 2),
                    flops=nL * (2 * rows * (2 * d * d + 2 * dkv * d + 3 * F * d) + 4 * g * (L_total + rows) * d),
                    bound="hbm")
    if cls == "draft_step":  # block build, every layer, out_norm and out_proj of a batch-1 draft in one launch
        layers = class_work("draft_layers", cfg, T, L_total, B)
        return dict(bytes=layers["bytes"] + d * H * 2 + V * d * 2 + rows * V * 4,
                    flops=layers["flops"] + 2 * B * d * H + 2 * rows * V * d, bound="hbm")
    if cls == "block_build":
        return dict(bytes=d * H * 2, flops=2 * B * d * H, bound="hbm")
    # (qkv_proj_beside_ingest, layer 0's QKV on the side stream, is not modelled: its event range spans
    # the ingest it overlaps, so it never ranks as the dominant class)
    return dict(bytes=0, flops=0, bound="hbm")


def dominant_class(prof_all, cfg, L_total, B):
    """The kernel class with the most device time per step among those with a work model (a class
    without one, such as a launch overlapped with another stream, is taken only if none has one).
    prof_all: {class: (ms, ranges, launches, index)} from the profiled pass."""
    modelled = [k for k in prof_all
                if class_work(k, cfg, 1, L_total, B)["bytes"] or class_work(k, cfg, 1, L_total, B)["flops"]]
    return max(modelled or list(prof_all), key=lambda k: prof_all[k][0])


def draft_bytes_min(cfg, L_total, B=1):
    """Algorithmic bytes of one draft call: every weight once (w2 once), the
    caches of all layers for every sequence, the embedding rows."""
    d, F, H, V, r, nL = cfg.d_draft, cfg.ff, cfg.hidden, cfg.vocab, cfg.markov_rank, cfg.n_layers
    dkv = cfg.d_kv
    layers = nL * (2 * d * d + 2 * dkv * d + 3 * F * d) * 2
    return (layers + d * H * 2 + V * d * 2 + V * r * 2 + B * cfg.gamma * r * 2
            + nL * 2 * (L_total + B * cfg.gamma) * dkv * 2 + B * H * 2)


def ingest_flops(cfg, T):
    d, mH, nL = cfg.d_draft, cfg.feat_dim, cfg.n_layers
    return 2 * T * mH * d + nL * 2 * T * d * 2 * cfg.d_kv


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
    """DRAM bytes per range of a kernel class from the committed ncu table (profiles/traffic.json,
    written by `bench.py --record-traffic` from an ncu capture), if its entry still matches the hash
    of the kernel's source file; None otherwise."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    for e in table.get("entries", []):
        if e.get("workload") != workload or e.get("class") != kernel_class:
            continue
        try:
            digest = hashlib.sha256(open(os.path.join(ROOT, e["source"]), "rb").read()).hexdigest()[:16]
        except OSError:
            return None
        if digest != e.get("source_sha16"):
            return None
        return int(e["dram_bytes_per_launch"]) * int(e.get("launches_per_range", 1))
    return None


def record_traffic(csv_path, kernel_class, workload, source, launches_per_range, capture):
    """Write (or replace) the entry of (workload, kernel_class) in profiles/traffic.json from an ncu
    raw-page CSV (``ncu -i X.ncu-rep --page raw --csv``) of the kernel's captured launches: the
    mean of dram__bytes_read.sum + dram__bytes_write.sum over them, keyed to the source file's hash."""
    import csv
    import hashlib
    with open(csv_path, newline="") as f:
        rows = list(csv.reader(f))
    head = rows[0]
    ir, iw = head.index("dram__bytes_read.sum"), head.index("dram__bytes_write.sum")
    # the second row names the units ncu chose (byte, Kbyte, Mbyte, Gbyte; decimal prefixes)
    scale = {"byte": 1.0, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "": 1.0}
    ur = rows[1] if len(rows) > 1 else []
    sr = scale.get(ur[ir].strip().lower(), 1.0) if len(ur) > ir else 1.0
    sw = scale.get(ur[iw].strip().lower(), 1.0) if len(ur) > iw else 1.0
    vals = []
    for r in rows[1:]:
        try:
            vals.append(float(r[ir].replace(",", "")) * sr + float(r[iw].replace(",", "")) * sw)
        except (ValueError, IndexError):
            continue  # the units row
    if not vals:
        raise SystemExit(f"no DRAM byte counters in {csv_path}")
    digest = hashlib.sha256(open(os.path.join(ROOT, source), "rb").read()).hexdigest()[:16]
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            table = json.load(f)
    except (OSError, ValueError):
        table = {"about": "DRAM bytes (ncu dram__bytes_read.sum + dram__bytes_write.sum) per launch of a bench "
                          "kernel class, valid while the kernel source's SHA-256 prefix matches; written by "
                          "bench.py --record-traffic", "entries": []}
    table["entries"] = [e for e in table["entries"] if not (e["workload"] == workload and e["class"] == kernel_class)]
    table["entries"].append({"workload": workload, "class": kernel_class, "source": source, "source_sha16": digest,
                             "launches_per_range": int(launches_per_range),
                             "dram_bytes_per_launch": int(round(sum(vals) / len(vals))), "launches_captured": len(vals),
                             "capture": capture})
    with open(p, "w") as f:
        json.dump(table, f, indent=1)
        f.write("\n")


def cpu_model():
    """The host CPU's model name (lscpu / /proc/cpuinfo), for the CPU-baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() == "Model name":
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu model")):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def bf16_dev(a, dev):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)
    return t.view(torch.bfloat16)


# --------------------------------------------------------------------------- workloads

class Runner:
    """One workload: its step (one pass of the whole hot path), its units, and its oracle sample."""
    metric = ""
    unit = "blocks/s"
    blocks_per_step = 1

    def __init__(self, wl, dev, seed=0):
        self.wl, self.cfg, self.dev, self.seed = wl, wl.cfg, dev, seed

    # GPU side
    def make_drafter(self, W, max_ctx, max_seqs=1):
        import torch

        import block_draft_model_gb300 as bdm
        cfg = self.cfg
        self.Wd = {k: (bf16_dev(v, self.dev) if v.dtype == np.uint16 else torch.from_numpy(v).to(self.dev))
                   for k, v in W.items()}
        return bdm.Drafter(hidden=cfg.hidden, n_taps=cfg.n_taps, d_draft=cfg.d_draft, n_heads=cfg.n_heads,
                           n_layers=cfg.n_layers, ff_mult=cfg.ff_mult, gamma=cfg.gamma, vocab=cfg.vocab,
                           markov_rank=cfg.markov_rank, eps=cfg.eps, dtype=bdm.BF16, max_ctx=max_ctx,
                           max_seqs=max_seqs, weights=self.Wd, n_kv_heads=cfg.n_kv_heads, qk_norm=cfg.qk_norm,
                           rope_theta=cfg.rope_theta)


class FreshContextRunner(Runner):
    """Batch 1: every step ingests a fresh context of L rows, then drafts `drafts` blocks."""

    def __init__(self, wl, dev, drafts=1, pool=POOL, seed=0):
        super().__init__(wl, dev, seed)
        self.T, self.drafts, self.npool = wl.ctx_len, drafts, pool
        self.blocks_per_step = drafts
        self.metric = (f"draft blocks/s (batch 1, fresh context of {self.T} rows ingested per step, "
                       f"{drafts} block{'s' if drafts > 1 else ''} per step)")
        self.ctx_tokens_per_step = self.T
        self.L_total = self.T

    def setup(self):
        import torch
        cfg = self.cfg
        self.W = syn.make_weights(cfg, seed=self.seed)
        self.g = self.make_drafter(self.W, max_ctx=self.T)
        self.pool_np = [syn.make_feats(cfg, self.T, seed=self.seed, step=i) for i in range(self.npool)]
        self.pool = [bf16_dev(x, self.dev) for x in self.pool_np]
        self.anchors = syn.uniform_int(self.seed, syn.STREAM_ANCHORS, (max(self.npool, 16) * self.drafts,), 0,
                                       cfg.vocab - 1)
        self.tok = torch.empty(cfg.gamma, dtype=torch.int32, device=self.dev)
        self.conf = torch.empty(cfg.gamma, dtype=torch.float32, device=self.dev)
        self.host_pool = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in self.pool_np[:2]]
        self.tok_h = torch.empty(cfg.gamma, dtype=torch.int32).pin_memory()
        self.conf_h = torch.empty(cfg.gamma, dtype=torch.float32).pin_memory()
        self.h2d = self.T * cfg.feat_dim * 2
        self.d2h = self.drafts * cfg.gamma * 8

    def step(self, i):
        g = self.g
        g.reset(0)
        # the context ingest and the first draft in one call (the block rows are built beside the ingest)
        g.ingest_and_draft(self.pool[i % self.npool], int(self.anchors[(i * self.drafts) % len(self.anchors)]),
                           self.tok, self.conf)
        for j in range(1, self.drafts):
            g.draft(int(self.anchors[(i * self.drafts + j) % len(self.anchors)]), self.tok, self.conf)

    def host_step(self, i):
        g = self.g
        g.reset(0)
        g.ingest_context_host(self.host_pool[i % len(self.host_pool)])
        for j in range(self.drafts):
            g.draft_host(int(self.anchors[(i * self.drafts + j) % len(self.anchors)]), self.tok_h, self.conf_h)

    def phases(self, timed):
        g, T = self.g, self.T
        ms_ingest = timed(lambda i: (g.reset(0), g.ingest_context(self.pool[i % self.npool])))
        g.reset(0)
        g.ingest_context(self.pool[0])
        ms_draft = timed(lambda i: g.draft(int(self.anchors[i % len(self.anchors)]), self.tok, self.conf))
        bm = draft_bytes_min(self.cfg, T)
        return {"ingest_ms": ms_ingest, "ingest_ctx_tokens_per_s": T / (ms_ingest / 1e3),
                "ingest_tflops": ingest_flops(self.cfg, T) / (ms_ingest / 1e3) / 1e12,
                "draft_ms": ms_draft, "draft_blocks_per_s": 1e3 / ms_draft, "draft_bytes_min": bm,
                "draft_gbs_of_bytes_min": bm / (ms_draft / 1e3) / 1e9}

    def oracle_baseline(self, seconds, max_steps, rows=4096):
        """The CPU oracle on a bounded sample of this workload, scaled to blocks/s of the full step:
        ingest of up to `rows` rows and one draft are timed separately, the step time is
        T / rows * t_ingest + drafts * t_draft."""
        import oracle
        dr = oracle.Drafter(self.cfg, self.W)
        rows = min(self.T, rows)
        n, t_in, t_dr, t0 = 0, 0.0, 0.0, time.perf_counter()
        while n < max_steps:
            dr.reset(0)
            a = time.perf_counter()
            dr.ingest(self.pool_np[n % self.npool][:rows])
            b = time.perf_counter()
            dr.draft(int(self.anchors[n % len(self.anchors)]))
            c = time.perf_counter()
            t_in += b - a
            t_dr += c - b
            n += 1
            if c - t0 >= seconds:
                break
        step_s = (t_in / n) * self.T / rows + (t_dr / n) * self.drafts
        sample = (f"{n} x (ingest {rows} rows + 1 block) of the same drafter, fp64"
                  + ("" if rows == self.T and self.drafts == 1 else
                     f"; scaled to a step of {self.T} rows + {self.drafts} blocks"))
        return self.drafts / step_s, sample


class StreamRunner(Runner):
    """Batch 1: a context of L rows is ingested once; every step ingests 1-6 new rows and drafts one block."""

    def __init__(self, wl, dev, seed=0):
        super().__init__(wl, dev, seed)
        self.metric = f"draft blocks/s (batch 1, context {wl.ctx_len} rows growing by 1-6 rows per step)"

    def setup(self):
        import torch
        cfg, wl = self.cfg, self.wl
        self.W = syn.make_weights(cfg, seed=self.seed)
        self.max_ctx = wl.ctx_len + 6 * 4096
        self.g = self.make_drafter(self.W, max_ctx=self.max_ctx)
        self.g.ingest_context(bf16_dev(syn.make_feats(cfg, wl.ctx_len, seed=self.seed), self.dev))
        counts = syn.uniform_int(self.seed, syn.STREAM_COUNTS, (256,), 1, 6)
        new_np = [syn.make_feats(cfg, int(c), seed=self.seed, step=i) for i, c in enumerate(counts)]
        self.new = [bf16_dev(x, self.dev) for x in new_np]
        self.new_h = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in new_np[:32]]
        self.length = wl.ctx_len
        self.tok_h = torch.empty(cfg.gamma, dtype=torch.int32).pin_memory()
        self.conf_h = torch.empty(cfg.gamma, dtype=torch.float32).pin_memory()
        self.anchors = syn.uniform_int(self.seed, syn.STREAM_ANCHORS, (256,), 0, cfg.vocab - 1)
        self.tok = torch.empty(cfg.gamma, dtype=torch.int32, device=self.dev)
        self.conf = torch.empty(cfg.gamma, dtype=torch.float32, device=self.dev)
        self.ctx_tokens_per_step = float(counts.mean())
        self.L_total = wl.ctx_len
        self.h2d = int(self.ctx_tokens_per_step * cfg.feat_dim * 2)
        self.d2h = cfg.gamma * 8

    def step(self, i):
        x = self.new[i % len(self.new)]
        self.length += x.shape[0]
        if self.length > self.max_ctx:
            raise RuntimeError("context capacity exhausted; lower --steps")
        self.g.ingest_and_draft(x, int(self.anchors[i % len(self.anchors)]), self.tok, self.conf)

    def host_step(self, i):
        x = self.new_h[i % len(self.new_h)]
        self.length += x.shape[0]
        if self.length > self.max_ctx:
            raise RuntimeError("context capacity exhausted; lower --steps")
        self.g.ingest_context_host(x)
        self.g.draft_host(int(self.anchors[i % len(self.anchors)]), self.tok_h, self.conf_h)

    def phases(self, timed):
        return {}


class BatchedRunner(Runner):
    """64 sequences with ragged contexts; every step ingests 1-6 rows per sequence and drafts one block each."""

    def __init__(self, wl, dev, seed=0):
        super().__init__(wl, dev, seed)
        self.blocks_per_step = wl.n_seqs
        self.metric = (f"draft blocks/s ({wl.n_seqs} sequences per step, ragged contexts "
                       f"{wl.ctx_len_range[0]}-{wl.ctx_len_range[1]} rows, 1-6 new rows per sequence per step)")

    def setup(self):
        import torch
        cfg, wl = self.cfg, self.wl
        n = wl.n_seqs
        self.W = syn.make_weights(cfg, seed=self.seed)
        lens = syn.ctx_lengths(wl, seed=self.seed)
        self.max_ctx = int(lens.max()) + 6 * 2048
        self.g = self.make_drafter(self.W, max_ctx=self.max_ctx, max_seqs=n)
        self.ids = torch.arange(n, dtype=torch.int32, device=self.dev)
        for i in range(n):  # one-shot contexts, one sequence at a time to bound host memory
            feats = bf16_dev(syn.make_feats(cfg, int(lens[i]), seed=self.seed, seq=i), self.dev)
            cu = torch.tensor([0, int(lens[i])], dtype=torch.int32, device=self.dev)
            self.g.ingest_context_batched(self.ids[i:i + 1], cu, feats)
        self.L_total = int(lens.sum())
        counts = syn.uniform_int(self.seed, syn.STREAM_COUNTS, (64, n), 1, 6)
        self.steps_in = []
        for s in range(counts.shape[0]):
            feats = np.concatenate([syn.make_feats(cfg, int(c), seed=self.seed, step=s, seq=i)
                                    for i, c in enumerate(counts[s])])
            cu = np.concatenate([[0], np.cumsum(counts[s])]).astype(np.int32)
            self.steps_in.append((bf16_dev(feats, self.dev), torch.from_numpy(cu).to(self.dev),
                                  torch.from_numpy(feats.view(np.int16)).pin_memory(), torch.from_numpy(cu).pin_memory()))
        anchors = syn.uniform_int(self.seed, syn.STREAM_ANCHORS, (64, n), 0, cfg.vocab - 1)
        self.anchors = [torch.from_numpy(a.copy()).to(self.dev) for a in anchors]
        self.anchors_h = [torch.from_numpy(a.copy()).pin_memory() for a in anchors]
        self.tok = torch.empty(n, cfg.gamma, dtype=torch.int32, device=self.dev)
        self.conf = torch.empty(n, cfg.gamma, dtype=torch.float32, device=self.dev)
        self.tok_h = torch.empty(n, cfg.gamma, dtype=torch.int32).pin_memory()
        self.conf_h = torch.empty(n, cfg.gamma, dtype=torch.float32).pin_memory()
        self.ctx_tokens_per_step = float(counts.sum(axis=1).mean())
        self.h2d = int(self.ctx_tokens_per_step * cfg.feat_dim * 2 + (n + 1) * 4 + n * 4)
        self.d2h = n * cfg.gamma * 8

    def step(self, i):
        feats, cu, _, _ = self.steps_in[i % len(self.steps_in)]
        self.g.ingest_context_batched(self.ids, cu, feats)
        self.g.draft_batched(self.ids, self.anchors[i % len(self.anchors)], self.tok, self.conf)

    def host_step(self, i):
        _, _, feats_h, cu_h = self.steps_in[i % len(self.steps_in)]
        feats = feats_h.to(self.dev, non_blocking=True).view(__import__("torch").bfloat16)
        cu = cu_h.to(self.dev, non_blocking=True)
        anchors = self.anchors_h[i % len(self.anchors_h)].to(self.dev, non_blocking=True)
        self.g.ingest_context_batched(self.ids, cu, feats)
        self.g.draft_batched(self.ids, anchors, self.tok, self.conf)
        self.tok_h.copy_(self.tok)
        self.conf_h.copy_(self.conf)

    def phases(self, timed):
        return {}


def make_runner(name, dev, variant=None):
    wl = syn.WORKLOADS[name]
    if variant:  # the same workload on the grouped-query / QK-norm / rotary drafter
        wl = dataclasses.replace(wl, cfg=dataclasses.replace(wl.cfg, **variant))
    if name == "minicpm_L1024":
        return FreshContextRunner(wl, dev)
    if name == "gemma_L32768_ingest":
        return FreshContextRunner(wl, dev, drafts=wl.steps, pool=2)
    if name == "gemma_L4096_stream":
        return StreamRunner(wl, dev)
    if name == "gemma_batched64":
        return BatchedRunner(wl, dev)
    raise SystemExit(f"unknown workload {name}")


def oracle_single_thread(args):
    """The same oracle on one host thread: a child process with the BLAS / OpenMP pools at one thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-single-thread", "--workload", args.workload,
           "--cpu-seconds", str(args.cpu_seconds)]
    try:
        out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600).stdout
        j = json.loads(out.strip().splitlines()[-1])
        return {"value": j["value"], "unit": "blocks/s", "cores": 1, "sample": j["sample"]}
    except (subprocess.SubprocessError, ValueError, IndexError, KeyError, OSError) as e:
        return {"value": None, "unit": "blocks/s", "cores": 1, "error": str(e)[:200]}


# --------------------------------------------------------------------------- tensor-core phases

def tc_phases(dev, peaks, reps=5, only=None):
    """The two contractions the drafter runs on the tensor cores at scale, on the Gemma-shaped
    drafter (H 2560, m 4, d 1024, 5 layers, V 262144): a fresh 32768-row context ingested in one call
    (Eq 2 projection + Eq 3 K/V of every layer, 1.374 TFLOP) and the batched out_proj product of 64
    sequences x 5 block rows (320 x 1024 x 262144, 171.8 GFLOP).  Each is timed with CUDA events over
    `reps` calls after one warm-up call and reported against the measured dense bf16 peak."""
    import torch

    import block_draft_model_gb300 as bdm
    wl = syn.WORKLOADS["gemma_L32768_ingest"]
    cfg, T = wl.cfg, wl.ctx_len
    W = syn.make_weights(cfg, seed=0)
    run = Runner(wl, dev)
    g = run.make_drafter(W, max_ctx=T)
    X = bf16_dev(syn.make_feats(cfg, T, seed=0), dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    ms_in = timed(lambda: (g.reset(0), g.ingest_context(X))) if only in (None, "ingest_L32768") else float("nan")
    fl_in = ingest_flops(cfg, T)
    rows = 64 * cfg.gamma
    A = bf16_dev(syn.normal_bf16(5, 7, (rows, cfg.d_draft)), dev)
    out = torch.empty(rows, cfg.vocab, dtype=torch.float32, device=dev)
    Wo = run.Wd["out_proj"]
    ms_op = (timed(lambda: bdm.linear(A, Wo, out, kernel=bdm.KERNEL_AUTO)) if only in (None, "batched_out_proj")
             else float("nan"))
    fl_op = 2.0 * rows * cfg.d_draft * cfg.vocab
    g.close()
    del g, X, A, out, run
    torch.cuda.empty_cache()
    peak = peaks["bf16_tflops"]
    res = {}
    for name, ms, fl, note in (
            ("ingest_L32768", ms_in, fl_in, "Gemma-shaped: fresh 32768-row context, Eq 2 + Eq 3 of 5 layers"),
            ("batched_out_proj_320x1024x262144", ms_op, fl_op, "64 sequences x 5 rows against the 262144-row out_proj")):
        tf = fl / (ms / 1e3) / 1e12
        res[name] = {"ms": ms, "tflops": tf, "frac_of_bf16_peak": tf / peak, "flops": fl, "note": note}
    res["peak_tflops"] = peak
    res["peak_src"] = peaks["src"] + " (burst)"
    return res


# --------------------------------------------------------------------------- main

def variant_of(args):
    """The grouped-query / QK-norm / rotary options given on the command line."""
    return {k: v for k, v in (("n_kv_heads", args.n_kv_heads), ("qk_norm", args.qk_norm),
                              ("rope_theta", args.rope_theta)) if v}


def arm_config(wl, world, args, variant=None):
    """The `config` object both arms print for a workload."""
    cfg = wl.cfg
    return {"workload": wl.name, "ctx_len": wl.ctx_len, "sequences": wl.n_seqs, "gamma": cfg.gamma,
            "d_draft": cfg.d_draft, "vocab": cfg.vocab,
            "parallelism": f"replicas{world}" if world > 1 else "single",
            **({"layers": args.layers} if getattr(args, "layers", "auto") != "auto" else {}),
            "token_choice": (f"sampled (temperature {args.temperature}, top-k {args.top_k})"
                             if args.temperature > 0 else "argmax"),
            **({"variant": variant} if variant else {}),
            "l2": "inputs larger than L2 (weights, caches and features stream > 1 GB per step)"}


def reference_arm(args):
    """The CPU oracle on the default workload, timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    variant = variant_of(args)
    wl = syn.WORKLOADS[args.workload]
    if variant:
        wl = dataclasses.replace(wl, cfg=dataclasses.replace(wl.cfg, **variant))
    cfg = wl.cfg
    T = wl.ctx_len or 1024
    W = syn.make_weights(cfg, seed=0)
    pool = [syn.make_feats(cfg, min(T, 4096), seed=0, step=i) for i in range(2)]
    anchors = syn.uniform_int(0, syn.STREAM_ANCHORS, (64,), 0, cfg.vocab - 1)
    import oracle
    dr = oracle.Drafter(cfg, W)

    sample = (args.temperature, args.top_k, 2024, 0) if args.temperature > 0 else None

    def one(i):
        dr.reset(0)
        dr.ingest(pool[i % 2])
        dr.draft(int(anchors[i % 64]), sample=sample)

    n_w = max(1, args.warmup)
    for i in range(n_w):
        one(i)
    t0 = time.perf_counter()
    n = 0
    while n < args.steps:
        one(n)
        n += 1
        if time.perf_counter() - t0 > 240:
            break
    dt = time.perf_counter() - t0
    v = n / dt
    sample = f"{n} steps of ingest {min(T, 4096)} rows + 1 block (fp64 numpy, {cpu_cores()} threads)"
    # the same metric, unit, direction and config as this workload's GPU line
    line = {"impl": "reference", "metric": make_runner(args.workload, None, variant).metric, "value": v,
            "unit": "blocks/s", "n_gpus": args.gpus, "steps": n, "warmup": n_w, "ms_per_step": 1e3 * dt / n,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": arm_config(wl, 1, args, variant),
            "cpu_baseline": {"value": v, "unit": "blocks/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": v, "unit": "blocks/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.record_traffic:
        record_traffic(*args.record_traffic)
        return
    if args.oracle_single_thread:
        # run with the BLAS and OpenMP pools at one thread (set by the parent before numpy loads)
        wl = syn.WORKLOADS[args.workload]
        run = FreshContextRunner(wl, None)
        run.W = syn.make_weights(wl.cfg, seed=0)
        run.pool_np = [syn.make_feats(wl.cfg, min(run.T, 128), seed=0, step=i) for i in range(2)]
        run.npool = 2
        run.anchors = syn.uniform_int(0, syn.STREAM_ANCHORS, (16,), 0, wl.cfg.vocab - 1)
        v, sample = run.oracle_baseline(args.cpu_seconds, 20, rows=128)
        print(json.dumps({"value": v, "sample": sample}), flush=True)
        return
    if args.impl == "reference":
        reference_arm(args)
        return
    rank, world, local = dist_setup(args.gpus)
    import torch

    import block_draft_model_gb300 as bdm
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    bdm.build()
    bdm.load()
    if args.tc_phase:
        print(json.dumps({"tc_phase": args.tc_phase, **tc_phases(dev, load_peaks(), reps=2, only=args.tc_phase)}),
              flush=True)
        return
    variant = variant_of(args)
    run = make_runner(args.workload, dev, variant)
    run.setup()
    layers = {"auto": bdm.LAYERS_AUTO, "per_kernel": bdm.LAYERS_PER_KERNEL,
              "persistent_mma": bdm.LAYERS_PERSISTENT_MMA, "step_tc": bdm.LAYERS_STEP_TC}[args.layers]
    if layers != bdm.LAYERS_AUTO:
        run.g.set_path(bdm.PATH_LAYERS, layers)
    if args.temperature > 0:
        run.g.set_sampling(args.temperature, args.top_k, 2024)
    cfg, g = run.cfg, run.g
    stream = torch.cuda.current_stream(dev)
    B = run.wl.n_seqs

    # warm-up, with a profile of every kernel class to find the dominant one
    nw = max(3, args.warmup)
    for i in range(nw):
        run.step(i)
    torch.cuda.synchronize()
    g.profile(-1)
    nprof = 2
    for i in range(nprof):
        run.step(nw + i)
    torch.cuda.synchronize()
    prof_all = g.profile_read()
    g.profile(0)
    dominant = dominant_class(prof_all, cfg, run.L_total, B)

    # timed region: K steps, no profiling (event pairs inside the draft graph would break the launch overlap)
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    l0 = g.launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    base = nw + nprof
    ev0.record(stream)
    for i in range(args.steps):
        run.step(base + i)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = g.launch_count() - l0
    ms = ev0.elapsed_time(ev1)
    # the dominant kernel class over a second run of the same K steps, with event pairs around its launches
    g.profile(1 << prof_all[dominant][3])
    for i in range(args.steps):
        run.step(base + args.steps + i)
    torch.cuda.synchronize()
    prof = g.profile_read()
    g.profile(0)
    ms_max = reduce_max(ms, world, dev)
    clk = clocks.stop() if rank == 0 else None

    # the dominant kernel class, timed live (event pairs on the launching stream inside the timed region)
    dms, dranges, dlaunch, _ = prof[dominant]
    peaks = load_peaks()
    T_range = getattr(run, "T", int(round(run.ctx_tokens_per_step)))
    work = class_work(dominant, cfg, T_range, run.L_total, B)
    per_range_s = dms / 1e3 / max(dranges, 1)
    if work["bound"] == "tensor":
        ach = work["flops"] / per_range_s / 1e12
        peak, unit = peaks["bf16_tflops"], "TFLOP/s"
    else:
        ach = work["bytes"] / per_range_s / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
    roofline = {"kernel": dominant, "bound": work["bound"], "achieved": ach, "peak": peak, "unit": unit,
                "frac": ach / peak, "peak_src": peaks["src"], "traffic": load_traffic(dominant, run.wl.name),
                "algorithmic_per_launch": work["bytes"] if work["bound"] == "hbm" else work["flops"],
                "avg_range_us": per_range_s * 1e6, "launches_per_range": dlaunch / max(dranges, 1),
                "share_of_step": prof_all[dominant][0] / sum(v[0] for v in prof_all.values())}

    def timed(fn, n=max(10, min(args.steps, 50))):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(n):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    phases = run.phases(timed) if hasattr(run, "phases") else {}
    if not args.no_tc_phases and world == 1 and args.workload == "minicpm_L1024":
        phases["tensor_core"] = tc_phases(dev, load_peaks())
    phases["per_class_ms_per_step"] = {k: round(v[0] / nprof, 4) for k, v in prof_all.items() if v[1]}
    phases["note"] = ("per-class times come from a separate profiled pass whose event pairs break the "
                      "launch overlap; they rank the kernels, the step time is the timed region's")

    # end to end through the public API with host buffers (pinned): copies inside the timed region
    e2e = None
    if getattr(run, "host_step", None):
        ne = max(5, min(args.steps, 30))
        for i in range(2):
            run.host_step(i)
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        for i in range(ne):
            run.host_step(i)
        torch.cuda.synchronize()
        e2e_s = reduce_max(time.perf_counter() - t0, world, dev)
        e2e = {"value": world * ne * run.blocks_per_step / e2e_s, "unit": "blocks/s",
               "h2d_bytes_per_step": int(run.h2d), "d2h_bytes_per_step": int(run.d2h)}
    assert g.check() == 0

    value = world * args.steps * run.blocks_per_step / (ms_max / 1e3)
    line = {"metric": run.metric, "value": value, "unit": "blocks/s", "n_gpus": world, "steps": args.steps,
            "warmup": nw, "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": arm_config(run.wl, world, args, variant),
            "ctx_tokens_per_s": world * args.steps * run.ctx_tokens_per_step / (ms_max / 1e3),
            "phases": phases, "roofline": roofline, "clocks": clk, "gpu_launches": launches, "e2e": e2e}
    if rank == 0 and world == 1 and not args.no_cpu_baseline and isinstance(run, FreshContextRunner):
        v, sample = run.oracle_baseline(args.cpu_seconds, 50)
        line["cpu_baseline"] = {"value": v, "unit": "blocks/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": sample, "cpu_model": cpu_model(),
                                "single_thread": oracle_single_thread(args)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    g.close()


if __name__ == "__main__":
    main()
