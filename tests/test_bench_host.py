"""Host logic of the benchmark (no GPU): the algorithmic work model behind the
roofline fields and the lookup of ncu DRAM traffic, which must refuse a row
whose kernel source changed since the capture."""
import dataclasses
import hashlib
import importlib.util
import os
import sys

import pytest

import synthetic as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def test_draft_bytes_of_the_minicpm_shape(bench):
    """Every weight once (w2 once) plus the caches of a 1024-row context: the
    layers 419.4 MB, tok_proj 8.4, out_proj 300.8, w2 37.6, caches 41.9 MB."""
    cfg = syn.MINICPM
    d, F, nL = cfg.d_draft, cfg.ff, cfg.n_layers
    layers = nL * (4 * d * d + 3 * F * d) * 2
    assert abs(layers / 1e6 - 419.4) < 0.1
    caches = nL * 2 * (1024 + cfg.gamma) * d * 2
    assert abs(caches / 1e6 - 42.3) < 0.1
    assert abs(bench.draft_bytes_min(cfg, 1024) / 1e6 - 808.5) < 0.1


def test_class_work_counts_kv_width(bench):
    mha = syn.MINICPM
    gqa = dataclasses.replace(mha, n_kv_heads=4)
    d, dkv = mha.d_draft, gqa.d_kv
    assert dkv == d // 4
    assert bench.class_work("qkv_proj", mha, 1, 1024, 1)["bytes"] == 3 * d * d * 2
    assert bench.class_work("qkv_proj", gqa, 1, 1024, 1)["bytes"] == (d + 2 * dkv) * d * 2
    a_mha = bench.class_work("attention", mha, 1, 1024, 1)["bytes"]
    a_gqa = bench.class_work("attention", gqa, 1, 1024, 1)["bytes"]
    assert a_mha == 4 * a_gqa
    # batch-1 projections stream their weights; many rows make them contractions
    assert bench.class_work("gate_up_proj", mha, 1, 1024, 1)["bound"] == "hbm"
    assert bench.class_work("gate_up_proj", mha, 1, 1024, 8)["bound"] == "tensor"
    assert bench.draft_bytes_min(gqa, 1024) < bench.draft_bytes_min(mha, 1024)


def test_dominant_class_skips_unmodelled_overlap(bench):
    """Layer 0's QKV projection beside the ingest has no work model (its event range spans the
    ingest it overlaps): it is never the roofline's class, even with the longest range."""
    cfg = syn.MINICPM
    assert bench.class_work("qkv_proj_beside_ingest", cfg, 1, 1024, 1)["bytes"] == 0
    prof = {"ingest_kv": (0.074, 2, 2, 2), "gate_up_proj": (0.073, 5, 5, 8),
            "qkv_proj_beside_ingest": (0.2, 1, 1, 14)}
    assert bench.dominant_class(prof, cfg, 1024, 1) == "ingest_kv"
    assert bench.dominant_class({"qkv_proj_beside_ingest": (0.2, 1, 1, 14)}, cfg, 1024, 1) == \
        "qkv_proj_beside_ingest"


def test_traffic_rows_follow_the_kernel_source(bench, tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k() {}\n")
    (tmp_path / "profiles").mkdir()
    # an ncu raw-page CSV of two captured launches of the kernel: the table keeps their mean
    csv = tmp_path / "raw.csv"
    csv.write_text('"ID","Kernel Name","dram__bytes_read.sum","dram__bytes_write.sum"\n'
                   '"","","byte","byte"\n'
                   '"0","k","900","100"\n'
                   '"1","k","1100","100"\n')
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    bench.record_traffic(str(csv), "c", "w", "k.cu", 3, "x.md")
    assert bench.load_traffic("c", "w") == 3 * 1100
    # counters exported in scaled units
    csv.write_text('"ID","Kernel Name","dram__bytes_read.sum","dram__bytes_write.sum"\n'
                   '"","","Mbyte","Kbyte"\n'
                   '"0","k","33.5","1.5"\n')
    bench.record_traffic(str(csv), "c", "w", "k.cu", 1, "x.md")
    assert bench.load_traffic("c", "w") == 33501500
    assert bench.load_traffic("c", "other") is None
    src.write_text("__global__ void k() { /* changed */ }\n")
    assert bench.load_traffic("c", "w") is None
