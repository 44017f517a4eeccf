"""The C-ABI library builds, loads without a GPU and exports every function
that include/dspark.h declares.  No compute call is made here."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import block_draft_model_gb300 as bdm
    bdm.build()
    return bdm.load()


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for must in ("dspark_create", "dspark_destroy", "dspark_ingest_context", "dspark_draft",
                 "dspark_ingest_context_batched", "dspark_draft_batched", "dspark_reset",
                 "dspark_context_length", "dspark_last_error"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    import block_draft_model_gb300 as bdm
    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(bdm.EXPORTED) == names
    out = subprocess.run(["nm", "-D", "--defined-only", bdm.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (dspark_[a-z_]+)\b", out))
    assert set(names) <= exported


def test_library_needs_no_libcuda_at_load():
    import block_draft_model_gb300 as bdm
    out = subprocess.run(["readelf", "-d", bdm.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out


def test_host_side_errors_without_gpu(lib):
    """Calls that fail argument checks return a status before touching the GPU."""
    import block_draft_model_gb300 as bdm
    assert lib.dspark_version().decode().startswith("dspark")
    h = ctypes.c_void_p(0)
    cfg = bdm.Config(256, 3, 128, 3, 2, 2, 4, 1024, 32, 1e-6, 1, 0, 64, 1)   # 128 % 3 != 0
    st = lib.dspark_create(ctypes.byref(cfg), None, None, ctypes.byref(h))
    assert st == bdm.ERR_INVALID_ARG and not h.value
    assert b"not divisible" in lib.dspark_last_error(None)
    cfg = bdm.Config(256, 3, 128, 4, 2, 2, 4, 1024, 32, 1e-6, 1, 0, 64, 1)
    assert lib.dspark_create(ctypes.byref(cfg), None, None, ctypes.byref(h)) == bdm.ERR_INVALID_ARG
    assert b"NULL" in lib.dspark_last_error(None)
    cfg = bdm.Config(256, 3, 128, 4, 2, 2, 17, 1024, 32, 1e-6, 1, 0, 64, 1)    # gamma > 16
    assert lib.dspark_create(ctypes.byref(cfg), None, None, ctypes.byref(h)) == bdm.ERR_UNSUPPORTED
    assert lib.dspark_ingest_context(None, None, 4, None) == bdm.ERR_INVALID_ARG
    assert lib.dspark_draft(None, 0, None, None, None, None) == bdm.ERR_INVALID_ARG
    lib.dspark_destroy(None)


def test_variant_and_sampling_arguments_without_gpu(lib):
    """The grouped-query / QK-norm / rotary config fields, the sampler and the wait
    self-test reject bad arguments before any device work."""
    import block_draft_model_gb300 as bdm
    h = ctypes.c_void_p(0)

    def create(**kw):
        cfg = bdm.Config(256, 3, 128, 4, 2, 2, 4, 1024, 32, 1e-6, 0, 0, 64, 1)
        for k, v in kw.items():
            setattr(cfg, k, v)
        return lib.dspark_create(ctypes.byref(cfg), None, None, ctypes.byref(h))

    assert create(n_kv_heads=3) == bdm.ERR_INVALID_ARG
    assert b"multiple of n_kv_heads" in lib.dspark_last_error(None)
    assert create(n_kv_heads=-1) == bdm.ERR_INVALID_ARG
    assert create(qk_norm=2) == bdm.ERR_INVALID_ARG
    assert create(rope_theta=-1.0) == bdm.ERR_INVALID_ARG
    assert create(rope_theta=float("inf")) == bdm.ERR_INVALID_ARG
    # a valid variant config gets past the config check to the weight check
    assert create(n_kv_heads=2, qk_norm=1, rope_theta=10000.0) == bdm.ERR_INVALID_ARG
    assert b"weights are NULL" in lib.dspark_last_error(None)
    assert not h.value
    assert lib.dspark_set_sampling(None, ctypes.c_float(1.0), 0, 0, None) == bdm.ERR_INVALID_ARG
    for which in (-1, 6, 100):
        assert lib.dspark_selftest_wait(which, None) == bdm.ERR_INVALID_ARG


def test_set_path_rejects_bad_choices_without_gpu(lib):
    """dspark_set_path checks the handle before anything else."""
    import block_draft_model_gb300 as bdm
    assert lib.dspark_set_path(None, bdm.PATH_LAYERS, 0) == bdm.ERR_INVALID_ARG
    assert b"NULL" in lib.dspark_last_error(None)
