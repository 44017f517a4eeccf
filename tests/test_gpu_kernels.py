"""Kernel-level parity of the contraction behind every projection
(dspark_linear: out = A W^T) for each GEMM implementation, against the
oracle's float64 definition, on shapes that span several tiles and ragged
tails.  bf16 inputs, fp32 accumulation: max|d| <= 1e-4 * max|ref|."""
import numpy as np
import pytest

import oracle
import synthetic as syn
from helpers import to_torch

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_draft_model_gb300 as bdm
    bdm.build()
    bdm.load()


SHAPES = [(1, 64, 64), (5, 1000, 1024), (8, 4096, 2048), (16, 3072, 1024), (17, 300, 136), (3, 73448, 2048),
          (8, 2048, 10240), (2, 130, 200),
          (128, 256, 64), (129, 257, 192), (320, 1000, 1024), (1024, 1024, 10240), (777, 2048, 1024)]


@pytest.mark.parametrize("kernel", [1, 2, 3, 4])
@pytest.mark.parametrize("shape", SHAPES)
def test_linear_kernels(kernel, shape):
    import block_draft_model_gb300 as bdm
    M, N, K = shape
    if kernel in (2, 4) and M > 16:
        pytest.skip("weight streaming takes M <= 16")
    if kernel in (3, 4) and K < 64:
        pytest.skip("tensor-core path takes K >= 64")
    A = syn.normal_bf16(7, 1, (M, K))
    W = syn.normal_bf16(7, 2, (N, K), 0.05)
    ref = oracle.linear(A, W)
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    bdm.linear(to_torch(A), to_torch(W), out, kernel=kernel)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.max(np.abs(got - ref))
    assert err <= 1e-4 * np.max(np.abs(ref)), (kernel, shape, err)


# The wide form (kernel 5): one row group (M <= 160) and two (161..320, 112-row groups at M = 208),
# ragged M, N and K tails, fewer tiles than SMs and more; and kernel 0, which picks the wide form
# where N has at least one 128-row tile per SM (and M is not in 161..256), the tiles elsewhere.
WIDE_SHAPES = [(1, 4099, 136), (17, 1000, 1024), (160, 2176, 520), (161, 4099, 1024), (200, 19457, 264),
               (208, 4099, 1024), (320, 73448, 1024), (320, 1000, 2048)]


@pytest.mark.parametrize("kernel", [5, 0])
@pytest.mark.parametrize("shape", WIDE_SHAPES)
def test_linear_wide(kernel, shape):
    import block_draft_model_gb300 as bdm
    M, N, K = shape
    A = syn.normal_bf16(9, 1, (M, K))
    W = syn.normal_bf16(9, 2, (N, K), 0.05)
    ref = oracle.linear(A, W)
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    bdm.linear(to_torch(A), to_torch(W), out, kernel=kernel)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.max(np.abs(got - ref))
    assert err <= 1e-4 * np.max(np.abs(ref)), (kernel, shape, err)


def test_linear_wide_batched_out_proj_sampled():
    """The batched vocabulary projection at full size (320 x 1024 against 262144 rows), through
    kernel 0 (which takes the wide form there): 2048 sampled vocabulary rows against the oracle,
    every entry finite; and 321 rows, one past the wide form's limit, refused by kernel 5."""
    import block_draft_model_gb300 as bdm
    M, N, K = 320, 262144, 1024
    A = syn.normal_bf16(10, 1, (M, K))
    W = syn.normal_bf16(10, 2, (N, K), 0.02)
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    bdm.linear(to_torch(A), to_torch(W), out, kernel=bdm.KERNEL_AUTO)
    torch.cuda.synchronize()
    cols = np.sort(np.random.default_rng(0).choice(N, 2048, replace=False))
    cols[-1] = N - 1
    ref = oracle.linear(A, W[cols])
    got = out[:, torch.as_tensor(cols, device="cuda")].double().cpu().numpy()
    assert np.max(np.abs(got - ref)) <= 1e-4 * np.max(np.abs(ref))
    assert bool(torch.isfinite(out).all())
    A2 = torch.zeros((321, K), dtype=torch.bfloat16, device="cuda")
    out2 = torch.empty((321, 4096), dtype=torch.float32, device="cuda")
    with pytest.raises(bdm.DsparkError):
        bdm.linear(A2, to_torch(W[:4096]), out2, kernel=bdm.KERNEL_TC_WIDE)


def test_linear_fp32_simt_and_streaming():
    import block_draft_model_gb300 as bdm
    for kernel, (M, N, K) in ((1, (70, 130, 200)), (2, (4, 1024, 256))):
        A = syn.normal_f32(8, 1, (M, K))
        W = syn.normal_f32(8, 2, (N, K), 0.05)
        out = torch.empty((M, N), dtype=torch.float32, device="cuda")
        bdm.linear(to_torch(A), to_torch(W), out, kernel=kernel)
        torch.cuda.synchronize()
        ref = oracle.linear(A, W)
        assert np.max(np.abs(out.double().cpu().numpy() - ref)) <= 1e-5 * np.max(np.abs(ref))
