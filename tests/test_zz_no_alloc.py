"""The weight-streaming linear call that allocates no device memory.

Callers that cannot call cudaMalloc (code running inside another runtime's
memory pool, allocator-free serving loops) use dspark_linear_stream_noalloc,
whose split-K scratch is a static device array of the library.  Its output
must match the allocating entry point (dspark_linear, kernel 4) within the
kernel tests' tolerance, on two calls in a row (the second call reuses the
array the first one left behind).  This file is collected last on purpose.
"""
import numpy as np
import pytest

import oracle
import synthetic as syn

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _bf16(a):
    return torch.from_numpy(a.view(np.int16).copy()).cuda().view(torch.bfloat16)


# (8, 1024, 320) and (4, 2000, 384): K split five and six ways, splits that a thread-block
# cluster cannot reduce, so the partial sums go through the static scratch array and the
# tile tickets (the other shapes reduce inside clusters or do not split K).
@pytest.mark.parametrize("shape", [(8, 2048, 2048), (5, 1000, 1024), (16, 6144, 2048), (1, 73448, 256),
                                   (8, 1024, 320), (4, 2000, 384)])
def test_noalloc_matches_allocating_entry_point_twice(shape):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_draft_model_gb300 as bdm
    bdm.build()
    bdm.load()
    M, N, K = shape
    A = syn.normal_bf16(31, 1, (M, K))
    W = syn.normal_bf16(31, 2, (N, K), 0.05)
    Ad, Wd = _bf16(A), _bf16(W)
    ref = torch.empty(M, N, dtype=torch.float32, device="cuda")
    bdm.linear(Ad, Wd, ref, kernel=bdm.KERNEL_TC_STREAM)
    torch.cuda.synchronize()
    want = oracle.linear(A, W)
    scale = np.max(np.abs(want))
    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        bdm.linear_stream_noalloc(Ad, Wd, out)
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        assert np.isfinite(got).all(), call
        assert np.max(np.abs(got - ref.double().cpu().numpy())) <= 1e-4 * scale, call
        assert np.max(np.abs(got - want)) <= 1e-4 * scale, call
        assert bdm.noalloc_check() == 0, call   # no bounded wait gave up


def test_noalloc_rejects_oversize_shapes():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_draft_model_gb300 as bdm
    bdm.load()
    A = torch.zeros(17, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(17, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(bdm.DsparkError) as e:
        bdm.linear_stream_noalloc(A, W, out)
    assert e.value.status == bdm.ERR_INVALID_ARG


def test_noalloc_rejects_n_beyond_the_static_tickets():
    """N > 128 * DSPARK_NOALLOC_MAX_TILES rows needs more tile tickets than the static array
    holds: DSPARK_ERR_CAPACITY before anything is launched."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_draft_model_gb300 as bdm
    bdm.load()
    N = 128 * 4096 + 1
    A = torch.zeros(1, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(N, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, N, dtype=torch.float32, device="cuda")
    with pytest.raises(bdm.DsparkError) as e:
        bdm.linear_stream_noalloc(A, W, out)
    assert e.value.status == bdm.ERR_CAPACITY
    assert bdm.noalloc_check() == 0
