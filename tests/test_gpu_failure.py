"""Failure detection without a fault: every kind of bounded device wait the
library uses is run on words that nothing completes; each gives up after its
limit (about a second), the kernel returns normally with the timeout bit in the
error word, and the device keeps working (a draft afterwards matches the
oracle).
"""
import numpy as np
import pytest

import oracle
import synthetic as syn
from helpers import check_block, make_gpu_drafter, to_torch, weights_to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="session", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_draft_model_gb300 as bdm
    bdm.build()
    bdm.load()


# 0: the single-sequence Markov chain's arrival count, 1: the resident chain's barrier,
# 2: the cooperative chain's barrier, 3: the one-launch layers' grid barrier,
# 4: the tensor-core kernels' mbarrier wait, 5: the one-launch step's grid barrier
@pytest.mark.parametrize("which", range(6))
def test_bounded_wait_gives_up_and_reports(which):
    import block_draft_model_gb300 as bdm
    word = bdm.selftest_wait(which)
    assert word & bdm.DEVERR_TIMEOUT, word


def test_selftest_rejects_unknown_wait():
    import block_draft_model_gb300 as bdm
    with pytest.raises(bdm.DsparkError):
        bdm.selftest_wait(6)


def test_device_usable_after_the_timeouts():
    import block_draft_model_gb300 as bdm
    assert bdm.selftest_wait(1) & bdm.DEVERR_TIMEOUT
    cfg = syn.DrafterConfig(hidden=128, n_taps=2, d_draft=128, n_heads=2, n_layers=1, ff_mult=2, gamma=4, vocab=500,
                            markov_rank=32)
    W = syn.make_weights(cfg, seed=61)
    X = syn.make_feats(cfg, 12, seed=61)
    dr = oracle.Drafter(cfg, W)
    dr.ingest(X)
    gd = make_gpu_drafter(cfg, weights_to_device(W), max_ctx=16)
    gd.ingest_context(to_torch(X))
    tok = torch.empty(cfg.gamma, dtype=torch.int32, device="cuda")
    conf = torch.empty(cfg.gamma, dtype=torch.float32, device="cuda")
    lg = torch.empty(cfg.gamma, cfg.vocab, dtype=torch.float32, device="cuda")
    gd.draft(9, tok, conf, lg)
    torch.cuda.synchronize()
    check_block(dr, 0, 9, tok.cpu().numpy(), conf.cpu().numpy(), lg.cpu().numpy())
    assert gd.check() == 0
