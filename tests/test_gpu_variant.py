"""GPU parity of the grouped-query / QK-norm / rotary variant (the oracle's
reading R11) through the C ABI: every cache row (the K rows normalised and
turned at their context positions), every logit, token and confidence of the
drafted blocks, for single-sequence and batched ingest and draft, bf16 and
fp32, several K/V head counts.
"""
import numpy as np
import pytest

import oracle
import synthetic as syn
from helpers import (check_block, check_cache, make_gpu_drafter, rel_tol, to_torch, weights_to_device)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="session", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_draft_model_gb300 as bdm
    bdm.build()
    bdm.load()


def _draft(gdr, cfg, anchor):
    tok = torch.empty(cfg.gamma, dtype=torch.int32, device="cuda")
    conf = torch.empty(cfg.gamma, dtype=torch.float32, device="cuda")
    lg = torch.empty(cfg.gamma, cfg.vocab, dtype=torch.float32, device="cuda")
    gdr.draft(anchor, tok, conf, lg)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), conf.cpu().numpy(), lg.cpu().numpy()


def _single(cfg, L, seed, chunks, anchors):
    W = syn.make_weights(cfg, seed=seed, norm_std=0.2)
    X = syn.make_feats(cfg, L, seed=seed)
    dr = oracle.Drafter(cfg, W)
    dr.ingest(X)
    gdr = make_gpu_drafter(cfg, weights_to_device(W), max_ctx=L + 8)
    lo = 0
    Xd = to_torch(X)
    for hi in chunks + [L]:
        gdr.ingest_context(Xd[lo:hi])
        lo = hi
    rel = rel_tol(cfg)
    check_cache(dr, gdr, cfg, 0, np.arange(L), rel, label="cache")
    for a in anchors:
        tok, conf, lg = _draft(gdr, cfg, a)
        check_block(dr, 0, a, tok, conf, lg, rel=rel, label=f"anchor {a}")
    assert gdr.check() == 0


@pytest.mark.parametrize("d,n_heads,n_kv,qk,theta,L,gamma", [
    (256, 4, 2, True, 10000.0, 300, 6),       # GQA 2:1, norm and rotation, tensor-core ingest and attention
    (1024, 8, 1, False, 500000.0, 1500, 8),   # one K/V head, rotation only, many key ranges
    (512, 8, 4, False, 0.0, 120, 5),          # GQA alone (the batch-1 norm chain streams QKV of width d + 2 d_kv)
])
def test_variant_single_sequence(d, n_heads, n_kv, qk, theta, L, gamma):
    cfg = syn.DrafterConfig(hidden=256, n_taps=2, d_draft=d, n_heads=n_heads, n_layers=2, ff_mult=2, gamma=gamma,
                            vocab=1000, markov_rank=64, n_kv_heads=n_kv, qk_norm=qk, rope_theta=theta)
    _single(cfg, L, seed=51, chunks=[L // 3, L // 2], anchors=[3, 998])


def test_variant_fp32_drafter():
    cfg = syn.DrafterConfig(hidden=128, n_taps=3, d_draft=128, n_heads=4, n_layers=2, ff_mult=2, gamma=4, vocab=700,
                            markov_rank=32, dtype="fp32", n_kv_heads=2, qk_norm=True, rope_theta=10000.0)
    _single(cfg, 40, seed=52, chunks=[7], anchors=[5, 600])


def test_variant_batched_ragged():
    """Three sequences in slots (2, 0, 1) with ragged contexts, ingested together
    (positions from the batched row table) and drafted together."""
    cfg = syn.DrafterConfig(hidden=128, n_taps=2, d_draft=256, n_heads=4, n_layers=2, ff_mult=2, gamma=5, vocab=900,
                            markov_rank=32, n_kv_heads=2, qk_norm=True, rope_theta=10000.0)
    W = syn.make_weights(cfg, seed=53, norm_std=0.2)
    dr = oracle.Drafter(cfg, W)
    gd = make_gpu_drafter(cfg, weights_to_device(W), max_ctx=80, max_seqs=3)
    slots = [2, 0, 1]
    lens = [33, 7, 60]
    feats = [syn.make_feats(cfg, n, seed=53, seq=s) for s, n in zip(slots, lens)]
    for s, f in zip(slots, feats):
        dr.ingest(f, seq=s)
    ids = torch.tensor(slots, dtype=torch.int32, device="cuda")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    gd.ingest_context_batched(ids, cu, to_torch(np.concatenate(feats, axis=0)))
    for s, n in zip(slots, lens):
        check_cache(dr, gd, cfg, s, np.arange(n), label=f"slot {s}")
    anchors = torch.tensor([4, 899, 450], dtype=torch.int32, device="cuda")
    tok = torch.empty(3, cfg.gamma, dtype=torch.int32, device="cuda")
    conf = torch.empty(3, cfg.gamma, dtype=torch.float32, device="cuda")
    lg = torch.empty(3, cfg.gamma, cfg.vocab, dtype=torch.float32, device="cuda")
    gd.draft_batched(ids, anchors, tok, conf, lg)
    torch.cuda.synchronize()
    for b, s in enumerate(slots):
        check_block(dr, s, int(anchors[b]), tok[b].cpu().numpy(), conf[b].cpu().numpy(), lg[b].cpu().numpy(),
                    label=f"slot {s}")
    assert gd.check() == 0


def test_variant_config_errors():
    import block_draft_model_gb300 as bdm
    cfg = syn.DrafterConfig(hidden=128, n_taps=2, d_draft=256, n_heads=4, n_layers=1, ff_mult=2, gamma=4, vocab=300,
                            markov_rank=32, n_kv_heads=3)
    W = syn.make_weights(syn.DrafterConfig(hidden=128, n_taps=2, d_draft=256, n_heads=4, n_layers=1, ff_mult=2,
                                           gamma=4, vocab=300, markov_rank=32), seed=1)
    with pytest.raises(bdm.DsparkError):
        make_gpu_drafter(cfg, weights_to_device(W), max_ctx=16)
