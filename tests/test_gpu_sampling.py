"""GPU parity of the sampling form of the Markov chain (the oracle's reading R10)
through the C ABI.

For every drawn position the check is teacher-forced on the GPU's own chain:
the GPU's logits of position k must match the oracle's Markov logits for the
GPU's token k-1 (within the logit tolerance), and the GPU's token k must be the
oracle sampler's draw on exactly those GPU logits (same candidates, same
uniforms), except where two Gumbel keys lie closer than the fp32 rounding of
the keys, where either is accepted.  Confidences follow the same chain.
"""
import numpy as np
import pytest

import oracle
import synthetic as syn
from helpers import make_gpu_drafter, rel_tol, to_torch, weights_to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="session", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_draft_model_gb300 as bdm
    bdm.build()
    bdm.load()


def check_sampled(dr, slot, anchor, tok, conf, lg, t, top_k, seed, draw0, rel, label=""):
    y = dr.backbone(anchor, slot)
    U = dr.base_logits(y)
    prev = int(anchor)
    for k in range(U.shape[0]):
        ref, e = dr.markov_step(U[k], prev)
        gl = np.asarray(lg[k], np.float64)
        err = np.max(np.abs(gl - ref))
        assert err <= rel * np.max(np.abs(ref)), f"{label} k {k}: logits max|d| {err:.3e}"
        keys = []
        want = oracle.sample_token(gl, t, top_k, seed, slot, draw0 + k, keys_out=keys)
        got = int(tok[k])
        if got != want:
            cand, z = keys[0]
            assert got in set(cand.tolist()), f"{label} k {k}: token {got} is not a candidate"
            zg = z[list(cand).index(got)]
            assert z.max() - zg <= 1e-4 * max(1.0, abs(z.max())), f"{label} k {k}: {got} vs {want}"
        cf = dr.confidence(y[k], e)
        assert abs(float(conf[k]) - cf) <= rel, f"{label} k {k}: conf {conf[k]} vs {cf}"
        prev = got


def _setup(cfg, L, seed, max_seqs=1, n_seq=1):
    W = syn.make_weights(cfg, seed=seed, norm_std=0.2)
    dr = oracle.Drafter(cfg, W)
    gd = make_gpu_drafter(cfg, weights_to_device(W), max_ctx=L + 8, max_seqs=max_seqs)
    feats = []
    for s in range(n_seq):
        X = syn.make_feats(cfg, L + s, seed=seed, seq=s)
        dr.ingest(X, seq=s)
        feats.append(X)
    if n_seq == 1 and max_seqs == 1:
        gd.ingest_context(to_torch(feats[0]))
    else:
        lens = [f.shape[0] for f in feats]
        ids = torch.arange(n_seq, dtype=torch.int32, device="cuda")
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
        gd.ingest_context_batched(ids, cu, to_torch(np.concatenate(feats, axis=0)))
    return dr, gd


def _draft(gd, cfg, anchor):
    tok = torch.empty(cfg.gamma, dtype=torch.int32, device="cuda")
    conf = torch.empty(cfg.gamma, dtype=torch.float32, device="cuda")
    lg = torch.empty(cfg.gamma, cfg.vocab, dtype=torch.float32, device="cuda")
    gd.draft(anchor, tok, conf, lg)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), conf.cpu().numpy(), lg.cpu().numpy()


@pytest.mark.parametrize("t,top_k", [(0.8, 0), (1.3, 8), (0.5, 64), (2.0, 1)])
def test_sampled_draft_matches_oracle(t, top_k):
    """bf16 drafter, V 1000 over 152 CTAs (7 rows each, so local lists shorter
    than top_k are padded), three calls in a row (the draw counter advances by
    gamma), then the sampler reset replays the first call's draws."""
    cfg = syn.DrafterConfig(hidden=256, n_taps=2, d_draft=256, n_heads=2, n_layers=2, ff_mult=2, gamma=6, vocab=1000,
                            markov_rank=64)
    dr, gd = _setup(cfg, 40, seed=41)
    seed = 0xC0FFEE + top_k
    gd.set_sampling(t, top_k, seed)
    first = None
    for call, anchor in enumerate([3, 999, 500]):
        tok, conf, lg = _draft(gd, cfg, anchor)
        check_sampled(dr, 0, anchor, tok, conf, lg, t, top_k, seed, call * cfg.gamma, rel_tol(cfg),
                      label=f"call {call}")
        if call == 0:
            first = tok.copy()
    assert gd.check() == 0
    gd.set_sampling(t, top_k, seed)
    tok, _, _ = _draft(gd, cfg, 3)
    assert np.array_equal(tok, first)
    if top_k == 1:  # the top candidate only: the greedy chain
        gd.set_sampling(0.0)
        gtok, _, _ = _draft(gd, cfg, 3)
        assert np.array_equal(gtok, first)


@pytest.mark.parametrize("vocab,rank,top_k", [(100, 32, 16), (262144, 128, 64), (70001, 256, 0)])
def test_sampled_draft_vocabulary_shapes(vocab, rank, top_k):
    """V 100 (most CTAs own no row), V 262144 (1725 rows per CTA, the 2048-word
    local sort), V 70001 with the whole vocabulary as candidates."""
    cfg = syn.DrafterConfig(hidden=128, n_taps=2, d_draft=128, n_heads=2, n_layers=1, ff_mult=2, gamma=4, vocab=vocab,
                            markov_rank=rank)
    dr, gd = _setup(cfg, 20, seed=42)
    gd.set_sampling(1.1, top_k, 77)
    tok, conf, lg = _draft(gd, cfg, vocab // 3)
    check_sampled(dr, 0, vocab // 3, tok, conf, lg, 1.1, top_k, 77, 0, rel_tol(cfg))
    assert gd.check() == 0


def test_sampled_fp32_drafter():
    cfg = syn.TINY
    dr, gd = _setup(cfg, 30, seed=43)
    gd.set_sampling(0.9, 5, 1234)
    for call in range(2):
        tok, conf, lg = _draft(gd, cfg, 17 + call)
        check_sampled(dr, 0, 17 + call, tok, conf, lg, 0.9, 5, 1234, call * cfg.gamma, rel_tol(cfg))
    assert gd.check() == 0


def test_sampled_batched_draft_uses_each_slot():
    """Three sequences in slots (2, 0, 1): each draws with its own slot and counter."""
    cfg = syn.DrafterConfig(hidden=128, n_taps=2, d_draft=128, n_heads=2, n_layers=2, ff_mult=2, gamma=5, vocab=3000,
                            markov_rank=64)
    dr, gd = _setup(cfg, 30, seed=44, max_seqs=3, n_seq=3)
    gd.set_sampling(1.0, 32, 99)
    ids = torch.tensor([2, 0, 1], dtype=torch.int32, device="cuda")
    anchors = torch.tensor([7, 2999, 1500], dtype=torch.int32, device="cuda")
    tok = torch.empty(3, cfg.gamma, dtype=torch.int32, device="cuda")
    conf = torch.empty(3, cfg.gamma, dtype=torch.float32, device="cuda")
    lg = torch.empty(3, cfg.gamma, cfg.vocab, dtype=torch.float32, device="cuda")
    for call in range(2):
        gd.draft_batched(ids, anchors, tok, conf, lg)
        torch.cuda.synchronize()
        for b in range(3):
            slot = int(ids[b])
            check_sampled(dr, slot, int(anchors[b]), tok[b].cpu().numpy(), conf[b].cpu().numpy(),
                          lg[b].cpu().numpy(), 1.0, 32, 99, call * cfg.gamma, rel_tol(cfg), label=f"call {call} b {b}")
    assert gd.check() == 0


def test_sampling_arguments_are_checked():
    import block_draft_model_gb300 as bdm
    cfg = syn.DrafterConfig(hidden=128, n_taps=2, d_draft=128, n_heads=2, n_layers=1, ff_mult=2, gamma=4, vocab=500,
                            markov_rank=32)
    _, gd = _setup(cfg, 10, seed=45)
    for args in [(-1.0, 0), (float("nan"), 0), (1.0, -1), (1.0, 65)]:
        with pytest.raises(bdm.DsparkError):
            gd.set_sampling(*args)
