"""Pins for the oracle's sampler (reading R10 of the oracle): the counter-based
generator against its published reference outputs, the uniform's lattice, the
drawn frequencies against softmax(l / t) over the top-k candidates (a
chi-square test over many draws), and the special cases that reduce to the
argmax.  Planted mistakes in the sampler must fail at least one pin.
"""
import os

import numpy as np
import pytest
import scipy.stats

import oracle
import oracle.dspark_oracle as od
import synthetic as syn

from test_oracle_pins import tiny_cfg


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "splitmix64_seed0.txt")


def test_splitmix64_reference_outputs():
    """SplitMix64 (Steele, Lea and Flood, OOPSLA 2014), stream seeded with 0: its
    first outputs as published with the reference implementation (tests/golden)."""
    want = [int(ln, 16) for ln in open(GOLDEN).read().split("\n") if ln.strip() and not ln.startswith("#")]
    assert len(want) == 3
    z = oracle.splitmix64(np.arange(len(want), dtype=np.uint64), 0)
    assert [int(v) for v in z] == want


def test_splitmix64_seed_is_a_stream_offset():
    """Seeding with s starts the stream s / golden-ratio-increment steps later:
    the stream seeded with the increment itself is the seed-0 stream shifted by one."""
    a = oracle.splitmix64(np.arange(1, 6, dtype=np.uint64), 0)
    b = oracle.splitmix64(np.arange(0, 5, dtype=np.uint64), 0x9E3779B97F4A7C15)
    assert np.array_equal(a, b)


def test_uniform_lattice_and_moments():
    v = np.arange(200000)
    u = oracle.sample_uniform(123, 3, 17, v)
    assert np.all(u > 0) and np.all(u < 1)
    k = u * (1 << 24) - 0.5                      # integers 0 .. 2^24 - 1
    assert np.array_equal(k, np.round(k))
    assert abs(u.mean() - 0.5) < 3e-3 and abs(u.var() - 1 / 12) < 2e-3
    # different slots, draws and seeds give different numbers for the same entry
    assert not np.array_equal(u[:100], oracle.sample_uniform(123, 4, 17, v[:100]))
    assert not np.array_equal(u[:100], oracle.sample_uniform(123, 3, 18, v[:100]))
    assert not np.array_equal(u[:100], oracle.sample_uniform(124, 3, 17, v[:100]))


LOGITS = np.array([1.3, -0.4, 2.1, 0.2, 2.1, -1.7, 0.9])


def _frequencies(logits, t, top_k, n, seed=99, slot=1):
    counts = np.zeros(logits.shape[0], np.int64)
    for draw in range(n):
        counts[oracle.sample_token(logits, t, top_k, seed, slot, draw)] += 1
    return counts


def _softmax_over(logits, t, idx):
    p = np.zeros(logits.shape[0])
    z = logits[idx] / t
    e = np.exp(z - z.max())
    p[idx] = e / e.sum()
    return p


@pytest.mark.parametrize("t,top_k", [(0.7, 0), (1.6, 0), (0.9, 3), (1.3, 5)])
def test_draws_follow_softmax_over_the_candidates(t, top_k):
    """Gumbel-max draws are exact samples of softmax(l / t) restricted to the
    top_k largest logits (the tie at 2.1 between entries 2 and 4 keeps both)."""
    n = 12000
    counts = _frequencies(LOGITS, t, top_k, n)
    idx = np.arange(LOGITS.shape[0]) if top_k == 0 else np.lexsort((np.arange(7), -LOGITS))[:top_k]
    p = _softmax_over(LOGITS, t, idx)
    assert counts[p == 0].sum() == 0
    keep = p > 0
    chi = scipy.stats.chisquare(counts[keep], n * p[keep])
    assert chi.pvalue > 1e-4, (counts, n * p)


def test_top_k_candidates_and_boundary_ties():
    l = np.array([0.5, 3.0, 1.0, 3.0, 1.0, 1.0])
    assert list(oracle.sample_candidates(l, 1)) == [1]
    assert list(oracle.sample_candidates(l, 2)) == [1, 3]
    assert list(oracle.sample_candidates(l, 3)) == [1, 3, 2]      # of the tied 1.0s, the lowest index
    assert list(oracle.sample_candidates(l, 4)) == [1, 3, 2, 4]
    assert list(oracle.sample_candidates(l, 0)) == list(range(6))
    assert list(oracle.sample_candidates(l, 9)) == list(range(6))


def test_top_one_and_cold_limit_are_the_argmax():
    rng = np.random.default_rng(5)
    for trial in range(50):
        l = rng.normal(size=40)
        best = int(np.argmax(l))
        assert oracle.sample_token(l, 2.5, 1, 7, 0, trial) == best
        assert oracle.sample_token(l, 1e-6, 0, 7, 0, trial) == best


def test_sampled_drafter_with_top_one_is_the_greedy_drafter():
    cfg = tiny_cfg(gamma=5)
    W = syn.make_weights(cfg, seed=31, norm_std=0.3, std=0.3)
    dr = oracle.Drafter(cfg, W)
    dr.ingest(syn.make_feats(cfg, 6, seed=31))
    g = dr.draft(3)
    s = dr.draft(3, sample=(0.8, 1, 11, 0))
    assert np.array_equal(g[0], s[0]) and np.allclose(g[1], s[1])


def test_sampled_drafter_uses_the_drawn_chain():
    """With sampling the chain follows the drawn tokens: position k's logits are
    the Markov logits of token k-1, and each token is sample_token of them."""
    cfg = tiny_cfg(gamma=5)
    W = syn.make_weights(cfg, seed=32, norm_std=0.3, std=0.3)
    dr = oracle.Drafter(cfg, W)
    dr.ingest(syn.make_feats(cfg, 6, seed=32))
    tok, conf, logits, y, U = dr.draft(7, sample=(1.5, 0, 5, 40))
    prev = 7
    for k in range(cfg.gamma):
        lk, _ = dr.markov_step(U[k], prev)
        assert np.array_equal(lk, logits[k])
        assert tok[k] == oracle.sample_token(lk, 1.5, 0, 5, 0, 40 + k)
        prev = int(tok[k])
    assert not np.array_equal(tok, dr.draft(7)[0])                 # not the greedy chain


# planted mistakes in the sampler, each caught by one of the pins above
def _no_temperature(logits, temperature, top_k, seed, slot, draw, keys_out=None):
    cand = np.sort(od.sample_candidates(logits, top_k))
    g = -np.log(-np.log(od.sample_uniform(seed, slot, draw, cand)))
    return int(cand[int(np.argmax(logits[cand] + g))])


def _wrong_gumbel_sign(logits, temperature, top_k, seed, slot, draw, keys_out=None):
    cand = np.sort(od.sample_candidates(logits, top_k))
    g = np.log(-np.log(od.sample_uniform(seed, slot, draw, cand)))
    return int(cand[int(np.argmax(logits[cand] / temperature + g))])


def _top_k_off_by_one(logits, top_k):
    V = logits.shape[0]
    if top_k <= 0 or top_k >= V:
        return np.arange(V)
    return np.lexsort((np.arange(V), -logits))[:top_k + 1]


def _ties_to_higher_index(logits, top_k):
    V = logits.shape[0]
    if top_k <= 0 or top_k >= V:
        return np.arange(V)
    return np.lexsort((-np.arange(V), -logits))[:top_k]


SAMPLER_MUTANTS = {
    "temperature ignored": ("sample_token", _no_temperature),
    "Gumbel noise with the wrong sign": ("sample_token", _wrong_gumbel_sign),
    "one candidate too many": ("sample_candidates", _top_k_off_by_one),
    "boundary ties to the higher index": ("sample_candidates", _ties_to_higher_index),
}


def _pins_pass():
    try:
        test_top_k_candidates_and_boundary_ties()
        for t, k in [(0.7, 0), (0.9, 3), (1.3, 5)]:
            test_draws_follow_softmax_over_the_candidates(t, k)
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("name", sorted(SAMPLER_MUTANTS))
def test_sampler_pins_catch_planted_mistake(monkeypatch, name):
    assert _pins_pass()
    attr, fn = SAMPLER_MUTANTS[name]
    monkeypatch.setattr(od, attr, fn)
    monkeypatch.setattr(oracle, attr, fn)
    assert not _pins_pass(), name
