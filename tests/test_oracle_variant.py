"""Pins for the oracle's grouped-query / QK-norm / rotary variant (reading R11):
closed forms of the rotation, GQA against multi-head attention with repeated
K/V heads, invariance under a common shift of every position, invariance of
the normalised Q and K to the scale of W_q and W_k, and the attention
probabilities of a tiny drafter against explicit loops over heads, keys and
rotation pairs (which fixes where the block rows sit relative to the context).
"""
import math

import numpy as np
import pytest

import oracle
import synthetic as syn


def vcfg(**kw):
    base = dict(hidden=48, n_taps=2, d_draft=32, n_heads=4, n_layers=2, ff_mult=2, gamma=3, vocab=50,
                markov_rank=8, dtype="fp32", n_kv_heads=2, qk_norm=True, rope_theta=10000.0)
    base.update(kw)
    return syn.DrafterConfig(**base)


def _drafter(cfg, W, L=6, seed=7):
    dr = oracle.Drafter(cfg, W)
    dr.ingest(syn.make_feats(cfg, L, seed=seed))
    return dr


def test_rope_closed_forms():
    """head_dim 4, base theta: a unit vector on entry 0 turns towards entry 2 (the
    rotate-half partner) by pos radians; entry 1 pairs with entry 3 at the
    frequency theta^(-1/2)."""
    th, p = 100.0, 0.7
    r0 = oracle.rope(np.array([[1.0, 0.0, 0.0, 0.0]]), np.array([p]), 1, th)[0]
    np.testing.assert_allclose(r0, [math.cos(p), 0.0, math.sin(p), 0.0], atol=1e-15)
    r1 = oracle.rope(np.array([[0.0, 1.0, 0.0, 0.0]]), np.array([p]), 1, th)[0]
    f = p / math.sqrt(th)
    np.testing.assert_allclose(r1, [0.0, math.cos(f), 0.0, math.sin(f)], atol=1e-15)
    r3 = oracle.rope(np.array([[0.0, 0.0, 0.0, 1.0]]), np.array([p]), 1, th)[0]
    np.testing.assert_allclose(r3, [0.0, -math.sin(f), 0.0, math.cos(f)], atol=1e-15)


def test_rope_is_a_rotation_per_pair():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(5, 24))
    pos = np.array([0, 1, 17, 300, 4096])
    y = oracle.rope(x, pos, 3, 500.0)
    np.testing.assert_allclose(y[0], x[0], atol=1e-15)                        # position 0
    xh, yh = x.reshape(5, 3, 8), y.reshape(5, 3, 8)
    np.testing.assert_allclose(xh[..., :4] ** 2 + xh[..., 4:] ** 2, yh[..., :4] ** 2 + yh[..., 4:] ** 2, rtol=1e-12)
    np.testing.assert_allclose(oracle.rope(y, -pos, 3, 500.0), x, atol=1e-12)  # the inverse turn
    # dot products of turned vectors depend on the position difference only
    a, b = rng.normal(size=(1, 8)), rng.normal(size=(1, 8))
    d1 = oracle.rope(a, [40], 1, 500.0) @ oracle.rope(b, [15], 1, 500.0).T
    d2 = oracle.rope(a, [125], 1, 500.0) @ oracle.rope(b, [100], 1, 500.0).T
    np.testing.assert_allclose(d1, d2, rtol=1e-12)


def test_gqa_equals_mha_with_repeated_kv_heads():
    """Query heads 2j and 2j+1 share K/V head j: the same drafter with one K/V head
    per query head, whose W_k and W_v rows repeat head j for both, gives the same
    draft (and QK-norm and rotation act per head, so they commute with it)."""
    cfg = vcfg()
    W = syn.make_weights(cfg, seed=3, norm_std=0.3, std=0.3)
    mha = vcfg(n_kv_heads=0)
    Wm = dict(W)
    hd = cfg.head_dim
    for i in range(cfg.n_layers):
        for m in ("k", "v"):
            rows = W[f"bb.{i}.{m}"].reshape(cfg.kv_heads, hd, -1)
            Wm[f"bb.{i}.{m}"] = np.repeat(rows, cfg.n_heads // cfg.kv_heads, axis=0).reshape(cfg.d_draft, -1)
    a = _drafter(cfg, W).draft(5)
    b = _drafter(mha, Wm).draft(5)
    assert np.array_equal(a[0], b[0])
    np.testing.assert_allclose(a[2], b[2], rtol=0, atol=1e-12)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-12)


def test_common_position_shift_changes_nothing():
    cfg = vcfg()
    W = syn.make_weights(cfg, seed=4, norm_std=0.3, std=0.3)
    d0 = _drafter(cfg, W)
    d1 = oracle.Drafter(cfg, W)
    d1.pos_offset = 1234
    d1.ingest(syn.make_feats(cfg, 6, seed=7))
    a, b = d0.draft(9), d1.draft(9)
    np.testing.assert_allclose(a[2], b[2], rtol=0, atol=1e-9)
    assert np.array_equal(a[0], b[0])
    # but the rotation is active: without it the draft differs
    c = _drafter(vcfg(rope_theta=0.0), W).draft(9)
    assert np.max(np.abs(a[2] - c[2])) > 1e-6


def test_qk_norm_removes_the_scale_of_wq_and_wk():
    cfg = vcfg()
    W = syn.make_weights(cfg, seed=5, norm_std=0.3, std=0.3)
    W2 = dict(W)
    for i in range(cfg.n_layers):
        W2[f"bb.{i}.q"] = W[f"bb.{i}.q"] * np.float32(4.0)
        W2[f"bb.{i}.k"] = W[f"bb.{i}.k"] * np.float32(4.0)
    a, b = _drafter(cfg, W).draft(2), _drafter(cfg, W2).draft(2)
    np.testing.assert_allclose(a[2], b[2], rtol=0, atol=1e-4 * np.max(np.abs(a[2])))
    # without QK-norm the scale matters
    nq = vcfg(qk_norm=False)
    Wn = {k: v for k, v in W.items() if not k.endswith(("q_norm", "k_norm"))}
    Wn2 = {k: v for k, v in W2.items() if not k.endswith(("q_norm", "k_norm"))}
    assert np.max(np.abs(_drafter(nq, Wn).draft(2)[2] - _drafter(nq, Wn2).draft(2)[2])) > 1e-4


def test_first_layer_attention_against_loops():
    """Layer 0's attention probabilities of a one-layer drafter, rebuilt with
    explicit loops: RMSNorm per head, the rotation pair by pair at the context
    position t and the block position L + j, GQA head h // 2."""
    cfg = vcfg(n_layers=1)
    W = syn.make_weights(cfg, seed=6, norm_std=0.3, std=0.3)
    L = 5
    dr = _drafter(cfg, W, L=L)
    probs = []
    dr.backbone(11, 0, probs_out=probs)
    w = {k: oracle.to_f64(v) for k, v in W.items() if k != "embed"}
    hd, eps, th = cfg.head_dim, cfg.eps, cfg.rope_theta
    X = oracle.to_f64(syn.make_feats(cfg, L, seed=7))
    Hc = oracle.context_features(X, w["W_c"], w["ctx_norm"], eps)
    x = dr.block_input(11)

    def norm_rows(a, g):
        return [[a[r][c] / math.sqrt(sum(v * v for v in a[r]) / len(a[r]) + eps) * g[c] for c in range(len(a[r]))]
                for r in range(len(a))]

    def head_vec(row, W_, head, which, pos):
        v = [sum(W_[head * hd + e][c] * row[c] for c in range(len(row))) for e in range(hd)]
        ms = sum(t * t for t in v) / hd
        v = [v[e] / math.sqrt(ms + eps) * w[f"bb.0.{which}_norm"][e] for e in range(hd)]
        out = list(v)
        for e in range(hd // 2):
            ang = pos * th ** (-2.0 * e / hd)
            out[e] = v[e] * math.cos(ang) - v[e + hd // 2] * math.sin(ang)
            out[e + hd // 2] = v[e + hd // 2] * math.cos(ang) + v[e] * math.sin(ang)
        return out

    nc = norm_rows(Hc.tolist(), w["bb.0.attn_norm"])
    nb = norm_rows(x.tolist(), w["bb.0.attn_norm"])
    for h in range(cfg.n_heads):
        kvh = h // (cfg.n_heads // cfg.kv_heads)
        keys = [head_vec(nc[t], w["bb.0.k"], kvh, "k", t) for t in range(L)] + \
               [head_vec(nb[j], w["bb.0.k"], kvh, "k", L + j) for j in range(cfg.gamma)]
        for j in range(cfg.gamma):
            q = head_vec(nb[j], w["bb.0.q"], h, "q", L + j)
            s = [sum(q[e] * k[e] for e in range(hd)) / math.sqrt(hd) for k in keys]
            m = max(s)
            p = [math.exp(v - m) for v in s]
            tot = sum(p)
            np.testing.assert_allclose(probs[h][j], [v / tot for v in p], rtol=0, atol=1e-12)


def test_variant_configs_are_checked():
    with pytest.raises(ValueError):
        oracle.Drafter(vcfg(n_kv_heads=3), {})


# planted mistakes in the variant, each caught by a pin above
def _interleaved_rope(x, positions, n_heads, theta):
    rows, width = x.shape
    hd = width // n_heads
    ang = np.asarray(positions, np.float64)[:, None] * theta ** (-2.0 * np.arange(hd // 2) / hd)[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    xh = x.reshape(rows, n_heads, hd // 2, 2)
    a, b = xh[..., 0], xh[..., 1]
    return np.stack([a * c - b * s, b * c + a * s], axis=-1).reshape(rows, width)


def _modulo_gqa_attention(Q, K, V, n_heads, probs_out=None, n_kv_heads=0):
    g, d = Q.shape
    hd = d // n_heads
    nkv = n_kv_heads or n_heads
    O = np.empty((g, d))
    for h in range(n_heads):
        sl, kv = slice(h * hd, (h + 1) * hd), slice((h % nkv) * hd, (h % nkv + 1) * hd)
        P = oracle.softmax((Q[:, sl] @ K[:, kv].T) * hd ** -0.5)
        if probs_out is not None:
            probs_out.append(P)
        O[:, sl] = P @ V[:, kv]
    return O


def _block_from_zero_layer(self, i, x, Kc, Vc, probs_out=None):
    cfg, w = self.cfg, self.w
    n = oracle.rmsnorm(x, w[f"bb.{i}.attn_norm"], cfg.eps)
    pos = np.arange(cfg.gamma)
    Q = self.qk_transform(n @ w[f"bb.{i}.q"].T, i, "q", pos, cfg.n_heads)
    Kb = self.qk_transform(n @ w[f"bb.{i}.k"].T, i, "k", pos, cfg.kv_heads)
    O = oracle.attention(Q, np.concatenate([Kc, Kb]), np.concatenate([Vc, n @ w[f"bb.{i}.v"].T]), cfg.n_heads,
                         probs_out, cfg.kv_heads)
    x = x + O @ w[f"bb.{i}.o"].T
    n2 = oracle.rmsnorm(x, w[f"bb.{i}.ff_norm"], cfg.eps)
    return x + oracle.ffn(n2, w[f"bb.{i}.gate"], w[f"bb.{i}.up"], w[f"bb.{i}.down"], cfg.act)


def _fails(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_variant_pins_catch_planted_mistakes(monkeypatch):
    import oracle.dspark_oracle as od
    with monkeypatch.context() as m:
        m.setattr(od, "rope", _interleaved_rope)
        m.setattr(oracle, "rope", _interleaved_rope)
        assert _fails(test_rope_closed_forms)
    with monkeypatch.context() as m:
        m.setattr(od, "attention", _modulo_gqa_attention)
        assert _fails(test_gqa_equals_mha_with_repeated_kv_heads)
        assert _fails(test_first_layer_attention_against_loops)
    with monkeypatch.context() as m:
        m.setattr(od.Drafter, "layer", _block_from_zero_layer)
        assert _fails(test_first_layer_attention_against_loops)
