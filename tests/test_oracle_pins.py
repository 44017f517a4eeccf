"""Pins of the CPU oracle against things other than itself.

* brute force: the dense form of "module-dflash.ts" (``forwardInfer`` calls
  ``#backbone``, which rebuilds H_ctx from the FULL context and re-projects the
  context K/V inside every ``#layer``), written as plain Python loops on tiny
  inputs, against the oracle's cached, incremental form;
* invariants stated or implied by the pages (W2 = 0 gives pure parallel
  DFlash, conf head zero gives sigmoid(b), context is read-only memory with no
  positional encoding, so row order does not matter and ingest is row-wise);
* closed forms (uniform attention, a hand-worked two-dimensional drafter);
* library routines for the scalar pieces (scipy's expit / erf, numpy argmax).
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle
import synthetic as syn


def tiny_cfg(**kw):
    base = dict(hidden=6, n_taps=2, d_draft=8, n_heads=2, n_layers=2, ff_mult=2, gamma=3,
                vocab=11, markov_rank=3, eps=1e-6, dtype="fp32")
    base.update(kw)
    return syn.DrafterConfig(**base)


# --------------------------------------------------------------------------- brute force

def _f(a):
    """numpy (float32 or bf16 bits) -> nested Python floats."""
    return oracle.to_f64(a).tolist()


def _matvec(W, x):
    return [sum(W[o][k] * x[k] for k in range(len(x))) for o in range(len(W))]


def _rms(x, w, eps):
    ms = sum(v * v for v in x) / len(x)
    s = 1.0 / math.sqrt(ms + eps)
    return [x[i] * s * w[i] for i in range(len(x))]


def _act(g, kind):
    if kind == "silu":
        return g / (1.0 + math.exp(-g))
    return 0.5 * g * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (g + 0.044715 * g * g * g)))


def brute_force_draft(cfg, W, ctx_rows, anchor):
    """Dense recomputation of one draft block, loop by loop, from all context rows."""
    d, nh, eps = cfg.d_draft, cfg.n_heads, cfg.eps
    hd = d // nh
    P = {k: _f(v) for k, v in W.items() if k not in ("embed",)}
    E = _f(W["embed"])
    # Eq 2 over the full context
    Hctx = [_rms(_matvec(P["W_c"], row), P["ctx_norm"], eps) for row in ctx_rows]
    # block
    x = []
    x0 = _matvec(P["tok_proj"], E[anchor])
    x.append([x0[c] + P["block_pos"][0][c] for c in range(d)])
    for j in range(1, cfg.gamma):
        x.append([P["mask_emb"][j - 1][c] + P["block_pos"][j][c] for c in range(d)])
    for i in range(cfg.n_layers):
        pre = f"bb.{i}."
        nd = [_rms(r, P[pre + "attn_norm"], eps) for r in x]
        nc = [_rms(r, P[pre + "attn_norm"], eps) for r in Hctx]
        q = [_matvec(P[pre + "q"], r) for r in nd]
        keys = [_matvec(P[pre + "k"], r) for r in nc] + [_matvec(P[pre + "k"], r) for r in nd]
        vals = [_matvec(P[pre + "v"], r) for r in nc] + [_matvec(P[pre + "v"], r) for r in nd]
        att = [[0.0] * d for _ in range(cfg.gamma)]
        for h in range(nh):
            lo = h * hd
            for j in range(cfg.gamma):
                s = [sum(q[j][lo + c] * kk[lo + c] for c in range(hd)) / math.sqrt(hd) for kk in keys]
                mx = max(s)
                ex = [math.exp(v - mx) for v in s]
                den = sum(ex)
                for c in range(hd):
                    att[j][lo + c] = sum(ex[t] / den * vals[t][lo + c] for t in range(len(keys)))
        o = [_matvec(P[pre + "o"], r) for r in att]
        x = [[x[j][c] + o[j][c] for c in range(d)] for j in range(cfg.gamma)]
        n2 = [_rms(r, P[pre + "ff_norm"], eps) for r in x]
        out = []
        for j in range(cfg.gamma):
            g = _matvec(P[pre + "gate"], n2[j])
            u = _matvec(P[pre + "up"], n2[j])
            hmid = [_act(g[c], cfg.act) * u[c] for c in range(len(g))]
            dn = _matvec(P[pre + "down"], hmid)
            out.append([x[j][c] + dn[c] for c in range(d)])
        x = out
    y = [_rms(r, P["out_norm"], eps) for r in x]
    U = [_matvec(P["out_proj"], r) for r in y]
    w1, w2 = P["markov.w1"], P["markov.w2"]
    prev = anchor
    toks, confs, logits = [], [], []
    for k in range(cfg.gamma):
        e = w1[prev]
        lk = [U[k][v] + sum(w2[v][c] * e[c] for c in range(len(e))) for v in range(cfg.vocab)]
        best = 0
        for v in range(1, cfg.vocab):
            if lk[v] > lk[best]:
                best = v
        z = sum(a * b for a, b in zip(y[k] + e, P["conf.w"])) + P["conf.b"][0]
        confs.append(1.0 / (1.0 + math.exp(-z)))
        toks.append(best)
        logits.append(lk)
        prev = best
    return toks, confs, logits


@pytest.mark.parametrize("variant", [
    dict(),
    dict(act="gelu_tanh"),
    dict(dtype="bf16"),
    dict(gamma=1, n_layers=1),
    dict(n_heads=1, d_draft=4, hidden=5, n_taps=3),
])
def test_cached_oracle_matches_dense_brute_force(variant):
    cfg = tiny_cfg(**variant)
    W = syn.make_weights(cfg, seed=3, norm_std=0.1, std=0.3)
    L = 5
    X = syn.make_feats(cfg, L, seed=3)
    drafter = oracle.Drafter(cfg, W)
    # ingest in two uneven pieces: the cache must equal a one-shot recompute
    drafter.ingest(X[:2])
    drafter.ingest(X[2:])
    rows = oracle.to_f64(X).tolist()
    for anchor in (0, 7):
        tok, conf, logits, _, _ = drafter.draft(anchor)
        btok, bconf, blogits = brute_force_draft(cfg, W, rows, anchor)
        np.testing.assert_allclose(logits, np.array(blogits), rtol=0, atol=1e-12)
        np.testing.assert_allclose(conf, np.array(bconf), rtol=0, atol=1e-12)
        assert list(tok) == btok


def test_empty_context_matches_brute_force():
    cfg = tiny_cfg()
    W = syn.make_weights(cfg, seed=4, norm_std=0.1, std=0.3)
    drafter = oracle.Drafter(cfg, W)
    tok, conf, logits, _, _ = drafter.draft(3)
    btok, bconf, blogits = brute_force_draft(cfg, W, [], 3)
    np.testing.assert_allclose(logits, np.array(blogits), rtol=0, atol=1e-12)
    assert list(tok) == btok


# --------------------------------------------------------------------------- invariants

def _setup(seed=5, **kw):
    cfg = tiny_cfg(**kw)
    W = syn.make_weights(cfg, seed=seed, norm_std=0.1, std=0.3)
    X = syn.make_feats(cfg, 7, seed=seed)
    return cfg, W, X


def test_context_permutation_invariance():
    """No positional encoding on the context: row order does not change the draft."""
    cfg, W, X = _setup()
    a = oracle.Drafter(cfg, W)
    a.ingest(X)
    perm = np.array([3, 0, 6, 1, 5, 2, 4])
    b = oracle.Drafter(cfg, W)
    b.ingest(X[perm])
    ra, rb = a.draft(2), b.draft(2)
    np.testing.assert_allclose(ra[2], rb[2], rtol=0, atol=1e-12)
    np.testing.assert_allclose(ra[1], rb[1], rtol=0, atol=1e-12)
    assert list(ra[0]) == list(rb[0])


def test_zero_projection_gives_zero_context_and_cache():
    cfg, W, X = _setup()
    W["W_c"] = np.zeros_like(W["W_c"])
    dr = oracle.Drafter(cfg, W)
    Hc = oracle.context_features(oracle.to_f64(X), dr.w["W_c"], dr.w["ctx_norm"], cfg.eps)
    assert np.all(Hc == 0.0)
    dr.ingest(X)
    for i in range(cfg.n_layers):
        K, V = dr.cache(0, i)
        assert K.shape == (7, cfg.d_draft) and np.all(K == 0.0) and np.all(V == 0.0)


def test_zero_markov_factor_leaves_base_logits():
    """W2 = 0 makes the drafter pure parallel DFlash (``initFromDims``)."""
    cfg, W, X = _setup()
    W["markov.w2"] = np.zeros_like(W["markov.w2"])
    dr = oracle.Drafter(cfg, W)
    dr.ingest(X)
    tok, conf, logits, y, U = dr.draft(4)
    assert np.array_equal(logits, U)
    assert list(tok) == [int(np.argmax(U[k])) for k in range(cfg.gamma)]


def test_zero_confidence_head_gives_sigmoid_of_bias():
    cfg, W, X = _setup()
    W["conf.w"] = np.zeros_like(W["conf.w"])
    W["conf.b"] = np.array([0.0], np.float32)
    dr = oracle.Drafter(cfg, W)
    dr.ingest(X)
    assert np.all(dr.draft(1)[1] == 0.5)
    W["conf.b"] = np.array([1.25], np.float32)
    dr = oracle.Drafter(cfg, W)
    dr.ingest(X)
    np.testing.assert_allclose(dr.draft(1)[1], scipy.special.expit(1.25), rtol=0, atol=1e-15)


def test_attention_rows_sum_to_one():
    cfg, W, X = _setup()
    dr = oracle.Drafter(cfg, W)
    dr.ingest(X)
    probs = []
    dr.backbone(5, probs_out=probs)
    assert len(probs) == cfg.n_layers * cfg.n_heads
    for P in probs:
        assert P.shape == (cfg.gamma, 7 + cfg.gamma)
        assert np.all(P > 0)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def test_chunked_ingest_equals_one_shot():
    cfg, W, X = _setup()
    a = oracle.Drafter(cfg, W)
    a.ingest(X)
    b = oracle.Drafter(cfg, W)
    for lo, hi in ((0, 1), (1, 4), (4, 4), (4, 7)):
        b.ingest(X[lo:hi])
    for i in range(cfg.n_layers):
        for x, y in zip(a.cache(0, i), b.cache(0, i)):
            np.testing.assert_allclose(x, y, rtol=0, atol=1e-13)
    assert b.context_length() == 7


def test_identical_feature_rows_give_identical_cache_rows():
    cfg, W, X = _setup()
    X = X.copy()
    X[4] = X[1]
    dr = oracle.Drafter(cfg, W)
    dr.ingest(X)
    for i in range(cfg.n_layers):
        K, V = dr.cache(0, i)
        assert np.array_equal(K[4], K[1]) and np.array_equal(V[4], V[1])
        assert not np.array_equal(K[4], K[2])


def test_sequences_are_independent():
    cfg, W, X = _setup()
    X2 = syn.make_feats(cfg, 3, seed=9)
    a = oracle.Drafter(cfg, W)
    a.ingest(X, seq=0)
    a.ingest(X2, seq=5)
    b = oracle.Drafter(cfg, W)
    b.ingest(X)
    ra, rb = a.draft(2, seq=0), b.draft(2)
    assert np.array_equal(ra[2], rb[2])
    assert a.context_length(5) == 3


# --------------------------------------------------------------------------- closed forms

def test_zero_query_weights_give_uniform_attention():
    """W_q = 0 => all scores 0 => every probability 1/(L+gamma) and O = mean of the value rows."""
    cfg, W, X = _setup()
    for i in range(cfg.n_layers):
        W[f"bb.{i}.q"] = np.zeros_like(W[f"bb.{i}.q"])
    dr = oracle.Drafter(cfg, W)
    dr.ingest(X)
    probs = []
    dr.backbone(3, probs_out=probs)
    for P in probs:
        np.testing.assert_allclose(P, 1.0 / (7 + cfg.gamma), rtol=0, atol=1e-15)
    Q = np.zeros((cfg.gamma, cfg.d_draft))
    rng = np.random.default_rng(0)
    K, V = rng.normal(size=(9, cfg.d_draft)), rng.normal(size=(9, cfg.d_draft))
    O = oracle.attention(Q, K, V, cfg.n_heads)
    np.testing.assert_allclose(O, np.broadcast_to(V.mean(axis=0), O.shape), rtol=0, atol=1e-14)


def test_single_position_empty_context_is_a_pre_norm_mlp():
    """gamma = 1, L = 0, one head: the only key is the block row itself, so the
    softmax weight is 1 and attention returns W_v n; the layer is
    x + W_o W_v n followed by the gated FFN."""
    cfg = tiny_cfg(gamma=1, n_layers=1, n_heads=1)
    W = syn.make_weights(cfg, seed=8, norm_std=0.2, std=0.3)
    dr = oracle.Drafter(cfg, W)
    w = {k: oracle.to_f64(v) for k, v in W.items()}
    x = w["tok_proj"] @ w["embed"][6] + w["block_pos"][0]
    n = x / np.sqrt(np.mean(x * x) + cfg.eps) * w["bb.0.attn_norm"]
    x = x + w["bb.0.o"] @ (w["bb.0.v"] @ n)
    n2 = x / np.sqrt(np.mean(x * x) + cfg.eps) * w["bb.0.ff_norm"]
    g = w["bb.0.gate"] @ n2
    x = x + w["bb.0.down"] @ (g * scipy.special.expit(g) * (w["bb.0.up"] @ n2))
    y = x / np.sqrt(np.mean(x * x) + cfg.eps) * w["out_norm"]
    np.testing.assert_allclose(dr.backbone(6)[0], y, rtol=0, atol=1e-12)


def test_hand_worked_two_dimensional_drafter():
    """A drafter small enough to evaluate by hand (eps = 0).

    Context row X = [3, 4], W_c = I: P = [3, 4], rms = sqrt(12.5), so
    H_ctx = [3, 4] / sqrt(12.5) = [0.6 sqrt 2, 0.8 sqrt 2] and its mean square is 1.
    W_k = W_v = I, attn_norm = 1: K_c = V_c = H_ctx.
    Anchor 1, E[1] = [1, 0], tok_proj = I, block_pos = 0, mask_emb = [[0, 1]]:
    x = [[1, 0], [0, 1]], normalised rows n = [[sqrt 2, 0], [0, sqrt 2]] = K_b = V_b.
    W_q = 0: uniform attention over 3 keys, O_j = (V_c + n_0 + n_1) / 3 for both j.
    W_o = I, gate = 0 (FFN output 0): x' = x + O.
    out_norm = 1, out_proj rows [1, 0], [0, 1], [1, 1]: U = y out_proj^T.
    w1 = [[1], [2], [3]], w2 = [[0], [0.5], [-1]] (rank 1):
    logits_k = U_k + w2 * w1[prev_k].
    conf.w = [1, 0, 1], conf.b = -1: conf_k = sigmoid(y_k[0] + w1[prev_k] - 1).
    """
    cfg = syn.DrafterConfig(hidden=2, n_taps=1, d_draft=2, n_heads=1, n_layers=1, ff_mult=1, gamma=2,
                            vocab=3, markov_rank=1, eps=0.0, dtype="fp32")
    I2 = np.eye(2, dtype=np.float32)
    z2 = np.zeros((2, 2), np.float32)
    one = np.ones(2, np.float32)
    W = {"bb.0.attn_norm": one, "bb.0.q": z2, "bb.0.k": I2, "bb.0.v": I2, "bb.0.o": I2,
         "bb.0.ff_norm": one, "bb.0.gate": z2, "bb.0.up": I2, "bb.0.down": I2,
         "W_c": I2, "ctx_norm": one, "tok_proj": I2, "mask_emb": np.array([[0, 1]], np.float32),
         "block_pos": z2, "out_norm": one, "out_proj": np.array([[1, 0], [0, 1], [1, 1]], np.float32),
         "markov.w1": np.array([[1], [2], [3]], np.float32),
         "markov.w2": np.array([[0], [0.5], [-1]], np.float32),
         "conf.w": np.array([1, 0, 1], np.float32), "conf.b": np.array([-1], np.float32),
         "embed": np.array([[0, 0], [1, 0], [0, 1]], np.float32)}
    dr = oracle.Drafter(cfg, W)
    dr.ingest(np.array([[3, 4]], np.float32))
    r2 = math.sqrt(2.0)
    Hc = [0.6 * r2, 0.8 * r2]
    K, V = dr.cache(0, 0)
    np.testing.assert_allclose(K[0], Hc, atol=1e-15)
    np.testing.assert_allclose(V[0], Hc, atol=1e-15)
    O = [(Hc[0] + r2) / 3.0, (Hc[1] + r2) / 3.0]
    xs = [[1 + O[0], O[1]], [O[0], 1 + O[1]]]
    ys = []
    for x in xs:
        s = math.sqrt((x[0] ** 2 + x[1] ** 2) / 2.0)
        ys.append([x[0] / s, x[1] / s])
    U = [[y[0], y[1], y[0] + y[1]] for y in ys]
    tok, conf, logits, y, _ = dr.draft(1)
    np.testing.assert_allclose(y, ys, atol=1e-14)
    # k = 0: prev = anchor 1, w1[1] = 2: bias = [0, 1, -2]
    l0 = [U[0][0], U[0][1] + 1.0, U[0][2] - 2.0]
    np.testing.assert_allclose(logits[0], l0, atol=1e-14)
    t0 = int(np.argmax(l0))
    assert tok[0] == t0
    e1 = [1.0, 2.0, 3.0][t0]
    l1 = [U[1][0], U[1][1] + 0.5 * e1, U[1][2] - e1]
    np.testing.assert_allclose(logits[1], l1, atol=1e-14)
    assert tok[1] == int(np.argmax(l1))
    np.testing.assert_allclose(conf[0], 1 / (1 + math.exp(-(ys[0][0] + 2.0 - 1.0))), atol=1e-15)
    np.testing.assert_allclose(conf[1], 1 / (1 + math.exp(-(ys[1][0] + e1 - 1.0))), atol=1e-15)


# --------------------------------------------------------------------------- scalar pieces

def check_gelu_tanh(fn):
    """The tanh form of GELU that MLX calls ``geluApprox`` (``#layer`` of "module-dflash.ts")
    against PyTorch's own tanh-approximate GELU in float64.  The erf form differs from it by
    up to ~5e-4 on [-8, 8], far above this tolerance, so substituting one for the other fails."""
    torch = pytest.importorskip("torch")
    z = np.concatenate([np.linspace(-8, 8, 1601), [-30.0, -1e-3, 1e-3, 30.0]])
    ref = torch.nn.functional.gelu(torch.from_numpy(z), approximate="tanh").numpy()
    np.testing.assert_allclose(fn(z), ref, rtol=1e-12, atol=1e-12)


def test_scalar_functions_against_library_routines():
    z = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(oracle.sigmoid(z), scipy.special.expit(z), rtol=1e-14, atol=1e-300)
    np.testing.assert_allclose(oracle.silu(z), z * scipy.special.expit(z), rtol=1e-14, atol=1e-300)
    # tanh-GELU is within 1e-3 of the exact erf GELU on this range (known approximation error)
    exact = 0.5 * z * (1 + scipy.special.erf(z / math.sqrt(2)))
    assert np.max(np.abs(oracle.gelu_tanh(z) - exact)) < 1e-3
    assert oracle.gelu_tanh(np.array([0.0]))[0] == 0.0
    check_gelu_tanh(oracle.gelu_tanh)
    np.testing.assert_allclose(oracle.softmax(np.array([[0.0, math.log(3.0)]])), [[0.25, 0.75]], atol=1e-15)
    x = np.array([[3.0, 4.0]])
    np.testing.assert_allclose(oracle.rmsnorm(x, np.array([1.0, 2.0]), 0.0),
                               [[3 / math.sqrt(12.5), 8 / math.sqrt(12.5)]], atol=1e-15)


def test_bf16_widening_is_exact():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0001, 0x7F7F, 0x0000, 0x8000], np.uint16)
    vals = oracle.bf16_bits_to_f64(bits)
    assert vals[0] == 1.0 and vals[1] == -1.0
    assert vals[2] == 3.140625
    assert vals[3] == 2.0 ** -133
    assert vals[4] == (2 - 2 ** -7) * 2.0 ** 127
    assert vals[5] == 0.0 and math.copysign(1, vals[6]) == -1


def test_argmax_ties_take_the_lowest_index():
    """Two vocabulary rows with identical out_proj and w2 rows tie exactly; the
    greedy chain must pick the lower index (numpy's first-maximum rule)."""
    cfg = tiny_cfg()
    W = syn.make_weights(cfg, seed=11, std=0.3)
    dr0 = oracle.Drafter(cfg, W)
    dr0.ingest(syn.make_feats(cfg, 4, seed=11))
    t0 = int(dr0.draft(2)[0][0])
    lo = 0 if t0 != 0 else 1
    hi = t0
    if lo > hi:
        lo, hi = hi, lo
    W2 = dict(W)
    W2["out_proj"] = W["out_proj"].copy()
    W2["markov.w2"] = W["markov.w2"].copy()
    W2["out_proj"][lo] = W["out_proj"][t0]
    W2["markov.w2"][lo] = W["markov.w2"][t0]
    W2["out_proj"][hi] = W["out_proj"][t0]
    W2["markov.w2"][hi] = W["markov.w2"][t0]
    dr = oracle.Drafter(cfg, W2)
    dr.ingest(syn.make_feats(cfg, 4, seed=11))
    tok, _, logits, _, _ = dr.draft(2)
    assert logits[0][lo] == logits[0][hi] == logits[0].max()
    assert tok[0] == lo


def test_bad_config_is_rejected():
    with pytest.raises(ValueError):
        oracle.Drafter(tiny_cfg(d_draft=9, n_heads=2), {})


def test_linear_against_loops():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(3, 5)).astype(np.float32)
    W = rng.normal(size=(4, 5)).astype(np.float32)
    out = oracle.linear(x, W)
    for m in range(3):
        for n in range(4):
            assert abs(out[m, n] - sum(float(x[m, k]) * float(W[n, k]) for k in range(5))) < 1e-12
