"""Plant plausible mistakes in the oracle (on the CPU) and check that the
brute-force pin notices each of them.  This shows the pins are sharp enough
to catch a dropped term, a wrong operand or a wrong index."""
import numpy as np
import pytest

import oracle
import oracle.dspark_oracle as od
import synthetic as syn

from test_oracle_pins import brute_force_draft, check_gelu_tanh, tiny_cfg


def _no_scale_attention(Q, K, V, n_heads, probs_out=None, n_kv_heads=0):
    g, d = Q.shape
    hd = d // n_heads
    O = np.empty((g, d))
    for h in range(n_heads):
        sl = slice(h * hd, (h + 1) * hd)
        O[:, sl] = od.softmax(Q[:, sl] @ K[:, sl].T) @ V[:, sl]
    return O


def _column_softmax(s):
    z = s - np.max(s, axis=0, keepdims=True)
    e = np.exp(z)
    return e / np.sum(e, axis=0, keepdims=True)


def _swapped_ffn(n2, Wg, Wu, Wd, act="silu"):
    g = n2 @ Wg.T
    u = n2 @ Wu.T
    return (od.silu(u) * g) @ Wd.T


def _unnormed_context_kv(H_ctx, attn_norm, Wk, Wv, eps):
    return H_ctx @ Wk.T, H_ctx @ Wv.T


def _rms_without_weight(x, w, eps):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)



MUTANTS = {
    "attention scale dropped": ("attention", _no_scale_attention),
    "softmax over the wrong axis": ("softmax", _column_softmax),
    "gate and up swapped": ("ffn", _swapped_ffn),
    "context rows not normalised before W_k/W_v": ("context_kv", _unnormed_context_kv),
    "norm weight ignored": ("rmsnorm", _rms_without_weight),
}


def _max_diff(cfg, W, X, anchor):
    dr = oracle.Drafter(cfg, W)
    dr.ingest(X)
    tok, conf, logits, _, _ = dr.draft(anchor)
    btok, bconf, blogits = brute_force_draft(cfg, W, oracle.to_f64(X).tolist(), anchor)
    return max(np.max(np.abs(logits - np.array(blogits))), np.max(np.abs(conf - np.array(bconf))))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_brute_force_pin_catches_planted_mistake(monkeypatch, name):
    cfg = tiny_cfg()
    W = syn.make_weights(cfg, seed=21, norm_std=0.3, std=0.3)
    X = syn.make_feats(cfg, 5, seed=21)
    assert _max_diff(cfg, W, X, 4) < 1e-12
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(od, attr, fn)
    assert _max_diff(cfg, W, X, 4) > 1e-6, name


def test_brute_force_pin_catches_wrong_markov_index(monkeypatch):
    """Feeding the anchor to every chain position instead of the drafted token."""
    cfg = tiny_cfg(gamma=4)
    W = syn.make_weights(cfg, seed=22, norm_std=0.3, std=0.3)
    X = syn.make_feats(cfg, 5, seed=22)
    orig = od.Drafter.markov_step
    anchor = 4

    def mutant(self, U_k, prev):
        return orig(self, U_k, anchor)

    monkeypatch.setattr(od.Drafter, "markov_step", mutant)
    dr = oracle.Drafter(cfg, W)
    dr.ingest(X)
    tok = dr.draft(anchor)[0]
    btok = brute_force_draft(cfg, W, oracle.to_f64(X).tolist(), anchor)[0]
    assert any(t != anchor for t in btok[:-1])      # the chain really moves
    assert _max_diff(cfg, W, X, anchor) > 1e-6


def test_brute_force_pin_catches_transposed_query(monkeypatch):
    cfg = tiny_cfg()
    W = syn.make_weights(cfg, seed=23, norm_std=0.3, std=0.3)
    X = syn.make_feats(cfg, 5, seed=23)
    dr = oracle.Drafter(cfg, W)
    for i in range(cfg.n_layers):
        dr.w[f"bb.{i}.q"] = dr.w[f"bb.{i}.q"].T.copy()
    dr.ingest(X)
    logits = dr.draft(4)[2]
    blogits = brute_force_draft(cfg, W, oracle.to_f64(X).tolist(), 4)[2]
    assert np.max(np.abs(logits - np.array(blogits))) > 1e-6


def _layer_norm(x, w, eps):
    c = x - np.mean(x, axis=-1, keepdims=True)
    return c / np.sqrt(np.mean(c * c, axis=-1, keepdims=True) + eps) * w


def _confidence_without_e(self, y_k, e):
    return od.confidence(y_k, np.zeros_like(e), self.w["conf.w"], self.w["conf.b"][0])


def _block_without_positions(self, anchor):
    cfg, w = self.cfg, self.w
    x = np.empty((cfg.gamma, cfg.d_draft))
    x[0] = w["tok_proj"] @ od.to_f64(self.raw["embed"][anchor])
    for j in range(1, cfg.gamma):
        x[j] = w["mask_emb"][j - 1]
    return x


def _backbone_without_out_norm(self, anchor, seq=0, probs_out=None):
    Ks, Vs = self._cache(seq)
    x = self.block_input(anchor)
    for i in range(self.cfg.n_layers):
        x = self.layer(i, x, Ks[i], Vs[i], probs_out)
    return x


MORE_MUTANTS = {
    "LayerNorm (mean subtracted) instead of RMSNorm": (od, "rmsnorm", _layer_norm),
    "confidence without the previous token's w1 row": (od.Drafter, "confidence", _confidence_without_e),
    "block position rows dropped": (od.Drafter, "block_input", _block_without_positions),
    "out_norm skipped": (od.Drafter, "backbone", _backbone_without_out_norm),
}


@pytest.mark.parametrize("name", sorted(MORE_MUTANTS))
def test_brute_force_pin_catches_more_mistakes(monkeypatch, name):
    cfg = tiny_cfg(gamma=3)
    W = syn.make_weights(cfg, seed=24, norm_std=0.3, std=0.3)
    X = syn.make_feats(cfg, 5, seed=24)
    assert _max_diff(cfg, W, X, 4) < 1e-12
    owner, attr, fn = MORE_MUTANTS[name]
    monkeypatch.setattr(owner, attr, fn)
    assert _max_diff(cfg, W, X, 4) > 1e-6, name


def _gelu_erf(g):
    """The exact (erf) GELU, a plausible stand-in for the tanh form."""
    import scipy.special
    return 0.5 * g * (1.0 + scipy.special.erf(g / np.sqrt(2.0)))


def test_gelu_pin_catches_erf_for_tanh(monkeypatch):
    """The brute force restates the tanh formula, so it cannot tell the two GELU forms
    apart; the library-routine pin must."""
    check_gelu_tanh(od.gelu_tanh)
    monkeypatch.setattr(od, "gelu_tanh", _gelu_erf)
    with pytest.raises(AssertionError):
        check_gelu_tanh(od.gelu_tanh)
