"""Host-side helpers shared by the tests: moving synthetic inputs to the GPU,
building the library handle, and checking a drafted block against the oracle.

The oracle decides what is correct: where the greedy chain meets a near-tie
(two tokens within the tolerance of the maximum), every token within the
tolerance is a correct draft, and the chain branches.  ``valid_paths``
enumerates the branches from the oracle alone; the GPU's block must be one of
them, and its logits and confidences are compared with that branch's values.
"""
from __future__ import annotations

import numpy as np

import oracle
import synthetic as syn

# parity tolerances: max|dlogit| <= REL * max|logit| (bf16 weights and caches; fp32 drafter)
REL_BF16 = 2e-2
REL_FP32 = 1e-4


def rel_tol(cfg) -> float:
    return REL_FP32 if cfg.dtype == "fp32" else REL_BF16


def to_torch(a: np.ndarray, device="cuda"):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def weights_to_device(W: dict, device="cuda") -> dict:
    return {k: to_torch(v, device) for k, v in W.items()}


def make_gpu_drafter(cfg, Wd: dict, max_ctx: int, max_seqs: int = 1):
    import block_draft_model_gb300 as bdm
    return bdm.Drafter(hidden=cfg.hidden, n_taps=cfg.n_taps, d_draft=cfg.d_draft, n_heads=cfg.n_heads,
                       n_layers=cfg.n_layers, ff_mult=cfg.ff_mult, gamma=cfg.gamma, vocab=cfg.vocab,
                       markov_rank=cfg.markov_rank, eps=cfg.eps, dtype=bdm.FP32 if cfg.dtype == "fp32" else bdm.BF16,
                       act=bdm.ACT_GELU_TANH if cfg.act == "gelu_tanh" else bdm.ACT_SILU, max_ctx=max_ctx,
                       max_seqs=max_seqs, weights=Wd, n_kv_heads=cfg.n_kv_heads, qk_norm=cfg.qk_norm,
                       rope_theta=cfg.rope_theta)


def tensor_to_f64(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return oracle.bf16_bits_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.double().cpu().numpy()


def valid_paths(dr: oracle.Drafter, y: np.ndarray, U: np.ndarray, anchor: int, rel: float, max_paths: int = 256):
    """Every greedy chain the oracle accepts: at each position, the tokens whose
    logit is within rel*max|logit| of the maximum.  Returns a list of
    (tokens, logits [gamma, V], conf [gamma])."""
    gamma = U.shape[0]
    out = []

    def rec(k, prev, toks, lgs, cfs):
        if len(out) > max_paths:
            return
        if k == gamma:
            out.append((list(toks), np.array(lgs), np.array(cfs)))
            return
        lk, e = dr.markov_step(U[k], prev)
        tol = rel * np.max(np.abs(lk))
        cand = np.flatnonzero(lk >= np.max(lk) - tol)
        c = dr.confidence(y[k], e)
        for t in cand:
            rec(k + 1, int(t), toks + [int(t)], lgs + [lk], cfs + [c])

    rec(0, int(anchor), [], [], [])
    assert len(out) <= max_paths, "too many near-ties to enumerate"
    return out


def check_block(dr: oracle.Drafter, seq: int, anchor: int, tokens, conf, logits=None, rel=REL_BF16,
                label=""):
    """Compare one drafted block (tokens [gamma], conf [gamma], logits [gamma, V] or None)
    with the oracle's draft of (seq, anchor)."""
    y = dr.backbone(anchor, seq)
    U = dr.base_logits(y)
    paths = valid_paths(dr, y, U, anchor, rel)
    toks = [int(t) for t in tokens]
    match = [p for p in paths if p[0] == toks]
    assert match, f"{label}: GPU tokens {toks} not among the oracle's valid chains {[p[0] for p in paths][:8]}"
    _, lg, cf = match[0]
    # the greedy (lowest-index, exact-max) chain must be the first path when it is unique
    greedy = dr.draft(anchor, seq)[0].tolist()
    if len(paths) == 1:
        assert toks == greedy, f"{label}: {toks} vs greedy {greedy}"
    np.testing.assert_allclose(np.asarray(conf, np.float64), cf, rtol=0, atol=rel, err_msg=f"{label}: conf")
    if logits is not None:
        L = np.asarray(logits, np.float64)
        for k in range(lg.shape[0]):
            tol = rel * np.max(np.abs(lg[k]))
            err = np.max(np.abs(L[k] - lg[k]))
            assert err <= tol, f"{label}: logits row {k}: max|d| {err:.3e} > {tol:.3e}"
    return len(paths)


def check_cache(dr: oracle.Drafter, gdr, cfg, seq: int, rows, rel=None, label=""):
    """Compare cache rows (all layers) of the GPU handle with the oracle's."""
    rel = rel if rel is not None else rel_tol(cfg)
    n = dr.context_length(seq)
    rows = np.asarray(rows)
    assert rows.max(initial=-1) < n
    for i in range(cfg.n_layers):
        K, V = dr.cache(seq, i)
        gk, gv = gdr.cache(seq, i, n)
        gk = tensor_to_f64(gk)[rows]
        gv = tensor_to_f64(gv)[rows]
        for name, a, b in (("K", gk, K[rows]), ("V", gv, V[rows])):
            tol = rel * np.max(np.abs(b))
            err = np.max(np.abs(a - b)) if a.size else 0.0
            assert err <= tol, f"{label}: layer {i} {name}: max|d| {err:.3e} > {tol:.3e}"
