"""Plain fp64 CPU oracle of the DSpark/DFlash block-drafter step.

TEST INFRASTRUCTURE ONLY (see the package docstring): no product code imports
this module.

Sources, by page and section:
  * "module-dflash.ts" (page "mlx-bun 0.0.7 -> 0.0.9"; a DFlash drafter after
    the DSpark paper section 3.1, Eq 2-3): header comment (Eq 2, Eq 3),
    ``#buildContext``, ``#buildBlock``, ``#maskBias``, ``#layer``,
    ``#backbone``, ``#baseLogits``, ``#markov``, ``#confidence``,
    ``forwardInfer``.  This page is the authority on the arithmetic.
  * "src/dspark-runtime.js" (page "minicpm5-2b-webgpu"): ``updateContext``
    (the context K/V is computed once per context token and stored in a
    per-layer cache) and ``propose`` (the draft step, with the Markov chain
    kept greedy and sequential).

Every value is computed in float64 from the exact values handed to the GPU
(bf16 bit patterns are widened exactly).  Nothing is blocked, fused or
reordered beyond what the definitions state; numpy's matmul is the only
library primitive used for the contractions.

Readings where the pages are silent or disagree (each is listed, with its
reason, in the design notes of the repository):
  R1 out_proj maps d -> V directly (one [V, d] matrix): the composed head.
  R2 FFN activation: SiLU(gate) * up by default; tanh-GELU as an option.
  R3 RMSNorm(x, w) = x / sqrt(mean(x^2) + eps) * w, eps = 1e-6.
  R4 the context rows and the block rows use the same attn_norm of layer i.
  R5 no positional encoding besides block_pos; no QK-norm.
  R6 nothing is masked inside [context ++ block] for one sequence.
  R7 block position k yields draft token k; prev_0 is the anchor token, and
     later positions use the previously drafted token (greedy).
  R8 argmax ties resolve to the lowest index.
  R9 conf_k = sigmoid(conf_w . [y_k ; w1[prev_k]] + conf_b), y_k after out_norm.
  R10 sampling instead of argmax (both pages name a temperature, a top-k and a
     seeded key stream, "module-dflash.ts" ``forwardInfer`` / "src/dspark-
     runtime.js" ``propose``, but define none of them): with temperature t > 0
     the candidates are the top_k largest logits (ties to the lower index; all
     V when top_k = 0), and the token is drawn from softmax(logits / t) over
     them by the Gumbel-max rule, argmax_v (l_v / t + g_v), g_v = -ln(-ln u_v).
     u_v comes from the counter-based SplitMix64 generator (Steele, Lea and
     Flood, 2014): the (c + 1)-th output of the stream seeded with `seed`, for
     the counter c = slot * 2^48 + draw * 2^24 + v, top 24 bits, centred:
     u = (floor(z / 2^40) + 0.5) / 2^24.  `draw` numbers the tokens drawn for
     one sequence slot since the sampler was set (gamma per draft call), taken
     modulo 2^24 so that the three fields of c never overlap (v < 2^24).
  R11 the variant of "src/dspark-runtime.js" (kernels ``noiseNormRope`` for the
     block rows and ``contextNormRope`` for the context rows, ``qNorm`` /
     ``kNorm`` bindings, K/V widths KV != H): grouped-query attention with
     n_kv_heads K/V heads, query head h reading K/V head h // (n_heads /
     n_kv_heads); optional per-head RMSNorm of Q and K (weight [head_dim]
     shared by the heads, the same eps) followed by rotary embedding in the
     rotate-half layout, entries e and e + hd/2 turned by pos * theta^(-2e/hd);
     V is neither normalised nor rotated.  Positions: context row t of a
     sequence at t, block row j at L + j (L = context length), so the block
     continues the context.
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------- values

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns: the pattern is the top half of a float32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(a: np.ndarray) -> np.ndarray:
    """float32 arrays widen as they are; uint16 arrays are bf16 bit patterns."""
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------- primitives

def linear(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """The contraction of every projection (MLX ``ops.matmul(x, W)`` with W stored
    [out, in] here): x W^T in float64."""
    return to_f64(x) @ to_f64(W).T


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """MLX ``rmsNorm(x, w, eps)`` as used by ``#buildContext`` and ``#layer``:
    each row divided by the root of (its mean square + eps), times w (R3)."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def softmax(s: np.ndarray) -> np.ndarray:
    """Row softmax, written with the row maximum subtracted (exact in real arithmetic)."""
    z = s - np.max(s, axis=-1, keepdims=True)
    e = np.exp(z)
    return e / np.sum(e, axis=-1, keepdims=True)


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def silu(g):
    """SiLU(g) = g * sigmoid(g) ("src/dspark-runtime.js", ``silu`` kernel in ``propose``)."""
    return g * sigmoid(g)


def gelu_tanh(g):
    """Tanh-approximated GELU (MLX ``geluApprox`` in ``#layer``):
    0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3)))."""
    return 0.5 * g * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (g + 0.044715 * g ** 3)))


# --------------------------------------------------------------------------- Eq 2 / Eq 3

def context_features(X: np.ndarray, W_c: np.ndarray, ctx_norm: np.ndarray, eps: float) -> np.ndarray:
    """Eq 2, ``#buildContext``: H_ctx = RMSNorm(W_c [H^l1; ...; H^lm]) * ctx_norm.

    X: [T, m*H] (the m tapped hidden states concatenated on the feature axis),
    W_c: [d, m*H].  Returns H_ctx [T, d]."""
    P = X @ W_c.T
    return rmsnorm(P, ctx_norm, eps)


def context_kv(H_ctx: np.ndarray, attn_norm: np.ndarray, Wk: np.ndarray, Wv: np.ndarray, eps: float):
    """Eq 3, context half of ``#layer``: the context rows are normalised with the
    layer's attn_norm (the same norm as the block, R4) and projected by the
    layer's own W^K, W^V.  Row-wise, hence cacheable per token
    ("src/dspark-runtime.js", ``updateContext``)."""
    n = rmsnorm(H_ctx, attn_norm, eps)
    return n @ Wk.T, n @ Wv.T


def attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray, n_heads: int, probs_out: list | None = None,
              n_kv_heads: int = 0):
    """Scaled dot-product attention of ``#layer``: per head, softmax(Q K^T / sqrt(hd)) V
    over every key row (no mask, R6).  Q: [g, d]; K, V: [n, d_kv] (context first,
    then block); query head h reads K/V head h // (n_heads / n_kv_heads) (R11;
    n_kv_heads = 0: one K/V head per query head).  Returns O [g, d] with heads
    concatenated."""
    g, d = Q.shape
    hd = d // n_heads
    group = n_heads // (n_kv_heads or n_heads)
    O = np.empty((g, d), dtype=np.float64)
    for h in range(n_heads):
        sl = slice(h * hd, (h + 1) * hd)
        kv = slice((h // group) * hd, (h // group + 1) * hd)
        S = (Q[:, sl] @ K[:, kv].T) * (hd ** -0.5)
        P = softmax(S)
        if probs_out is not None:
            probs_out.append(P)
        O[:, sl] = P @ V[:, kv]
    return O


def head_rmsnorm(x: np.ndarray, w: np.ndarray, n_heads: int, eps: float) -> np.ndarray:
    """R11: RMSNorm of every head's slice of the rows of x, weight w [head_dim]."""
    rows, width = x.shape
    hd = width // n_heads
    return rmsnorm(x.reshape(rows, n_heads, hd), w, eps).reshape(rows, width)


def rope(x: np.ndarray, positions: np.ndarray, n_heads: int, theta: float) -> np.ndarray:
    """R11: rotary embedding, rotate-half layout: in every head, entries e and
    e + hd/2 (e < hd/2) are turned by the angle pos * theta^(-2e/hd)."""
    rows, width = x.shape
    hd = width // n_heads
    half = hd // 2
    ang = np.asarray(positions, np.float64)[:, None] * theta ** (-2.0 * np.arange(half) / hd)[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    xh = x.reshape(rows, n_heads, hd)
    a, b = xh[..., :half], xh[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1).reshape(rows, width)


def ffn(n2: np.ndarray, Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray, act: str = "silu") -> np.ndarray:
    """Gated FFN of ``#layer``: (act(n2 Wg^T) * (n2 Wu^T)) Wd^T (R2)."""
    g = n2 @ Wg.T
    u = n2 @ Wu.T
    a = silu(g) if act == "silu" else gelu_tanh(g)
    return (a * u) @ Wd.T


# --------------------------------------------------------------------------- sampling (R10)

SPLITMIX_GAMMA = np.uint64(0x9E3779B97F4A7C15)


def splitmix64(counter: np.ndarray, seed: int) -> np.ndarray:
    """Output number counter + 1 of the SplitMix64 stream that starts at `seed`
    (state advanced by the golden-ratio increment, then the two xor-shift-
    multiply rounds and a final xor-shift), for an array of counters."""
    c = np.asarray(counter, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + (c + np.uint64(1)) * SPLITMIX_GAMMA
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def sample_uniform(seed: int, slot: int, draw: int, v: np.ndarray) -> np.ndarray:
    """u in (0, 1) for vocabulary entries v of draw `draw` of sequence `slot` (R10)."""
    c = ((np.uint64(slot) << np.uint64(48)) | (np.uint64(draw % (1 << 24)) << np.uint64(24))
         | np.asarray(v, dtype=np.uint64))
    return ((splitmix64(c, seed) >> np.uint64(40)).astype(np.float64) + 0.5) / float(1 << 24)


def sample_candidates(logits: np.ndarray, top_k: int) -> np.ndarray:
    """Indices of the top_k largest logits, larger first, ties to the lower index; all when top_k = 0."""
    V = logits.shape[0]
    if top_k <= 0 or top_k >= V:
        return np.arange(V)
    order = np.lexsort((np.arange(V), -logits))
    return order[:top_k]


def sample_token(logits: np.ndarray, temperature: float, top_k: int, seed: int, slot: int, draw: int,
                 keys_out: list | None = None) -> int:
    """R10: argmax over the candidates of logits / t + Gumbel noise (ties to the lower index)."""
    cand = np.sort(sample_candidates(logits, top_k))
    g = -np.log(-np.log(sample_uniform(seed, slot, draw, cand)))
    z = logits[cand] / temperature + g
    if keys_out is not None:
        keys_out.append((cand, z))
    return int(cand[int(np.argmax(z))])


def confidence(y_k: np.ndarray, e: np.ndarray, conf_w: np.ndarray, conf_b: float) -> float:
    """``#confidence``: sigmoid([y_k ; e] . conf_w + conf_b) (R9)."""
    z = float(np.concatenate([y_k, e]) @ conf_w) + float(conf_b)
    return float(sigmoid(z))


# --------------------------------------------------------------------------- drafter

class Drafter:
    """The drafter with per-sequence, per-layer context K/V caches.

    ``weights`` maps the parameter names of ``buildNames`` (plus ``embed``, the
    target's token embedding [V, H]) to arrays in ``[out, in]`` layout: float32
    values or bf16 bit patterns (uint16).
    """

    def __init__(self, cfg, weights: dict):
        self.cfg = cfg
        d = cfg.d_draft
        if d % cfg.n_heads != 0:
            raise ValueError(f"d_draft {d} not divisible by n_heads {cfg.n_heads}")
        if cfg.n_heads % cfg.kv_heads != 0:
            raise ValueError(f"n_heads {cfg.n_heads} not a multiple of n_kv_heads {cfg.kv_heads}")
        if cfg.rope_theta > 0 and cfg.head_dim % 2 != 0:
            raise ValueError("rotary embedding needs an even head_dim")
        self.raw = weights
        w = {}
        for name, arr in weights.items():
            if name in ("embed", "markov.w1"):
                continue                     # row-gathered on use
            w[name] = to_f64(arr)
        self.w = w
        self.seqs: dict[int, list] = {}      # seq -> [ [K_i], [V_i] ] per layer, lists of row blocks
        self.pos_offset = 0                  # added to every position of R11 (a pin shifts it)

    # ------------------------------------------------------------------ ingest
    def _cache(self, seq: int):
        if seq not in self.seqs:
            dkv = self.cfg.d_kv
            self.seqs[seq] = [[np.zeros((0, dkv)) for _ in range(self.cfg.n_layers)],
                              [np.zeros((0, dkv)) for _ in range(self.cfg.n_layers)]]
        return self.seqs[seq]

    def reset(self, seq: int = 0):
        self.seqs.pop(seq, None)

    def context_length(self, seq: int = 0) -> int:
        c = self.seqs.get(seq)
        return 0 if c is None else c[0][0].shape[0]

    def ingest(self, X: np.ndarray, seq: int = 0, chunk: int = 2048):
        """Eq 2 then Eq 3 for T new context rows, appended to the caches of ``seq``."""
        cfg, w = self.cfg, self.w
        L0 = self.context_length(seq)
        Ks, Vs = self._cache(seq)
        T = X.shape[0]
        newK = [[] for _ in range(cfg.n_layers)]
        newV = [[] for _ in range(cfg.n_layers)]
        for t0 in range(0, T, chunk):
            Xc = to_f64(X[t0:t0 + chunk])
            Hc = context_features(Xc, w["W_c"], w["ctx_norm"], cfg.eps)
            pos = L0 + t0 + np.arange(Hc.shape[0])
            for i in range(cfg.n_layers):
                k, v = context_kv(Hc, w[f"bb.{i}.attn_norm"], w[f"bb.{i}.k"], w[f"bb.{i}.v"], cfg.eps)
                k = self.qk_transform(k, i, "k", pos, cfg.kv_heads)
                newK[i].append(k)
                newV[i].append(v)
        for i in range(cfg.n_layers):
            Ks[i] = np.concatenate([Ks[i]] + newK[i], axis=0)
            Vs[i] = np.concatenate([Vs[i]] + newV[i], axis=0)

    def qk_transform(self, x: np.ndarray, layer: int, which: str, positions: np.ndarray, n_heads: int):
        """R11 on Q or K rows: per-head RMSNorm (if configured), then rotary
        embedding at `positions` (if configured); identity otherwise."""
        cfg = self.cfg
        if cfg.qk_norm:
            x = head_rmsnorm(x, self.w[f"bb.{layer}.{which}_norm"], n_heads, cfg.eps)
        if cfg.rope_theta > 0:
            x = rope(x, np.asarray(positions) + self.pos_offset, n_heads, cfg.rope_theta)
        return x

    def cache(self, seq: int, layer: int):
        Ks, Vs = self._cache(seq)
        return Ks[layer], Vs[layer]

    # ------------------------------------------------------------------ draft
    def block_input(self, anchor: int) -> np.ndarray:
        """``#buildBlock``: x_0 = tok_proj E[anchor] + block_pos[0];
        x_j = mask_emb[j-1] + block_pos[j] for j = 1..gamma-1."""
        cfg, w = self.cfg, self.w
        x = np.empty((cfg.gamma, cfg.d_draft))
        e_anchor = to_f64(self.raw["embed"][anchor])
        x[0] = w["tok_proj"] @ e_anchor + w["block_pos"][0]
        for j in range(1, cfg.gamma):
            x[j] = w["mask_emb"][j - 1] + w["block_pos"][j]
        return x

    def layer(self, i: int, x: np.ndarray, Kc: np.ndarray, Vc: np.ndarray, probs_out: list | None = None):
        """``#layer`` i: pre-norm attention of the block over [context ++ block],
        residual, then pre-norm gated FFN, residual."""
        cfg, w = self.cfg, self.w
        n = rmsnorm(x, w[f"bb.{i}.attn_norm"], cfg.eps)
        Q = n @ w[f"bb.{i}.q"].T
        Kb = n @ w[f"bb.{i}.k"].T
        Vb = n @ w[f"bb.{i}.v"].T
        pos = Kc.shape[0] + np.arange(cfg.gamma)      # R11: the block continues the context
        Q = self.qk_transform(Q, i, "q", pos, cfg.n_heads)
        Kb = self.qk_transform(Kb, i, "k", pos, cfg.kv_heads)
        K = np.concatenate([Kc, Kb], axis=0)
        V = np.concatenate([Vc, Vb], axis=0)
        O = attention(Q, K, V, cfg.n_heads, probs_out, cfg.kv_heads)
        x = x + O @ w[f"bb.{i}.o"].T
        n2 = rmsnorm(x, w[f"bb.{i}.ff_norm"], cfg.eps)
        return x + ffn(n2, w[f"bb.{i}.gate"], w[f"bb.{i}.up"], w[f"bb.{i}.down"], cfg.act)

    def backbone(self, anchor: int, seq: int = 0, probs_out: list | None = None) -> np.ndarray:
        """``#backbone`` on the cached context: block, every layer, out_norm -> y [gamma, d]."""
        Ks, Vs = self._cache(seq)
        x = self.block_input(anchor)
        for i in range(self.cfg.n_layers):
            x = self.layer(i, x, Ks[i], Vs[i], probs_out)
        return rmsnorm(x, self.w["out_norm"], self.cfg.eps)

    def base_logits(self, y: np.ndarray) -> np.ndarray:
        """``#baseLogits`` under R1: U = y out_proj^T, [gamma, V]."""
        return y @ self.w["out_proj"].T

    def markov_step(self, U_k: np.ndarray, prev: int):
        """Logits of one block position given the previous token: (logits, e)."""
        e = to_f64(self.raw["markov.w1"][prev])
        return U_k + self.w["markov.w2"] @ e, e

    def confidence(self, y_k: np.ndarray, e: np.ndarray) -> float:
        return confidence(y_k, e, self.w["conf.w"], self.w["conf.b"][0])

    def draft(self, anchor: int, seq: int = 0, sample: tuple | None = None):
        """``forwardInfer``: the parallel backbone once, then the sequential Markov
        chain, greedy (R8) or, with sample = (temperature, top_k, seed, draw0),
        drawn by R10 with draw number draw0 + k at position k for slot `seq`.
        Returns (tokens [gamma] int64, conf [gamma], logits [gamma, V],
        y [gamma, d], U [gamma, V])."""
        cfg = self.cfg
        y = self.backbone(anchor, seq)
        U = self.base_logits(y)
        tokens = np.empty(cfg.gamma, np.int64)
        conf = np.empty(cfg.gamma)
        logits = np.empty((cfg.gamma, cfg.vocab))
        prev = int(anchor)
        for k in range(cfg.gamma):
            lk, e = self.markov_step(U[k], prev)
            if sample is not None and sample[0] > 0:
                t, top_k, seed, draw0 = sample
                tok = sample_token(lk, t, top_k, seed, seq, draw0 + k)
            else:
                tok = int(np.argmax(lk))       # R8: first maximum
            logits[k] = lk
            conf[k] = self.confidence(y[k], e)
            tokens[k] = tok
            prev = tok
        return tokens, conf, logits, y, U
