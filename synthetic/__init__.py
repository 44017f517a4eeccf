"""Seeded synthetic inputs for the DSpark/DFlash block drafter.

This module is shared by the CPU oracle, the tests and the benchmark.  It
holds no arithmetic of the drafter itself: it only draws numbers (see
``gen.c`` for the generator's definition) and knows the tensor shapes and the
workload sizes.

Weights follow the drafter's parameter list (``DflashDrafter`` parameter
names, "module-dflash.ts", page "mlx-bun 0.0.7 -> 0.0.9", ``buildNames``) in
the ``[out, in]`` row-major layout that the C-ABI takes.  Values: every
non-norm weight N(0, 0.02), norms 1 (optionally 1 + N(0, norm_std) so that
tests can tell the norm vectors apart), context features and the target's
token embedding N(0, 1).  bf16 tensors are returned as their raw 16-bit
patterns (``numpy.uint16``); each consumer widens them itself.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_gen.so")
_lock = threading.Lock()
_lib_handle = None


def build(force: bool = False) -> str:
    """Compile gen.c into _gen.so (gcc, OpenMP, -O2, no arch flags)."""
    src = os.path.join(_HERE, "gen.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
                               "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _lib():
    global _lib_handle
    with _lock:
        if _lib_handle is None:
            lib = ctypes.CDLL(build())
            u64, i64, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
            vp = ctypes.c_void_p
            lib.synth_normal_f32.argtypes = [u64, u64, i64, dbl, vp]
            lib.synth_normal_bf16.argtypes = [u64, u64, i64, dbl, vp]
            lib.synth_uniform_int.argtypes = [u64, u64, i64, i64, i64, vp]
            lib.synth_words.argtypes = [u64, u64, i64, vp]
            for f in (lib.synth_normal_f32, lib.synth_normal_bf16, lib.synth_uniform_int, lib.synth_words):
                f.restype = None
            _lib_handle = lib
    return _lib_handle


def _n(shape) -> int:
    n = 1
    for s in shape:
        n *= int(s)
    return n


def normal_f32(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    out = np.empty(_n(shape), dtype=np.float32)
    _lib().synth_normal_f32(seed, stream, out.size, std, out.ctypes.data)
    return out.reshape(shape)


def normal_bf16(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    """Raw bf16 bit patterns (uint16) of the RNE-rounded float draws."""
    out = np.empty(_n(shape), dtype=np.uint16)
    _lib().synth_normal_bf16(seed, stream, out.size, std, out.ctypes.data)
    return out.reshape(shape)


def uniform_int(seed: int, stream: int, shape, lo: int, hi: int) -> np.ndarray:
    """Integers uniform on the closed range [lo, hi] (int32)."""
    out = np.empty(_n(shape), dtype=np.int32)
    _lib().synth_uniform_int(seed, stream, out.size, lo, hi, out.ctypes.data)
    return out.reshape(shape)


def words(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _lib().synth_words(seed, stream, n, out.ctypes.data)
    return out


# --------------------------------------------------------------------------- shapes

@dataclasses.dataclass(frozen=True)
class DrafterConfig:
    """Drafter dimensions (``DflashConfig`` + ``TargetDims``, "module-dflash.ts")."""
    hidden: int          # H, target hidden size
    n_taps: int          # m, tapped target layers
    d_draft: int         # d
    n_heads: int
    n_layers: int
    ff_mult: int
    gamma: int           # block size
    vocab: int           # V
    markov_rank: int     # r
    eps: float = 1e-6
    dtype: str = "bf16"  # "bf16" or "fp32": storage type of weights, features and caches
    act: str = "silu"    # "silu" or "gelu_tanh"
    n_kv_heads: int = 0       # K/V heads; 0 = n_heads (fewer: grouped-query attention)
    qk_norm: bool = False     # per-head RMSNorm of Q and K (weights q_norm, k_norm [head_dim] per layer)
    rope_theta: float = 0.0   # > 0: rotary position embedding of Q and K with this base

    @property
    def head_dim(self) -> int:
        return self.d_draft // self.n_heads

    @property
    def kv_heads(self) -> int:
        return self.n_kv_heads or self.n_heads

    @property
    def d_kv(self) -> int:
        return self.kv_heads * self.head_dim

    @property
    def ff(self) -> int:
        return self.ff_mult * self.d_draft

    @property
    def feat_dim(self) -> int:
        return self.n_taps * self.hidden


def param_names(cfg: DrafterConfig) -> list[str]:
    """Parameter order of the drafter (``buildNames``), plus the target's embedding."""
    names = []
    for i in range(cfg.n_layers):
        names += [f"bb.{i}.{n}" for n in ("attn_norm", "q", "k", "v", "o", "ff_norm", "gate", "up", "down")]
    names += ["W_c", "ctx_norm", "tok_proj", "mask_emb", "block_pos", "out_norm", "out_proj",
              "markov.w1", "markov.w2", "conf.w", "conf.b"]
    if cfg.qk_norm:  # after the rest, so that the other parameters keep their streams
        for i in range(cfg.n_layers):
            names += [f"bb.{i}.q_norm", f"bb.{i}.k_norm"]
    return names


def param_shape(cfg: DrafterConfig, name: str) -> tuple:
    d, F, H, V, r, g = cfg.d_draft, cfg.ff, cfg.hidden, cfg.vocab, cfg.markov_rank, cfg.gamma
    if name.startswith("bb."):
        leaf = name.split(".")[2]
        dkv, hd = cfg.d_kv, cfg.head_dim
        return {"attn_norm": (d,), "ff_norm": (d,), "q": (d, d), "k": (dkv, d), "v": (dkv, d), "o": (d, d),
                "gate": (F, d), "up": (F, d), "down": (d, F), "q_norm": (hd,), "k_norm": (hd,)}[leaf]
    return {"W_c": (d, cfg.feat_dim), "ctx_norm": (d,), "tok_proj": (d, H), "mask_emb": (g - 1, d),
            "block_pos": (g, d), "out_norm": (d,), "out_proj": (V, d), "markov.w1": (V, r),
            "markov.w2": (V, r), "conf.w": (d + r,), "conf.b": (1,), "embed": (V, H)}[name]


def is_norm(name: str) -> bool:
    return name.endswith("norm")


STREAM_EMBED = 1000
STREAM_ANCHORS = 1001
STREAM_COUNTS = 1002
STREAM_LENGTHS = 1003
STREAM_FEATS = 1 << 32       # + (step + 1) << 16 | sequence


def make_weights(cfg: DrafterConfig, seed: int = 0, norm_std: float = 0.0, std: float = 0.02,
                 zero: tuple = ()) -> dict:
    """All drafter weights plus ``embed`` ([V, H], N(0, 1)).

    fp32 configs give float32 arrays; bf16 configs give uint16 bit patterns
    (norm vectors are always float32).  Names in ``zero`` are all-zero.
    """
    out = {}
    names = param_names(cfg)
    for sid, name in enumerate(names):
        shape = param_shape(cfg, name)
        if name in zero:
            out[name] = np.zeros(shape, np.float32) if (cfg.dtype == "fp32" or is_norm(name)) \
                else np.zeros(shape, np.uint16)
        elif is_norm(name):
            w = np.ones(shape, np.float32)
            if norm_std > 0:
                w = w + normal_f32(seed, sid, shape, norm_std)
            out[name] = w.astype(np.float32)
        elif cfg.dtype == "fp32":
            out[name] = normal_f32(seed, sid, shape, std)
        else:
            out[name] = normal_bf16(seed, sid, shape, std)
    shape = param_shape(cfg, "embed")
    if "embed" in zero:
        out["embed"] = np.zeros(shape, np.float32 if cfg.dtype == "fp32" else np.uint16)
    else:
        out["embed"] = (normal_f32 if cfg.dtype == "fp32" else normal_bf16)(seed, STREAM_EMBED, shape, 1.0)
    return out


def make_feats(cfg: DrafterConfig, T: int, seed: int = 0, step: int = -1, seq: int = 0) -> np.ndarray:
    """Context features ``[T, m*H]`` ~ N(0, 1) (tap-major on the feature axis).

    ``step = -1`` is the one-shot context of sequence ``seq``; ``step >= 0`` the
    tokens ingested before draft step ``step``.
    """
    assert 0 <= seq < (1 << 16) and -1 <= step < (1 << 15)
    shape = (T, cfg.feat_dim)
    stream = STREAM_FEATS + ((step + 1) << 16) + seq
    return (normal_f32 if cfg.dtype == "fp32" else normal_bf16)(seed, stream, shape, 1.0)


# --------------------------------------------------------------------------- workloads

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    cfg: DrafterConfig
    ctx_len: int = 0                 # one-shot context length (single sequence)
    steps: int = 0                   # draft steps after the one-shot ingest
    new_tokens: tuple = (0, 0)       # per-step ingest, uniform on [lo, hi] (0, 0: none)
    n_seqs: int = 1
    ctx_len_range: tuple = (0, 0)    # ragged one-shot lengths per sequence, uniform on [lo, hi]


TINY = DrafterConfig(hidden=256, n_taps=3, d_draft=128, n_heads=4, n_layers=2, ff_mult=2, gamma=4,
                     vocab=1024, markov_rank=32, dtype="fp32")
MINICPM = DrafterConfig(hidden=2048, n_taps=5, d_draft=2048, n_heads=16, n_layers=5, ff_mult=2, gamma=8,
                        vocab=73448, markov_rank=256)
GEMMA = DrafterConfig(hidden=2560, n_taps=4, d_draft=1024, n_heads=8, n_layers=5, ff_mult=2, gamma=5,
                      vocab=262144, markov_rank=256)

WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", TINY, ctx_len=64, steps=1),
    "minicpm_L1024": Workload("minicpm_L1024", MINICPM, ctx_len=1024, steps=1),
    "gemma_L4096_stream": Workload("gemma_L4096_stream", GEMMA, ctx_len=4096, steps=64, new_tokens=(1, 6)),
    "gemma_L32768_ingest": Workload("gemma_L32768_ingest", GEMMA, ctx_len=32768, steps=16),
    "gemma_batched64": Workload("gemma_batched64", GEMMA, steps=128, new_tokens=(1, 6), n_seqs=64,
                                ctx_len_range=(512, 8192)),
}


def anchors(wl: Workload, seed: int = 0) -> np.ndarray:
    """Anchor (last accepted) token per step and sequence, [steps, n_seqs] in [0, V)."""
    return uniform_int(seed, STREAM_ANCHORS, (max(wl.steps, 1), wl.n_seqs), 0, wl.cfg.vocab - 1)


def step_counts(wl: Workload, seed: int = 0) -> np.ndarray:
    """New context tokens ingested before each draft step, [steps, n_seqs]."""
    lo, hi = wl.new_tokens
    if hi == 0:
        return np.zeros((max(wl.steps, 1), wl.n_seqs), np.int32)
    return uniform_int(seed, STREAM_COUNTS, (wl.steps, wl.n_seqs), lo, hi)


def ctx_lengths(wl: Workload, seed: int = 0) -> np.ndarray:
    """One-shot context length per sequence."""
    lo, hi = wl.ctx_len_range
    if hi == 0:
        return np.full(wl.n_seqs, wl.ctx_len, np.int32)
    return uniform_int(seed, STREAM_LENGTHS, (wl.n_seqs,), lo, hi)
