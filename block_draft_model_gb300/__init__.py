"""Python binding of libdspark, the GB300 DSpark/DFlash block drafter.

Argument marshalling only: every step of ingest and draft runs in the CUDA
kernels of ``libdspark.so`` (see ``include/dspark.h`` for the ABI).  PyTorch
provides device memory and streams.  If the library is missing the import of
``Drafter`` methods fails loudly; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdspark.so")

OK, ERR_INVALID_ARG, ERR_CAPACITY, ERR_CUDA, ERR_UNSUPPORTED, ERR_TIMEOUT, ERR_OOM, ERR_DEVICE = range(8)
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "CAPACITY", 3: "CUDA", 4: "UNSUPPORTED", 5: "TIMEOUT", 6: "OOM",
                7: "DEVICE"}
BF16, FP32 = 0, 1
ACT_SILU, ACT_GELU_TANH = 0, 1

EXPORTED = ["dspark_create", "dspark_destroy", "dspark_ingest_context", "dspark_draft", "dspark_ingest_and_draft",
            "dspark_ingest_context_batched", "dspark_draft_batched", "dspark_ingest_context_host",
            "dspark_draft_host", "dspark_reset", "dspark_context_length", "dspark_check", "dspark_get_cache",
            "dspark_last_error", "dspark_launch_count", "dspark_version", "dspark_profile",
            "dspark_profile_read", "dspark_linear", "dspark_linear_stream_noalloc", "dspark_noalloc_last_error",
            "dspark_noalloc_check", "dspark_set_path",
            "dspark_set_sampling", "dspark_selftest_wait"]


class DsparkError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_taps", ctypes.c_int32), ("d_draft", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("n_layers", ctypes.c_int32), ("ff_mult", ctypes.c_int32),
                ("gamma", ctypes.c_int32), ("vocab", ctypes.c_int32), ("markov_rank", ctypes.c_int32),
                ("eps", ctypes.c_float), ("dtype", ctypes.c_int32), ("act", ctypes.c_int32),
                ("max_ctx", ctypes.c_int32), ("max_seqs", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("qk_norm", ctypes.c_int32), ("rope_theta", ctypes.c_float)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class Weights(ctypes.Structure):
    _fields_ = [("W_c", ctypes.c_void_p), ("ctx_norm", ctypes.c_void_p), ("embed", ctypes.c_void_p),
                ("tok_proj", ctypes.c_void_p), ("mask_emb", ctypes.c_void_p), ("block_pos", ctypes.c_void_p),
                ("attn_norm", _PP), ("wq", _PP), ("wk", _PP), ("wv", _PP), ("wo", _PP), ("ff_norm", _PP),
                ("w_gate", _PP), ("w_up", _PP), ("w_down", _PP), ("out_norm", ctypes.c_void_p),
                ("out_proj", ctypes.c_void_p), ("markov_w1", ctypes.c_void_p), ("markov_w2", ctypes.c_void_p),
                ("conf_w", ctypes.c_void_p), ("conf_b", ctypes.c_void_p), ("q_norm", _PP), ("k_norm", _PP)]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libdspark.so (built by ``build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with block_draft_model_gb300.build()")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sig = {
        "dspark_create": ([ctypes.POINTER(Config), ctypes.POINTER(Weights), vp, ctypes.POINTER(vp)], i32),
        "dspark_destroy": ([vp], None),
        "dspark_ingest_context": ([vp, vp, i32, vp], i32),
        "dspark_draft": ([vp, i32, vp, vp, vp, vp], i32),
        "dspark_ingest_and_draft": ([vp, vp, i32, i32, vp, vp, vp, vp], i32),
        "dspark_ingest_context_batched": ([vp, i32, vp, vp, vp, i32, vp], i32),
        "dspark_draft_batched": ([vp, i32, vp, vp, vp, vp, vp, vp], i32),
        "dspark_ingest_context_host": ([vp, vp, i32, vp], i32),
        "dspark_draft_host": ([vp, i32, vp, vp, vp, vp], i32),
        "dspark_reset": ([vp, i32, vp], i32),
        "dspark_set_sampling": ([vp, ctypes.c_float, i32, ctypes.c_uint64, vp], i32),
        "dspark_set_path": ([vp, i32, i32], i32),
        "dspark_selftest_wait": ([i32, ctypes.POINTER(i32)], i32),
        "dspark_context_length": ([vp, i32, ctypes.POINTER(i32)], i32),
        "dspark_check": ([vp, ctypes.POINTER(i32)], i32),
        "dspark_get_cache": ([vp, i32, i32, ctypes.POINTER(vp), ctypes.POINTER(vp)], i32),
        "dspark_last_error": ([vp], ctypes.c_char_p),
        "dspark_launch_count": ([vp], i64),
        "dspark_version": ([], ctypes.c_char_p),
        "dspark_profile": ([vp, i32], i32),
        "dspark_linear": ([i32, vp, i64, vp, i32, i32, i32, vp, i64, i32, vp], i32),
        "dspark_linear_stream_noalloc": ([vp, i64, vp, i32, i32, i32, vp, i64, vp], i32),
        "dspark_noalloc_last_error": ([], ctypes.c_char_p),
        "dspark_noalloc_check": ([ctypes.POINTER(i32)], i32),
        "dspark_profile_read": ([vp, i32, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_double),
                                 ctypes.POINTER(i64), ctypes.POINTER(i64)], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def build(force: bool = False) -> str:
    """Compile libdspark.so for sm_103a (nvcc); returns its path."""
    from . import buildlib
    return buildlib.build(force=force)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> int:
    import torch
    if stream is None:
        return int(torch.cuda.current_stream().cuda_stream)
    return int(getattr(stream, "cuda_stream", stream))


KERNEL_AUTO, KERNEL_SIMT, KERNEL_STREAM, KERNEL_TC, KERNEL_TC_STREAM, KERNEL_TC_WIDE = 0, 1, 2, 3, 4, 5


def linear(A, W, out, kernel: int = KERNEL_AUTO, stream=None):
    """out[m, n] = sum_k A[m, k] W[n, k] on the GPU (A, W bf16 or float32 CUDA tensors, out float32)."""
    import torch
    lib = load()
    dt = BF16 if A.dtype == torch.bfloat16 else FP32
    M, K = A.shape
    N = W.shape[0]
    st = lib.dspark_linear(dt, _ptr(A), A.stride(0), _ptr(W), M, N, K, _ptr(out), out.stride(0), int(kernel),
                           _stream(stream))
    if st != OK:
        raise DsparkError(st, lib.dspark_last_error(None).decode())


def linear_stream_noalloc(A, W, out, stream=None):
    """out = A W^T (bf16 A [M <= 16, K], W [N, K]; float out) through the entry point that allocates
    no device memory (its scratch is a static device array of the library)."""
    import torch
    lib = load()
    M, K = A.shape
    N = W.shape[0]
    if A.dtype != torch.bfloat16 or W.dtype != torch.bfloat16 or out.dtype != torch.float32:
        raise DsparkError(ERR_INVALID_ARG, "A and W must be bfloat16 and out float32")
    if (W.shape[1] != K or tuple(out.shape) != (M, N) or W.stride(1) != 1 or W.stride(0) != K
            or A.stride(1) != 1 or out.stride(1) != 1):
        raise DsparkError(ERR_INVALID_ARG, "W must be a contiguous [N, K] matrix, A and out row-major [M, K], [M, N]")
    st = lib.dspark_linear_stream_noalloc(_ptr(A), A.stride(0), _ptr(W), M, N, K, _ptr(out), out.stride(0),
                                          _stream(stream))
    if st != OK:
        raise DsparkError(st, lib.dspark_noalloc_last_error().decode())


def noalloc_check() -> int:
    """Read and clear the error word of the allocation-free entry point on the current device
    (synchronous); returns it, 0 when no bounded wait gave up since the last check."""
    lib = load()
    w = ctypes.c_int32(0)
    st = lib.dspark_noalloc_check(ctypes.byref(w))
    if st not in (OK, ERR_DEVICE):
        raise DsparkError(st, lib.dspark_noalloc_last_error().decode())
    return int(w.value)


class _CudaArray:
    """Wraps a device pointer for ``torch.as_tensor`` (``__cuda_array_interface__``)."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


def selftest_wait(which: int) -> int:
    """Run one of the library's bounded device waits on words that nothing completes;
    returns the error word it recorded (DEVERR_TIMEOUT when the wait gave up)."""
    lib = load()
    w = ctypes.c_int32(0)
    st = lib.dspark_selftest_wait(int(which), ctypes.byref(w))
    if st != OK:
        raise DsparkError(st, lib.dspark_last_error(None).decode())
    return int(w.value)


DEVERR_TIMEOUT = 16
PATH_LAYERS, PATH_MARKOV, PATH_NORM_CHAIN, PATH_GRAPHS = range(4)
LAYERS_AUTO, LAYERS_PER_KERNEL, LAYERS_PERSISTENT_MMA, LAYERS_STEP_TC = range(4)


class Drafter:
    """A drafter handle.  ``weights`` maps parameter names (``bb.{i}.q`` ...,
    ``W_c``, ``embed`` ...) to CUDA tensors in ``[out, in]`` layout; matrices
    in bf16 (or float32 for ``dtype=FP32``), norm vectors float32."""

    def __init__(self, *, hidden, n_taps, d_draft, n_heads, n_layers, ff_mult, gamma, vocab, markov_rank,
                 eps=1e-6, dtype=BF16, act=ACT_SILU, max_ctx=4096, max_seqs=1, weights=None, stream=None,
                 n_kv_heads=0, qk_norm=False, rope_theta=0.0):
        self.lib = load()
        self.cfg = Config(hidden, n_taps, d_draft, n_heads, n_layers, ff_mult, gamma, vocab, markov_rank, eps,
                          dtype, act, max_ctx, max_seqs, n_kv_heads, int(bool(qk_norm)), rope_theta)
        self.d_kv = (n_kv_heads or n_heads) * (d_draft // n_heads)
        self.gamma, self.vocab = gamma, vocab
        self._h = ctypes.c_void_p(0)
        w = weights or {}
        L = n_layers

        def arr(fmt):
            a = (ctypes.c_void_p * L)(*[_ptr(w.get(fmt.format(i))) for i in range(L)])
            return ctypes.cast(a, _PP), a

        self._keep = []
        fields = {}
        for key, fmt in (("attn_norm", "bb.{}.attn_norm"), ("wq", "bb.{}.q"), ("wk", "bb.{}.k"), ("wv", "bb.{}.v"),
                         ("wo", "bb.{}.o"), ("ff_norm", "bb.{}.ff_norm"), ("w_gate", "bb.{}.gate"),
                         ("w_up", "bb.{}.up"), ("w_down", "bb.{}.down"), ("q_norm", "bb.{}.q_norm"),
                         ("k_norm", "bb.{}.k_norm")):
            p, a = arr(fmt)
            fields[key] = p
            self._keep.append(a)
        self.w = Weights(_ptr(w.get("W_c")), _ptr(w.get("ctx_norm")), _ptr(w.get("embed")), _ptr(w.get("tok_proj")),
                         _ptr(w.get("mask_emb")), _ptr(w.get("block_pos")), fields["attn_norm"], fields["wq"],
                         fields["wk"], fields["wv"], fields["wo"], fields["ff_norm"], fields["w_gate"],
                         fields["w_up"], fields["w_down"], _ptr(w.get("out_norm")), _ptr(w.get("out_proj")),
                         _ptr(w.get("markov.w1")), _ptr(w.get("markov.w2")), _ptr(w.get("conf.w")),
                         _ptr(w.get("conf.b")), fields["q_norm"], fields["k_norm"])
        self._embed = w.get("embed")   # borrowed by the library: keep it alive
        st = self.lib.dspark_create(ctypes.byref(self.cfg), ctypes.byref(self.w), _stream(stream),
                                    ctypes.byref(self._h))
        if st != OK:
            raise DsparkError(st, self.lib.dspark_last_error(None).decode())

    # -- helpers
    def _check(self, st):
        if st != OK:
            raise DsparkError(st, self.lib.dspark_last_error(self._h).decode())

    def close(self):
        if self._h:
            self.lib.dspark_destroy(self._h)
            self._h = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- the ABI, one method per call
    def ingest_context(self, feats, stream=None):
        self._check(self.lib.dspark_ingest_context(self._h, _ptr(feats), int(feats.shape[0]), _stream(stream)))

    def draft(self, last_token: int, tokens, conf, logits=None, stream=None):
        self._check(self.lib.dspark_draft(self._h, int(last_token), _ptr(tokens), _ptr(conf), _ptr(logits),
                                          _stream(stream)))

    def ingest_context_batched(self, seq_ids, cu_tokens, feats, stream=None):
        self._check(self.lib.dspark_ingest_context_batched(self._h, int(seq_ids.shape[0]), _ptr(seq_ids),
                                                           _ptr(cu_tokens), _ptr(feats), int(feats.shape[0]),
                                                           _stream(stream)))

    def ingest_and_draft(self, feats, last_token: int, tokens, conf, logits=None, stream=None):
        """ingest_context(feats) then draft(last_token, ...) in one call, with the same results: the
        block rows, and layer 0's QKV projection where its norm comes through the block build, run on
        a side stream while the context is ingested."""
        self._check(self.lib.dspark_ingest_and_draft(self._h, _ptr(feats), int(feats.shape[0]), int(last_token),
                                                     _ptr(tokens), _ptr(conf), _ptr(logits), _stream(stream)))

    def draft_batched(self, seq_ids, last_tokens, tokens, conf, logits=None, stream=None):
        self._check(self.lib.dspark_draft_batched(self._h, int(seq_ids.shape[0]), _ptr(seq_ids), _ptr(last_tokens),
                                                  _ptr(tokens), _ptr(conf), _ptr(logits), _stream(stream)))

    def ingest_context_host(self, feats_host, stream=None):
        self._check(self.lib.dspark_ingest_context_host(self._h, _ptr(feats_host), int(feats_host.shape[0]),
                                                        _stream(stream)))

    def draft_host(self, last_token: int, tokens_host, conf_host, logits_host=None, stream=None):
        self._check(self.lib.dspark_draft_host(self._h, int(last_token), _ptr(tokens_host), _ptr(conf_host),
                                               _ptr(logits_host), _stream(stream)))

    def set_sampling(self, temperature: float, top_k: int = 0, seed: int = 0, stream=None):
        """temperature > 0: draw the Markov chain's tokens (top_k candidates, 0 = all) instead of argmax."""
        self._check(self.lib.dspark_set_sampling(self._h, float(temperature), int(top_k), int(seed) & (2**64 - 1),
                                                 _stream(stream)))

    def set_path(self, what: int, value: int):
        """Force one form of a computation (PATH_* / LAYERS_*; 0 = the library's choice)."""
        self._check(self.lib.dspark_set_path(self._h, int(what), int(value)))

    def reset(self, seq_id: int = 0, stream=None):
        self._check(self.lib.dspark_reset(self._h, int(seq_id), _stream(stream)))

    def context_length(self, seq_id: int = 0) -> int:
        out = ctypes.c_int32(0)
        self._check(self.lib.dspark_context_length(self._h, int(seq_id), ctypes.byref(out)))
        return out.value

    def check(self) -> int:
        """Read and clear the device error word; raises DsparkError if it was set."""
        out = ctypes.c_int32(0)
        st = self.lib.dspark_check(self._h, ctypes.byref(out))
        if st not in (OK, ERR_DEVICE):
            self._check(st)
        return out.value

    def cache(self, seq_id: int, layer: int, rows: int):
        """(K, V) views [rows, d_kv] of the library-owned cache of (seq_id, layer)."""
        import torch
        k, v = ctypes.c_void_p(0), ctypes.c_void_p(0)
        self._check(self.lib.dspark_get_cache(self._h, int(seq_id), int(layer), ctypes.byref(k), ctypes.byref(v)))
        d = self.d_kv
        if self.cfg.dtype == FP32:
            mk = lambda p: torch.as_tensor(_CudaArray(p, (rows, d), "<f4"), device="cuda")
        else:
            mk = lambda p: torch.as_tensor(_CudaArray(p, (rows, d), "<i2"), device="cuda").view(torch.bfloat16)
        return mk(k.value), mk(v.value)

    def launch_count(self) -> int:
        return int(self.lib.dspark_launch_count(self._h))

    def profile(self, mask: int):
        """Start CUDA-event timing of the kernel classes in ``mask`` (bit i = the
        i-th class of ``profile_read``; -1 = all; counters cleared), or stop (0)."""
        self._check(self.lib.dspark_profile(self._h, int(mask)))

    def profile_read(self) -> dict:
        """{class: (device ms, timed ranges, kernel launches)} of the recorded ranges."""
        n = 32
        names = (ctypes.c_char_p * n)()
        ms = (ctypes.c_double * n)()
        rng = (ctypes.c_int64 * n)()
        lc = (ctypes.c_int64 * n)()
        k = self.lib.dspark_profile_read(self._h, n, names, ms, rng, lc)
        if k < 0:
            raise DsparkError(ERR_CUDA, "profile_read failed")
        return {names[i].decode(): (ms[i], rng[i], lc[i], i) for i in range(min(k, n))}
