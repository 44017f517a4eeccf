"""CPU oracle for the DSpark/DFlash block drafter step.

TEST INFRASTRUCTURE ONLY.  This package is the slow, plain fp64 restatement of
what the drafter computes; the CUDA library is checked against it.  Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import it.  It shares no code with the CUDA path and the product never calls
it: there is no CPU fallback.
"""
from .dspark_oracle import (  # noqa: F401
    Drafter,
    attention,
    bf16_bits_to_f64,
    confidence,
    context_features,
    context_kv,
    ffn,
    gelu_tanh,
    head_rmsnorm,
    linear,
    rmsnorm,
    rope,
    sample_candidates,
    sample_token,
    sample_uniform,
    splitmix64,
    sigmoid,
    silu,
    softmax,
    to_f64,
)
