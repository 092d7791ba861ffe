"""Small numeric definitions used by the oracle (test infrastructure).

* ``bf16_round``: round fp64 values to the nearest bfloat16 value, ties to
  even, in one rounding step (bfloat16 = binary32 exponent range, 8
  significant bits).
* ``rms_norm``: x / sqrt(mean(x^2) + eps), gain 1.
* ``silu``: v / (1 + exp(-v)).

The pages do not give the synthetic decoder's normalisation, activation or
rounding points (the decoder itself is a stand-in for the pages' 27B-class
model, not taken from the pages); these are the plain textbook definitions.
"""

from __future__ import annotations

import numpy as np

_MIN_EXP = -126          # smallest normal binary exponent of bfloat16
_MANT_BITS = 7           # stored fraction bits of bfloat16


def bf16_round(v) -> np.ndarray:
    """Nearest bfloat16 value (ties to even) of each finite fp64 value, as fp64."""
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(v)
    nz = v != 0.0
    a = v[nz]
    _, e = np.frexp(a)              # a = m * 2^e with 0.5 <= |m| < 1
    e = e - 1                       # a = m' * 2^e with 1 <= |m'| < 2
    e = np.maximum(e, _MIN_EXP)     # subnormals share the smallest exponent
    ulp = np.ldexp(1.0, e - _MANT_BITS)
    out[nz] = np.rint(a / ulp) * ulp  # scaling by a power of two is exact
    return out


def bf16_bits_of(v) -> np.ndarray:
    """bf16 bit patterns of values that are already bfloat16 values."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)   # exact for bf16 values
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def rms_norm(x, eps: float = 1e-6) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps)


def silu(v) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))
