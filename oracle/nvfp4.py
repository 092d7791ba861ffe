"""NVFP4 linear layer (test infrastructure).

Context Studios, "TensorFold: The engine that makes local LLMs 2-3x faster":
the engine gained NVFP4 checkpoints on the RTX PRO 6000 Blackwell, and the
project reports those checkpoints' top-1 agreement with an fp32 reference.
The pages do not spell the format out; this follows NVIDIA's public
description of NVFP4:

* elements are FP4 E2M1 codes: bit 3 sign, bits 2..1 exponent (bias 1),
  bit 0 mantissa; exponent 0 is subnormal: value = (-1)^s * 0.5 * m, else
  (-1)^s * 2^(e - 1) * (1 + m / 2) -- the magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6;
* every 16 consecutive elements along K share one FP8 E4M3 scale: bit 7
  sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa; exponent 0 is
  subnormal (2^-6 * m / 8), the pattern S.1111.111 is NaN, there is no
  infinity (largest finite value 448);
* one fp32 scale per tensor.
* dequantised weight: w[n][k] = e2m1(c[n][k]) * e4m3(s[n][k // 16]) * global_scale.

Storage read here (the canonical layout of this library's API): codes uint8
[N][K/2], element 2j in the low nibble of byte j and element 2j + 1 in the
high nibble; block scales uint8 [N][K/16] holding E4M3 bit patterns; the
global scale as a Python float (an fp32 value).

The oracle is the definition written out: decode every element and every
scale from its bits, dequantise in fp64 (exact: each product has at most a
few significant bits) and take one fp64 matrix product with the bf16
activations.
"""

from __future__ import annotations

import math

import numpy as np

from .linear import bf16_to_f64

BLOCK = 16


def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code."""
    code = int(code) & 0xF
    s, e, m = code >> 3, (code >> 1) & 3, code & 1
    mag = 0.5 * m if e == 0 else math.ldexp(1.0 + 0.5 * m, e - 1)
    return -mag if s else mag


def e4m3_value(byte: int) -> float:
    """Value of an 8-bit E4M3 (FN) pattern; NaN for S.1111.111."""
    byte = int(byte) & 0xFF
    s, e, m = byte >> 7, (byte >> 3) & 0xF, byte & 7
    if e == 15 and m == 7:
        return math.nan
    mag = math.ldexp(m / 8.0, -6) if e == 0 else math.ldexp(1.0 + m / 8.0, e - 7)
    return -mag if s else mag


_E2M1 = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
_E4M3 = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


def unpack_codes(codes_u8: np.ndarray) -> np.ndarray:
    """uint8 [N][K] of the 4-bit codes in a canonical uint8 [N][K/2] array."""
    b = np.ascontiguousarray(codes_u8, dtype=np.uint8)
    out = np.empty((b.shape[0], 2 * b.shape[1]), dtype=np.uint8)
    out[:, 0::2] = b & 0xF
    out[:, 1::2] = b >> 4
    return out


def dequantize(codes_u8: np.ndarray, scales_u8: np.ndarray, global_scale: float) -> np.ndarray:
    """fp64 weights [N][K]."""
    c = unpack_codes(codes_u8)
    N, K = c.shape
    s = np.asarray(scales_u8, dtype=np.uint8)
    if K % BLOCK or s.shape != (N, K // BLOCK):
        raise ValueError("shape mismatch")
    scale = np.repeat(_E4M3[s], BLOCK, axis=1)
    if not np.all(np.isfinite(scale)):
        raise ValueError("NaN block scale")
    return _E2M1[c] * scale * float(np.float32(global_scale))


def nvfp4_linear(codes_u8: np.ndarray, scales_u8: np.ndarray, global_scale: float, x_bf16: np.ndarray,
                 cols=None) -> np.ndarray:
    """fp64 y [R][N] (or [R][len(cols)]) = x @ dequantize(...)^T."""
    codes_u8 = np.asarray(codes_u8)
    scales_u8 = np.asarray(scales_u8)
    if cols is not None:
        cols = np.asarray(cols, dtype=np.int64)
        codes_u8, scales_u8 = codes_u8[cols], scales_u8[cols]
    w = dequantize(codes_u8, scales_u8, global_scale)
    x = bf16_to_f64(np.atleast_2d(x_bf16))
    if x.shape[1] != w.shape[1]:
        raise ValueError("x has the wrong width")
    return x @ w.T
