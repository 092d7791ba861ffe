"""MLX-style affine 4-bit linear layer (test infrastructure).

TensorFold README, model list and "What each checkpoint needs": the engine
serves MLX 4-bit checkpoints.  The pages do not spell out that format; this
follows the public description of MLX's affine quantisation:

* codes: uint32 [N][K/8]; word j of row n holds q[n][8j + i] in bits
  [4i, 4i + 4); q is an unsigned integer in [0, 15];
* scales, biases: bf16 [N][K/G], one pair per group of G input features;
* dequantised weight: w[n][k] = scale[n][k // G] * q[n][k] + bias[n][k // G];
* y[r][n] = sum_k w[n][k] * x[r][k].

The oracle is that definition written out: dequantise in fp64, then one fp64
matrix product.
"""

from __future__ import annotations

import numpy as np

from .linear import bf16_to_f64


def unpack_u32_codes(codes_u32: np.ndarray) -> np.ndarray:
    """uint8 [N][K] of the unsigned codes in a uint32 [N][K/8] array."""
    c = np.ascontiguousarray(codes_u32, dtype=np.uint32)
    N, W = c.shape
    q = np.empty((N, W, 8), dtype=np.uint8)
    for i in range(8):
        q[:, :, i] = (c >> np.uint32(4 * i)) & np.uint32(0xF)
    return q.reshape(N, 8 * W)


def affine_w4_linear(codes_u32: np.ndarray, scales_bf16: np.ndarray, biases_bf16: np.ndarray,
                     x_bf16: np.ndarray, group: int, cols=None) -> np.ndarray:
    """fp64 y [R][N] (or [R][len(cols)])."""
    codes_u32 = np.asarray(codes_u32)
    if cols is not None:
        cols = np.asarray(cols, dtype=np.int64)
        codes_u32, scales_bf16, biases_bf16 = codes_u32[cols], np.asarray(scales_bf16)[cols], \
            np.asarray(biases_bf16)[cols]
    q = unpack_u32_codes(codes_u32).astype(np.float64)
    N, K = q.shape
    if K % group or np.asarray(scales_bf16).shape != (N, K // group) or \
            np.asarray(biases_bf16).shape != (N, K // group):
        raise ValueError("shape mismatch")
    s = np.repeat(bf16_to_f64(scales_bf16), group, axis=1)
    b = np.repeat(bf16_to_f64(biases_bf16), group, axis=1)
    w = s * q + b
    x = bf16_to_f64(np.atleast_2d(x_bf16))
    if x.shape[1] != K:
        raise ValueError("x has the wrong width")
    return x @ w.T
