"""ctypes front-end of the C W4 linear oracle (test infrastructure).

TensorFold README, "What each checkpoint needs": 4-bit weights quantised in
groups (64 for the dense model, 32 for the MoE model).  The scheme is read
as symmetric: code in [-8, 7] times one fp16 scale per group.  The C code
forms each group's integer-weighted partial sum in fp64 and adds
``scale * partial`` group by group in ascending order.
"""

from __future__ import annotations

import ctypes
import numpy as np

from .build import build

_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.oracle_w4_linear.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, P, ctypes.c_int, P]
        lib.oracle_w4_linear.restype = None
        lib.oracle_unpack_codes.argtypes = [P, ctypes.c_int, ctypes.c_int, P]
        lib.oracle_half_array.argtypes = [P, ctypes.c_int64, P]
        lib.oracle_bf16_array.argtypes = [P, ctypes.c_int64, P]
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def w4_linear(codes: np.ndarray, scales: np.ndarray, x_bf16: np.ndarray, group: int,
              cols=None) -> np.ndarray:
    """fp64 ``y[R][N]`` (or ``y[R][len(cols)]``) of the W4 linear layer.

    codes  uint8 [N][K/2] canonical packed codes
    scales uint16 [N][K/group] fp16 bits
    x_bf16 uint16 [R][K] bf16 bits
    """
    lib = _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    N, K2 = codes.shape
    K = 2 * K2
    R = x.shape[0]
    if x.shape[1] != K or scales.shape != (N, K // group) or K % group:
        raise ValueError("shape mismatch")
    if cols is None:
        ncols, cptr = N, None
    else:
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        if cols.size and (cols.min() < 0 or cols.max() >= N):
            raise ValueError("column out of range")
        ncols, cptr = cols.size, _ptr(cols)
    y = np.empty((R, ncols), dtype=np.float64)
    lib.oracle_w4_linear(_ptr(codes), _ptr(scales), _ptr(x), R, K, N, group, cptr, ncols, _ptr(y))
    return y


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    lib = _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    N, K2 = codes.shape
    out = np.empty((N, 2 * K2), dtype=np.int8)
    lib.oracle_unpack_codes(_ptr(codes), 2 * K2, N, _ptr(out))
    return out


def half_to_f64(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib.oracle_half_array(_ptr(b), b.size, _ptr(out))
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib.oracle_bf16_array(_ptr(b), b.size, _ptr(out))
    return out


def num_threads() -> int:
    return int(_load().oracle_num_threads())
