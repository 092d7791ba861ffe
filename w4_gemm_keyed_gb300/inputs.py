"""Seeded synthetic inputs for the verify pass.

This module only draws numbers.  It holds none of the method's arithmetic
(no dequantisation, no matvec, no hashing, no sampling), so the CUDA path
and the CPU oracle can both be fed from it without sharing any code that
computes a result.

Value distributions follow the workloads of the TensorFold pages (page
"git.imzlh.top/EugeneClaw/TensorFold", section "What each checkpoint
needs": 4-bit weights in groups of 64 for the 27B-class dense model and
groups of 32 for the MoE model), with the concrete recipe fixed here:

* int4 codes uniform in [-8, 7], stored in the canonical packed layout
  ``codes[N][K/2]`` (uint8; low nibble = even k; two's-complement nibble);
* fp16 scales ``|N(0, 0.02)| + 1e-3``, stored as raw fp16 bits
  ``scales[N][K/G]`` (uint16);
* bf16 activations ``N(0, 1)`` stored as raw bf16 bits (uint16), rounded
  from float32 to nearest-even;
* 64-bit sampling seeds, int64 positions, int32 draft tokens.

All generators take a ``numpy.random.Generator`` so every caller controls
the seed.  Bit patterns (not torch dtypes) are returned so that neither
side depends on a framework's conversion routines.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "rng_for",
    "bf16_bits_from_f32",
    "bf16_normal",
    "w4_weights",
    "mlx_affine_weights",
    "uniform_codes_packed",
    "fp16_scales",
    "logits_normal",
    "seeds_u64",
    "positions",
    "noisy_drafts",
    "router_logits",
    "CONFIGS",
]


def rng_for(*key: int) -> np.random.Generator:
    """A PCG64 generator keyed by a tuple of non-negative integers."""
    return np.random.default_rng(np.random.SeedSequence(list(key)))


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16 (nearest, ties to even); return uint16 bits.

    Only used to *produce* bf16 inputs; the oracle and the kernels read the
    resulting bit patterns with their own decoders.
    """
    f = np.ascontiguousarray(a, dtype=np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = (bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return rounded.astype(np.uint16)


def bf16_normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    """bf16 bits of N(0, std^2) samples."""
    return bf16_bits_from_f32(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def uniform_codes_packed(rng: np.random.Generator, N: int, K: int) -> np.ndarray:
    """Canonical packed int4 codes, uniform over [-8, 7].

    Every byte holds two independent uniform nibbles, so drawing uniform
    bytes is the same as drawing uniform codes and packing them.
    """
    if K % 2:
        raise ValueError("K must be even")
    buf = rng.bytes(N * (K // 2))
    return np.frombuffer(buf, dtype=np.uint8).reshape(N, K // 2).copy()


def fp16_scales(rng: np.random.Generator, N: int, n_groups: int) -> np.ndarray:
    """fp16 bits of |N(0, 0.02)| + 1e-3."""
    s = np.abs(rng.standard_normal((N, n_groups), dtype=np.float32)) * np.float32(0.02) + np.float32(1e-3)
    return s.astype(np.float16).view(np.uint16)


def w4_weights(rng: np.random.Generator, K: int, N: int, group: int):
    """(codes_packed uint8 [N][K/2], scales fp16-bits uint16 [N][K/group])."""
    if K % group:
        raise ValueError("K must be a multiple of the group size")
    codes = uniform_codes_packed(rng, N, K)
    scales = fp16_scales(rng, N, K // group)
    return codes, scales


def mlx_affine_weights(rng: np.random.Generator, K: int, N: int, group: int):
    """(codes uint32 [N][K/8], scales bf16 bits [N][K/group], biases bf16 bits [N][K/group]).

    MLX-style affine 4-bit layout: unsigned codes uniform in [0, 15], packed 8
    per word (element i in bits 4i..4i+3); scales |N(0, 0.02)| + 1e-3 and
    biases -scale * U(6, 9) (a group's minimum sits about 7.5 steps below its
    mean), both rounded to bf16.
    """
    if K % group or K % 8:
        raise ValueError("K must be a multiple of the group size and of 8")
    q = rng.integers(0, 16, size=(N, K), dtype=np.uint32)
    words = np.zeros((N, K // 8), dtype=np.uint32)
    for i in range(8):
        words |= q[:, i::8] << np.uint32(4 * i)
    s = (np.abs(rng.standard_normal((N, K // group), dtype=np.float32)) * np.float32(0.02) + np.float32(1e-3))
    b = -s * rng.uniform(6.0, 9.0, size=s.shape).astype(np.float32)
    return words, bf16_bits_from_f32(s), bf16_bits_from_f32(b)


def nvfp4_weights(rng: np.random.Generator, K: int, N: int, min_scale_exp: int = 8):
    """(codes uint8 [N][K/2], block-scale bytes uint8 [N][K/16], global scale).

    Two 4-bit E2M1 codes per byte, each of the 16 patterns equally likely
    (element 2j in the low nibble); one positive E4M3 scale byte per 16
    elements with its exponent field uniform in [min_scale_exp, 15] and its
    mantissa uniform in [0, 7], the one NaN pattern (0x7F) redrawn as 0x7E;
    global scale 2^-15.  With the default exponents the block scales span
    [2, 448] and the weights about 2^-15 .. 2^-3.5, the spread of a
    checkpoint quantised from N(0, 0.02)-sized weights.
    """
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    e = rng.integers(min_scale_exp, 16, size=(N, K // 16), dtype=np.uint8)
    m = rng.integers(0, 8, size=(N, K // 16), dtype=np.uint8)
    scales = (e << np.uint8(3)) | m
    scales[scales == 0x7F] = 0x7E
    return codes, scales, 2.0 ** -15


def logits_normal(rng: np.random.Generator, R: int, V: int, std: float = 3.0) -> np.ndarray:
    """float32 logits N(0, std^2) of shape [R][V]."""
    return (rng.standard_normal((R, V), dtype=np.float32) * np.float32(std)).astype(np.float32)


def seeds_u64(rng: np.random.Generator, n: int) -> np.ndarray:
    return rng.integers(0, 2**64 - 1, size=n, dtype=np.uint64, endpoint=True)


def positions(rng: np.random.Generator, n: int, hi: int = 65536) -> np.ndarray:
    return rng.integers(0, hi, size=n, dtype=np.int64)


def noisy_drafts(rng: np.random.Generator, true_tokens, p_match: float, V: int) -> np.ndarray:
    """Draft tokens that copy ``true_tokens`` with probability ``p_match``.

    Otherwise a uniform token in [0, V) is drawn (which may still equal the
    true token by chance, as a real drafter's guess could).
    """
    t = np.asarray(true_tokens, dtype=np.int64)
    keep = rng.random(t.shape) < p_match
    rand = rng.integers(0, V, size=t.shape, dtype=np.int64)
    return np.where(keep, t, rand).astype(np.int32)


def attention_inputs(rng: np.random.Generator, R: int, n_kv: int, group: int, L: int, head_dim: int = 128,
                     q_std: float = 1.0):
    """bf16 bits of verify-row queries [R][n_kv*group][head_dim] and a KV cache
    prefix k, v [n_kv][L][head_dim], all normal (keys and values N(0, 1))."""
    q = bf16_normal(rng, (R, n_kv * group, head_dim), q_std)
    k = bf16_normal(rng, (n_kv, L, head_dim))
    v = bf16_normal(rng, (n_kv, L, head_dim))
    return q, k, v


def router_logits(rng: np.random.Generator, R: int, n_experts: int) -> np.ndarray:
    return rng.standard_normal((R, n_experts), dtype=np.float32)


# Shapes of the five workloads (sizes only; no arithmetic).
CONFIGS = {
    "tiny": dict(K=256, N=1024, group=64, rows=(1, 2, 4), V=1024,
                 temperature=0.7, top_k=20, top_p=0.95, seed=1234, n_drafts=4, p_match=0.7),
    "dense27b": dict(shapes=((5120, 17408), (17408, 5120)), group=64, rows=(1, 2, 4, 8, 16)),
    "lmhead": dict(K=5120, V=151936, group=64, rows=tuple(range(1, 17)),
                   settings=((0.0, 0, 1.0), (0.6, 20, 0.95), (1.0, 50, 0.8)), p_match=0.6),
    "moe30b": dict(hidden=2048, ffn=768, n_experts=128, top_k=8, group=32, rows=(1, 4, 8, 16)),
    "decoder": dict(V=151936, hidden=5120, ffn=17408, n_blocks=8, group=64, n_tokens=64,
                    rows=8, temperature=0.7, top_k=20, top_p=0.95, seeds=(1234, 1235, 1236, 1237, 1238),
                    p_match=0.75),
}
