"""Pins of the MLX-style affine W4 oracle (oracle/affine.py)."""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import affine
from w4_gemm_keyed_gb300 import inputs


def test_nibble_order_hand_decoded():
    words = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32)
    assert affine.unpack_u32_codes(words).tolist() == [list(range(16))]


def test_one_hot_is_scale_times_code_plus_bias():
    rng = inputs.rng_for(801)
    K, N, G = 128, 37, 64
    codes, scales, biases = inputs.mlx_affine_weights(rng, K, N, G)
    q = affine.unpack_u32_codes(codes).astype(np.float64)
    s, b = oracle.bf16_to_f64(scales), oracle.bf16_to_f64(biases)
    for k in (0, 1, 7, 8, 63, 64, 127):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, k] = 0x3F80
        y = affine.affine_w4_linear(codes, scales, biases, x, G)[0]
        assert np.array_equal(y, s[:, k // G] * q[:, k] + b[:, k // G])


def test_equals_symmetric_oracle_when_bias_is_minus_eight_scales():
    """q = c + 8 with bias -8 * scale is the symmetric code c times scale.
    Scales are chosen exactly representable in both bf16 and fp16."""
    rng = inputs.rng_for(802)
    K, N, G, R = 256, 50, 64, 3
    c = rng.integers(-8, 8, size=(N, K))
    sv = rng.integers(1, 128, size=(N, K // G)).astype(np.float32) / np.float32(1024)   # <= 7 significant bits
    scales_bf16 = (sv.view(np.uint32) >> 16).astype(np.uint16)
    biases_bf16 = ((-8 * sv).view(np.uint32) >> 16).astype(np.uint16)
    scales_f16 = sv.astype(np.float16).view(np.uint16)
    q = (c + 8).astype(np.uint32)
    words = np.zeros((N, K // 8), dtype=np.uint32)
    for i in range(8):
        words |= q[:, i::8] << np.uint32(4 * i)
    nib = (c & 0xF).astype(np.uint8)
    sym = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    x = inputs.bf16_normal(rng, (R, K))
    ya = affine.affine_w4_linear(words, scales_bf16, biases_bf16, x, G)
    ys = oracle.w4_linear(sym, scales_f16, x, G)
    assert np.allclose(ya, ys, rtol=1e-12, atol=1e-12)


def test_exact_rational_brute_force():
    rng = inputs.rng_for(803)
    K, N, G, R = 64, 3, 32, 2
    codes, scales, biases = inputs.mlx_affine_weights(rng, K, N, G)
    x = inputs.bf16_normal(rng, (R, K))
    q = affine.unpack_u32_codes(codes)
    s, b = oracle.bf16_to_f64(scales), oracle.bf16_to_f64(biases)
    xf = oracle.bf16_to_f64(x)
    y = affine.affine_w4_linear(codes, scales, biases, x, G)
    for r in range(R):
        for n in range(N):
            exact = sum((Fraction(s[n, k // G]) * int(q[n, k]) + Fraction(b[n, k // G])) * Fraction(xf[r, k])
                        for k in range(K))
            assert abs(Fraction(y[r, n]) - exact) <= abs(exact) * Fraction(1, 10**12) + Fraction(1, 10**15)


def test_column_subset_equals_full():
    rng = inputs.rng_for(804)
    K, N, G = 128, 40, 32
    codes, scales, biases = inputs.mlx_affine_weights(rng, K, N, G)
    x = inputs.bf16_normal(rng, (4, K))
    cols = np.array([0, 5, 39, 17])
    full = affine.affine_w4_linear(codes, scales, biases, x, G)
    assert np.array_equal(affine.affine_w4_linear(codes, scales, biases, x, G, cols=cols), full[:, cols])


@pytest.mark.parametrize("mutant", ["nibble_order", "no_bias"])
def test_planted_mistakes_are_caught(monkeypatch, mutant):
    if mutant == "nibble_order":
        orig = affine.unpack_u32_codes
        monkeypatch.setattr(affine, "unpack_u32_codes", lambda c: orig(c)[:, ::-1].copy())
        with pytest.raises(AssertionError):
            test_nibble_order_hand_decoded()
    else:
        real = affine.bf16_to_f64
        calls = {"n": 0}

        def zero_second(bits):   # scales are decoded first, biases second
            calls["n"] += 1
            out = real(bits)
            return out * 0.0 if calls["n"] % 3 == 2 else out
        monkeypatch.setattr(affine, "bf16_to_f64", zero_second)
        with pytest.raises(AssertionError):
            test_one_hot_is_scale_times_code_plus_bias()
