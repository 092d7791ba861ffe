"""Pins of the W4 linear oracle against things other than itself.

* the fp16 / bf16 decoders against numpy's and torch's conversions (all 65536 patterns);
* the canonical nibble decoding against a hand-decoded byte and a test-local packer;
* one-hot activations, where the layer reduces to ``code * scale`` exactly;
* a dequantise-then-matmul restatement (numpy BLAS, a different algorithm);
* exact rational brute force on tiny shapes;
* planted mistakes in a copy of the C source, each caught by one of the above.
"""

import ctypes
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import linear as olin
from w4_gemm_keyed_gb300 import inputs


def unpack_local(packed):
    """Test-local decoder of the canonical layout (independent of the oracle's C)."""
    b = np.asarray(packed, dtype=np.uint8).astype(np.int16)
    lo, hi = b & 0xF, b >> 4
    out = np.empty((b.shape[0], 2 * b.shape[1]), dtype=np.int16)
    out[:, 0::2], out[:, 1::2] = lo, hi
    return np.where(out >= 8, out - 16, out).astype(np.int8)


def pack_canonical(codes_i8):
    """Test-local packer: low nibble = even k, two's complement."""
    c = np.asarray(codes_i8, dtype=np.int16) & 0xF
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def test_half_decoder_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.half_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_bf16_decoder_all_patterns():
    torch = pytest.importorskip("torch")
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_nibble_order_hand_decoded():
    # byte 0x8F: low nibble 0xF -> -1 (k even), high nibble 0x8 -> -8 (k odd)
    # byte 0x70: low nibble 0x0 ->  0,          high nibble 0x7 ->  7
    codes = np.array([[0x8F, 0x70]], dtype=np.uint8)
    assert oracle.unpack_codes(codes).tolist() == [[-1, -8, 0, 7]]


def test_unpack_round_trip():
    rng = inputs.rng_for(11, 1)
    c = rng.integers(-8, 8, size=(37, 128), dtype=np.int8)
    assert np.array_equal(oracle.unpack_codes(pack_canonical(c)), c)
    # the generator's packed bytes decode to uniform codes over the full range
    packed, _ = inputs.w4_weights(rng, 256, 64, 64)
    u = oracle.unpack_codes(packed)
    assert np.array_equal(u, unpack_local(packed))
    assert u.min() == -8 and u.max() == 7


@pytest.mark.parametrize("G", [32, 64])
def test_one_hot_reduces_to_code_times_scale(G):
    rng = inputs.rng_for(11, 2, G)
    K, N = 4 * G, 40
    codes, scales = inputs.w4_weights(rng, K, N, G)
    ks = [0, 1, G - 1, G, 2 * G + 3, K - 1]
    x = np.zeros((len(ks), K), dtype=np.uint16)
    for r, k in enumerate(ks):
        x[r, k] = 0x3F80  # bf16 1.0
    y = oracle.w4_linear(codes, scales, x, G)
    c = unpack_local(codes).astype(np.float64)
    s = scales.view(np.float16).astype(np.float64)
    for r, k in enumerate(ks):
        assert np.array_equal(y[r], c[:, k] * s[:, k // G])


@pytest.mark.parametrize("G,K,N,R", [(64, 256, 96, 3), (32, 192, 70, 5), (64, 64, 33, 1)])
def test_matches_dequantise_then_matmul(G, K, N, R):
    rng = inputs.rng_for(11, 3, G, K)
    codes, scales = inputs.w4_weights(rng, K, N, G)
    x = inputs.bf16_normal(rng, (R, K))
    y = oracle.w4_linear(codes, scales, x, G)
    c = unpack_local(codes).astype(np.float64)
    s = np.repeat(scales.view(np.float16).astype(np.float64), G, axis=1)
    W = c * s  # exact in fp64
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = xf @ W.T
    assert c.shape == (N, K)
    tol = 1e-12 * np.sqrt(np.mean(ref ** 2))
    assert np.max(np.abs(y - ref)) <= tol


def test_column_subset_equals_full():
    rng = inputs.rng_for(11, 4)
    codes, scales = inputs.w4_weights(rng, 128, 64, 64)
    x = inputs.bf16_normal(rng, (2, 128))
    full = oracle.w4_linear(codes, scales, x, 64)
    cols = np.array([63, 0, 17, 17, 40])
    assert np.array_equal(oracle.w4_linear(codes, scales, x, 64, cols=cols), full[:, cols])


def test_exact_rational_brute_force():
    rng = inputs.rng_for(11, 5)
    G, K, N, R = 32, 64, 6, 2
    codes, scales = inputs.w4_weights(rng, K, N, G)
    x = inputs.bf16_normal(rng, (R, K))
    y = oracle.w4_linear(codes, scales, x, G)
    c = unpack_local(codes)
    s = scales.view(np.float16).astype(np.float64)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for r in range(R):
        for n in range(N):
            exact = sum(Fraction(s[n, k // G]) * int(c[n, k]) * Fraction(xf[r, k]) for k in range(K))
            # fp64 evaluation of a sum of 64 exact terms: well inside 64 ulps of the scale
            assert abs(Fraction(y[r, n]) - exact) <= Fraction(2.0 ** -40)


# ----------------------------------------------------------------------------
# Planted mistakes: each mutant of the C source must fail a pin above.
# ----------------------------------------------------------------------------
MUTANTS = {
    "nibble_order_swapped": ("(k % 2 == 0) ? (byte & 0x0f) : (byte >> 4)",
                             "(k % 2 == 0) ? (byte >> 4) : (byte & 0x0f)"),
    "unsigned_codes": ("return nib >= 8 ? nib - 16 : nib;", "return nib;"),
    "scale_group_index_off_by_one": ("scales[(size_t)n * n_groups + g]",
                                     "scales[(size_t)n * n_groups + (g + 1) % n_groups]"),
    "last_element_of_group_dropped": ("k < (g + 1) * G; ++k", "k < (g + 1) * G - 1; ++k"),
    "half_exponent_bias": ("expo - 25", "expo - 24"),
}


def _build_mutant(tmp_path, name):
    src = open(os.path.join(os.path.dirname(olin.__file__), "w4_ref.c")).read()
    old, new = MUTANTS[name]
    assert old in src, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-o", str(lib), str(path), "-lm"], check=True)
    return ctypes.CDLL(str(lib))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, monkeypatch, name):
    lib = _build_mutant(tmp_path, name)
    P = ctypes.c_void_p
    lib.oracle_w4_linear.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     P, ctypes.c_int, P]
    lib.oracle_unpack_codes.argtypes = [P, ctypes.c_int, ctypes.c_int, P]
    lib.oracle_half_array.argtypes = [P, ctypes.c_int64, P]
    lib.oracle_bf16_array.argtypes = [P, ctypes.c_int64, P]
    monkeypatch.setattr(olin, "_lib", lib)
    pins = [test_half_decoder_all_patterns, test_nibble_order_hand_decoded,
            lambda: test_one_hot_reduces_to_code_times_scale(64),
            lambda: test_matches_dequantise_then_matmul(32, 192, 70, 5)]
    failures = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError):
            failures += 1
    assert failures >= 1, f"mutant {name} passed every pin"
