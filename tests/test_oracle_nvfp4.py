"""Pins of the NVFP4 linear oracle (oracle/nvfp4.py) against things other than itself.

* every E2M1 code against the value table of the format (magnitudes 0, 0.5, 1,
  1.5, 2, 3, 4, 6 and their negatives);
* every E4M3 byte against torch's float8_e4m3fn conversion (NaN where it has NaN);
* the nibble order on a hand-decoded byte;
* one-hot activations, where the layer reduces to one dequantised weight exactly;
* the block size: a scale byte changes exactly its 16 input features;
* exact rational brute force on tiny shapes;
* planted mistakes, each caught by one of the above.
"""

import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import nvfp4 as NV
from w4_gemm_keyed_gb300 import inputs

E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def _bf16(v):
    return inputs.bf16_bits_from_f32(np.asarray(v, dtype=np.float32))


def test_e2m1_every_code():
    for c, want in enumerate(E2M1_TABLE):
        got = NV.e2m1_value(c)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), c


def test_e4m3_every_byte_against_torch():
    torch = pytest.importorskip("torch")
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([NV.e4m3_value(b) for b in range(256)])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert NV.e4m3_value(0x7E) == 448.0 and NV.e4m3_value(0x01) == 2.0 ** -9


def test_nibble_order_hand_decoded():
    # byte 0x2F: low nibble 0xF -> -6 (element 0), high nibble 0x2 -> 1.0 (element 1)
    codes = np.full((1, 8), 0x00, dtype=np.uint8)
    codes[0, 0] = 0x2F
    w = NV.dequantize(codes, np.array([[0x38]], dtype=np.uint8), 1.0)   # scale byte 0x38 = 1.0
    assert w[0, 0] == -6.0 and w[0, 1] == 1.0 and np.all(w[0, 2:] == 0.0)


def test_one_hot_reduces_to_one_weight():
    rng = inputs.rng_for(811)
    K, N = 64, 5
    codes, scales, gs = inputs.nvfp4_weights(rng, K, N, min_scale_exp=0)
    for k in (0, 1, 15, 16, 33, 63):
        x = np.zeros((1, K), dtype=np.float32)
        x[0, k] = 1.0
        y = NV.nvfp4_linear(codes, scales, gs, _bf16(x))
        for n in range(N):
            c = (codes[n, k // 2] >> (4 * (k % 2))) & 0xF
            want = E2M1_TABLE[c] * NV.e4m3_value(scales[n, k // 16]) * gs
            assert y[0, n] == want


def test_block_scale_covers_sixteen_features():
    K, N = 64, 1
    codes = np.full((N, K // 2), 0x22, dtype=np.uint8)         # every element 1.0
    scales = np.full((N, K // 16), 0x38, dtype=np.uint8)       # every block scale 1.0
    scales[0, 1] = 0x40                                        # block 1 (k 16..31) scale 2.0
    w = NV.dequantize(codes, scales, 1.0)
    assert np.all(w[0, :16] == 1.0) and np.all(w[0, 16:32] == 2.0) and np.all(w[0, 32:] == 1.0)


def _fr_e2m1(c):
    s, e, m = c >> 3, (c >> 1) & 3, c & 1
    mag = Fraction(m, 2) if e == 0 else Fraction(2 + m, 2) * Fraction(2) ** (e - 1)
    return -mag if s else mag


def _fr_e4m3(b):
    s, e, m = b >> 7, (b >> 3) & 15, b & 7
    mag = Fraction(m, 8) * Fraction(1, 64) if e == 0 else Fraction(8 + m, 8) * Fraction(2) ** (e - 7)
    return -mag if s else mag


def test_exact_rational_brute_force():
    rng = inputs.rng_for(812)
    K, N, R = 32, 3, 2
    codes, scales, gs = inputs.nvfp4_weights(rng, K, N, min_scale_exp=0)
    x_bits = inputs.bf16_normal(rng, (R, K))
    xf = (x_bits.astype(np.uint32) << 16).view(np.float32)
    y = NV.nvfp4_linear(codes, scales, gs, x_bits)
    for r in range(R):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                c = int((codes[n, k // 2] >> (4 * (k % 2))) & 0xF)
                acc += _fr_e2m1(c) * _fr_e4m3(int(scales[n, k // 16])) * Fraction(gs) * Fraction(float(xf[r, k]))
            assert abs(y[r, n] - float(acc)) <= 1e-12 * max(1e-30, abs(float(acc)))


def test_column_subset_equals_full():
    rng = inputs.rng_for(813)
    codes, scales, gs = inputs.nvfp4_weights(rng, 128, 40)
    x = inputs.bf16_normal(rng, (3, 128))
    cols = np.array([0, 7, 39, 12])
    assert np.array_equal(NV.nvfp4_linear(codes, scales, gs, x, cols=cols), NV.nvfp4_linear(codes, scales, gs, x)[:, cols])


# ------------------------------------------------------------------ planted mistakes
def _mutants():
    def swapped_nibbles(codes_u8):
        b = np.ascontiguousarray(codes_u8, dtype=np.uint8)
        out = np.empty((b.shape[0], 2 * b.shape[1]), dtype=np.uint8)
        out[:, 0::2], out[:, 1::2] = b >> 4, b & 0xF
        return out

    def bias_off(code):
        code = int(code) & 0xF
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = 0.5 * m if e == 0 else math.ldexp(1.0 + 0.5 * m, e)
        return -mag if s else mag

    def e4m3_no_subnormal(byte):
        byte = int(byte) & 0xFF
        s, e, m = byte >> 7, (byte >> 3) & 0xF, byte & 7
        if e == 15 and m == 7:
            return math.nan
        mag = math.ldexp(1.0 + m / 8.0, e - 7)
        return -mag if s else mag

    return {"swapped_nibbles": ("unpack_codes", swapped_nibbles),
            "e2m1_bias": ("_E2M1", np.array([bias_off(c) for c in range(16)])),
            "e4m3_subnormal": ("_E4M3", np.array([e4m3_no_subnormal(b) for b in range(256)])),
            "block_32": ("BLOCK", 32)}


@pytest.mark.parametrize("name", ["swapped_nibbles", "e2m1_bias", "e4m3_subnormal", "block_32"])
def test_planted_mistake_is_caught(monkeypatch, name):
    attr, value = _mutants()[name]
    monkeypatch.setattr(NV, attr, value)
    pins = [test_nibble_order_hand_decoded, test_one_hot_reduces_to_one_weight, test_block_scale_covers_sixteen_features,
            test_exact_rational_brute_force, test_e4m3_every_byte_against_torch]
    caught = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError):
            caught += 1
    assert caught >= 1, f"mutant {name} passed every pin"


def test_planted_global_scale_dropped_is_caught(monkeypatch):
    orig = NV.dequantize
    monkeypatch.setattr(NV, "dequantize", lambda c, s, g: orig(c, s, 1.0))
    with pytest.raises(AssertionError):
        test_one_hot_reduces_to_one_weight()
