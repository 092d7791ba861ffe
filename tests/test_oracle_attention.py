"""Pins of the attention oracle (oracle/attention.py): closed forms and
invariants of causal grouped-head softmax attention, each chosen so that a
plausible slip (no 1/sqrt(D) scale, a mask off by one, a wrong head mapping,
a missing normalisation) fails at least one of them."""

import numpy as np
import pytest

from oracle import attention
from oracle.linear import bf16_to_f64
from w4_gemm_keyed_gb300 import inputs

D = attention.HEAD_DIM


def bf16(x):
    a = np.asarray(x, dtype=np.float32)
    bits = inputs.bf16_bits_from_f32(a).reshape(a.shape)
    return int(bits) if bits.ndim == 0 else bits


def test_single_key_returns_its_value():
    rng = inputs.rng_for(901)
    q, k, v = inputs.attention_inputs(rng, 1, 2, 4, 8)
    out = attention.attention_verify(q, k, v, 0, 4)
    for h in range(8):
        assert np.array_equal(out[0, h], bf16_to_f64(v[h // 4, 0]))


def test_zero_query_is_the_mean_of_the_visible_values():
    rng = inputs.rng_for(902)
    _, k, v = inputs.attention_inputs(rng, 3, 1, 1, 40)
    q = np.zeros((3, 1, D), dtype=np.uint16)
    out = attention.attention_verify(q, k, v, 20, 1)
    for r in range(3):
        expect = bf16_to_f64(v[0, : 21 + r]).mean(axis=0)
        assert np.allclose(out[r, 0], expect, rtol=0, atol=1e-12)


def test_two_keys_weighted_three_to_one():
    # q = 4 e0, k0 = 0, k1 = 3.109375 e0: the score gap is 12.4375 / sqrt(128)
    # = 1.09934, and exp(1.09934) = 3.0022, so the weights are 0.2498 / 0.7502.
    q = np.zeros((1, 1, D), dtype=np.uint16)
    q[0, 0, 0] = bf16(4.0)
    k = np.zeros((1, 2, D), dtype=np.uint16)
    k[0, 1, 0] = bf16(3.109375)
    v = np.zeros((1, 2, D), dtype=np.uint16)
    v[0, 0, 1] = bf16(1.0)
    v[0, 1, 2] = bf16(1.0)
    out = attention.attention_verify(q, k, v, 1, 1)[0, 0]
    assert abs(out[1] - 0.25) < 1e-3 and abs(out[2] - 0.75) < 1e-3
    assert np.all(out[3:] == 0) and out[0] == 0


def test_a_key_component_shared_by_all_positions_cancels():
    rng = np.random.default_rng(903)
    q = rng.standard_normal(D)
    k = rng.standard_normal((30, D))
    v = rng.standard_normal((30, D))
    u = 3.0 * rng.standard_normal(D)
    a = attention.attention_row(q, k, v, 29)
    b = attention.attention_row(q, k + u, v, 29)
    assert np.allclose(a, b, rtol=0, atol=1e-12)
    # and the result is a convex combination of the visible values
    assert np.all(a <= v.max(axis=0) + 1e-12) and np.all(a >= v.min(axis=0) - 1e-12)


def test_row_sees_its_own_position_and_nothing_later():
    rng = inputs.rng_for(904)
    q, k, v = inputs.attention_inputs(rng, 4, 1, 2, 64)
    pos0 = 50
    base = attention.attention_verify(q, k, v, pos0, 2)
    # entries after a row's position do not matter
    for r in range(4):
        k2, v2 = k.copy(), v.copy()
        k2[:, pos0 + r + 1:] = bf16(7.0)
        v2[:, pos0 + r + 1:] = bf16(-5.0)
        out = attention.attention_verify(q, k2, v2, pos0, 2)
        assert np.array_equal(out[r], base[r])
    # a key aligned with the query at the row's own position dominates
    q1 = np.zeros((1, 1, D), dtype=np.uint16)
    q1[0, 0, :] = bf16(1.0)
    k1 = np.zeros((1, 10, D), dtype=np.uint16)
    k1[0, 7, :] = bf16(4.0)          # score 512 / sqrt(128) = 45.25 above the others
    v1 = inputs.bf16_normal(rng, (1, 10, D))
    out = attention.attention_verify(q1, k1, v1, 7, 1)[0, 0]
    assert np.allclose(out, bf16_to_f64(v1[0, 7]), rtol=0, atol=1e-15 + 1e-18)


def test_query_head_h_reads_kv_head_h_div_group():
    rng = inputs.rng_for(905)
    q, k, v = inputs.attention_inputs(rng, 2, 2, 2, 16)
    k[1] = k[0]
    v[1] = bf16(bf16_to_f64(v[0]) + 64.0)
    out = attention.attention_verify(q, k, v, 10, 2)
    q_swapped = q.copy()
    q_swapped[:, 2:4] = q[:, 0:2]
    out2 = attention.attention_verify(q_swapped, k, v, 10, 2)
    # heads 2, 3 (kv head 1) with the queries of heads 0, 1 (kv head 0): the
    # same weights, values shifted by 64 up to the bf16 rounding of v + 64
    assert np.allclose(out2[:, 2:4], out[:, 0:2] + 64.0, rtol=0, atol=0.26)
    assert np.all(np.abs(out[:, 0:2]) < 8)


def test_rows_equal_single_row_calls():
    rng = inputs.rng_for(906)
    q, k, v = inputs.attention_inputs(rng, 5, 2, 4, 300)
    out = attention.attention_verify(q, k, v, 250, 4)
    for r in range(5):
        one = attention.attention_verify(q[r:r + 1], k, v, 250 + r, 4)
        assert np.array_equal(one[0], out[r])


@pytest.mark.parametrize("mutant", ["no_scale", "mask_excludes_self", "mask_one_late", "head_mod", "no_norm"])
def test_planted_mistakes_are_caught(monkeypatch, mutant):
    import math
    real_row = attention.attention_row

    def no_scale(q, k, v, p):
        s = k[: p + 1] @ q
        w = np.exp(s - s.max())
        return (w @ v[: p + 1]) / w.sum()

    def excl_self(q, k, v, p):
        return real_row(q, k, v, max(p - 1, 0))

    def one_late(q, k, v, p):
        return real_row(q, k, v, min(p + 1, k.shape[0] - 1))

    def no_norm(q, k, v, p):
        s = (k[: p + 1] @ q) / math.sqrt(q.shape[0])
        return np.exp(s) @ v[: p + 1]

    checks = [test_single_key_returns_its_value, test_zero_query_is_the_mean_of_the_visible_values,
              test_two_keys_weighted_three_to_one, test_a_key_component_shared_by_all_positions_cancels,
              test_row_sees_its_own_position_and_nothing_later, test_query_head_h_reads_kv_head_h_div_group]
    if mutant == "head_mod":
        real_verify = attention.attention_verify

        def head_mod(q_bits, k_bits, v_bits, pos0, group, heads=None):
            n_kv = k_bits.shape[0]
            out = np.empty(q_bits.shape, dtype=np.float64)
            for r in range(q_bits.shape[0]):
                for h in range(q_bits.shape[1]):
                    out[r, h] = real_row(bf16_to_f64(q_bits[r, h]), bf16_to_f64(k_bits[h % n_kv]),
                                         bf16_to_f64(v_bits[h % n_kv]), pos0 + r)
            return out
        monkeypatch.setattr(attention, "attention_verify", head_mod)
        assert real_verify is not head_mod
    else:
        monkeypatch.setattr(attention, "attention_row",
                            {"no_scale": no_scale, "mask_excludes_self": excl_self, "mask_one_late": one_late,
                             "no_norm": no_norm}[mutant])
    failed = 0
    for check in checks:
        try:
            check()
        except AssertionError:
            failed += 1
    assert failed >= 1, f"no pin caught the planted mistake {mutant}"


def test_properties_on_random_shapes():
    """Over random small shapes: outputs are convex combinations of the visible
    values, a key component shared by all positions cancels, verify rows equal
    single-row calls, and entries after a row's position never matter."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    @hyp.settings(max_examples=25, deadline=None)
    @hyp.given(R=st.integers(1, 4), n_kv=st.integers(1, 2), group=st.sampled_from([1, 2]),
               pos0=st.integers(0, 30), seed=st.integers(0, 2**31 - 1))
    def check(R, n_kv, group, pos0, seed):
        rng = np.random.default_rng(seed)
        L = pos0 + R + 3
        q, k, v = inputs.attention_inputs(rng, R, n_kv, group, L, q_std=2.0)
        out = attention.attention_verify(q, k, v, pos0, group)
        kf, vf = bf16_to_f64(k), bf16_to_f64(v)
        for r in range(R):
            p = pos0 + r
            for h in range(n_kv * group):
                vis = vf[h // group, : p + 1]
                assert np.all(out[r, h] <= vis.max(axis=0) + 1e-12)
                assert np.all(out[r, h] >= vis.min(axis=0) - 1e-12)
                u = rng.standard_normal(D)
                shifted = attention.attention_row(bf16_to_f64(q[r, h]), kf[h // group] + u, vf[h // group], p)
                assert np.allclose(shifted, out[r, h], rtol=0, atol=1e-9)
            one = attention.attention_verify(q[r:r + 1], k, v, p, group)
            assert np.array_equal(one[0], out[r])
        k2, v2 = k.copy(), v.copy()
        k2[:, pos0 + R:] = bf16(3.0)
        v2[:, pos0 + R:] = bf16(-9.0)
        assert np.array_equal(attention.attention_verify(q, k2, v2, pos0, group), out)

    check()
