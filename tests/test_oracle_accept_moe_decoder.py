"""Pins of the acceptance, MoE, numerics and synthetic-decoder oracles.

* acceptance brute-forced over every draft/sample combination for R <= 4, V <= 3,
  against a restatement (length of the longest matching prefix);
* bf16 rounding against torch's float32 -> bfloat16 conversion, plus fp64
  tie cases in closed form; rms_norm and silu in closed form / scipy;
* MoE routing against scipy's softmax and a stable argsort; the MoE block
  against the invariant that rows are independent and the closed form
  "identical experts => output equals one expert's output";
* drafted decoding equals serial decoding (token_sha) on a tiny synthetic
  decoder, with perfect, noisy and useless drafters, at several widths R;
* planted mistakes, each caught by one of these.
"""

import itertools
import math

import numpy as np
import pytest

import oracle
from oracle import accept as A
from oracle import decoder as D
from oracle import moe as M
from oracle import numerics as NUM
from w4_gemm_keyed_gb300 import inputs


# ------------------------------------------------------------------ accept
def _restated_accept(d, t):
    n = len(list(itertools.takewhile(lambda p: p[0] == p[1], zip(d, t))))
    return n, t[n]


def test_accept_brute_force():
    for R in range(1, 5):
        for V in range(1, 4):
            for t in itertools.product(range(V), repeat=R):
                for d in itertools.product(range(V), repeat=R - 1):
                    assert A.accept(d, t) == _restated_accept(d, t)
                    c = A.committed(d, t)
                    assert 1 <= len(c) <= R and c == list(t[: len(c)])


def test_accept_rejects_bad_shapes():
    with pytest.raises(ValueError):
        A.accept([1, 2], [1, 2])
    with pytest.raises(ValueError):
        A.accept([], [])


# ------------------------------------------------------------------ numerics
def test_bf16_round_matches_torch_on_float32_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    # force exact ties (low half 0x8000) with both parities of the kept bit
    bits[:2000] = (bits[:2000] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    f = bits.view(np.float32)
    f = f[np.isfinite(f) & (np.abs(f) < 3.0e38)]
    ours = NUM.bf16_round(f.astype(np.float64))
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


def test_bf16_round_fp64_ties_closed_form():
    e8, e7, e6 = 2.0 ** -8, 2.0 ** -7, 2.0 ** -6
    assert NUM.bf16_round(1.0 + e8) == 1.0                  # tie -> even
    assert NUM.bf16_round(1.0 + 3 * e8) == 1.0 + e6         # tie -> even (upwards)
    assert NUM.bf16_round(1.0 + e8 + 2.0 ** -40) == 1.0 + e7  # just above the tie
    assert NUM.bf16_round(-(1.0 + e8 + 2.0 ** -40)) == -(1.0 + e7)
    assert NUM.bf16_round(2.0 ** -133) == 2.0 ** -133       # smallest subnormal
    assert NUM.bf16_round(0.0) == 0.0


def test_rms_norm_and_silu_closed_forms():
    scipy_special = pytest.importorskip("scipy.special")
    c = 0.37
    x = np.full((1, 64), c)
    assert np.allclose(NUM.rms_norm(x, 1e-6), c / math.sqrt(c * c + 1e-6), rtol=0, atol=1e-15)
    x = np.array([[3.0, 4.0]])  # mean square 12.5
    assert np.allclose(NUM.rms_norm(x, 0.0), x / math.sqrt(12.5), rtol=1e-15)
    v = np.linspace(-30, 30, 1001)
    assert np.allclose(NUM.silu(v), v * scipy_special.expit(v), rtol=1e-14, atol=1e-300)
    assert NUM.silu(0.0) == 0.0


# ------------------------------------------------------------------ MoE
def _moe_weights(rng, E, H, F, G, identical=False):
    def mats(K, N):
        c, s = inputs.w4_weights(rng, K, N, G)
        return c, s
    W = {k: [] for k in ("gate_codes", "gate_scales", "up_codes", "up_scales", "down_codes", "down_scales")}
    first = None
    for e in range(E):
        if identical and first is not None:
            blob = first
        else:
            blob = (mats(H, F), mats(H, F), mats(F, H))
            first = first or blob
        (gc, gs), (uc, us), (dc, ds) = blob
        for k, v in zip(W, (gc, gs, uc, us, dc, ds)):
            W[k].append(v)
    return {k: np.stack(v) for k, v in W.items()}


def test_route_matches_scipy_softmax():
    scipy_special = pytest.importorskip("scipy.special")
    rng = inputs.rng_for(21, 1)
    z = inputs.router_logits(rng, 16, 128)
    z[3, 10] = z[3, 20] = z[3].max() + 1.0  # a tie at the top: lower id first
    ids, w = M.route(z, 8)
    for r in range(16):
        ref_ids = np.argsort(-z[r].astype(np.float64), kind="stable")[:8]
        assert ids[r].tolist() == ref_ids.tolist()
        p = scipy_special.softmax(z[r].astype(np.float64))[ref_ids]
        assert np.allclose(w[r], p / p.sum(), rtol=1e-13, atol=0)
    assert ids[3, 0] == 10 and ids[3, 1] == 20


def test_moe_rows_independent_and_identical_experts():
    rng = inputs.rng_for(21, 2)
    E, H, F, G = 6, 64, 64, 32
    W = _moe_weights(rng, E, H, F, G)
    x = inputs.bf16_normal(rng, (5, H))
    z = inputs.router_logits(rng, 5, E)
    out, ids, w, ysel = M.moe(x, z, W, G, top_k=3)
    for r in range(5):
        o1, *_ = M.moe(x[r:r + 1], z[r:r + 1], W, G, top_k=3)
        assert np.array_equal(o1[0], out[r])
    Wi = _moe_weights(rng, E, H, F, G, identical=True)
    out_i, _, _, ysel_i = M.moe(x, z, Wi, G, top_k=3)
    assert np.allclose(out_i, ysel_i[:, 0, :], rtol=1e-14, atol=1e-14)


# ------------------------------------------------------------------ decoder
def tiny_model(seed=31, V=64, H=128, F=192, n_blocks=2, G=64):
    rng = inputs.rng_for(seed)
    blocks = []
    for _ in range(n_blocks):
        gc, gs = inputs.w4_weights(rng, H, F, G)
        uc, us = inputs.w4_weights(rng, H, F, G)
        dc, ds = inputs.w4_weights(rng, F, H, G)
        blocks.append(dict(gate_codes=gc, gate_scales=gs, up_codes=uc, up_scales=us,
                           down_codes=dc, down_scales=ds))
    lc, ls = inputs.w4_weights(rng, H, V, G)
    return dict(emb=inputs.bf16_normal(rng, (V, H), 0.02), blocks=blocks, lm_codes=lc, lm_scales=ls, group=G)


@pytest.mark.parametrize("R,p_match", [(2, 1.0), (4, 0.75), (8, 0.75), (8, 0.0)])
def test_drafted_equals_serial_token_sha(R, p_match):
    model = tiny_model()
    T, k, p, seed, n = 0.7, 20, 0.95, 1234, 24
    serial = D.serial_decode(model, 5, n, T, k, p, seed)
    rng = inputs.rng_for(32, R, int(p_match * 100))
    future = np.array(serial + [0] * R)

    def drafts(pos0, m):
        return inputs.noisy_drafts(rng, future[pos0 - 1: pos0 - 1 + m], p_match, 64)

    drafted, lens = D.drafted_decode(model, 5, n, R, T, k, p, seed, drafts)
    assert D.token_sha(drafted) == D.token_sha(serial)
    assert drafted == serial
    if p_match == 1.0:
        assert all(a == R - 1 for a in lens[:-1])
    if p_match == 0.0:
        assert np.mean(lens) < 0.5


def test_decoder_logits_row_independent():
    model = tiny_model()
    l4 = D.logits(model, [1, 2, 3, 2])
    assert np.array_equal(l4[1], l4[3])
    assert np.array_equal(D.logits(model, [3])[0], l4[2])


# ------------------------------------------------------------------ planted mistakes
def test_planted_accept_off_by_one_is_caught(monkeypatch):
    orig = A.accept

    def mutant(d, t):
        a, _ = orig(d, t)
        a = min(a + 1, len(t) - 1)
        return a, t[a]
    monkeypatch.setattr(A, "accept", mutant)
    with pytest.raises(AssertionError):
        test_accept_brute_force()


def test_planted_route_without_renormalisation_is_caught(monkeypatch):
    orig = M.route

    def mutant(z, top_k=8):
        ids, w = orig(z, top_k)
        zz = np.asarray(z, np.float64)
        full = np.exp(zz - zz.max(axis=1, keepdims=True))
        full /= full.sum(axis=1, keepdims=True)
        return ids, np.take_along_axis(full, ids, axis=1)
    monkeypatch.setattr(M, "route", mutant)
    with pytest.raises(AssertionError):
        test_route_matches_scipy_softmax()


def test_planted_decoder_bonus_mistake_is_caught(monkeypatch):
    orig = A.accept

    def mutant(d, t):  # feeds the last draft instead of the bonus token
        a, b = orig(d, t)
        return a, (d[a] if a < len(d) else b)
    monkeypatch.setattr(A, "accept", mutant)
    with pytest.raises(AssertionError):
        test_drafted_equals_serial_token_sha(4, 0.75)


# ------------------------------------------------------------------ compositions in closed form
# Hand-sized weights whose results follow from the definitions alone: SwiGLU
# (Shazeer 2020, "GLU Variants Improve Transformer": silu of the gate
# projection times the up projection), RMSNorm with gain 1 and eps 1e-6, the
# residual add, and the rank-order combine of the renormalised top-k router
# weights.  The expected numbers below were worked out once from those
# definitions (bf16 values are exact binary fractions).
_BF16_ONE = 0x3F80
_FP16_ONE, _FP16_HALF, _FP16_QUARTER = 0x3C00, 0x3800, 0x3400


def _pack_rows(codes_i8):
    """Canonical packed codes of a small int matrix (low nibble = even k)."""
    c = np.asarray(codes_i8, dtype=np.int16) & 0xF
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def _mat(N, K, G, entries, scale_bits):
    """codes [N][K] zero except entries {(n, k): code}; every group scale = scale_bits[n]."""
    c = np.zeros((N, K), dtype=np.int8)
    for (n, k), v in entries.items():
        c[n, k] = v
    s = np.zeros((N, K // G), dtype=np.uint16)
    for n, b in enumerate(scale_bits):
        s[n, :] = b
    return _pack_rows(c), s


def _expert(H, F, G, gate, up, down, down_scales):
    gc, gs = _mat(F, H, G, gate, [_FP16_ONE] * F)
    uc, us = _mat(F, H, G, up, [_FP16_ONE] * F)
    dc, ds = _mat(H, F, G, down, down_scales)
    return dict(gate_codes=gc, gate_scales=gs, up_codes=uc, up_scales=us, down_codes=dc, down_scales=ds)


def _stack(experts):
    return {k: np.stack([e[k] for e in experts]) for k in experts[0]}


def _one_hot_row(H):
    x = np.zeros((1, H), dtype=np.uint16)
    x[0, 0] = _BF16_ONE
    return x


def test_expert_swiglu_closed_form():
    # x = e_0; gate row 0 reads 2 * x_0, up row 0 reads -3 * x_0:
    #   h_0 = bf16(silu(2) * -3) = bf16(-5.2847824678...) = -5.28125  (silu of the GATE)
    #   (silu of the up projection instead would give bf16(silu(-3) * 2) = -0.28515625)
    # down rows: y_0 = 0.5 * 1 * h_0, y_1 = 0.25 * -2 * h_0; every other output is 0.
    H = F = G = 32
    e = _expert(H, F, G, {(0, 0): 2}, {(0, 0): -3}, {(0, 0): 1, (1, 0): -2},
                [_FP16_HALF, _FP16_QUARTER] + [_FP16_ONE] * (H - 2))
    h_bits, y = M.expert_forward(_one_hot_row(H), _stack([e]), 0, G)
    h = oracle.bf16_to_f64(h_bits)
    assert h[0, 0] == -5.28125 and np.all(h[0, 1:] == 0.0)
    assert y[0, 0] == -2.640625 and y[0, 1] == 2.640625 and np.all(y[0, 2:] == 0.0)


def test_moe_combine_rank_order_closed_form():
    # expert 0: y_0[0] = bf16(silu(1)) = 0.73046875; expert 1: y_1[0] = 2 * bf16(silu(2)) = 3.515625.
    # router logits (0, 1): expert 1 ranks first with weight e / (1 + e), expert 0 second with 1 / (1 + e).
    H = F = G = 32
    e0 = _expert(H, F, G, {(0, 0): 1}, {(0, 0): 1}, {(0, 0): 1}, [_FP16_ONE] * H)
    e1 = _expert(H, F, G, {(0, 0): 2}, {(0, 0): 1}, {(0, 0): 2}, [_FP16_ONE] * H)
    z = np.array([[0.0, 1.0]], dtype=np.float32)
    out, ids, w, ysel = M.moe(_one_hot_row(H), z, _stack([e0, e1]), G, top_k=2)
    assert ids[0].tolist() == [1, 0]
    assert ysel[0, 0, 0] == 3.515625 and ysel[0, 1, 0] == 0.73046875
    w_first, w_second = 0.7310585786300049, 0.2689414213699951   # e/(1+e), 1/(1+e)
    assert w[0, 0] == pytest.approx(w_first, rel=1e-15) and w[0, 1] == pytest.approx(w_second, rel=1e-15)
    assert out[0, 0] == pytest.approx(w_first * 3.515625 + w_second * 0.73046875, rel=1e-15)
    assert np.all(out[0, 1:] == 0.0)


def _block(H, F, G, gate, up, down, down_scale_bits):
    return _expert(H, F, G, gate, up, down, [down_scale_bits] * H)


def test_block_residual_kept_when_down_is_zero():
    # zero down-projection codes: the block adds nothing and x comes back unchanged
    H = F = G = 64
    rng = inputs.rng_for(33)
    x = rng.standard_normal((3, H))
    blk = _block(H, F, G, {(0, 0): 3, (5, 7): -2}, {(0, 0): 1, (5, 9): 4}, {}, _FP16_ONE)
    assert np.array_equal(D.block_forward(x, blk, G), x)


def test_block_rmsnorm_swiglu_residual_closed_form():
    # a constant row c = 2^-10: RMSNorm gives c / sqrt(c^2 + 1e-6) = 0.698672998985... -> bf16 0.69921875
    # in every entry (without the norm the GEMMs would see 2^-10).  Gate row 0 reads 1 * n_0,
    # up row 0 reads 2 * n_0 = 1.3984375; h_0 = bf16(silu(0.69921875) * 1.3984375)
    # = bf16(0.65319377915...) = 0.65234375; down row 0 reads 0.25 * h_0 = 0.1630859375,
    # added to the residual: x_0 = 2^-10 + 0.1630859375 = 0.1640625, every other entry stays 2^-10.
    H = F = G = 64
    c = 2.0 ** -10
    assert c / math.sqrt(c * c + 1e-6) == pytest.approx(0.6986729989854964, rel=1e-15)
    blk = _block(H, F, G, {(0, 0): 1}, {(0, 0): 2}, {(0, 0): 1}, _FP16_QUARTER)
    x = np.full((2, H), c)
    out = D.block_forward(x, blk, G)
    assert np.all(out[:, 0] == 0.1640625)
    assert np.all(out[:, 1:] == c)


def _mutant_block(kind):
    def block_forward(x, blk, group):
        n = x if kind == "no_norm" else NUM.rms_norm(x, D.EPS)
        n_bits = NUM.bf16_bits_of(NUM.bf16_round(n))
        g = oracle.w4_linear(blk["gate_codes"], blk["gate_scales"], n_bits, group)
        u = oracle.w4_linear(blk["up_codes"], blk["up_scales"], n_bits, group)
        act = NUM.silu(u) * g if kind == "silu_on_up" else NUM.silu(g) * u
        h_bits = NUM.bf16_bits_of(NUM.bf16_round(act))
        d = oracle.w4_linear(blk["down_codes"], blk["down_scales"], h_bits, group)
        return d if kind == "no_residual" else x + d
    return block_forward


@pytest.mark.parametrize("kind", ["no_norm", "silu_on_up", "no_residual"])
def test_planted_block_mistakes_are_caught(monkeypatch, kind):
    monkeypatch.setattr(D, "block_forward", _mutant_block(kind))
    with pytest.raises(AssertionError):
        test_block_residual_kept_when_down_is_zero()
        test_block_rmsnorm_swiglu_residual_closed_form()


def test_planted_expert_silu_on_up_is_caught(monkeypatch):
    def expert_forward(x_bits, W, e, group):
        g = oracle.w4_linear(W["gate_codes"][e], W["gate_scales"][e], x_bits, group)
        u = oracle.w4_linear(W["up_codes"][e], W["up_scales"][e], x_bits, group)
        h_bits = NUM.bf16_bits_of(NUM.bf16_round(NUM.silu(u) * g))
        return h_bits, oracle.w4_linear(W["down_codes"][e], W["down_scales"][e], h_bits, group)
    monkeypatch.setattr(M, "expert_forward", expert_forward)
    with pytest.raises(AssertionError):
        test_expert_swiglu_closed_form()


def test_planted_combine_weights_permuted_is_caught(monkeypatch):
    orig = M.route

    def mutant(z, top_k=8):
        ids, w = orig(z, top_k)
        return ids, w[:, ::-1].copy()
    monkeypatch.setattr(M, "route", mutant)
    with pytest.raises(AssertionError):
        test_moe_combine_rank_order_closed_form()
