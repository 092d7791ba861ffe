"""Pins of the keyed-sampling oracle.

* SplitMix64 against its published output sequence (tests/golden);
* the uniform / Gumbel maps at their closed-form extremes, and a
  Kolmogorov-Smirnov test of g against the Gumbel CDF;
* the candidate set against hand-computed closed forms and against a
  set-based restatement, brute-forced over tiny vocabularies with ties;
* Gumbel-max frequencies against softmax(l / T) restricted to the
  candidates (chi-square), for several vocabularies and settings;
* planted mistakes in the oracle, each caught by one of the pins.
"""

import itertools
import math
import os

import numpy as np
import pytest

from oracle import sampling as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "splitmix64_seed1234567.txt")


def _golden_values():
    return [int(l) for l in open(GOLDEN) if l.strip() and not l.startswith("#")]


def test_splitmix64_published_sequence():
    state = 1234567
    got = []
    for _ in range(5):
        got.append(S.splitmix64(state))
        state = (state + 0x9E3779B97F4A7C15) % 2**64
    assert got == _golden_values()


def test_key_hash_composition_and_word_widths():
    sm = S.splitmix64
    assert S.key_hash(7, 3, 11) == sm(sm(sm(7) ^ 3) ^ 11)
    # negative positions are 64-bit two's complement words, tokens 32-bit words
    assert S.key_hash(7, -1, 5) == sm(sm(sm(7) ^ (2**64 - 1)) ^ 5)
    assert S.key_hash(7, 2, -1) == sm(sm(sm(7) ^ 2) ^ 0xFFFFFFFF)
    # the three inputs are not interchangeable
    assert len({S.key_hash(1, 2, 3), S.key_hash(2, 1, 3), S.key_hash(3, 2, 1)}) == 3


def test_uniform_extremes_closed_form():
    assert S.uniform_of(0) == 2.0 ** -54
    assert S.uniform_of((1 << 11) - 1) == 2.0 ** -54          # low 11 bits are dropped
    assert S.uniform_of(1 << 11) == 1.5 * 2.0 ** -53
    # m = 2^53 - 2: m + 0.5 is a tie in fp64 and rounds to the even m
    assert S.uniform_of((2**53 - 2) << 11) == (2**53 - 2) / 2.0**53
    # m = 2^53 - 1: m + 0.5 rounds (ties to even) to 2^53, so u = 1 and g = +inf
    assert S.uniform_of(2**64 - 1) == 1.0
    assert S.gumbel_of(2**64 - 1) == math.inf
    assert S.gumbel_of(0) == -math.log(-math.log(2.0 ** -54))


def test_gumbel_distribution_ks():
    scipy_stats = pytest.importorskip("scipy.stats")
    g = np.array([S.gumbel(99, pos, tok) for pos in range(200) for tok in range(100)])
    res = scipy_stats.kstest(g, "gumbel_r")
    assert res.pvalue > 1e-3
    assert abs(g.mean() - 0.5772156649) < 0.03


def test_greedy_ties_and_signed_zero():
    assert S.sample_row(np.array([1, 3, 3, 2], np.float32), 0.0, 20, 0.9, 1, 1)[0] == 1
    assert S.sample_row(np.array([-0.0, 0.0], np.float32), 0.0, 0, 1.0, 1, 1)[0] == 0
    assert S.sample_row(np.array([0.0, -0.0, 5.0], np.float32), 0.0, 0, 1.0, 1, 1)[0] == 2


def test_candidate_set_closed_forms():
    flat = np.zeros(4, np.float32)  # q = 1/4 each, sums exact in binary
    assert S.candidate_set(flat, 1.0, 0, 0.5).tolist() == [0, 1]      # S_2 = 0.5 >= 0.5
    assert S.candidate_set(flat, 1.0, 0, 0.6).tolist() == [0, 1, 2]
    assert S.candidate_set(flat, 1.0, 0, 0.0).tolist() == [0]
    assert S.candidate_set(flat, 1.0, 0, 1.0).tolist() == [0, 1, 2, 3]
    assert S.candidate_set(flat, 1.0, 3, 1.0).tolist() == [0, 1, 2]  # ties at the k-th: lower ids
    l = np.array([0.0, math.log(3.0), 0.0, 5.0], np.float32)
    assert S.candidate_set(l, 1.0, 2, 1.0).tolist() == [3, 1]
    assert S.candidate_set(l, 1.0, 10, 1.0).tolist() == [3, 1, 0, 2]  # k >= V keeps all
    # two tokens with masses 3/4 and 1/4 after top-k=2 renormalisation (T=1)
    two = np.array([math.log(3.0), 0.0, -50.0], np.float32)
    assert S.candidate_set(two, 1.0, 2, 0.7).tolist() == [0]
    assert S.candidate_set(two, 1.0, 2, 0.8).tolist() == [0, 1]


def _restated_candidates(l32, T, top_k, top_p):
    """Set-based restatement: token i is kept iff its rank is below k' and the
    renormalised mass of the tokens ranked strictly before it is below top_p
    (the top-ranked token is always kept: the prefix has at least one token)."""
    V = l32.size
    key = sorted(range(V), key=lambda i: (-float(l32[i]), i))
    rank = {i: r for r, i in enumerate(key)}
    kk = V if (top_k <= 0 or top_k >= V) else top_k
    top = [i for i in range(V) if rank[i] < kk]
    p = float(np.float32(top_p))
    if p >= 1.0:
        return set(top)
    l0 = float(l32[key[0]])
    e = {i: math.exp((float(l32[i]) - l0) / T) for i in top}
    Z = 0.0
    for i in key[:kk]:
        Z += e[i]
    keep = set()
    for i in top:
        before = 0.0
        for j in key[: rank[i]]:
            before += e[j] / Z
        if before < p or rank[i] == 0:
            keep.add(i)
    return keep


def test_candidate_set_brute_force_tiny_vocab():
    grid = [-1.0, 0.0, 0.5, 2.0]
    count = 0
    for V in (1, 2, 3, 4):
        for vals in itertools.product(grid, repeat=V):
            l = np.array(vals, np.float32)
            for top_k in range(0, V + 2):
                for top_p in (0.0, 0.3, 0.5, 0.9, 0.95, 1.0):
                    for T in (0.5, 1.0, 2.0):
                        got = S.candidate_set(l, T, top_k, top_p)
                        assert len(got) >= 1
                        assert set(got.tolist()) == _restated_candidates(l, T, top_k, top_p)
                        # rank order within the returned list
                        keys = [(-float(l[i]), int(i)) for i in got]
                        assert keys == sorted(keys)
                        count += 1
    assert count > 10000


@pytest.mark.parametrize("V,T,top_k,top_p", [(4, 1.0, 0, 1.0), (16, 0.7, 10, 0.9), (64, 0.6, 20, 0.95),
                                             (64, 1.0, 50, 0.8)])
def test_gumbel_max_frequencies_match_softmax(V, T, top_k, top_p):
    scipy_stats = pytest.importorskip("scipy.stats")
    rng = np.random.default_rng(V * 1000 + top_k)
    l = (rng.standard_normal(V) * 0.5).astype(np.float32)
    cand = S.candidate_set(l, T, top_k, top_p)
    assert len(cand) >= 3  # a distribution worth testing
    ll = l[cand].astype(np.float64) / np.float64(np.float32(T))
    p = np.exp(ll - ll.max())
    p /= p.sum()
    n = 20000
    counts = {int(i): 0 for i in cand}
    for pos in range(n):
        t, _ = S.sample_row(l, T, top_k, top_p, seed=424242, pos=pos)
        assert t in counts
        counts[t] += 1
    obs = np.array([counts[int(i)] for i in cand], dtype=np.float64)
    exp = p * n
    # pool tiny-expectation cells so the chi-square approximation holds
    big = exp >= 5
    obs_b = np.append(obs[big], obs[~big].sum())
    exp_b = np.append(exp[big], exp[~big].sum())
    if exp_b[-1] == 0:
        obs_b, exp_b = obs_b[:-1], exp_b[:-1]
    res = scipy_stats.chisquare(obs_b, exp_b)
    assert res.pvalue > 1e-3


# ----------------------------------------------------------------------------
# Planted mistakes in the oracle (on the CPU): each must fail a pin.
# ----------------------------------------------------------------------------
def _mutant_hash_order(seed, pos, token):
    s = S.splitmix64(int(seed) & S.M64)
    s = S.splitmix64(s ^ (int(token) & 0xFFFFFFFF))
    return S.splitmix64(s ^ (int(pos) & S.M64))


_ORIG_CANDIDATES = S.candidate_set


def _mutant_candidate_exclusive(l, T, top_k, top_p):
    order = _ORIG_CANDIDATES(l, T, top_k, 1.0)
    full = _ORIG_CANDIDATES(l, T, top_k, top_p)
    return full[:-1] if (len(full) > 1 and len(full) < len(order)) else full


@pytest.mark.parametrize("mutant", ["gumbel_sign", "hash_order", "crossing_token_dropped", "temperature_ignored"])
def test_planted_mistakes_are_caught(monkeypatch, mutant):
    if mutant == "gumbel_sign":
        monkeypatch.setattr(S, "gumbel_of", lambda h: math.log(-math.log(S.uniform_of(h))))
        pins = [test_uniform_extremes_closed_form, test_gumbel_distribution_ks]
    elif mutant == "hash_order":
        monkeypatch.setattr(S, "key_hash", _mutant_hash_order)
        pins = [test_key_hash_composition_and_word_widths]
    elif mutant == "crossing_token_dropped":
        monkeypatch.setattr(S, "candidate_set", _mutant_candidate_exclusive)
        pins = [test_candidate_set_closed_forms, test_candidate_set_brute_force_tiny_vocab]
    else:
        orig = S.sample_row

        def no_temp(l, T, k, p, seed, pos):
            return orig(l, 1.0 if T > 0 else 0.0, k, p, seed, pos)
        monkeypatch.setattr(S, "sample_row", no_temp)
        pins = [lambda: test_gumbel_max_frequencies_match_softmax(64, 0.6, 20, 0.95)]
    caught = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError):
            caught += 1
    assert caught >= 1
