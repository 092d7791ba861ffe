"""Keyed sampler and acceptance on the GPU against the oracle.

Given identical logits the token ids must be identical; a mismatch is only
tolerated as a logged near-tie (oracle score gap < 1e-9, where the fp64 log /
exp of the two sides may round differently).
"""

import math

import numpy as np
import pytest
import torch

from oracle import accept as oacc
from oracle import sampling as osamp
from w4_gemm_keyed_gb300 import inputs

pytestmark = pytest.mark.gpu

SETTINGS = [(0.0, 0, 1.0), (0.6, 20, 0.95), (1.0, 50, 0.8), (0.7, 20, 0.95), (1.3, 64, 0.99), (0.9, 7, 1.0),
            (0.5, 33, 0.3)]


def gpu_sample(tf, logits, T, k, p, seed, pos):
    t = tf.keyed_sample(torch.from_numpy(logits).cuda(), T, k, p, seed, torch.from_numpy(pos).cuda())
    return t.cpu().numpy()


def check_tokens(gpu, logits, T, k, p, seed, pos, near_tie=None):
    ref, gaps = osamp.sample(logits, T, k, p, seed, pos)
    for r in range(len(ref)):
        if gpu[r] != ref[r]:
            assert gaps[r] < 1e-9, f"row {r}: gpu {gpu[r]} oracle {ref[r]} gap {gaps[r]}"
            if near_tie is not None:
                near_tie(f"V={logits.shape[1]} T={T} k={k} p={p} row {r}", gaps[r])


@pytest.mark.parametrize("T,k,p", SETTINGS)
@pytest.mark.parametrize("V", [1024, 151936, 8193])
def test_tokens_match_oracle(tf, near_tie, V, T, k, p):
    rng = inputs.rng_for(201, V, int(T * 10), k)
    R = 16
    logits = inputs.logits_normal(rng, R, V, std=2.0)
    seed = int(inputs.seeds_u64(rng, 1)[0])
    pos = inputs.positions(rng, R)
    check_tokens(gpu_sample(tf, logits, T, k, p, seed, pos), logits, T, k, p, seed, pos, near_tie)


@pytest.mark.parametrize("T,k,p", SETTINGS)
def test_ties_follow_the_lower_id(tf, near_tie, T, k, p):
    rng = inputs.rng_for(202, k)
    R, V = 16, 5000
    logits = rng.integers(-3, 2, size=(R, V)).astype(np.float32)   # massive ties
    logits[3, :] = 0.0
    logits[4, ::2] = -0.0                                            # signed zeros tie with +0
    seed = 1234
    pos = np.arange(R, dtype=np.int64)
    check_tokens(gpu_sample(tf, logits, T, k, p, seed, pos), logits, T, k, p, seed, pos, near_tie)


@pytest.mark.parametrize("n_top,p", [(4, 0.5), (4, 0.25), (4, 0.75), (8, 0.125), (8, 0.5 + 1e-6), (8, 0.5 - 1e-6)])
def test_top_p_cut_on_a_mass_boundary(tf, near_tie, n_top, p):
    """n_top equal leading logits (the rest negligible) put the cumulative mass
    exactly on, or within 1e-6 of, p at the cut: the fp32 pass cannot decide
    there and the fp64 sums must give the oracle's prefix."""
    R, V = 16, 3000
    logits = np.full((R, V), -1.0e4, dtype=np.float32)
    rng = inputs.rng_for(205, n_top, int(p * 1e6))
    for r in range(R):
        ids = rng.choice(V, size=n_top, replace=False)
        logits[r, ids] = 1.5
    seed, pos = 77, np.arange(R, dtype=np.int64) * 3
    for T, k in ((1.0, 20), (0.7, 64), (2.0, 0)):
        check_tokens(gpu_sample(tf, logits, T, k, p, seed, pos), logits, T, k, p, seed, pos, near_tie)


@pytest.mark.parametrize("T,k,p", [(1.0, 64, 1.0), (1.0, 20, 0.9), (3.0, 50, 0.95)])
def test_large_logits_take_the_fp64_decision(tf, near_tie, T, k, p):
    """Logits near 1e5 widen the fp32 scores' error bound to ~0.05, so several
    candidates often survive the fp32 filter and the fp64 scores decide."""
    rng = inputs.rng_for(206, k, int(T * 10))
    R, V = 16, 2048
    for _ in range(4):
        logits = (1.0e5 + rng.normal(0.0, 0.3, size=(R, V))).astype(np.float32)
        seed = int(inputs.seeds_u64(rng, 1)[0])
        pos = inputs.positions(rng, R)
        check_tokens(gpu_sample(tf, logits, T, k, p, seed, pos), logits, T, k, p, seed, pos, near_tie)


@pytest.mark.parametrize("V", [1, 2, 5, 63, 64, 4096, 4097])
def test_small_and_ragged_vocabularies(tf, near_tie, V):
    rng = inputs.rng_for(203, V)
    R = 4
    logits = inputs.logits_normal(rng, R, V, std=1.0)
    pos = inputs.positions(rng, R)
    for T, k, p in [(0.0, 0, 1.0), (0.8, 0 if V <= 64 else 64, 0.9), (1.0, 3, 0.5)]:
        check_tokens(gpu_sample(tf, logits, T, k, p, 77, pos), logits, T, k, p, 77, pos, near_tie)


def test_nonfinite_logits_flag_the_row(tf):
    R, V = 3, 3000
    logits = np.zeros((R, V), np.float32)
    logits[1, 2999] = np.nan
    logits[2, 5] = np.inf
    ws = tf.workspace(tf.keyed_sample_workspace_bytes(R, V))
    t = tf.keyed_sample(torch.from_numpy(logits).cuda(), 0.7, 20, 0.9, 5,
                        torch.zeros(R, dtype=torch.int64, device="cuda"), ws=ws).cpu().numpy()
    assert t[1] == -1 and t[2] == -1 and t[0] >= 0
    assert tf.workspace_status(ws) == tf.TF_DEV_NONFINITE_LOGIT
    # the workspace is clean again: a finite call reports OK
    tf.keyed_sample(torch.zeros((R, V), device="cuda"), 0.7, 20, 0.9, 5,
                    torch.zeros(R, dtype=torch.int64, device="cuda"), ws=ws)
    assert tf.workspace_status(ws) == tf.TF_DEV_OK


# ---------------------------------------------------------------- general candidate path (k' > 64)
def check_tokens_general(gpu, logits, T, k, p, seed, pos, near_tie):
    """Identical tokens, except where the oracle itself sits on a knife edge:
    a top-2 score gap below 1e-9, or a top-p cut whose running sum lies within
    1e-9 of top_p (the general path sums the mass in another fixed order)."""
    ref, gaps = osamp.sample(logits, T, k, p, seed, pos)
    for r in range(len(ref)):
        if gpu[r] != ref[r]:
            margin = osamp.topp_margin(logits[r], T, k, p)
            assert gaps[r] < 1e-9 or margin < 1e-9, \
                f"row {r}: gpu {gpu[r]} oracle {ref[r]} gap {gaps[r]} top-p margin {margin}"
            near_tie(f"general V={logits.shape[1]} T={T} k={k} p={p} row {r}", min(gaps[r], margin))


@pytest.mark.parametrize("k", [0, 65, 1000, 151936])
@pytest.mark.parametrize("T,p", [(0.7, 0.95), (1.0, 0.8), (0.6, 1.0)])
def test_general_candidate_path_matches_oracle(tf, near_tie, k, T, p):
    rng = inputs.rng_for(205, k, int(T * 10), int(p * 100))
    R, V = 4, 151936
    logits = inputs.logits_normal(rng, R, V, std=2.0)
    seed = int(inputs.seeds_u64(rng, 1)[0])
    pos = inputs.positions(rng, R)
    check_tokens_general(gpu_sample(tf, logits, T, k, p, seed, pos), logits, T, k, p, seed, pos, near_tie)


def test_general_path_ties_and_small_vocabularies(tf, near_tie):
    rng = inputs.rng_for(206)
    for V in (65, 66, 1000, 4097):
        logits = rng.integers(-3, 3, size=(3, V)).astype(np.float32)   # heavy ties at every boundary
        pos = inputs.positions(rng, 3)
        for T, k, p in ((0.8, 0, 0.9), (1.0, 65, 0.5), (0.5, V - 1, 1.0), (1.3, 100, 0.99)):
            check_tokens_general(gpu_sample(tf, logits, T, k, p, 17, pos), logits, T, k, p, 17, pos, near_tie)


@pytest.mark.parametrize("dist", ["narrow", "wide", "quantised"])
@pytest.mark.parametrize("k,T,p", [(0, 0.7, 0.01), (0, 1.0, 0.999999), (3000, 0.9, 0.9), (0, 0.05, 0.5)])
def test_general_path_logit_shapes(tf, near_tie, dist, k, T, p):
    """Logit distributions that take the radix select and the top-p walk
    through their gathering steps at different depths: a narrow spread (the
    leading digits never split), a wide one, and coarse steps (long runs of
    equal logits, broken by id)."""
    rng = inputs.rng_for(208, ["narrow", "wide", "quantised"].index(dist), k, int(p * 1e6))
    R, V = 3, 151936
    if dist == "narrow":
        logits = (1.5 + 0.01 * rng.standard_normal((R, V))).astype(np.float32)
    elif dist == "wide":
        logits = (10.0 * rng.standard_normal((R, V))).astype(np.float32)
    else:
        logits = np.round(2.0 * rng.standard_normal((R, V)) * 8.0).astype(np.float32) / 8.0
    pos = inputs.positions(rng, R)
    check_tokens_general(gpu_sample(tf, logits, T, k, p, 23, pos), logits, T, k, p, 23, pos, near_tie)


@pytest.mark.parametrize("T", [1.0, 0.05, 30.0])
def test_general_path_noise_decides(tf, near_tie, T):
    """Equal logits over the whole vocabulary (top-k <= 0, top-p 1): the token
    is the argmax of the Gumbel noise alone, which the general path first
    estimates in fp32 with an error bound and then settles in fp64; 16 rows
    x 4 seeds against the oracle."""
    R, V = 16, 151936
    rng = inputs.rng_for(209, int(T * 100))
    logits = np.full((R, V), 0.25, dtype=np.float32)
    for seed in inputs.seeds_u64(rng, 4):
        pos = inputs.positions(rng, R)
        check_tokens_general(gpu_sample(tf, logits, T, 0, 1.0, int(seed), pos), logits, T, 0, 1.0, int(seed), pos,
                             near_tie)


def test_general_path_rows_independent_of_R_and_nan_rows(tf):
    rng = inputs.rng_for(207)
    V = 151936
    logits = inputs.logits_normal(rng, 16, V, std=2.0)
    pos = inputs.positions(rng, 16)
    full = gpu_sample(tf, logits, 0.8, 0, 0.9, 31, pos)
    for r in (0, 9, 15):
        assert gpu_sample(tf, logits[r:r + 1], 0.8, 0, 0.9, 31, pos[r:r + 1])[0] == full[r]
    logits[3, 1234] = np.nan
    ws = tf.workspace(tf.keyed_sample_workspace_bytes(16, V))
    t = tf.keyed_sample(torch.from_numpy(logits).cuda(), 0.8, 0, 0.9, 31, torch.from_numpy(pos).cuda(), ws=ws)
    t = t.cpu().numpy()
    assert t[3] == -1 and np.array_equal(np.delete(t, 3), np.delete(full, 3))
    assert tf.workspace_status(ws) == tf.TF_DEV_NONFINITE_LOGIT


def test_rows_independent_of_R(tf):
    rng = inputs.rng_for(204)
    V = 151936
    logits = inputs.logits_normal(rng, 16, V, std=2.0)
    pos = inputs.positions(rng, 16)
    full = gpu_sample(tf, logits, 0.6, 20, 0.95, 99, pos)
    for r in (0, 7, 15):
        one = gpu_sample(tf, logits[r:r + 1], 0.6, 20, 0.95, 99, pos[r:r + 1])
        assert one[0] == full[r]


def test_accept_brute_force(tf):
    import itertools
    for R in range(1, 5):
        for V in range(1, 4):
            combos_t = list(itertools.product(range(V), repeat=R))
            combos_d = list(itertools.product(range(V), repeat=R - 1))
            for t in combos_t:
                for d in combos_d:
                    dd = torch.tensor(list(d) or [0], dtype=torch.int32, device="cuda")
                    tt = torch.tensor(list(t), dtype=torch.int32, device="cuda")
                    a, b = tf.accept(dd, tt)
                    assert (int(a.item()), int(b.item())) == oacc.accept(d, t)


def test_accept_sixteen_rows(tf):
    rng = np.random.default_rng(5)
    for _ in range(50):
        t = rng.integers(0, 3, 16)
        d = np.where(rng.random(15) < 0.8, t[:15], rng.integers(0, 3, 15))
        a, b = tf.accept(torch.from_numpy(d.astype(np.int32)).cuda(), torch.from_numpy(t.astype(np.int32)).cuda())
        assert (int(a.item()), int(b.item())) == oacc.accept(d, t)
