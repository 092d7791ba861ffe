"""The LM-head verify step at full size: W4 group-64 5120 -> 151936, R = 1..16.

* logits against the fp64 oracle on sampled columns (max |err| <= 1e-3 * rms);
* every row byte-equal to its own 1-row launch, for every R in 1..16;
* the GPU sampler on the GPU's logits gives the oracle sampler's tokens on the
  same logits (greedy, T=0.6/top-k 20/top-p 0.95, T=1.0/top-k 50/top-p 0.8;
  64-bit seeds, positions in [0, 65536)); a mismatch is only allowed as a
  logged near-tie;
* acceptance of drafts that copy the oracle token with probability 0.6:
  accepted length and bonus token equal the oracle's.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import accept as oacc
from oracle import sampling as osamp
from w4_gemm_keyed_gb300 import inputs
from gpu_util import assert_close_rows, dev_bits16, pack

pytestmark = pytest.mark.gpu

K, V, G = 5120, 151936, 64
SETTINGS = [(0.0, 0, 1.0), (0.6, 20, 0.95), (1.0, 50, 0.8)]


@pytest.fixture(scope="module")
def lmhead(tf):
    rng = inputs.rng_for(3, K, V)
    codes, scales = inputs.w4_weights(rng, K, V, G)
    x = inputs.bf16_normal(rng, (16, K))
    W = pack(tf, codes, scales, G)
    logits = tf.lane_gemm_w4(W, dev_bits16(x))
    return codes, scales, x, W, logits


def test_logits_match_oracle_on_sampled_columns(tf, lmhead):
    codes, scales, x, W, logits = lmhead
    rng = np.random.default_rng(31)
    cols = np.unique(np.concatenate([[0, 1, 255, 256, V // 2, V - 2, V - 1], rng.integers(0, V, 512)]))
    ref = oracle.w4_linear(codes, scales, x, G, cols=cols)
    assert_close_rows(logits.cpu().numpy()[:, cols], ref)


def test_rows_are_invariant_to_R(tf, lmhead):
    codes, scales, x, W, logits = lmhead
    xd = dev_bits16(x)
    single = np.stack([tf.lane_gemm_w4(W, xd[r:r + 1]).cpu().numpy()[0] for r in range(16)])
    for R in range(1, 17):
        y = tf.lane_gemm_w4(W, xd[:R]).cpu().numpy()
        assert np.array_equal(y.view(np.uint32), single[:R].view(np.uint32)), f"R={R}"


@pytest.mark.parametrize("T,k,p", SETTINGS)
@pytest.mark.parametrize("R", [1, 2, 4, 8, 16])
def test_sample_and_accept_match_oracle(tf, lmhead, near_tie, R, T, k, p):
    codes, scales, x, W, _ = lmhead
    rng = inputs.rng_for(301, R, int(T * 10), k)
    logits = tf.lane_gemm_w4(W, dev_bits16(x[:R]))
    seed = int(inputs.seeds_u64(rng, 1)[0])
    pos = inputs.positions(rng, R)
    tokens = tf.keyed_sample(logits, T, k, p, seed, torch.from_numpy(pos).cuda()).cpu().numpy()
    host_logits = logits.cpu().numpy()
    ref, gaps = osamp.sample(host_logits, T, k, p, seed, pos)
    for r in range(R):
        if tokens[r] != ref[r]:
            assert gaps[r] < 1e-9, f"row {r}: gpu {tokens[r]} oracle {ref[r]} gap {gaps[r]}"
            near_tie(f"LM head R={R} T={T} k={k} p={p} row {r}", gaps[r])
    if R > 1:
        drafts = inputs.noisy_drafts(rng, ref[:R - 1], 0.6, V)
        acc, bonus = tf.accept(torch.from_numpy(drafts).cuda(), torch.from_numpy(tokens.astype(np.int32)).cuda())
        a_ref, bonus_ref = oacc.accept(drafts, tokens)
        assert (int(acc.item()), int(bonus.item())) == (a_ref, bonus_ref)
