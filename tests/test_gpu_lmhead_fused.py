"""tf_lmhead_sample: the LM head with its candidate epilogue, then the finaliser.

* full size (W4 group-64 5120 -> 151936, R = 1..16, greedy / T=0.6 top-k 20
  top-p 0.95 / T=1.0 top-k 50 top-p 0.8): the tokens equal the oracle
  sampler's on the same logits (a mismatch only as a logged near-tie) and the
  tokens of tf_lane_gemm_w4 followed by tf_keyed_sample bit for bit; the
  logits it stores on request are byte-equal to tf_lane_gemm_w4's;
* each row's token is the same whatever R is;
* small ragged shapes (grids of 1-152 CTAs, CTAs that store no block, k' up to
  the vocabulary, V below one tile) against the oracle and the unfused path;
* a k' too large for the candidate pool, and top_k <= 0, take the unfused
  path and still give the same tokens;
* a non-finite logit gives that row -1 and TF_DEV_NONFINITE_LOGIT; the
  workspace is clean for the next call;
* with `accepted`, acceptance inside the call gives tf_accept's result on the
  same tokens (fused, unfused fast and general paths).
"""

import numpy as np
import pytest
import torch

from oracle import sampling as osamp
from w4_gemm_keyed_gb300 import inputs
from gpu_util import dev_bits16, pack

pytestmark = pytest.mark.gpu

K, V, G = 5120, 151936, 64
SETTINGS = [(0.0, 0, 1.0), (0.6, 20, 0.95), (1.0, 50, 0.8)]


@pytest.fixture(scope="module")
def head(tf):
    rng = inputs.rng_for(3, K, V)
    codes, scales = inputs.w4_weights(rng, K, V, G)
    x = inputs.bf16_normal(rng, (16, K))
    W = pack(tf, codes, scales, G)
    return W, dev_bits16(x)


def check_oracle(tokens, logits, T, k, p, seed, pos, near_tie, what):
    ref, gaps = osamp.sample(logits, T, k, p, seed, pos)
    for r in range(len(ref)):
        if tokens[r] != ref[r]:
            assert gaps[r] < 1e-9, f"{what} row {r}: gpu {tokens[r]} oracle {ref[r]} gap {gaps[r]}"
            near_tie(f"{what} row {r}", gaps[r])


@pytest.mark.parametrize("T,k,p", SETTINGS)
@pytest.mark.parametrize("R", [1, 2, 4, 8, 16])
def test_full_size_matches_oracle_and_unfused(tf, head, near_tie, R, T, k, p):
    W, x = head
    rng = inputs.rng_for(311, R, int(T * 10), k)
    seed = int(inputs.seeds_u64(rng, 1)[0])
    pos = inputs.positions(rng, R)
    pd = torch.from_numpy(pos).cuda()
    logits = torch.empty((R, V), device="cuda")
    fused = tf.lmhead_sample(W, x[:R], T, k, p, seed, pd, logits=logits).cpu().numpy()
    ref_logits = tf.lane_gemm_w4(W, x[:R])
    assert torch.equal(logits.view(torch.int32), ref_logits.view(torch.int32))
    unfused = tf.keyed_sample(ref_logits, T, k, p, seed, pd).cpu().numpy()
    assert np.array_equal(fused, unfused)
    check_oracle(fused, logits.cpu().numpy(), T, k, p, seed, pos, near_tie, f"fused LM head R={R} T={T} k={k}")


def test_rows_do_not_depend_on_R(tf, head):
    W, x = head
    pos = torch.arange(100, 116, dtype=torch.int64, device="cuda")
    single = [int(tf.lmhead_sample(W, x[r:r + 1], 0.6, 20, 0.95, 77, pos[r:r + 1]).item()) for r in range(16)]
    for R in (2, 5, 8, 9, 16):
        t = tf.lmhead_sample(W, x[:R], 0.6, 20, 0.95, 77, pos[:R]).cpu().numpy()
        assert list(t) == single[:R], f"R={R}"


@pytest.mark.parametrize("Ks,N", [(128, 1), (128, 37), (128, 128), (192, 129), (128, 1000), (256, 4097),
                                  (64, 19584)])
@pytest.mark.parametrize("R", [1, 3, 9, 16])
def test_ragged_shapes(tf, near_tie, Ks, N, R):
    rng = inputs.rng_for(313, Ks, N, R)
    codes, scales = inputs.w4_weights(rng, Ks, N, G)
    W = pack(tf, codes, scales, G)
    x = dev_bits16(inputs.bf16_normal(rng, (R, Ks)))
    pos = inputs.positions(rng, R)
    pd = torch.from_numpy(pos).cuda()
    logits = tf.lane_gemm_w4(W, x)
    host = logits.cpu().numpy()
    for T, k, p in [(0.0, 0, 1.0), (0.8, 5, 0.9), (0.7, 20, 0.95), (1.2, 53, 1.0), (0.9, N, 0.5)]:
        seed = 1000 + k
        fused = tf.lmhead_sample(W, x, T, k, p, seed, pd).cpu().numpy()
        unfused = tf.keyed_sample(logits, T, k, p, seed, pd).cpu().numpy()
        assert np.array_equal(fused, unfused), f"T={T} k={k}"
        if k <= 64:
            check_oracle(fused, host, T, k, p, seed, pos, near_tie, f"fused {Ks}x{N} R={R} T={T} k={k}")


@pytest.mark.parametrize("k", [60, 64, 0])
def test_large_k_takes_the_unfused_path(tf, head, k):
    W, x = head
    R = 4
    pd = torch.arange(7, 7 + R, dtype=torch.int64, device="cuda")
    fused = tf.lmhead_sample(W, x[:R], 0.8, k, 0.9, 4242, pd).cpu().numpy()
    unfused = tf.keyed_sample(tf.lane_gemm_w4(W, x[:R]), 0.8, k, 0.9, 4242, pd).cpu().numpy()
    assert np.array_equal(fused, unfused)


def test_nonfinite_row_and_clean_workspace(tf):
    rng = inputs.rng_for(317)
    Ks, N, R = 128, 3000, 3
    codes, scales = inputs.w4_weights(rng, Ks, N, G)
    W = pack(tf, codes, scales, G)
    xb = inputs.bf16_normal(rng, (R, Ks))
    xb[1, 7] = 0x7F80   # +inf
    x = dev_bits16(xb)
    pd = torch.zeros(R, dtype=torch.int64, device="cuda")
    ws = tf.workspace(tf.lmhead_sample_workspace_bytes(W, R))
    t = tf.lmhead_sample(W, x, 0.7, 20, 0.9, 5, pd, ws=ws).cpu().numpy()
    assert t[1] == -1 and t[0] >= 0 and t[2] >= 0
    assert tf.workspace_status(ws) == tf.TF_DEV_NONFINITE_LOGIT
    xb[1, 7] = 0x3F80   # 1.0
    t2 = tf.lmhead_sample(W, dev_bits16(xb), 0.7, 20, 0.9, 5, pd, ws=ws).cpu().numpy()
    assert tf.workspace_status(ws) == tf.TF_DEV_OK
    ref = tf.keyed_sample(tf.lane_gemm_w4(W, dev_bits16(xb)), 0.7, 20, 0.9, 5, pd).cpu().numpy()
    assert np.array_equal(t2, ref)


def test_repeat_calls_reuse_the_workspace(tf, head):
    W, x = head
    R = 8
    pd = torch.arange(R, dtype=torch.int64, device="cuda")
    ws = tf.workspace(tf.lmhead_sample_workspace_bytes(W, R))
    a = tf.lmhead_sample(W, x[:R], 0.6, 20, 0.95, 9, pd, ws=ws).clone()
    b = tf.lmhead_sample(W, x[:R], 0.6, 20, 0.95, 9, pd, ws=ws).clone()
    c = tf.lmhead_sample(W, x[:R], 0.0, 0, 1.0, 9, pd, ws=ws).clone()
    assert torch.equal(a, b)
    assert torch.equal(c, tf.keyed_sample(tf.lane_gemm_w4(W, x[:R]), 0.0, 0, 1.0, 9, pd))


@pytest.mark.parametrize("k", [20, 60, 0])
@pytest.mark.parametrize("R", [1, 2, 7, 16])
def test_acceptance_in_the_call(tf, head, R, k):
    """With `accepted`, the finaliser (or, for the general path, a launch after
    it) accepts the drafts: the same accepted length and bonus as tf_accept on
    the same tokens; drafts copy the tokens up to a chosen point."""
    W, x = head
    pd = torch.arange(30, 30 + R, dtype=torch.int64, device="cuda")
    ref_tokens = tf.lmhead_sample(W, x[:R], 0.8, k, 0.9, 99, pd).clone()
    for cut in sorted({0, R // 2, R - 1}):
        drafts = ref_tokens[:max(R - 1, 1)].clone()
        if cut < R - 1:
            drafts[cut] = (drafts[cut] + 1) % 151936
        acc = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        bonus = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        t = tf.lmhead_sample(W, x[:R], 0.8, k, 0.9, 99, pd, drafts=drafts, accepted=acc, bonus=bonus)
        assert torch.equal(t, ref_tokens)
        a_ref, b_ref = tf.accept(drafts, t)
        assert (int(acc.item()), int(bonus.item())) == (int(a_ref.item()), int(b_ref.item())), f"cut={cut}"
