"""W4 lane GEMM on the GPU against the fp64 oracle, and row invariance.

* one-hot activations: every output is a single code * scale product, so the
  GPU must match the oracle bit for bit (checks packing, nibble order, scale
  placement, stream-K fixup and ragged tails exactly);
* seeded workloads (tiny, ragged, group 32, the 27B-class projections at full
  size on sampled columns): max |err| <= 1e-3 * rms(oracle row);
* row invariance: each row of an R-row launch is byte-equal to its own 1-row
  launch, at the full 27B-class sizes, for every R in 1..16.
"""

import numpy as np
import pytest

import oracle
from w4_gemm_keyed_gb300 import inputs
from gpu_util import assert_close_rows, dev_bits16, pack

pytestmark = pytest.mark.gpu


def run(tf, W, x_bits, ws=None):
    return tf.lane_gemm_w4(W, dev_bits16(x_bits), ws=ws).cpu().numpy()


@pytest.mark.parametrize("K,N,G", [(256, 1024, 64), (192, 300, 32), (64, 1, 64), (1024, 777, 32), (5120, 640, 64)])
def test_one_hot_is_bit_exact(tf, K, N, G):
    rng = inputs.rng_for(101, K, N, G)
    codes, scales = inputs.w4_weights(rng, K, N, G)
    W = pack(tf, codes, scales, G)
    ks = sorted(k for k in set([0, 1, 15, 16, 17, G - 1, G, K // 2 + 3, K - 2, K - 1]) if k < K)[:16]
    x = np.zeros((len(ks), K), dtype=np.uint16)
    for r, k in enumerate(ks):
        x[r, k] = 0x3F80  # 1.0
    y = run(tf, W, x)
    ref = oracle.w4_linear(codes, scales, x, G).astype(np.float32)
    assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("K,N,G,R", [(256, 1024, 64, 1), (256, 1024, 64, 2), (256, 1024, 64, 4),
                                     (192, 300, 32, 5), (64, 1, 64, 16), (2048, 1536, 32, 9),
                                     (768, 2048, 32, 16), (512, 1000, 64, 8), (1024, 4096, 64, 13)])
def test_matches_oracle(tf, K, N, G, R):
    rng = inputs.rng_for(102, K, N, G, R)
    codes, scales = inputs.w4_weights(rng, K, N, G)
    x = inputs.bf16_normal(rng, (R, K))
    W = pack(tf, codes, scales, G)
    assert_close_rows(run(tf, W, x), oracle.w4_linear(codes, scales, x, G))


@pytest.fixture(scope="module", params=[(5120, 17408), (17408, 5120)], ids=["5120x17408", "17408x5120"])
def dense27b(request, tf):
    K, N = request.param
    rng = inputs.rng_for(2, K, N)
    codes, scales = inputs.w4_weights(rng, K, N, 64)
    x = inputs.bf16_normal(rng, (16, K))
    return K, N, codes, scales, x, pack(tf, codes, scales, 64)


def test_dense27b_matches_oracle_on_sampled_columns(tf, dense27b):
    K, N, codes, scales, x, W = dense27b
    rng = np.random.default_rng(7)
    cols = np.unique(np.concatenate([[0, 1, 255, 256, N // 2, N - 2, N - 1], rng.integers(0, N, 384)]))
    for R in (1, 2, 4, 8, 16):
        y = run(tf, W, x[:R])
        ref = oracle.w4_linear(codes, scales, x[:R], 64, cols=cols)
        # normalise by the full-row rms of the oracle estimate from the sampled columns
        assert_close_rows(y[:, cols], ref)


def test_dense27b_rows_are_invariant_to_R(tf, dense27b):
    K, N, codes, scales, x, W = dense27b
    single = np.stack([run(tf, W, x[r:r + 1])[0] for r in range(16)])
    for R in range(1, 17):
        y = run(tf, W, x[:R])
        assert np.array_equal(y.view(np.uint32), single[:R].view(np.uint32)), f"R={R}"


def test_workspace_reuse_and_status(tf):
    K, N, G = 1024, 2048, 64
    rng = inputs.rng_for(103)
    codes, scales = inputs.w4_weights(rng, K, N, G)
    W = pack(tf, codes, scales, G)
    ws = tf.workspace(tf.lane_gemm_workspace_bytes(K, N, G))
    x = inputs.bf16_normal(rng, (7, K))
    a = run(tf, W, x, ws)
    b = run(tf, W, x, ws)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert tf.workspace_status(ws) == tf.TF_DEV_OK
    # counters are left zero for the next call
    assert int(ws[256:256 + (1 << 18)].count_nonzero()) == 0


def test_strided_activations_and_outputs(tf):
    import torch
    K, N, G, R = 512, 768, 64, 6
    rng = inputs.rng_for(104)
    codes, scales = inputs.w4_weights(rng, K, N, G)
    W = pack(tf, codes, scales, G)
    x = inputs.bf16_normal(rng, (R, K))
    xbig = torch.zeros((R, K + 64), dtype=torch.int16, device="cuda")
    xbig[:, :K] = dev_bits16(x)
    ybig = torch.full((R, N + 5), 7.0, device="cuda")
    tf.lane_gemm_w4(W, xbig[:, :K], y=ybig[:, :N])
    yb = ybig.cpu().numpy()
    assert np.all(yb[:, N:] == 7.0)
    assert_close_rows(yb[:, :N], oracle.w4_linear(codes, scales, x, G))


@pytest.mark.parametrize("m", [1, 2, 3, 4])
def test_whole_tile_ranges_match_oracle_and_are_row_invariant(tf, m):
    """Shapes whose tiles split evenly into nearly one share per SM take whole
    tiles per CTA (no split-K): 140 * m tiles of 128 features."""
    K, G = 128, 64
    N = 128 * 140 * m
    rng = inputs.rng_for(104, m)
    codes, scales = inputs.w4_weights(rng, K, N, G)
    x = inputs.bf16_normal(rng, (16, K))
    W = pack(tf, codes, scales, G)
    y16 = run(tf, W, x)
    assert_close_rows(y16[:3], oracle.w4_linear(codes, scales, x[:3], G))
    y1 = run(tf, W, x[:1])
    assert np.array_equal(y1.view(np.uint32), y16[:1].view(np.uint32))


def test_selfcheck_row_invariance_entry_point(tf):
    """The library's own row-invariance self-check passes on the 5120 -> 17408
    projection (group 64) and on a ragged 777-feature matrix (group 32)."""
    for K, N, G in ((5120, 17408, 64), (2048, 777, 32)):
        rng = inputs.rng_for(77, K, N)
        codes, scales = inputs.w4_weights(rng, K, N, G)
        W = pack(tf, codes, scales, G)
        x = dev_bits16(inputs.bf16_normal(rng, (16, K)))
        assert tf.selfcheck_row_invariance(W, x) == 0
