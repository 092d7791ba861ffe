"""MLX-style affine W4 lane GEMM (unsigned codes, bf16 scale and bias per group)
on the GPU against the fp64 oracle (oracle/affine.py).

* one-hot activations: each output is scale * code + bias in one rounding, so
  the GPU must match the oracle bit for bit;
* seeded shapes across tiles and ragged tails, G = 32 and 64, R up to 16:
  max |err| <= 1e-3 * rms(oracle row);
* row invariance: every row of an R-row launch byte-equal to its 1-row launch
  (the 5120 -> 17408 projection at G = 64, and G = 32 where R > 8 runs the
  3-stage pipeline);
* the no-alloc entry point gives the same bytes.
"""

import numpy as np
import pytest
import torch

from oracle import affine
from w4_gemm_keyed_gb300 import inputs
from gpu_util import assert_close_rows, dev_bits16

pytestmark = pytest.mark.gpu


def pack_affine(tf, codes, scales, biases, G):
    return tf.pack_w4_affine(torch.from_numpy(codes.view(np.int32)).cuda(), dev_bits16(scales), dev_bits16(biases), G)


def run(tf, W, x_bits):
    return tf.lane_gemm_w4(W, dev_bits16(x_bits)).cpu().numpy()


@pytest.mark.parametrize("K,N,G", [(128, 300, 64), (64, 1, 32), (256, 1024, 32)])
def test_one_hot_is_bit_exact(tf, K, N, G):
    rng = inputs.rng_for(811, K, N, G)
    codes, scales, biases = inputs.mlx_affine_weights(rng, K, N, G)
    W = pack_affine(tf, codes, scales, biases, G)
    ks = [k for k in (0, 1, 15, 16, 31, 32, 63, K - 1) if k < K][:16]
    x = np.zeros((len(ks), K), dtype=np.uint16)
    for r, k in enumerate(ks):
        x[r, k] = 0x3F80
    y = run(tf, W, x)
    ref = affine.affine_w4_linear(codes, scales, biases, x, G).astype(np.float32)
    assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("K,N,G,R", [(256, 1024, 64, 1), (192, 300, 32, 5), (512, 1000, 64, 8),
                                     (2048, 1536, 32, 9), (768, 777, 64, 16), (1024, 4096, 32, 16)])
def test_matches_oracle(tf, K, N, G, R):
    rng = inputs.rng_for(812, K, N, G, R)
    codes, scales, biases = inputs.mlx_affine_weights(rng, K, N, G)
    x = inputs.bf16_normal(rng, (R, K))
    W = pack_affine(tf, codes, scales, biases, G)
    assert_close_rows(run(tf, W, x), affine.affine_w4_linear(codes, scales, biases, x, G))


@pytest.mark.parametrize("K,N,G", [(5120, 17408, 64), (2048, 3072, 32)])
def test_rows_invariant_to_R_and_oracle_on_sampled_columns(tf, K, N, G):
    rng = inputs.rng_for(813, K, N, G)
    codes, scales, biases = inputs.mlx_affine_weights(rng, K, N, G)
    x = inputs.bf16_normal(rng, (16, K))
    W = pack_affine(tf, codes, scales, biases, G)
    xd = dev_bits16(x)
    single = np.stack([tf.lane_gemm_w4(W, xd[r:r + 1]).cpu().numpy()[0] for r in range(16)])
    for R in (1, 2, 7, 8, 9, 16):
        y = tf.lane_gemm_w4(W, xd[:R]).cpu().numpy()
        assert np.array_equal(y.view(np.uint32), single[:R].view(np.uint32)), f"R={R}"
    cols = np.unique(np.concatenate([[0, N // 2, N - 1], np.random.default_rng(5).integers(0, N, 256)]))
    assert_close_rows(single[:, cols], affine.affine_w4_linear(codes, scales, biases, x, G, cols=cols))


def test_noalloc_entry_gives_the_same_bytes(tf):
    K, N, G, R = 1024, 2048, 64, 12
    rng = inputs.rng_for(814)
    codes, scales, biases = inputs.mlx_affine_weights(rng, K, N, G)
    x = dev_bits16(inputs.bf16_normal(rng, (R, K)))
    W = pack_affine(tf, codes, scales, biases, G)
    want = tf.lane_gemm_w4(W, x).cpu().numpy()
    y = torch.empty((R, N), dtype=torch.float32, device="cuda")
    got = tf.lane_gemm_w4_noalloc(W, x, y).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
