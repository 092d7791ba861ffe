"""NVFP4 lane GEMM on the GPU against the oracle (oracle/nvfp4.py).

* one-hot activations: the output is one dequantised weight, bit for bit
  (each weight times its block scale and the tensor scale is exact in fp32);
* seeded shapes spanning several tiles and ragged tails, R = 1 .. 16, within
  max |err| <= 1e-3 * rms(oracle row);
* activations up to 60000 in magnitude (inside the fp16 range the kernel
  computes in) and block scales down in the E4M3 subnormals;
* row invariance: every row of an R-row launch equals its one-row launch byte
  for byte at 5120 -> 17408, with sampled columns against the oracle.
"""

import numpy as np
import pytest
import torch

from oracle import nvfp4 as onv
from w4_gemm_keyed_gb300 import inputs
from gpu_util import assert_close_rows, dev_u8, dev_bits16

pytestmark = pytest.mark.gpu


def pack(tf, codes, scales, gs):
    return tf.pack_nvfp4(dev_u8(codes), dev_u8(scales), gs)


def run(tf, W, x_bits):
    return tf.lane_gemm_nvfp4(W, dev_bits16(x_bits)).cpu().numpy()


@pytest.mark.parametrize("R", [1, 5, 16])
def test_one_hot_is_bit_exact(tf, R):
    rng = inputs.rng_for(821, R)
    K, N = 256, 300
    codes, scales, gs = inputs.nvfp4_weights(rng, K, N, min_scale_exp=0)
    W = pack(tf, codes, scales, gs)
    ks = rng.choice(K, R, replace=False)
    x = np.zeros((R, K), dtype=np.float32)
    x[np.arange(R), ks] = 1.0
    xb = inputs.bf16_bits_from_f32(x)
    y = run(tf, W, xb)
    ref = onv.nvfp4_linear(codes, scales, gs, xb).astype(np.float32)
    assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("K,N", [(64, 1), (128, 300), (256, 1000), (5120, 777), (1024, 4096)])
@pytest.mark.parametrize("R", [1, 3, 8, 9, 16])
def test_matches_oracle_on_ragged_shapes(tf, K, N, R):
    rng = inputs.rng_for(822, K, N, R)
    codes, scales, gs = inputs.nvfp4_weights(rng, K, N)
    x = inputs.bf16_normal(rng, (R, K))
    W = pack(tf, codes, scales, gs)
    assert_close_rows(run(tf, W, x), onv.nvfp4_linear(codes, scales, gs, x))


def test_large_activations_and_subnormal_scales(tf):
    rng = inputs.rng_for(823)
    K, N, R = 512, 256, 4
    codes, scales, gs = inputs.nvfp4_weights(rng, K, N, min_scale_exp=0)
    scales[:, ::3] = rng.integers(1, 8, size=scales[:, ::3].shape, dtype=np.uint8)   # E4M3 subnormals
    x = inputs.bf16_normal(rng, (R, K), std=2000.0)
    x[0, :8] = inputs.bf16_bits_from_f32(np.array([60000, -60000, 32768, -1e-5, 3e-6, 0, -0.0, 65000], np.float32))
    W = pack(tf, codes, scales, gs)
    assert_close_rows(run(tf, W, x), onv.nvfp4_linear(codes, scales, gs, x))


def test_rows_invariant_at_27b_shape(tf):
    rng = inputs.rng_for(824)
    K, N = 5120, 17408
    codes, scales, gs = inputs.nvfp4_weights(rng, K, N)
    x = inputs.bf16_normal(rng, (16, K))
    W = pack(tf, codes, scales, gs)
    xd = dev_bits16(x)
    single = np.stack([tf.lane_gemm_nvfp4(W, xd[r:r + 1]).cpu().numpy()[0] for r in range(16)])
    for R in range(1, 17):
        y = tf.lane_gemm_nvfp4(W, xd[:R]).cpu().numpy()
        assert np.array_equal(y.view(np.uint32), single[:R].view(np.uint32)), f"R={R}"
    cols = np.sort(rng.choice(N, 256, replace=False))
    assert_close_rows(single[:, cols], onv.nvfp4_linear(codes, scales, gs, x, cols=cols))


def test_split_k_shape_against_oracle(tf):
    # 17408 -> 5120 runs the stream-K cut with the split-K fixup
    rng = inputs.rng_for(825)
    K, N, R = 17408, 5120, 16
    codes, scales, gs = inputs.nvfp4_weights(rng, K, N)
    x = inputs.bf16_normal(rng, (R, K))
    W = pack(tf, codes, scales, gs)
    y = run(tf, W, x)
    cols = np.sort(rng.choice(N, 128, replace=False))
    assert_close_rows(y[:, cols], onv.nvfp4_linear(codes, scales, gs, x, cols=cols))
