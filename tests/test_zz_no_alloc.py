"""tf_lane_gemm_w4_noalloc (the lane GEMM on the library's built-in scratch)
against tf_lane_gemm_w4 with a caller workspace.

Two calls in a row on the shared scratch -- a full-size 27B-class projection,
then a small ragged one with another tile count and group size -- must each
give the workspace entry point's result: within the GEMM tests' tolerance and,
because both launches cut the work the same way, byte for byte.  The file is
named to run last so that it also sees whatever earlier tests left on the
device.
"""

import numpy as np
import pytest
import torch

from w4_gemm_keyed_gb300 import inputs
from gpu_util import TOL, assert_close_rows, dev_bits16, pack

pytestmark = pytest.mark.gpu

CASES = [(5120, 17408, 64, 16), (1024, 777, 32, 5)]


def test_two_calls_in_a_row_match_workspace_entry(tf):
    problems = []
    for K, N, G, R in CASES:
        rng = inputs.rng_for(401, K, N, G, R)
        codes, scales = inputs.w4_weights(rng, K, N, G)
        x = dev_bits16(inputs.bf16_normal(rng, (R, K)))
        problems.append((pack(tf, codes, scales, G), x, R, N))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for W, x, R, N in problems:
        want = tf.lane_gemm_w4(W, x).cpu().numpy()
        y = torch.full((R, N), float("nan"), dtype=torch.float32, device="cuda")
        got = tf.lane_gemm_w4_noalloc(W, x, y, status=status).cpu().numpy()
        assert int(status.item()) == 0
        assert_close_rows(got, want, TOL)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_repeat_without_status_pointer(tf):
    K, N, G, R = 768, 2048, 32, 9
    rng = inputs.rng_for(402, K, N, G, R)
    codes, scales = inputs.w4_weights(rng, K, N, G)
    W = pack(tf, codes, scales, G)
    x = dev_bits16(inputs.bf16_normal(rng, (R, K)))
    want = tf.lane_gemm_w4(W, x).cpu().numpy()
    y = torch.empty((R, N), dtype=torch.float32, device="cuda")
    for _ in range(2):
        y.fill_(float("nan"))
        got = tf.lane_gemm_w4_noalloc(W, x, y).cpu().numpy()
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
