"""Decoding with the verify passes chained on the device and replayed as a
CUDA graph (drafts from a device table, committed tokens into a device log).

The graph run must write exactly the tokens of eager serial decoding, for
serial (R = 1) and drafted runs alike, and agree with the eager drafted run.
"""

import numpy as np
import pytest
import torch

from w4_gemm_keyed_gb300 import inputs
from test_gpu_moe_decoder import tiny_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny(tf):
    from w4_gemm_keyed_gb300 import decode
    model = decode.upload_model(tiny_weights())
    return decode.Decoder(model)


def draft_table(serial, p_match, V, seed, length):
    """table[q] proposes position q: a noisy copy of the serial token there."""
    rng = inputs.rng_for(601, seed)
    truth = np.zeros(length, dtype=np.int64)
    truth[1:1 + len(serial)] = serial[: length - 1]
    return torch.from_numpy(inputs.noisy_drafts(rng, truth, p_match, V)).cuda()


def test_graph_serial_equals_eager_serial(tf, tiny):
    from w4_gemm_keyed_gb300 import decode
    T, k, p, seed, n = 0.7, 20, 0.95, 1234, 24
    eager = decode.serial_decode(tiny, 11, n, T, k, p, seed)
    graph, passes = decode.graph_decode(tiny, 11, n, 1, T, k, p, seed, passes_per_graph=8)
    assert graph == eager and passes >= n


@pytest.mark.parametrize("R,p_match", [(2, 0.9), (8, 0.75), (16, 0.5), (8, 1.0)])
def test_graph_drafted_equals_serial(tf, tiny, R, p_match):
    from w4_gemm_keyed_gb300 import decode
    T, k, p, seed, n = 0.7, 20, 0.95, 1235, 40
    serial = decode.serial_decode(tiny, 11, n + 3 * R, T, k, p, seed)
    table = draft_table(serial, p_match, 3000, seed, n + 8 * R + 2 * R)
    graph, passes = decode.graph_decode(tiny, 11, n, R, T, k, p, seed, draft_table=table, passes_per_graph=4)
    assert decode.token_sha(graph) == decode.token_sha(serial[:n])
    host_table = table.cpu().numpy()
    eager, lens = decode.drafted_decode(tiny, 11, n, R, T, k, p, seed,
                                        lambda pos0, m: host_table[pos0: pos0 + m])
    assert graph == eager
    if p_match == 1.0:
        assert all(a == R - 1 for a in lens[:-1])
    assert tf.workspace_status(tiny.ws) == tf.TF_DEV_OK


@pytest.mark.parametrize("R,p_match", [(1, 0.0), (8, 0.75)])
def test_graph_decode_matches_oracle_tokens(tf, tiny, R, p_match):
    """The graph-replayed loop (serial and drafted) against the fp64 oracle decoder
    on the same tiny model: identical committed tokens."""
    from oracle import decoder as odec
    from w4_gemm_keyed_gb300 import decode
    T, k, p, seed, n = 0.7, 20, 0.95, 1236, 24
    ref = odec.serial_decode(tiny_weights(), 11, n + 3 * R, T, k, p, seed)
    table = draft_table(ref, p_match, 3000, seed, n + 8 * R + 2 * R) if R > 1 else None
    graph, _ = decode.graph_decode(tiny, 11, n, R, T, k, p, seed, draft_table=table, passes_per_graph=4)
    assert graph == ref[:n]
    assert tf.workspace_status(tiny.ws) == tf.TF_DEV_OK
