"""The 27B-class synthetic decoder at full size: one block teacher-forced
against the oracle on sampled columns, and drafted decoding writing the same
tokens as serial decoding.

bf16 embedding 151936 x 5120 N(0, 0.02); 8 residual blocks of RMSNorm + W4
group-64 SwiGLU MLP 5120 -> 17408 -> 5120; W4 LM head 5120 -> 151936.  For
seeds 1234..1238: 64 tokens decoded one row per step, and the same 64 tokens
decoded by verify passes of R = 8 rows whose drafts copy the serial tokens
with probability 0.75 (else a uniform token); token_sha must be equal, and
the device status must stay clean.
"""

import numpy as np
import pytest
import torch

from w4_gemm_keyed_gb300 import inputs

pytestmark = pytest.mark.gpu

V, H, F, N_BLOCKS, G = 151936, 5120, 17408, 8, 64


@pytest.fixture(scope="module")
def decoder27b(tf):
    from w4_gemm_keyed_gb300 import decode
    rng = inputs.rng_for(5)
    blocks = []
    for _ in range(N_BLOCKS):
        gc, gs = inputs.w4_weights(rng, H, F, G)
        uc, us = inputs.w4_weights(rng, H, F, G)
        dc, ds = inputs.w4_weights(rng, F, H, G)
        blocks.append(dict(gate_codes=gc, gate_scales=gs, up_codes=uc, up_scales=us, down_codes=dc, down_scales=ds))
    lc, ls = inputs.w4_weights(rng, H, V, G)
    weights = dict(emb=inputs.bf16_normal(rng, (V, H), 0.02), blocks=blocks, lm_codes=lc, lm_scales=ls, group=G)
    model = decode.upload_model(weights)
    del weights, blocks
    return model, decode.Decoder(model)


@pytest.mark.parametrize("seed", [1234, 1235, 1236, 1237, 1238])
def test_drafted_equals_serial(tf, decoder27b, seed):
    from w4_gemm_keyed_gb300 import decode
    model, dec = decoder27b
    T, k, p, n, R, prompt = 0.7, 20, 0.95, 64, 8, 11
    serial = decode.serial_decode(dec, prompt, n, T, k, p, seed)
    assert tf.workspace_status(dec.ws) == tf.TF_DEV_OK
    rng = inputs.rng_for(502, seed)
    future = np.array(serial + [0] * (R + 1))
    drafted, lens = decode.drafted_decode(
        dec, prompt, n, R, T, k, p, seed,
        lambda pos0, m: inputs.noisy_drafts(rng, future[pos0 - 1: pos0 - 1 + m], 0.75, V))
    assert decode.token_sha(drafted) == decode.token_sha(serial)
    assert len(lens) < n  # the drafts were used
    assert tf.workspace_status(dec.ws) == tf.TF_DEV_OK


def test_graph_drafted_equals_serial(tf, decoder27b):
    from w4_gemm_keyed_gb300 import decode
    model, dec = decoder27b
    T, k, p, n, R, prompt, seed = 0.7, 20, 0.95, 64, 8, 11, 1234
    serial = decode.serial_decode(dec, prompt, n + 2 * R, T, k, p, seed)
    rng = inputs.rng_for(602, seed)
    truth = np.zeros(n + 12 * R, dtype=np.int64)
    truth[1:1 + len(serial)] = serial[: len(truth) - 1]
    table = torch.from_numpy(inputs.noisy_drafts(rng, truth, 0.75, V)).cuda()
    graph, passes = decode.graph_decode(dec, prompt, n, R, T, k, p, seed, draft_table=table, passes_per_graph=8)
    assert decode.token_sha(graph) == decode.token_sha(serial[:n])
    assert tf.workspace_status(dec.ws) == tf.TF_DEV_OK


@pytest.mark.parametrize("R", [3, 16])
def test_block0_teacher_forced_against_oracle(tf, decoder27b, R):
    """Block 0 at full size (hidden 5120, FFN 17408): RMSNorm output on every
    entry, the SwiGLU output h on 512 sampled FFN columns (gate/up launch with
    the SwiGLU epilogue) and the residual increment on 256 sampled hidden
    columns (17408 -> 5120, split across SMs with the split-K fixup), each
    against the fp64 oracle fed the GPU's own bf16 inputs."""
    from oracle import numerics as onum
    import oracle
    from test_gpu_moe_decoder import assert_bf16_close, assert_rounded_close
    from gpu_util import assert_close_rows
    model, dec = decoder27b
    rng = inputs.rng_for(5)                # block 0 is the first draw of the model's generator
    gc, gs = inputs.w4_weights(rng, H, F, G)
    uc, us = inputs.w4_weights(rng, H, F, G)
    dc, ds = inputs.w4_weights(rng, F, H, G)
    toks = [5, 151935, 0, 42, 7, 1234, 3, 99999, 9, 64, 1, 2, 77, 512, 150000, 31][:R]
    last = torch.tensor(toks[:1], dtype=torch.int32, device="cuda")
    drafts = torch.tensor(toks[1:] or [0], dtype=torch.int32, device="cuda")
    x = torch.empty((R, H), dtype=torch.float32, device="cuda")
    ws = tf.workspace(model.block_workspace_bytes())
    model.embed_rows(last, drafts, R, x, ws)
    x_in = x.cpu().numpy().astype(np.float64)
    n = torch.empty((R, H), dtype=torch.int16, device="cuda")
    h = torch.empty((R, F), dtype=torch.int16, device="cuda")
    model.block(0, x, n, h, ws)
    assert tf.workspace_status(ws) == tf.TF_DEV_OK
    n_g = n.cpu().numpy().view(np.uint16)
    h_g = h.cpu().numpy().view(np.uint16)
    assert_bf16_close(n_g, onum.bf16_bits_of(onum.bf16_round(onum.rms_norm(x_in, 1e-6))))
    srng = inputs.rng_for(503, R)
    cf = np.sort(srng.choice(F, 512, replace=False))
    g = oracle.w4_linear(gc, gs, n_g, G, cols=cf)
    u = oracle.w4_linear(uc, us, n_g, G, cols=cf)
    assert_rounded_close(h_g[:, cf], onum.silu(g) * u)
    ch = np.sort(srng.choice(H, 256, replace=False))
    ch[0], ch[-1] = 0, H - 1               # both ends of the output
    inc = x.cpu().numpy().astype(np.float64)[:, ch] - x_in[:, ch]
    assert_close_rows(inc, oracle.w4_linear(dc, ds, h_g, G, cols=ch))
