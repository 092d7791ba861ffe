"""The synthetic decoder with an attention sub-block per block, on the GPU.

Two blocks of hidden 5120: attention with 64 query heads over 8 KV heads
(group 8, head dim 128; fused QKV projection 5120 -> 10240, output projection
8192 -> 5120), then the SwiGLU MLP 5120 -> 17408 -> 5120; W4 group 64
throughout; vocabulary 32768; KV caches of 1024 positions.

* prefill: after a 600-token prompt (three 256-key partitions) the caches are
  byte-equal whether the prompt goes in one row per pass, in 16-row passes on
  the fixed grid, or resumed part-way with one-row passes first;
* drafted == serial: 48 tokens decoded one row per pass and by R = 8 passes
  whose drafts copy the serial tokens with probability 0.75 have equal
  token_sha (seeds 1234, 1235) -- rejected rows' cache entries are rewritten
  by the next pass before any row reads them;
* teacher-forced parity of block 0's attention sub-block against the oracle:
  the QKV projection (oracle W4 linear of the GPU's bf16 norm), the attention
  (oracle over the GPU's bf16 queries and cache) and the residual increment
  (oracle W4 linear of the GPU's bf16 attention output), each within
  1e-3 * rms of the oracle row;
* the oracle decoder with attention's tiny pinned model, teacher-forced
  through both blocks and the LM head (every bf16 cast exact against
  round-to-nearest-even of the GPU's fp32 values), and drafted decoding equal
  to serial decoding.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oatt
from w4_gemm_keyed_gb300 import inputs
from gpu_util import assert_close_rows, dev_bits16, kv_unswizzle

pytestmark = pytest.mark.gpu

V, H, F, N_BLOCKS, G = 32768, 5120, 17408, 2, 64
N_KV, GROUP, MAX_LEN, P = 8, 8, 1024, 600
N_Q = N_KV * GROUP
T, K_TOP, P_TOP = 0.7, 20, 0.95


@pytest.fixture(scope="module")
def attn_model(tf):
    from w4_gemm_keyed_gb300 import decode
    rng = inputs.rng_for(7)
    blocks, attn = [], []
    for _ in range(N_BLOCKS):
        gc, gs = inputs.w4_weights(rng, H, F, G)
        uc, us = inputs.w4_weights(rng, H, F, G)
        dc, ds = inputs.w4_weights(rng, F, H, G)
        blocks.append(dict(gate_codes=gc, gate_scales=gs, up_codes=uc, up_scales=us, down_codes=dc, down_scales=ds))
        qc, qs = inputs.w4_weights(rng, H, (N_Q + 2 * N_KV) * 128, G)
        oc, os_ = inputs.w4_weights(rng, N_Q * 128, H, G)
        attn.append(dict(qkv_codes=qc, qkv_scales=qs, o_codes=oc, o_scales=os_))
    lc, ls = inputs.w4_weights(rng, H, V, G)
    weights = dict(emb=inputs.bf16_normal(rng, (V, H), 0.02), blocks=blocks, attn=attn, lm_codes=lc, lm_scales=ls,
                   group=G)
    model = decode.upload_attn_model(weights, N_KV, GROUP, MAX_LEN)
    prompt = rng.integers(0, V, P).tolist()
    return model, attn, prompt


def caches_bytes(model):
    return [(c.k.clone(), c.v.clone()) for c in model.caches]


def clear(model):
    for c in model.caches:
        c.k.zero_()
        c.v.zero_()


def test_prefill_bits_do_not_depend_on_chunking(tf, attn_model):
    from w4_gemm_keyed_gb300 import decode
    model, _, prompt = attn_model
    dec = decode.AttnDecoder(model)
    clear(model)
    dec.prefill(prompt, block=16)
    grid = caches_bytes(model)
    clear(model)
    dec.prefill(prompt, block=1)
    single = caches_bytes(model)
    clear(model)
    dec.prefill(prompt[:37], block=1)          # a conversation resumed part-way
    dec.prefill(prompt, block=16, first=37)
    resumed = caches_bytes(model)
    for (kg, vg), (ks, vs), (kr, vr) in zip(grid, single, resumed):
        assert torch.equal(kg[:, :P], ks[:, :P]) and torch.equal(vg[:, :P], vs[:, :P])
        assert torch.equal(kg[:, :P], kr[:, :P]) and torch.equal(vg[:, :P], vr[:, :P])
    assert tf.workspace_status(dec.ws_status) == tf.TF_DEV_OK


@pytest.mark.parametrize("seed", [1234, 1235])
def test_drafted_equals_serial_with_attention(tf, attn_model, seed):
    from w4_gemm_keyed_gb300 import decode
    model, _, prompt = attn_model
    dec = decode.AttnDecoder(model)
    clear(model)
    dec.prefill(prompt)
    n, R = 48, 8
    serial = decode.attn_serial_decode(dec, prompt[-1], P, n, T, K_TOP, P_TOP, seed)
    rng = inputs.rng_for(702, seed)
    future = np.array(serial + [0] * (R + 1))
    drafted, lens = decode.attn_drafted_decode(
        dec, prompt[-1], P, n, R, T, K_TOP, P_TOP, seed,
        lambda pos0, m: inputs.noisy_drafts(rng, future[pos0 - P: pos0 - P + m], 0.75, V))
    assert decode.token_sha(drafted) == decode.token_sha(serial)
    assert len(lens) < n and max(lens) > 0
    assert tf.workspace_status(dec.ws_status) == tf.TF_DEV_OK
    assert tf.workspace_status(dec.ws_attn) == tf.TF_DEV_OK


def test_attention_block_matches_oracle_teacher_forced(tf, attn_model):
    from w4_gemm_keyed_gb300 import decode
    model, attn, prompt = attn_model
    dec = decode.AttnDecoder(model)
    clear(model)
    dec.prefill(prompt)
    R, b = 4, model.base
    dec.reset(prompt[-1], P)
    dec.h_drafts[: R - 1] = torch.tensor(prompt[:R - 1], dtype=torch.int32)
    dec.drafts[: R - 1].copy_(dec.h_drafts[: R - 1])
    dec._set_positions(R, P - 1, P)
    x = dec.x[:R]
    b.embed_rows(dec.last, dec.drafts, R, x, dec.ws_status)
    x0 = x.clone()
    tf.rmsnorm_bf16(x, b.rms_eps, out=dec.n[:R])
    tf.lane_gemm_w4(model.qkv[0], dec.n[:R], y=dec.qkv[:R], ws=dec.ws_gemm)
    n_bits = dec.n[:R].cpu().numpy().view(np.uint16)
    ref_qkv = oracle.w4_linear(attn[0]["qkv_codes"], attn[0]["qkv_scales"], n_bits, G)
    assert_close_rows(dec.qkv[:R].cpu().numpy(), ref_qkv)

    tf.cast_bf16(dec.qkv[:R], out=dec.qkv_b[:R])
    ko, vo = N_Q * 128, (N_Q + N_KV) * 128
    cache = model.caches[0]
    cache.append(dec.qkv_b[:R, ko:vo], dec.qkv_b[:R, vo:], dec.kv_pos, ws=dec.ws_status)
    cache.attention(dec.qkv_b[:R, :ko], GROUP, dec.kv_pos, out=dec.att[:R], ws=dec.ws_attn)
    q_bits = dec.qkv_b[:R, :ko].cpu().numpy().view(np.uint16).reshape(R, N_Q, 128)
    kc = kv_unswizzle(cache.k.cpu().numpy().view(np.uint16))
    vc = kv_unswizzle(cache.v.cpu().numpy().view(np.uint16))
    ref_att = oatt.attention_verify(q_bits, kc, vc, P - 1, GROUP).reshape(R, -1)
    assert_close_rows(dec.att[:R].cpu().numpy(), ref_att)

    tf.cast_bf16(dec.att[:R], out=dec.att_b[:R])
    tf.lane_gemm_w4_accumulate(model.o[0], dec.att_b[:R], x, ws=dec.ws_gemm)
    a_bits = dec.att_b[:R].cpu().numpy().view(np.uint16)
    ref_inc = oracle.w4_linear(attn[0]["o_codes"], attn[0]["o_scales"], a_bits, G)
    inc = x.double().cpu().numpy() - x0.double().cpu().numpy()
    assert_close_rows(inc, ref_inc)
    assert tf.workspace_status(dec.ws_status) == tf.TF_DEV_OK


def test_tiny_attention_decoder_matches_oracle_teacher_forced(tf):
    """The pinned oracle's tiny decoder with attention (hidden 128, one KV head,
    group 2, vocabulary 500) after a 40-token prompt, one verify pass of 4 rows
    through both blocks and the LM head.  A deep bf16 pipeline is not comparable
    end to end: one rounding-boundary flip (fp32 on the GPU, fp64 in the oracle)
    cascades through the later roundings to about 1 % of the logits.  So every
    stage is compared with the oracle fed the GPU's own rounded inputs; every
    bf16 cast is checked exactly against round-to-nearest-even of the GPU's fp32
    values.  The GPU's drafted decoding must equal its serial decoding."""
    from w4_gemm_keyed_gb300 import decode
    from oracle import attn_decoder as oad
    from oracle import numerics as onum
    from test_gpu_moe_decoder import assert_bf16_close, assert_rounded_close
    from test_oracle_attn_decoder import tiny_attn_model, T as T_TINY, K_TOP as K_TINY, P_TOP as P_TINY
    weights, prompt = tiny_attn_model()
    P_T, V_T, Gt = len(prompt), weights["emb"].shape[0], weights["group"]
    n_q = weights["n_kv"] * weights["attn_group"]
    model = decode.upload_attn_model(weights, weights["n_kv"], weights["attn_group"], 256)
    b = model.base
    dec = decode.AttnDecoder(model)
    dec.prefill(prompt)
    R, rows = 4, [prompt[-1], 11, 12, 13]
    dec.reset(prompt[-1], P_T)
    dec.h_drafts[: R - 1] = torch.tensor(rows[1:], dtype=torch.int32)
    dec.drafts[: R - 1].copy_(dec.h_drafts[: R - 1])
    dec._set_positions(R, P_T - 1, P_T)
    x = dec.x[:R]
    b.embed_rows(dec.last, dec.drafts, R, x, dec.ws_status)
    assert np.array_equal(x.cpu().numpy().astype(np.float64), oracle.bf16_to_f64(weights["emb"][rows]))
    ko, vo = n_q * 128, (n_q + weights["n_kv"]) * 128

    def bits(t):
        return t.cpu().numpy().view(np.uint16)

    for i, (blk, att) in enumerate(zip(weights["blocks"], weights["attn"])):
        x_in = x.cpu().numpy().astype(np.float64)
        tf.rmsnorm_bf16(x, b.rms_eps, out=dec.n[:R])
        n_g = bits(dec.n[:R])
        assert_bf16_close(n_g, onum.bf16_bits_of(onum.bf16_round(onum.rms_norm(x_in, 1e-6))))
        tf.lane_gemm_w4(model.qkv[i], dec.n[:R], y=dec.qkv[:R], ws=dec.ws_gemm)
        qkv_g = dec.qkv[:R].cpu().numpy()
        assert_close_rows(qkv_g, oracle.w4_linear(att["qkv_codes"], att["qkv_scales"], n_g, Gt))
        tf.cast_bf16(dec.qkv[:R], out=dec.qkv_b[:R])
        qkv_b = bits(dec.qkv_b[:R])
        assert np.array_equal(qkv_b, inputs.bf16_bits_from_f32(qkv_g))
        cache = model.caches[i]
        cache.append(dec.qkv_b[:R, ko:vo], dec.qkv_b[:R, vo:], dec.kv_pos, ws=dec.ws_status)
        cache.attention(dec.qkv_b[:R, :ko], model.group, dec.kv_pos, out=dec.att[:R], ws=dec.ws_attn)
        att_g = dec.att[:R].cpu().numpy()
        kc = kv_unswizzle(cache.k.cpu().numpy().view(np.uint16))
        vc = kv_unswizzle(cache.v.cpu().numpy().view(np.uint16))
        ref_att = oatt.attention_verify(qkv_b[:, :ko].reshape(R, n_q, 128), kc, vc, P_T - 1, model.group)
        assert_close_rows(att_g, ref_att.reshape(R, -1))
        tf.cast_bf16(dec.att[:R], out=dec.att_b[:R])
        att_b = bits(dec.att_b[:R])
        assert np.array_equal(att_b, inputs.bf16_bits_from_f32(att_g))
        x_mid0 = x.cpu().numpy().astype(np.float64)
        tf.lane_gemm_w4_accumulate(model.o[i], dec.att_b[:R], x, ws=dec.ws_gemm)
        x_mid = x.cpu().numpy().astype(np.float64)
        assert_close_rows(x_mid - x_mid0, oracle.w4_linear(att["o_codes"], att["o_scales"], att_b, Gt))
        b.block(i, x, dec.n_out[:R], dec.h_out[:R], dec.ws_block)
        n2_g, h_g = bits(dec.n_out[:R]), bits(dec.h_out[:R])
        assert_bf16_close(n2_g, onum.bf16_bits_of(onum.bf16_round(onum.rms_norm(x_mid, 1e-6))))
        g = oracle.w4_linear(blk["gate_codes"], blk["gate_scales"], n2_g, Gt)
        u = oracle.w4_linear(blk["up_codes"], blk["up_scales"], n2_g, Gt)
        assert_rounded_close(h_g, onum.silu(g) * u)
        x_ref = x_mid + oracle.w4_linear(blk["down_codes"], blk["down_scales"], h_g, Gt)
        assert_close_rows(x.cpu().numpy(), x_ref)
    x_fin = x.cpu().numpy().astype(np.float64)
    n_fin = tf.rmsnorm_bf16(x, b.rms_eps)
    n_fin_g = bits(n_fin)
    assert_bf16_close(n_fin_g, onum.bf16_bits_of(onum.bf16_round(onum.rms_norm(x_fin, 1e-6))))
    logits = tf.lane_gemm_w4(b.lm_head, n_fin).cpu().numpy()
    assert_close_rows(logits, oracle.w4_linear(weights["lm_codes"], weights["lm_scales"], n_fin_g, Gt))

    serial = decode.attn_serial_decode(dec, prompt[-1], P_T, 32, T_TINY, K_TINY, P_TINY, 1234)
    rng = inputs.rng_for(813)
    future = np.array(serial + [0] * 5)
    drafted, lens = decode.attn_drafted_decode(
        dec, prompt[-1], P_T, 32, 4, T_TINY, K_TINY, P_TINY, 1234,
        lambda pos0, m: inputs.noisy_drafts(rng, future[pos0 - P_T: pos0 - P_T + m], 0.6, V_T))
    assert decode.token_sha(drafted) == decode.token_sha(serial)
    assert tf.workspace_status(dec.ws_status) == tf.TF_DEV_OK
