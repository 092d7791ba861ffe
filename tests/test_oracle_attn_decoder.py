"""Pins of the oracle decoder with attention (oracle/attn_decoder.py).

* the pages' invariant: drafted decoding (rejections included) emits exactly
  the serial tokens;
* entries left by rejected rows are never read: overwriting every entry at or
  after the next pass's first position with garbage leaves that pass's logits
  bit-identical;
* a planted mistake (attention reading one position past the row's own) is
  caught by the stale-entry pin.
"""

import numpy as np
import pytest

from oracle import attn_decoder as oad
from oracle import attention as oatt
from oracle import decoder as odec
from w4_gemm_keyed_gb300 import inputs

V, H, F, G, N_KV, GRP, N_BLOCKS = 500, 128, 256, 64, 1, 2, 2
T, K_TOP, P_TOP = 0.8, 20, 0.95


def tiny_attn_model(seed=811):
    rng = inputs.rng_for(seed)
    blocks, attn = [], []
    n_q = N_KV * GRP
    for _ in range(N_BLOCKS):
        gc, gs = inputs.w4_weights(rng, H, F, G)
        uc, us = inputs.w4_weights(rng, H, F, G)
        dc, ds = inputs.w4_weights(rng, F, H, G)
        blocks.append(dict(gate_codes=gc, gate_scales=gs, up_codes=uc, up_scales=us, down_codes=dc, down_scales=ds))
        qc, qs = inputs.w4_weights(rng, H, (n_q + 2 * N_KV) * 128, G)
        oc, os_ = inputs.w4_weights(rng, n_q * 128, H, G)
        attn.append(dict(qkv_codes=qc, qkv_scales=qs, o_codes=oc, o_scales=os_))
    lc, ls = inputs.w4_weights(rng, H, V, G)
    model = dict(emb=inputs.bf16_normal(rng, (V, H), 0.02), blocks=blocks, attn=attn, lm_codes=lc, lm_scales=ls,
                 group=G, n_kv=N_KV, attn_group=GRP)
    prompt = rng.integers(0, V, 40).tolist()
    return model, prompt


@pytest.fixture(scope="module")
def tiny():
    return tiny_attn_model()


def test_drafted_equals_serial(tiny):
    model, prompt = tiny
    P, n, R = len(prompt), 24, 4
    cache = oad.new_cache(model, 256)
    oad.prefill(model, cache, prompt)
    serial = oad.serial_decode(model, cache, prompt[-1], P, n, T, K_TOP, P_TOP, 1234)
    rng = inputs.rng_for(812)
    future = np.array(serial + [0] * (R + 1))
    cache = oad.new_cache(model, 256)
    oad.prefill(model, cache, prompt)
    drafted, lens = oad.drafted_decode(model, cache, prompt[-1], P, n, R, T, K_TOP, P_TOP, 1234,
                                       lambda pos0, m: inputs.noisy_drafts(rng, future[pos0 - P: pos0 - P + m], 0.6, V))
    assert odec.token_sha(drafted) == odec.token_sha(serial)
    assert any(a < R - 1 for a in lens) and any(a > 0 for a in lens)   # rejections and acceptances both occurred


def stale_entries_unread(model, prompt):
    """A drafted pass with a rejection, then the next pass run twice: on the cache
    as left, and with every entry at or after its first position overwritten."""
    P = len(prompt)
    cache = oad.new_cache(model, 256)
    oad.prefill(model, cache, prompt)
    last, pos = prompt[-1], P
    d = [7, 8, 9]                                   # drafts that will mostly be rejected
    l = oad.logits_of(model, oad.pass_rows(model, cache, [last] + d, pos - 1))
    t = [int(np.argmax(l[i])) for i in range(4)]
    a, bonus = 0, t[0]                              # accept nothing beyond row 0
    nxt = pos + a + 1
    import copy
    garbage = copy.deepcopy(cache)
    for c in garbage:
        c["k"][:, nxt - 1:] = 0x4200                # bf16 32.0
        c["v"][:, nxt - 1:] = 0xC2C8                # bf16 -100.0
    rows = [bonus, 3, 4, 5]
    l1 = oad.logits_of(model, oad.pass_rows(model, cache, rows, nxt - 1))
    l2 = oad.logits_of(model, oad.pass_rows(model, garbage, rows, nxt - 1))
    return np.array_equal(l1.view(np.uint32), l2.view(np.uint32))


def test_stale_entries_are_never_read(tiny):
    model, prompt = tiny
    assert stale_entries_unread(model, prompt)


def test_planted_read_past_own_position_is_caught(tiny, monkeypatch):
    model, prompt = tiny
    real = oatt.attention_verify
    # every row sees one position too many: the last row of a pass reaches an entry it did not write
    monkeypatch.setattr(oatt, "attention_verify",
                        lambda q, k, v, pos0, group, heads=None: real(q, k, v, pos0 + 1, group, heads))
    assert not stale_entries_unread(model, prompt)
