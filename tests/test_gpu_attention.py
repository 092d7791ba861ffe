"""Attention of the verify rows over a KV cache, on the GPU, through the C ABI,
against the fp64 oracle (oracle/attention.py).

* tf_kv_append writes the documented position-swizzled layout, bit for bit;
* outputs within 1e-3 * rms(oracle row) on shapes spanning several 256-key
  partitions and ragged tails (group 1/2/4/8, R = 1..16, positions on and
  around partition boundaries, the first position and the last one);
* row invariance: every row of an R-row launch byte-equal to the one-row
  launch at its position, R = 1..16, 8 KV heads x group 8 (128 query vectors);
* drafted == serial: passes that append R rows, of which only a prefix is
  accepted, leave every accepted row's output byte-equal to serial one-row
  decoding (rejected entries are rewritten by the next pass, never read);
* the full-size cache (8 KV heads, 64 query heads, 32768 positions) on
  sampled (row, head) pairs; a bad position sets the device status; a CUDA
  graph of append + attention replays with a moved position.
"""

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from w4_gemm_keyed_gb300 import inputs
from gpu_util import assert_close_rows, dev_bits16

pytestmark = pytest.mark.gpu
D = 128


def rows_of(kv):
    """[n_kv][L][128] -> the append call's [L][n_kv*128] rows."""
    n_kv, L, _ = kv.shape
    return np.ascontiguousarray(kv.transpose(1, 0, 2).reshape(L, n_kv * D))


def dev_pos(p):
    return torch.tensor([p], dtype=torch.int64, device="cuda")


def make_cache(tf, n_kv, max_len, k, v, n_entries):
    """A cache holding entries 0..n_entries-1 of the logical arrays k, v."""
    cache = tf.KVCache(n_kv, max_len)
    ws = cache.append(dev_bits16(rows_of(k[:, :n_entries])), dev_bits16(rows_of(v[:, :n_entries])), dev_pos(0))
    assert tf.workspace_status(ws) == tf.TF_DEV_OK
    return cache


def unswizzle(phys):
    """Device layout [n_kv][max_len][128] -> logical, by the rule in tf.h."""
    n_kv, L, _ = phys.shape
    t = np.arange(L)[:, None]
    d = np.arange(D)[None, :]
    src = 8 * ((d // 8) ^ (t % 8)) + d % 8
    return np.take_along_axis(phys, np.broadcast_to(src, (n_kv, L, D)), axis=2)


def test_append_writes_the_documented_layout(tf):
    rng = inputs.rng_for(1001)
    _, k, v = inputs.attention_inputs(rng, 1, 2, 1, 512)
    cache = make_cache(tf, 2, 512, k, v, 300)
    ws = cache.append(dev_bits16(rows_of(k[:, 300:305])), dev_bits16(rows_of(v[:, 300:305])), dev_pos(300))
    assert tf.workspace_status(ws) == tf.TF_DEV_OK
    kc = unswizzle(cache.k.cpu().numpy().view(np.uint16))
    vc = unswizzle(cache.v.cpu().numpy().view(np.uint16))
    assert np.array_equal(kc[:, :305], k[:, :305]) and np.array_equal(vc[:, :305], v[:, :305])
    assert not kc[:, 305:].any() and not vc[:, 305:].any()


CASES = [  # (n_kv, group, R, pos0, max_len)
    (1, 1, 1, 0, 256),          # one key
    (1, 1, 16, 0, 256),         # first rows, growing prefixes
    (2, 4, 3, 300, 512),
    (4, 2, 16, 248, 512),       # rows straddle the 256 boundary
    (2, 8, 7, 505, 768),
    (8, 8, 16, 1000, 1024),     # 128 query vectors; last rows end at max_len - 8
    (3, 1, 5, 1019, 1024),      # pos0 + R = max_len
    (8, 8, 1, 4095, 4096),      # one row at the last position, 16 partitions
]


@pytest.mark.parametrize("n_kv,group,R,pos0,max_len", CASES)
def test_matches_oracle(tf, n_kv, group, R, pos0, max_len):
    rng = inputs.rng_for(1002, n_kv, group, R, pos0)
    q, k, v = inputs.attention_inputs(rng, R, n_kv, group, max_len, q_std=2.0)
    cache = make_cache(tf, n_kv, max_len, k, v, pos0 + R)
    pos = dev_pos(pos0)
    ws = tf.workspace(cache.workspace_bytes(group, R))
    out = cache.attention(dev_bits16(q.reshape(R, -1)), group, pos, ws=ws)
    assert tf.workspace_status(ws) == tf.TF_DEV_OK
    ref = oatt.attention_verify(q, k, v, pos0, group)
    assert_close_rows(out.cpu().numpy(), ref.reshape(R, -1))


@pytest.mark.parametrize("pos0", [700, 250])
def test_rows_are_invariant_to_R(tf, pos0):
    n_kv, group, max_len = 8, 8, 1024
    rng = inputs.rng_for(1003, pos0)
    q, k, v = inputs.attention_inputs(rng, 16, n_kv, group, max_len, q_std=2.0)
    cache = make_cache(tf, n_kv, max_len, k, v, pos0 + 16)
    qd = dev_bits16(q.reshape(16, -1))
    single = [cache.attention(qd[r:r + 1], group, dev_pos(pos0 + r)).cpu().numpy()[0] for r in range(16)]
    for R in range(1, 17):
        out = cache.attention(qd[:R], group, dev_pos(pos0)).cpu().numpy()
        for r in range(R):
            assert np.array_equal(out[r].view(np.uint32), single[r].view(np.uint32)), f"R={R} row {r}"


def test_drafted_equals_serial_with_rollback(tf):
    n_kv, group, max_len, start, n = 2, 4, 1024, 200, 120
    rng = inputs.rng_for(1004)
    q, k, v = inputs.attention_inputs(rng, max_len, n_kv, group, max_len, q_std=2.0)
    qr = q.reshape(max_len, -1)
    truth_k, truth_v = rows_of(k), rows_of(v)
    # serial: one row per pass
    cache = make_cache(tf, n_kv, max_len, k, v, start)
    serial = {}
    for p in range(start, start + n):
        cache.append(dev_bits16(truth_k[p:p + 1]), dev_bits16(truth_v[p:p + 1]), dev_pos(p))
        serial[p] = cache.attention(dev_bits16(qr[p:p + 1]), group, dev_pos(p)).cpu().numpy()[0]
    # drafted: R = 8 rows per pass, rows after the accepted prefix carry wrong entries
    cache = make_cache(tf, n_kv, max_len, k, v, start)
    R, p = 8, start
    passes = 0
    while p < start + n:
        a = int(rng.integers(0, R))                     # rows 0..a are right
        kk, vv, qq = truth_k[p:p + R].copy(), truth_v[p:p + R].copy(), qr[p:p + R].copy()
        kk[a + 1:] = inputs.bf16_normal(rng, kk[a + 1:].shape, 3.0)
        vv[a + 1:] = inputs.bf16_normal(rng, vv[a + 1:].shape, 3.0)
        qq[a + 1:] = inputs.bf16_normal(rng, qq[a + 1:].shape, 2.0)
        cache.append(dev_bits16(kk), dev_bits16(vv), dev_pos(p))
        out = cache.attention(dev_bits16(qq), group, dev_pos(p)).cpu().numpy()
        for r in range(a + 1):
            if p + r < start + n:
                assert np.array_equal(out[r].view(np.uint32), serial[p + r].view(np.uint32)), f"pos {p + r}"
        p += a + 1
        passes += 1
    assert passes < n


def test_full_size_cache_on_sampled_heads(tf):
    n_kv, group, max_len, R = 8, 8, 32768, 16
    pos0 = max_len - R
    rng = inputs.rng_for(1005)
    q, k, v = inputs.attention_inputs(rng, R, n_kv, group, max_len, q_std=2.0)
    cache = make_cache(tf, n_kv, max_len, k, v, max_len)
    ws = tf.workspace(cache.workspace_bytes(group, R))
    out = cache.attention(dev_bits16(q.reshape(R, -1)), group, dev_pos(pos0), ws=ws).cpu().numpy()
    assert tf.workspace_status(ws) == tf.TF_DEV_OK
    pairs = [(0, 0), (0, 63), (5, 17), (15, 8), (15, 63), (9, 40)]
    ref = oatt.attention_verify(q, k, v, pos0, group, heads=pairs)
    got = out.reshape(R, n_kv * group, D)
    for r, h in pairs:
        assert_close_rows(got[r, h][None], ref[r, h][None])


def test_bad_position_sets_status_and_writes_nothing(tf):
    n_kv, group, max_len, R = 2, 2, 256, 4
    rng = inputs.rng_for(1006)
    q, k, v = inputs.attention_inputs(rng, R, n_kv, group, max_len)
    cache = make_cache(tf, n_kv, max_len, k, v, 200)
    for bad in (max_len - 2, -1):
        ws = tf.workspace(cache.workspace_bytes(group, R))
        out = torch.full((R, n_kv * group * D), 7.0, device="cuda")
        cache.attention(dev_bits16(q.reshape(R, -1)), group, dev_pos(bad), out=out, ws=ws)
        assert tf.workspace_status(ws) == tf.TF_DEV_BAD_POSITION
        assert bool((out == 7.0).all())
        before = cache.k.clone()
        ws2 = cache.append(dev_bits16(rows_of(k[:, :R])), dev_bits16(rows_of(v[:, :R])), dev_pos(bad))
        assert tf.workspace_status(ws2) == tf.TF_DEV_BAD_POSITION
        assert torch.equal(before, cache.k)


def test_graph_replay_follows_the_device_position(tf):
    n_kv, group, max_len, R = 4, 4, 1024, 8
    rng = inputs.rng_for(1007)
    q, k, v = inputs.attention_inputs(rng, R, n_kv, group, max_len, q_std=2.0)
    kr, vr = rows_of(k), rows_of(v)
    cache = make_cache(tf, n_kv, max_len, k, v, 300)
    pos = dev_pos(300)
    qd = dev_bits16(q.reshape(R, -1))
    knew, vnew = dev_bits16(kr[300:300 + R]), dev_bits16(vr[300:300 + R])
    ws = tf.workspace(cache.workspace_bytes(group, R))
    aws = tf.workspace(256)
    out = torch.empty((R, n_kv * group * D), device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        cache.append(knew, vnew, pos, ws=aws, stream=s)
        cache.attention(qd, group, pos, out=out, ws=ws, stream=s)
    s.synchronize()
    eager = out.cpu().numpy()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cache.append(knew, vnew, pos, ws=aws, stream=s)
        cache.attention(qd, group, pos, out=out, ws=ws, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint32), eager.view(np.uint32))
    # move the position on the device: the same graph now verifies rows at 600..607
    pos.fill_(600)
    knew.copy_(dev_bits16(kr[600:600 + R]))
    vnew.copy_(dev_bits16(vr[600:600 + R]))
    cache.append(dev_bits16(kr[300:600]), dev_bits16(vr[300:600]), dev_pos(300))
    g.replay()
    torch.cuda.synchronize()
    assert tf.workspace_status(ws) == tf.TF_DEV_OK
    ref = oatt.attention_verify(q, k, v, 600, group)
    assert_close_rows(out.cpu().numpy(), ref.reshape(R, -1))
