"""The sampler's key hash and Gumbel noise, read back from the device.

tf_keyed_hash evaluates the same device functions tf_keyed_sample uses
(TensorFold README, the two guarantees: Gumbel noise from a hash of the seed,
the position and the token id).  On a million seeded random triples --
64-bit seeds, positions over the whole int64 range, token ids over the whole
int32 range, plus hand-picked extremes -- the 64-bit keys must equal the
oracle's bit for bit.  The Gumbel values go through fp64 log on both sides
(CUDA's log on the device, the host's libm in the oracle), which may differ in
the last place.  With w = -ln u and g = -ln w, a last-place difference in w
moves g by about ulp(w) / w, an absolute amount: where w is near 1, g is near 0
and that amount is many ulps of g itself.  So the bound is absolute: |g_gpu -
g_oracle| <= 4 ulp(max(1, |g|)).  The share of bit-equal values is recorded.
"""

import numpy as np
import pytest
import torch

from oracle import sampling as osamp
from w4_gemm_keyed_gb300 import inputs

pytestmark = pytest.mark.gpu

N = 1_000_000


def _triples():
    rng = inputs.rng_for(901)
    seed = rng.integers(0, 2**64, size=N, dtype=np.uint64)
    pos = rng.integers(-2**63, 2**63 - 1, size=N, dtype=np.int64, endpoint=True)
    tok = rng.integers(-2**31, 2**31 - 1, size=N, dtype=np.int64, endpoint=True).astype(np.int32)
    # extremes: zero and all-ones words, the sampler's usual small positions and ids
    ext_s = np.array([0, 2**64 - 1, 1234, 0x9E3779B97F4A7C15, 2**63], dtype=np.uint64)
    ext_p = np.array([0, -1, 1, 65535, 2**63 - 1, -2**63], dtype=np.int64)
    ext_t = np.array([0, -1, 1, 151935, 2**31 - 1, -2**31], dtype=np.int32)
    k = 0
    for s in ext_s:
        for p in ext_p:
            for t in ext_t:
                seed[k], pos[k], tok[k] = s, p, t
                k += 1
    return seed, pos, tok


def test_key_hash_bit_exact_and_gumbel_within_4_ulp_of_max_1_g(tf, record_property):
    seed, pos, tok = _triples()
    h, g = tf.keyed_hash(torch.from_numpy(seed.view(np.int64)).cuda(), torch.from_numpy(pos).cuda(),
                         torch.from_numpy(tok).cuda())
    h = h.cpu().numpy().view(np.uint64)
    g = g.cpu().numpy()
    ref_h = np.array([osamp.key_hash(int(s), int(p), int(t)) for s, p, t in zip(seed.tolist(), pos.tolist(),
                                                                                tok.tolist())], dtype=np.uint64)
    bad = np.nonzero(h != ref_h)[0]
    assert bad.size == 0, f"{bad.size} keys differ, first at {bad[0]}: {h[bad[0]]:#x} vs {ref_h[bad[0]]:#x}"
    ref_g = np.array([osamp.gumbel_of(int(v)) for v in ref_h.tolist()])
    assert np.all(np.isfinite(g)) and np.all(np.isfinite(ref_g))
    ulp = np.spacing(np.maximum(1.0, np.abs(ref_g)))
    dist = np.abs(g - ref_g) / ulp
    exact = float(np.mean(g == ref_g))
    record_property("gumbel_bit_equal_share", exact)
    record_property("gumbel_max_ulp", float(dist.max()))
    assert dist.max() <= 4.0, f"Gumbel value {int(dist.argmax())} differs by {dist.max():.1f} ulp"


def test_uniform_never_zero_and_small_keys(tf):
    # keys whose top 53 bits are 0 give the smallest u = 0.5 / 2^53: g stays finite
    seed = torch.tensor([0, 1, 2], dtype=torch.int64, device="cuda")
    pos = torch.zeros(3, dtype=torch.int64, device="cuda")
    tok = torch.zeros(3, dtype=torch.int32, device="cuda")
    h, g = tf.keyed_hash(seed, pos, tok)
    for hv, gv in zip(h.cpu().numpy().view(np.uint64).tolist(), g.cpu().numpy().tolist()):
        ref = osamp.gumbel_of(int(hv))
        assert abs(gv - ref) <= 4 * np.spacing(max(1.0, abs(ref)))


def test_empty_call_is_a_no_op(tf):
    e = torch.empty(0, dtype=torch.int64, device="cuda")
    h, g = tf.keyed_hash(e, e, torch.empty(0, dtype=torch.int32, device="cuda"))
    assert h.numel() == 0 and g.numel() == 0
