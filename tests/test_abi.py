"""The C-ABI library builds, loads and exports every symbol include/tf.h declares;
host-side argument validation answers before any device work is enqueued.

These run without a GPU: no call here launches a kernel.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tf.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^TF_API\s+[\w\s\*]+?\b(tf_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from w4_gemm_keyed_gb300 import build, tf
    build.build()
    return tf.load()


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("tf_lane_gemm_w4", "tf_keyed_sample", "tf_accept", "tf_verify_step", "tf_pack_w4",
                 "tf_moe_w4", "tf_last_error", "tf_workspace_status"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    from w4_gemm_keyed_gb300 import tf
    for name in declared_symbols():
        assert hasattr(lib, name), name
    bound = {n for n, _, _ in tf.SIGNATURES}
    assert bound == set(declared_symbols())


def test_only_declared_symbols_are_exported(lib):
    import subprocess
    from w4_gemm_keyed_gb300 import tf
    out = subprocess.run(["nm", "-D", "--defined-only", tf.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l and l.split()[-1].startswith("tf_")}
    assert exported == set(declared_symbols())


def test_packed_size_and_status_strings(lib):
    from w4_gemm_keyed_gb300 import tf
    # 128-feature tiles x 64-wide k slices (N padded to a multiple of 128)
    assert tf.packed_bytes(5120, 17408, 64) == 68 * 80 * 4 * 2176
    assert tf.packed_bytes(256, 1000, 64) == 4 * 4 * 4 * 2176         # N padded to 1024
    assert tf.packed_bytes(2048, 1536, 32) == 6 * 32 * 4 * 2304
    assert tf.packed_bytes(100, 64, 64) == 0                           # K not a multiple of 64
    assert tf.packed_bytes(256, 64, 16) == 0                           # unsupported group
    assert lib.tf_status_string(0) == b"ok"
    assert lib.tf_version() >= 100


def test_host_validation_rejects_bad_arguments(lib):
    from w4_gemm_keyed_gb300 import tf
    W = tf.W4MatrixC(None, 256, 64, 64)
    st = lib.tf_lane_gemm_w4(ctypes.byref(W), None, 256, 1, None, 64, None, 0, None)
    assert st == tf.TF_ERR_INVALID_ARG and b"packed" in lib.tf_last_error()
    W = tf.W4MatrixC(256, 100, 64, 64)   # K not a multiple of 64
    assert lib.tf_lane_gemm_w4(ctypes.byref(W), 256, 128, 1, 256, 64, 256, 1 << 30, None) == tf.TF_ERR_UNSUPPORTED
    W = tf.W4MatrixC(256, 256, 64, 64)
    assert lib.tf_lane_gemm_w4(ctypes.byref(W), 256, 256, 0, 256, 64, 256, 1 << 30, None) == tf.TF_ERR_INVALID_ARG
    assert lib.tf_lane_gemm_w4(ctypes.byref(W), 256, 256, 17, 256, 64, 256, 1 << 30, None) == tf.TF_ERR_INVALID_ARG
    assert lib.tf_lane_gemm_w4(ctypes.byref(W), 258, 256, 1, 256, 64, 256, 1 << 30, None) == tf.TF_ERR_INVALID_ARG
    assert lib.tf_lane_gemm_w4(ctypes.byref(W), 256, 256, 1, 256, 64, None, 0, None) == tf.TF_ERR_WORKSPACE
    sp = tf.SamplingC(0.7, 0, 0.9)    # any k' is served; a vocabulary past the limit is not
    st = lib.tf_keyed_sample(256, 600000, 1, 600000, ctypes.byref(sp), 1, 256, 256, 256, 1 << 30, None)
    assert st == tf.TF_ERR_UNSUPPORTED
    sp = tf.SamplingC(-1.0, 20, 0.9)
    assert lib.tf_keyed_sample(256, 1000, 1, 1000, ctypes.byref(sp), 1, 256, 256, 256, 1 << 30, None) == \
        tf.TF_ERR_INVALID_ARG
    sp = tf.SamplingC(0.7, 20, 0.9)      # T > 0 needs positions
    assert lib.tf_keyed_sample(256, 1000, 1, 1000, ctypes.byref(sp), 1, None, 256, 256, 1 << 30, None) == \
        tf.TF_ERR_INVALID_ARG
    assert lib.tf_accept(None, 256, 2, 256, 256, None) == tf.TF_ERR_INVALID_ARG
    assert lib.tf_accept(None, 256, 0, 256, 256, None) == tf.TF_ERR_INVALID_ARG
    assert lib.tf_gather_drafts(None, 0, None, 0, None, None) == tf.TF_ERR_INVALID_ARG      # R = 0
    assert lib.tf_gather_drafts(None, 0, None, 1, None, None) == tf.TF_OK                   # R = 1: no drafts
    assert lib.tf_gather_drafts(None, 8, 256, 4, 256, None) == tf.TF_ERR_INVALID_ARG        # null table
    assert lib.tf_commit_tokens(256, 256, None, 256, 8, None) == tf.TF_ERR_INVALID_ARG      # null pos
    assert lib.tf_commit_tokens(256, 256, 256, 256, -1, None) == tf.TF_ERR_INVALID_ARG      # negative length
    L = tf.MoeLayerC(256, 256, 2048, 768, 128, 9, 32)   # top_k > 8
    assert lib.tf_moe_w4(ctypes.byref(L), 256, 256, 1, 256, 256, 1 << 30, None) == tf.TF_ERR_UNSUPPORTED
    assert lib.tf_last_error() != b""


def test_kv_cache_validation_rejects_bad_arguments(lib):
    from w4_gemm_keyed_gb300 import tf
    big = 1 << 30
    C = tf.KVCacheC(256, 512, 8, 4096)
    assert lib.tf_attention_workspace_bytes(ctypes.byref(C), 8, 16) == \
        256 + 16 * 16 * 64 * 128 * 4 + 16 * 16 * 64 * 2 * 4
    assert lib.tf_attention_workspace_bytes(ctypes.byref(C), 3, 16) == 0
    assert lib.tf_attention_workspace_bytes(ctypes.byref(C), 8, 17) == 0
    ok_args = (256, 1024, 1, 256, 256, 1024, 256, big, None)     # q, ldq, R, pos, out, ldo, ws, ws_bytes, stream
    for bad, code in [(tf.KVCacheC(None, 512, 8, 4096), tf.TF_ERR_INVALID_ARG),     # null k
                      (tf.KVCacheC(258, 512, 8, 4096), tf.TF_ERR_INVALID_ARG),      # misaligned k
                      (tf.KVCacheC(256, 512, 0, 4096), tf.TF_ERR_UNSUPPORTED),      # n_kv = 0
                      (tf.KVCacheC(256, 512, 8, 1000), tf.TF_ERR_UNSUPPORTED)]:     # max_len % 256
        assert lib.tf_attention_verify(ctypes.byref(bad), 1, *ok_args) == code
        assert lib.tf_kv_append(ctypes.byref(bad), 256, 256, 1024, 1, 256, 256, 256, None) == code
    assert lib.tf_attention_verify(ctypes.byref(C), 3, *ok_args) == tf.TF_ERR_UNSUPPORTED          # group 3
    assert lib.tf_attention_verify(ctypes.byref(C), 8, 256, 1024, 17, 256, 256, 8192, 256, big, None) == \
        tf.TF_ERR_INVALID_ARG                                                                       # R = 17
    assert lib.tf_attention_verify(ctypes.byref(C), 8, 256, 1000, 1, 256, 256, 8192, 256, big, None) == \
        tf.TF_ERR_INVALID_ARG                                                                       # ldq < n_q*128
    assert lib.tf_attention_verify(ctypes.byref(C), 1, 264, 1024, 1, 256, 256, 1024, 256, big, None) == \
        tf.TF_ERR_INVALID_ARG                                                                       # q not 16-B aligned
    assert lib.tf_attention_verify(ctypes.byref(C), 1, 256, 1024, 1, None, 256, 1024, 256, big, None) == \
        tf.TF_ERR_INVALID_ARG                                                                       # null pos
    assert lib.tf_attention_verify(ctypes.byref(C), 1, 256, 1024, 1, 256, 256, 1024, 256, 100, None) == \
        tf.TF_ERR_WORKSPACE                                                                         # ws too small
    assert lib.tf_kv_append(ctypes.byref(C), 256, 256, 1000, 1, 256, 256, 256, None) == tf.TF_ERR_INVALID_ARG
    assert lib.tf_kv_append(ctypes.byref(C), 256, 256, 1024, 4097, 256, 256, 256, None) == tf.TF_ERR_INVALID_ARG
    assert lib.tf_kv_append(ctypes.byref(C), 256, 256, 1024, 1, 256, 256, 128, None) == tf.TF_ERR_WORKSPACE
    huge = tf.KVCacheC(256, 512, 128, 0x7FFFFF00)          # a launch of 2^31 x 128 / 8 CTAs is refused
    assert lib.tf_kv_append(ctypes.byref(huge), 256, 256, 128 * 128, 0x7FFFFF00, 256, 256, 256, None) == \
        tf.TF_ERR_UNSUPPORTED


def test_generic_workspace_size_and_selfcheck_validation(lib):
    from w4_gemm_keyed_gb300 import tf
    assert tf.workspace_size(tf.TF_OP_LANE_GEMM, [5120, 17408, 64]) == tf.lane_gemm_workspace_bytes(5120, 17408, 64)
    assert tf.workspace_size(tf.TF_OP_KEYED_SAMPLE, [16, 151936]) == \
        int(lib.tf_keyed_sample_workspace_bytes(16, 151936))
    C = tf.KVCacheC(256, 512, 8, 4096)
    assert tf.workspace_size(tf.TF_OP_ATTENTION, [8, 4096, 8, 16]) == \
        lib.tf_attention_workspace_bytes(ctypes.byref(C), 8, 16)
    assert tf.workspace_size(99, [1, 2, 3]) == 0
    assert tf.workspace_size(tf.TF_OP_LANE_GEMM, [5120, 17408]) == 0
    assert tf.workspace_size(tf.TF_OP_LANE_GEMM, [5120, -1, 64]) == 0
    assert lib.tf_selfcheck_scratch_bytes(1000) == 256 + 2 * 16 * 1024 * 4
    assert lib.tf_selfcheck_scratch_bytes(0) == 0
    W = tf.W4MatrixC(256, 256, 64, 64, 0)
    res = tf.I32(7)
    assert lib.tf_selfcheck_row_invariance(ctypes.byref(W), 256, 256, 256, 1 << 30, 256, 1 << 30, None, None) == \
        tf.TF_ERR_INVALID_ARG                                                  # null result
    assert lib.tf_selfcheck_row_invariance(ctypes.byref(W), 256, 256, 256, 100, 256, 1 << 30, None,
                                           ctypes.byref(res)) == tf.TF_ERR_INVALID_ARG   # scratch too small
    assert lib.tf_selfcheck_row_invariance(ctypes.byref(W), 256, 256, 264, 1 << 30, 256, 1 << 30, None,
                                           ctypes.byref(res)) == tf.TF_ERR_INVALID_ARG   # scratch misaligned
    assert res.value == 7


def test_newer_entry_points_validate_before_launching(lib):
    from w4_gemm_keyed_gb300 import tf
    big = 1 << 30
    # bf16 cast
    assert lib.tf_cast_bf16(None, 1, 8, 8, 256, 8, None) == tf.TF_ERR_INVALID_ARG          # null x
    assert lib.tf_cast_bf16(256, 0, 8, 8, 256, 8, None) == tf.TF_ERR_INVALID_ARG           # R = 0
    assert lib.tf_cast_bf16(256, 65536, 8, 8, 256, 8, None) == tf.TF_ERR_INVALID_ARG       # R too large
    assert lib.tf_cast_bf16(256, 2, 8, 4, 256, 8, None) == tf.TF_ERR_INVALID_ARG           # ldx < N
    # accumulate GEMM: the same checks as tf_lane_gemm_w4
    W = tf.W4MatrixC(256, 100, 64, 64, 0)                                                # K % 64 != 0
    assert lib.tf_lane_gemm_w4_accumulate(ctypes.byref(W), 256, 128, 1, 256, 64, 256, big, None) == \
        tf.TF_ERR_UNSUPPORTED
    W = tf.W4MatrixC(256, 256, 64, 64, 0)
    assert lib.tf_lane_gemm_w4_accumulate(ctypes.byref(W), 256, 256, 17, 256, 64, 256, big, None) == \
        tf.TF_ERR_INVALID_ARG                                                           # R = 17
    assert lib.tf_lane_gemm_w4_accumulate(ctypes.byref(W), 256, 256, 1, 256, 64, None, 0, None) == \
        tf.TF_ERR_WORKSPACE
    W = tf.W4MatrixC(256, 256, 64, 64, 2)                                                # affine flag not 0/1
    assert lib.tf_lane_gemm_w4(ctypes.byref(W), 256, 256, 1, 256, 64, 256, big, None) == tf.TF_ERR_INVALID_ARG
    # affine packing
    assert lib.tf_pack_w4_affine(None, 256, 256, 256, 64, 64, 256, big, None) == tf.TF_ERR_INVALID_ARG
    assert lib.tf_pack_w4_affine(256, 256, 256, 100, 64, 64, 256, big, None) == tf.TF_ERR_UNSUPPORTED
    assert lib.tf_pack_w4_affine(256, 256, 256, 256, 64, 16, 256, big, None) == tf.TF_ERR_UNSUPPORTED
    assert lib.tf_pack_w4_affine(256, 256, 256, 256, 64, 64, 264, big, None) == tf.TF_ERR_INVALID_ARG
    need = lib.tf_w4_affine_packed_bytes(256, 64, 64)
    assert need > lib.tf_w4_packed_bytes(256, 64, 64)                                   # biases take room
    assert lib.tf_pack_w4_affine(256, 256, 256, 256, 64, 64, 256, need - 1, None) == tf.TF_ERR_INVALID_ARG


def test_lmhead_sample_validates_before_launching(lib):
    from w4_gemm_keyed_gb300 import tf
    big = 1 << 30
    W = tf.W4MatrixC(256, 256, 1000, 64, 0)
    sp = ctypes.byref(tf.SamplingC(0.7, 20, 0.9))
    greedy = ctypes.byref(tf.SamplingC(0.0, 0, 1.0))
    none3 = (None, None, None)

    def call(Wc, x, ldx, R, p, pos, tokens, logits=None, ldl=0, acc=none3, ws=256, ws_bytes=big):
        return lib.tf_lmhead_sample(ctypes.byref(Wc), x, ldx, R, p, 1, pos, tokens, logits, ldl, *acc, ws, ws_bytes,
                                    None)

    assert lib.tf_lmhead_sample_workspace_bytes(ctypes.byref(W), 0) == 0
    assert lib.tf_lmhead_sample_workspace_bytes(ctypes.byref(W), 17) == 0
    assert lib.tf_lmhead_sample_workspace_bytes(ctypes.byref(W), 16) > 16 * 1000 * 4
    bad = tf.TF_ERR_INVALID_ARG
    assert call(W, 256, 256, 0, sp, 256, 256) == bad                          # R = 0
    assert call(W, None, 256, 1, sp, 256, 256) == bad                         # null x
    assert call(W, 256, 200, 1, sp, 256, 256) == bad                          # ldx < K
    assert call(W, 256, 256, 1, sp, 256, None) == bad                         # null tokens
    assert call(W, 256, 256, 1, sp, None, 256) == bad                         # T > 0 without pos
    assert call(W, 256, 256, 1, sp, 256, 256, logits=256, ldl=999) == bad     # ldl < N
    assert call(W, 256, 256, 1, None, 256, 256) == bad                        # null sampling
    assert call(W, 256, 256, 2, sp, 256, 256, acc=(None, 256, 256)) == bad    # accepting 2 rows without drafts
    assert call(W, 256, 256, 1, greedy, None, 256, ws=None, ws_bytes=0) == tf.TF_ERR_WORKSPACE
    Wbig = tf.W4MatrixC(256, 256, 600000, 64, 0)
    assert call(Wbig, 256, 256, 1, sp, 256, 256) == tf.TF_ERR_UNSUPPORTED     # V above the limit


def test_binding_refuses_host_tensors(lib):
    """Every pointer the library takes is a device pointer: the binding raises
    for a host tensor (pinned or not) before anything reaches the library."""
    import torch
    from w4_gemm_keyed_gb300 import tf
    with pytest.raises(tf.TFError):
        tf.cast_bf16(torch.zeros(2, 8))
    with pytest.raises(tf.TFError):
        tf.rmsnorm_bf16(torch.zeros(2, 8), 1e-6)
    with pytest.raises(tf.TFError):
        tf.workspace_status(torch.zeros(256, dtype=torch.uint8))


def _start(p, q, rem):
    return p * q + min(p, rem)


def _owner(i, q, rem):
    big = rem * (q + 1)
    return i // (q + 1) if i < big else rem + (i - big) // q


@pytest.mark.parametrize("T,Kc,Pv", [(4, 4, 16), (68, 80, 152), (20, 272, 152), (594, 80, 152), (6, 32, 16),
                                     (8, 12, 16), (1, 1, 1), (3, 5, 11), (7, 9, 63)])
def test_stream_k_cut_formulas(T, Kc, Pv):
    """The split-K cut used by the GEMM kernel: Pv = min(Pv, T*Kc) contiguous
    ranges whose sizes differ by at most one tile the iteration space, owner()
    inverts them, and every tile's segment slots are distinct."""
    tot = T * Kc
    Pv = min(Pv, tot)
    q, rem = divmod(tot, Pv)
    b = [_start(p, q, rem) for p in range(Pv + 1)]
    assert b[0] == 0 and b[-1] == tot and all(q <= b[p + 1] - b[p] <= q + 1 for p in range(Pv))
    for i in range(tot):
        p = _owner(i, q, rem)
        assert b[p] <= i < b[p + 1]
    slots = set()
    for t in range(T):
        tb, te = t * Kc, (t + 1) * Kc
        lo, hi = _owner(tb, q, rem), _owner(te - 1, q, rem)
        segs = list(range(lo, hi + 1))
        covered = sum(min(b[p + 1], te) - max(b[p], tb) for p in segs)
        assert covered == Kc and all(min(b[p + 1], te) > max(b[p], tb) for p in segs)
        if len(segs) > 1:
            for p in segs:
                which = 0 if b[p] >= tb else 1
                assert (p, which) not in slots
                slots.add((p, which))


def test_keyed_hash_validates_before_launching(lib):
    from w4_gemm_keyed_gb300 import tf
    assert lib.tf_keyed_hash(None, None, None, 0, None, None, None) == tf.TF_OK          # nothing to do
    assert lib.tf_keyed_hash(256, 256, 256, -1, 256, 256, None) == tf.TF_ERR_INVALID_ARG
    assert lib.tf_keyed_hash(None, 256, 256, 4, 256, 256, None) == tf.TF_ERR_INVALID_ARG
    assert lib.tf_keyed_hash(256, 256, None, 4, 256, 256, None) == tf.TF_ERR_INVALID_ARG
    assert b"null" in lib.tf_last_error()


def test_binding_checks_output_shape_and_dtype(lib):
    import torch
    from w4_gemm_keyed_gb300 import tf
    W = tf.W4Matrix(torch.zeros(tf.packed_bytes(256, 128, 64), dtype=torch.uint8), 256, 128, 64)
    x = torch.zeros((4, 256), dtype=torch.int16)
    for y, what in ((torch.zeros((4, 128), dtype=torch.float16), "float32"),   # 16-bit output
                    (torch.zeros((3, 128), dtype=torch.float32), "rows"),      # fewer rows than R
                    (torch.zeros((4, 64), dtype=torch.float32), "rows"),       # fewer columns than N
                    (torch.zeros((128, 4), dtype=torch.float32).t(), "rows")):  # non-unit inner stride
        with pytest.raises(tf.TFError) as e:
            tf.lane_gemm_w4_noalloc(W, x, y)
        assert e.value.status == tf.TF_ERR_INVALID_ARG
    with pytest.raises(tf.TFError):
        tf.lane_gemm_w4(W, torch.zeros((4, 128), dtype=torch.int16))          # x narrower than K
