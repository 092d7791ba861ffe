"""Helpers shared by the GPU parity tests: move seeded numpy inputs to the
device and call the library through its binding.  No arithmetic of the method
lives here."""

import numpy as np
import torch

TOL = 1e-3  # max |gpu - oracle| <= TOL * rms(oracle row): the verify pass's logit tolerance


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def dev_bits16(a):
    """uint16 bit patterns (bf16 / fp16) as a device int16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).cuda()


def pack(tf, codes, scales, group, gate_up=False):
    return tf.pack_w4(dev_u8(codes), dev_bits16(scales), group, gate_up=gate_up)


def gate_up_canonical(gc, gs, uc, us):
    """Stack gate rows then up rows (the canonical input of the gate/up packer)."""
    return np.concatenate([gc, uc], axis=0), np.concatenate([gs, us], axis=0)


def assert_close_rows(gpu, ref, tol=TOL):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape
    rms = np.sqrt(np.mean(ref ** 2, axis=-1, keepdims=True))
    err = np.abs(gpu - ref)
    worst = float(np.max(err / rms))
    assert np.all(err <= tol * rms), f"max err / rms = {worst:.3e} > {tol}"
    return worst


def bits(a):
    return np.ascontiguousarray(a).view(np.uint32 if a.dtype.itemsize == 4 else np.uint16)


HEAD_DIM = 128


def kv_rows(kv):
    """[n_kv][L][128] -> the [L][n_kv*128] rows tf_kv_append takes."""
    n_kv, L, _ = kv.shape
    return np.ascontiguousarray(kv.transpose(1, 0, 2).reshape(L, n_kv * HEAD_DIM))


def kv_unswizzle(phys):
    """A KV cache array in the library's layout [n_kv][max_len][128] -> plain
    [n_kv][max_len][128], by the storage rule stated in include/tf.h."""
    n_kv, L, _ = phys.shape
    t = np.arange(L)[:, None]
    d = np.arange(HEAD_DIM)[None, :]
    src = 8 * ((d // 8) ^ (t % 8)) + d % 8
    return np.take_along_axis(phys, np.broadcast_to(src, (n_kv, L, HEAD_DIM)), axis=2)
