"""Thin Python binding of libtf (the C ABI in include/tf.h).

Argument marshalling only: every step of the verify pass runs in the
library's CUDA kernels.  PyTorch supplies device memory and the current
stream.  If the shared library is missing the functions raise -- there is
no CPU fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtf.so")

TF_OK, TF_ERR_INVALID_ARG, TF_ERR_UNSUPPORTED, TF_ERR_CUDA, TF_ERR_TIMEOUT, TF_ERR_WORKSPACE = range(6)
TF_DEV_OK, TF_DEV_TIMEOUT, TF_DEV_NONFINITE_LOGIT, TF_DEV_BAD_TOKEN, TF_DEV_BAD_POSITION = range(5)
HEAD_DIM = 128
TF_OP_LANE_GEMM, TF_OP_KEYED_SAMPLE, TF_OP_ATTENTION = 1, 2, 3
MAX_ROWS = 16
MAX_TOP_K = 64

P = ctypes.c_void_p
I32 = ctypes.c_int32
SZ = ctypes.c_size_t


class TFError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"tf status {status}: {message}")
        self.status = status


class W4MatrixC(ctypes.Structure):
    _fields_ = [("packed", P), ("K", I32), ("N", I32), ("group", I32), ("affine", I32)]


class Nvfp4MatrixC(ctypes.Structure):
    _fields_ = [("packed", P), ("K", I32), ("N", I32), ("global_scale", ctypes.c_float)]


class SamplingC(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", I32), ("top_p", ctypes.c_float)]


class MoeLayerC(ctypes.Structure):
    _fields_ = [("gate_up", P), ("down", P), ("hidden", I32), ("ffn", I32), ("n_experts", I32),
                ("top_k", I32), ("group", I32)]


class KVCacheC(ctypes.Structure):
    _fields_ = [("k", P), ("v", P), ("n_kv", I32), ("max_len", I32)]


class ModelC(ctypes.Structure):
    _fields_ = [("vocab", I32), ("hidden", I32), ("ffn", I32), ("n_blocks", I32), ("group", I32),
                ("rms_eps", ctypes.c_float), ("embedding", P), ("gate_up", ctypes.POINTER(W4MatrixC)),
                ("down", ctypes.POINTER(W4MatrixC)), ("lm_head", W4MatrixC)]


# (name, restype, argtypes) of every exported symbol
SIGNATURES = [
    ("tf_last_error", ctypes.c_char_p, []),
    ("tf_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("tf_version", ctypes.c_int, []),
    ("tf_device_sm_count", I32, []),
    ("tf_workspace_status", ctypes.c_int, [P, P, ctypes.POINTER(I32)]),
    ("tf_w4_packed_bytes", SZ, [I32, I32, I32]),
    ("tf_pack_w4", ctypes.c_int, [P, P, I32, I32, I32, P, SZ, P]),
    ("tf_w4_affine_packed_bytes", SZ, [I32, I32, I32]),
    ("tf_pack_w4_affine", ctypes.c_int, [P, P, P, I32, I32, I32, P, SZ, P]),
    ("tf_pack_w4_gate_up", ctypes.c_int, [P, P, I32, I32, I32, P, SZ, P]),
    ("tf_lane_gemm_workspace_bytes", SZ, [I32, I32, I32]),
    ("tf_nvfp4_packed_bytes", SZ, [I32, I32]),
    ("tf_pack_nvfp4", ctypes.c_int, [P, P, I32, I32, P, SZ, P]),
    ("tf_lane_gemm_nvfp4_workspace_bytes", SZ, [I32, I32]),
    ("tf_lane_gemm_nvfp4", ctypes.c_int, [ctypes.POINTER(Nvfp4MatrixC), P, I32, I32, P, I32, P, SZ, P]),
    ("tf_lane_gemm_w4", ctypes.c_int, [ctypes.POINTER(W4MatrixC), P, I32, I32, P, I32, P, SZ, P]),
    ("tf_lane_gemm_w4_noalloc", ctypes.c_int, [ctypes.POINTER(W4MatrixC), P, I32, I32, P, I32, P, P]),
    ("tf_lane_gemm_w4_accumulate", ctypes.c_int, [ctypes.POINTER(W4MatrixC), P, I32, I32, P, I32, P, SZ, P]),
    ("tf_cast_bf16", ctypes.c_int, [P, I32, I32, I32, P, I32, P]),
    ("tf_keyed_sample_workspace_bytes", SZ, [I32, I32]),
    ("tf_keyed_sample", ctypes.c_int, [P, I32, I32, I32, ctypes.POINTER(SamplingC), ctypes.c_uint64, P, P, P, SZ, P]),
    ("tf_keyed_hash", ctypes.c_int, [P, P, P, ctypes.c_int64, P, P, P]),
    ("tf_lmhead_sample_workspace_bytes", SZ, [ctypes.POINTER(W4MatrixC), I32]),
    ("tf_lmhead_sample", ctypes.c_int, [ctypes.POINTER(W4MatrixC), P, I32, I32, ctypes.POINTER(SamplingC),
                                        ctypes.c_uint64, P, P, P, I32, P, P, P, P, SZ, P]),
    ("tf_accept", ctypes.c_int, [P, P, I32, P, P, P]),
    ("tf_gather_drafts", ctypes.c_int, [P, ctypes.c_int64, P, I32, P, P]),
    ("tf_commit_tokens", ctypes.c_int, [P, P, P, P, ctypes.c_int64, P]),
    ("tf_kv_append", ctypes.c_int, [ctypes.POINTER(KVCacheC), P, P, I32, I32, P, P, SZ, P]),
    ("tf_attention_workspace_bytes", SZ, [ctypes.POINTER(KVCacheC), I32, I32]),
    ("tf_attention_verify", ctypes.c_int, [ctypes.POINTER(KVCacheC), I32, P, I32, I32, P, P, I32, P, SZ, P]),
    ("tf_selfcheck_scratch_bytes", SZ, [I32]),
    ("tf_selfcheck_row_invariance", ctypes.c_int, [ctypes.POINTER(W4MatrixC), P, I32, P, SZ, P, SZ, P,
                                                   ctypes.POINTER(I32)]),
    ("tf_workspace_size", SZ, [I32, ctypes.POINTER(ctypes.c_int64), I32]),
    ("tf_moe_workspace_bytes", SZ, [ctypes.POINTER(MoeLayerC), I32]),
    ("tf_moe_w4", ctypes.c_int, [ctypes.POINTER(MoeLayerC), P, P, I32, P, P, SZ, P]),
    ("tf_verify_step_workspace_bytes", SZ, [ctypes.POINTER(ModelC), I32]),
    ("tf_embed_rows", ctypes.c_int, [ctypes.POINTER(ModelC), P, P, I32, P, P, P]),
    ("tf_rmsnorm_bf16", ctypes.c_int, [P, I32, I32, ctypes.c_float, P, P]),
    ("tf_decoder_block_workspace_bytes", SZ, [ctypes.POINTER(ModelC)]),
    ("tf_decoder_block", ctypes.c_int, [ctypes.POINTER(ModelC), I32, P, I32, P, P, P, SZ, P]),
    ("tf_verify_step", ctypes.c_int, [ctypes.POINTER(ModelC), I32, P, P, P, ctypes.POINTER(SamplingC),
                                      ctypes.c_uint64, P, P, P, P, SZ, P]),
]

_lib = None


def load(path: str = LIB_PATH):
    """Load libtf.so (built by ``w4_gemm_keyed_gb300.build``); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise FileNotFoundError(f"{path} is missing: run __graft_entry__.build() first (no CPU fallback)")
        lib = ctypes.CDLL(path)
        for name, res, args in SIGNATURES:
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(status: int):
    if status != TF_OK:
        raise TFError(status, load().tf_last_error().decode())


def _ptr(t):
    """Device address of a CUDA tensor (None passes NULL).  Every pointer the
    library takes is a device pointer: a host tensor, pinned or not, is refused
    here rather than handed to a kernel."""
    if t is None:
        return None
    if not t.is_cuda:
        raise TFError(TF_ERR_INVALID_ARG, f"expected a CUDA tensor, got one on {t.device}")
    return t.data_ptr()


def _current_raw_stream():
    return torch.cuda.current_stream().cuda_stream


try:  # cheaper lookup of the current stream's handle where this torch version has it
    _raw = torch._C._cuda_getCurrentRawStream

    def _current_raw_stream():  # noqa: F811
        return _raw(torch.cuda.current_device())
except AttributeError:  # pragma: no cover
    pass


def _stream(stream=None):
    return stream.cuda_stream if stream is not None else _current_raw_stream()


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zero-filled device scratch (the caching allocator aligns to >= 256 B)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def workspace_status(ws: torch.Tensor, stream=None) -> int:
    code = I32(0)
    _check(load().tf_workspace_status(_ptr(ws), _stream(stream), ctypes.byref(code)))
    return int(code.value)


# ---------------------------------------------------------------- weights
class W4Matrix:
    """A packed W4 matrix living on the device."""

    def __init__(self, packed: torch.Tensor, K: int, N: int, group: int, gate_up: bool = False,
                 affine: bool = False):
        self.packed, self.K, self.N, self.group, self.gate_up, self.affine = packed, K, N, group, gate_up, affine
        self._c = W4MatrixC(packed.data_ptr(), K, N, group, int(affine))

    def c(self) -> W4MatrixC:
        return self._c


def packed_bytes(K: int, N: int, group: int) -> int:
    return int(load().tf_w4_packed_bytes(K, N, group))


def pack_w4(codes: torch.Tensor, scales: torch.Tensor, group: int, gate_up: bool = False,
            out: torch.Tensor = None, stream=None) -> W4Matrix:
    """codes uint8 [N][K/2] and scales fp16 (or int16/uint16 bits) [N][K/group], on the device."""
    lib = load()
    N, K2 = codes.shape
    K = 2 * K2
    nbytes = packed_bytes(K, N, group)
    if nbytes == 0:
        raise TFError(TF_ERR_UNSUPPORTED, f"unsupported shape K={K} N={N} group={group}")
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=codes.device)
    codes = codes.contiguous()
    scales = scales.contiguous()
    if gate_up:
        _check(lib.tf_pack_w4_gate_up(_ptr(codes), _ptr(scales), K, N // 2, group, _ptr(out), nbytes, _stream(stream)))
    else:
        _check(lib.tf_pack_w4(_ptr(codes), _ptr(scales), K, N, group, _ptr(out), nbytes, _stream(stream)))
    return W4Matrix(out, K, N, group, gate_up)


def pack_w4_affine(codes: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor, group: int,
                   out: torch.Tensor = None, stream=None) -> W4Matrix:
    """MLX-style affine weights on the device: codes uint32 (or int32 bits) [N][K/8],
    scales and biases bf16 (or int16 bits) [N][K/group]."""
    lib = load()
    N, K8 = codes.shape
    K = 8 * K8
    nbytes = int(lib.tf_w4_affine_packed_bytes(K, N, group))
    if nbytes == 0:
        raise TFError(TF_ERR_UNSUPPORTED, f"unsupported shape K={K} N={N} group={group}")
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=codes.device)
    codes, scales, biases = codes.contiguous(), scales.contiguous(), biases.contiguous()
    _check(lib.tf_pack_w4_affine(_ptr(codes), _ptr(scales), _ptr(biases), K, N, group, _ptr(out), nbytes,
                                 _stream(stream)))
    return W4Matrix(out, K, N, group, affine=True)


# ---------------------------------------------------------------- linear
def lane_gemm_workspace_bytes(K: int, N: int, group: int) -> int:
    return int(load().tf_lane_gemm_workspace_bytes(K, N, group))


def _check_rows_in(x: torch.Tensor, K: int):
    """x: CUDA bf16 (or int16 bits) [R][>= K] with unit inner stride."""
    if x.dim() != 2 or x.dtype not in (torch.bfloat16, torch.int16):
        raise TFError(TF_ERR_INVALID_ARG, f"x must be a 2-D bf16 / int16 tensor, got {tuple(x.shape)} {x.dtype}")
    if x.stride(1) != 1 or x.shape[1] < K:
        raise TFError(TF_ERR_INVALID_ARG, f"x must have unit inner stride and >= {K} columns")


def _check_rows_out(y: torch.Tensor, R: int, N: int, device, dtype=torch.float32):
    """y: CUDA tensor of `dtype` [>= R][>= N] with unit inner stride on x's device."""
    if y.dim() != 2 or y.dtype != dtype:
        raise TFError(TF_ERR_INVALID_ARG, f"y must be a 2-D {dtype} tensor, got {tuple(y.shape)} {y.dtype}")
    if not y.is_cuda or y.device != device:
        raise TFError(TF_ERR_INVALID_ARG, f"y must be on {device}, got {y.device}")
    if y.shape[0] < R or y.shape[1] < N or y.stride(1) != 1:
        raise TFError(TF_ERR_INVALID_ARG, f"y must hold >= {R} rows of >= {N} columns with unit inner stride")


def lane_gemm_w4(W: W4Matrix, x: torch.Tensor, y: torch.Tensor = None, ws: torch.Tensor = None,
                 stream=None) -> torch.Tensor:
    """y[R][N] fp32 = W4 linear of bf16 rows x[R][K] (x may be bf16 or int16 bits)."""
    lib = load()
    _check_rows_in(x, W.K)
    R = x.shape[0]
    if y is None:
        y = torch.empty((R, W.N), dtype=torch.float32, device=x.device)
    _check_rows_out(y, R, W.N, x.device)
    if ws is None:
        ws = workspace(lane_gemm_workspace_bytes(W.K, W.N, W.group), x.device)
    wc = W.c()
    _check(lib.tf_lane_gemm_w4(ctypes.byref(wc), _ptr(x), x.stride(0), R, _ptr(y), y.stride(0), _ptr(ws),
                               ws.numel(), _stream(stream)))
    return y


def lane_gemm_w4_noalloc(W: W4Matrix, x: torch.Tensor, y: torch.Tensor, status: torch.Tensor = None,
                         stream=None) -> torch.Tensor:
    """lane_gemm_w4 on the library's built-in scratch: the call allocates no device
    memory, so the output y[R][N] fp32 must be given.  status: optional device int32
    (zeroed by the caller) that receives a device-side error code."""
    lib = load()
    _check_rows_in(x, W.K)
    R = x.shape[0]
    _check_rows_out(y, R, W.N, x.device)
    if status is not None and (status.dtype != torch.int32 or status.device != x.device or status.numel() < 1):
        raise TFError(TF_ERR_INVALID_ARG, "status must be a CUDA int32 tensor on x's device")
    wc = W.c()
    _check(lib.tf_lane_gemm_w4_noalloc(ctypes.byref(wc), _ptr(x), x.stride(0), R, _ptr(y), y.stride(0),
                                       _ptr(status), _stream(stream)))
    return y


# ---------------------------------------------------------------- NVFP4
class Nvfp4Matrix:
    """A packed NVFP4 matrix living on the device."""

    def __init__(self, packed: torch.Tensor, K: int, N: int, global_scale: float):
        self.packed, self.K, self.N, self.global_scale = packed, K, N, float(global_scale)
        self._c = Nvfp4MatrixC(packed.data_ptr(), K, N, float(global_scale))

    def c(self) -> Nvfp4MatrixC:
        return self._c


def nvfp4_packed_bytes(K: int, N: int) -> int:
    return int(load().tf_nvfp4_packed_bytes(K, N))


def pack_nvfp4(codes: torch.Tensor, scales: torch.Tensor, global_scale: float, out: torch.Tensor = None,
               stream=None) -> Nvfp4Matrix:
    """codes uint8 [N][K/2] (E2M1, low nibble first) and E4M3 scale bytes uint8 [N][K/16], on the device."""
    N, K2 = codes.shape
    K = 2 * K2
    nbytes = nvfp4_packed_bytes(K, N)
    if nbytes == 0:
        raise TFError(TF_ERR_UNSUPPORTED, f"unsupported shape K={K} N={N}")
    if tuple(scales.shape) != (N, K // 16) or codes.dtype != torch.uint8 or scales.dtype != torch.uint8:
        raise TFError(TF_ERR_INVALID_ARG, "codes must be uint8 [N][K/2] and scales uint8 [N][K/16]")
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=codes.device)
    codes, scales = codes.contiguous(), scales.contiguous()
    _check(load().tf_pack_nvfp4(_ptr(codes), _ptr(scales), K, N, _ptr(out), nbytes, _stream(stream)))
    return Nvfp4Matrix(out, K, N, global_scale)


def lane_gemm_nvfp4(W: Nvfp4Matrix, x: torch.Tensor, y: torch.Tensor = None, ws: torch.Tensor = None,
                    stream=None) -> torch.Tensor:
    """y[R][N] fp32 = NVFP4 linear of bf16 rows x[R][K] (x may be bf16 or int16 bits)."""
    lib = load()
    _check_rows_in(x, W.K)
    R = x.shape[0]
    if y is None:
        y = torch.empty((R, W.N), dtype=torch.float32, device=x.device)
    _check_rows_out(y, R, W.N, x.device)
    if ws is None:
        ws = workspace(int(lib.tf_lane_gemm_nvfp4_workspace_bytes(W.K, W.N)), x.device)
    _check(lib.tf_lane_gemm_nvfp4(ctypes.byref(W.c()), _ptr(x), x.stride(0), R, _ptr(y), y.stride(0), _ptr(ws),
                                  ws.numel(), _stream(stream)))
    return y


# ---------------------------------------------------------------- sampling
def lane_gemm_w4_accumulate(W: W4Matrix, x: torch.Tensor, y: torch.Tensor, ws: torch.Tensor = None,
                            stream=None) -> torch.Tensor:
    """y[R][N] (fp32, in place) += W4 linear of bf16 rows x[R][K]."""
    lib = load()
    if ws is None:
        ws = workspace(lane_gemm_workspace_bytes(W.K, W.N, W.group), x.device)
    _check(lib.tf_lane_gemm_w4_accumulate(ctypes.byref(W.c()), _ptr(x), x.stride(0), x.shape[0], _ptr(y), y.stride(0),
                                          _ptr(ws), ws.numel(), _stream(stream)))
    return y


def cast_bf16(x: torch.Tensor, out: torch.Tensor = None, stream=None) -> torch.Tensor:
    """bf16 bits (int16 tensor) of the fp32 rows x [R][N], nearest-even."""
    R, N = x.shape
    if out is None:
        out = torch.empty((R, N), dtype=torch.int16, device=x.device)
    _check(load().tf_cast_bf16(_ptr(x), R, N, x.stride(0), _ptr(out), out.stride(0), _stream(stream)))
    return out


def keyed_sample_workspace_bytes(R: int, V: int) -> int:
    return int(load().tf_keyed_sample_workspace_bytes(R, V))


def keyed_sample(logits: torch.Tensor, temperature: float, top_k: int, top_p: float, seed: int,
                 pos: torch.Tensor = None, tokens: torch.Tensor = None, ws: torch.Tensor = None,
                 stream=None) -> torch.Tensor:
    lib = load()
    R, V = logits.shape
    if tokens is None:
        tokens = torch.empty(R, dtype=torch.int32, device=logits.device)
    if ws is None:
        ws = workspace(keyed_sample_workspace_bytes(R, V), logits.device)
    sp = SamplingC(temperature, top_k, top_p)
    _check(lib.tf_keyed_sample(_ptr(logits), logits.stride(0), R, V, ctypes.byref(sp), ctypes.c_uint64(seed & (2**64 - 1)),
                               _ptr(pos), _ptr(tokens), _ptr(ws), ws.numel(), _stream(stream)))
    return tokens


def lmhead_sample_workspace_bytes(W: W4Matrix, R: int) -> int:
    wc = W.c()
    return int(load().tf_lmhead_sample_workspace_bytes(ctypes.byref(wc), R))


def lmhead_sample(W: W4Matrix, x: torch.Tensor, temperature: float, top_k: int, top_p: float, seed: int,
                  pos: torch.Tensor = None, tokens: torch.Tensor = None, logits: torch.Tensor = None,
                  drafts: torch.Tensor = None, accepted: torch.Tensor = None, bonus: torch.Tensor = None,
                  ws: torch.Tensor = None, stream=None) -> torch.Tensor:
    """tokens[R] = keyed sample of the LM head's logits W x[R] in one call; logits
    (fp32 [R][>= N]) are also stored when given; with `accepted` (int32 [1]) the
    drafts are accepted against the tokens in the same call."""
    lib = load()
    _check_rows_in(x, W.K)
    R = x.shape[0]
    if tokens is None:
        tokens = torch.empty(R, dtype=torch.int32, device=x.device)
    if tokens.dtype != torch.int32 or tokens.numel() < R or not tokens.is_contiguous():
        raise TFError(TF_ERR_INVALID_ARG, "tokens must be a contiguous int32 tensor of >= R entries")
    if logits is not None:
        _check_rows_out(logits, R, W.N, x.device)
    if ws is None:
        ws = workspace(lmhead_sample_workspace_bytes(W, R), x.device)
    wc = W.c()
    sp = SamplingC(temperature, top_k, top_p)
    _check(lib.tf_lmhead_sample(ctypes.byref(wc), _ptr(x), x.stride(0), R, ctypes.byref(sp),
                                ctypes.c_uint64(seed & (2**64 - 1)), _ptr(pos), _ptr(tokens), _ptr(logits),
                                logits.stride(0) if logits is not None else 0, _ptr(drafts), _ptr(accepted),
                                _ptr(bonus), _ptr(ws), ws.numel(), _stream(stream)))
    return tokens


def keyed_hash(seed: torch.Tensor, pos: torch.Tensor, token: torch.Tensor, stream=None):
    """(h uint64 bits as int64, g fp64) of the sampler's key and Gumbel noise for
    device triples seed (int64 holding uint64 bits), pos int64, token int32."""
    n = seed.numel()
    if pos.numel() != n or token.numel() != n:
        raise TFError(TF_ERR_INVALID_ARG, "seed, pos and token must have the same length")
    for t, dt in ((seed, torch.int64), (pos, torch.int64), (token, torch.int32)):
        if t.dtype != dt or not t.is_contiguous():
            raise TFError(TF_ERR_INVALID_ARG, f"expected a contiguous {dt} tensor, got {t.dtype}")
    h = torch.empty(n, dtype=torch.int64, device=seed.device)
    g = torch.empty(n, dtype=torch.float64, device=seed.device)
    _check(load().tf_keyed_hash(_ptr(seed), _ptr(pos), _ptr(token), n, _ptr(h), _ptr(g), _stream(stream)))
    return h, g


def accept(drafts: torch.Tensor, sampled: torch.Tensor, accepted: torch.Tensor = None,
           bonus: torch.Tensor = None, stream=None):
    lib = load()
    R = sampled.shape[0]
    dev = sampled.device
    if accepted is None:
        accepted = torch.empty(1, dtype=torch.int32, device=dev)
    if bonus is None:
        bonus = torch.empty(1, dtype=torch.int32, device=dev)
    _check(lib.tf_accept(_ptr(drafts) if R > 1 else None, _ptr(sampled), R, _ptr(accepted), _ptr(bonus),
                         _stream(stream)))
    return accepted, bonus


def gather_drafts(table: torch.Tensor, pos: torch.Tensor, R: int, drafts: torch.Tensor, stream=None):
    """drafts[i] = table[pos + i] for i < R - 1 (device int32 table, device int64 pos)."""
    _check(load().tf_gather_drafts(_ptr(table), table.numel(), _ptr(pos), R, _ptr(drafts), _stream(stream)))
    return drafts


def commit_tokens(tokens: torch.Tensor, accepted: torch.Tensor, pos: torch.Tensor, log: torch.Tensor, stream=None):
    """Write a finished pass's committed tokens into the device log (index = position - 1)."""
    _check(load().tf_commit_tokens(_ptr(tokens), _ptr(accepted), _ptr(pos), _ptr(log), log.numel(),
                                   _stream(stream)))
    return log


def selfcheck_row_invariance(W: W4Matrix, x: torch.Tensor, stream=None) -> int:
    """0 if every row of every R in 1..16 matches its one-row launch bit for bit,
    else R * 256 + row of the first mismatch.  x: bf16 [16][K] on the device."""
    lib = load()
    scratch = workspace(int(lib.tf_selfcheck_scratch_bytes(W.N)), device=x.device)
    ws = workspace(lane_gemm_workspace_bytes(W.K, W.N, W.group), device=x.device)
    res = I32(-1)
    _check(lib.tf_selfcheck_row_invariance(ctypes.byref(W.c()), _ptr(x), x.stride(0), _ptr(scratch), scratch.numel(),
                                           _ptr(ws), ws.numel(), _stream(stream), ctypes.byref(res)))
    return int(res.value)


def workspace_size(op: int, dims) -> int:
    arr = (ctypes.c_int64 * len(dims))(*[int(d) for d in dims])
    return int(load().tf_workspace_size(op, arr, len(dims)))


# ---------------------------------------------------------------- KV cache attention
class KVCache:
    """A KV cache on the device: k, v bf16 bits (int16) [n_kv][max_len][128] in the
    library's position-swizzled layout (tf.h), zero-filled at creation."""

    def __init__(self, n_kv: int, max_len: int, device="cuda"):
        self.k = torch.zeros((n_kv, max_len, HEAD_DIM), dtype=torch.int16, device=device)
        self.v = torch.zeros((n_kv, max_len, HEAD_DIM), dtype=torch.int16, device=device)
        self.n_kv, self.max_len = n_kv, max_len
        self._c = KVCacheC(self.k.data_ptr(), self.v.data_ptr(), n_kv, max_len)

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, pos: torch.Tensor, ws: torch.Tensor = None,
               stream=None):
        """Entries at positions pos .. pos + R - 1 from k_new, v_new bf16 [R][n_kv*128]."""
        if ws is None:
            ws = workspace(256, device=k_new.device)
        R = k_new.shape[0]
        _check(load().tf_kv_append(ctypes.byref(self._c), _ptr(k_new), _ptr(v_new), k_new.stride(0), R, _ptr(pos),
                                   _ptr(ws), ws.numel(), _stream(stream)))
        return ws

    def workspace_bytes(self, group: int, R: int) -> int:
        return int(load().tf_attention_workspace_bytes(ctypes.byref(self._c), group, R))

    def attention(self, q: torch.Tensor, group: int, pos: torch.Tensor, out: torch.Tensor = None,
                  ws: torch.Tensor = None, stream=None) -> torch.Tensor:
        """fp32 [R][n_q*128]: rows at positions pos + r attending over entries 0..pos + r."""
        R = q.shape[0]
        n_q = self.n_kv * group
        if out is None:
            out = torch.empty((R, n_q * HEAD_DIM), dtype=torch.float32, device=q.device)
        if ws is None:
            ws = workspace(self.workspace_bytes(group, R), device=q.device)
        _check(load().tf_attention_verify(ctypes.byref(self._c), group, _ptr(q), q.stride(0), R, _ptr(pos), _ptr(out),
                                          out.stride(0), _ptr(ws), ws.numel(), _stream(stream)))
        return out


def rmsnorm_bf16(x: torch.Tensor, eps: float, out: torch.Tensor = None, stream=None) -> torch.Tensor:
    """bf16 bits (int16 tensor) of x / sqrt(mean(x^2) + eps), per row of fp32 x [R][H]."""
    R, H = x.shape
    if out is None:
        out = torch.empty((R, H), dtype=torch.int16, device=x.device)
    _check(load().tf_rmsnorm_bf16(_ptr(x), R, H, eps, _ptr(out), _stream(stream)))
    return out


# ---------------------------------------------------------------- MoE
class MoeLayer:
    def __init__(self, gate_up: torch.Tensor, down: torch.Tensor, hidden: int, ffn: int, n_experts: int,
                 top_k: int, group: int):
        self.gate_up, self.down = gate_up, down
        self.hidden, self.ffn, self.n_experts, self.top_k, self.group = hidden, ffn, n_experts, top_k, group

    def c(self) -> MoeLayerC:
        return MoeLayerC(self.gate_up.data_ptr(), self.down.data_ptr(), self.hidden, self.ffn, self.n_experts,
                         self.top_k, self.group)


def moe_workspace_bytes(layer: MoeLayer, R: int) -> int:
    lc = layer.c()
    return int(load().tf_moe_workspace_bytes(ctypes.byref(lc), R))


def moe_w4(layer: MoeLayer, x: torch.Tensor, router: torch.Tensor, out: torch.Tensor = None,
           ws: torch.Tensor = None, stream=None) -> torch.Tensor:
    lib = load()
    R = x.shape[0]
    if out is None:
        out = torch.empty((R, layer.hidden), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(moe_workspace_bytes(layer, R), x.device)
    lc = layer.c()
    _check(lib.tf_moe_w4(ctypes.byref(lc), _ptr(x), _ptr(router), R, _ptr(out), _ptr(ws), ws.numel(),
                         _stream(stream)))
    return out


# ---------------------------------------------------------------- synthetic decoder
class Model:
    """Device weights of the attention-free synthetic decoder."""

    def __init__(self, embedding: torch.Tensor, gate_up, down, lm_head: W4Matrix, vocab: int, hidden: int,
                 ffn: int, group: int, rms_eps: float = 1e-6):
        self.embedding, self.gate_up, self.down, self.lm_head = embedding, list(gate_up), list(down), lm_head
        self.vocab, self.hidden, self.ffn, self.group, self.rms_eps = vocab, hidden, ffn, group, rms_eps
        n = len(self.gate_up)
        self._gu = (W4MatrixC * max(n, 1))(*[m.c() for m in self.gate_up])
        self._dn = (W4MatrixC * max(n, 1))(*[m.c() for m in self.down])
        self._c = ModelC(vocab, hidden, ffn, n, group, rms_eps, embedding.data_ptr(), self._gu, self._dn,
                         lm_head.c())

    def workspace_bytes(self, R: int) -> int:
        return int(load().tf_verify_step_workspace_bytes(ctypes.byref(self._c), R))

    def embed_rows(self, last_token, drafts, R: int, x: torch.Tensor, ws: torch.Tensor, stream=None):
        _check(load().tf_embed_rows(ctypes.byref(self._c), _ptr(last_token), _ptr(drafts) if R > 1 else None, R,
                                    _ptr(x), _ptr(ws), _stream(stream)))

    def block_workspace_bytes(self) -> int:
        return int(load().tf_decoder_block_workspace_bytes(ctypes.byref(self._c)))

    def block(self, b: int, x: torch.Tensor, n_out: torch.Tensor, h_out: torch.Tensor, ws: torch.Tensor,
              stream=None):
        """In place on the fp32 residual x [R][hidden]; n_out/h_out receive the bf16 intermediates."""
        _check(load().tf_decoder_block(ctypes.byref(self._c), b, _ptr(x), x.shape[0], _ptr(n_out), _ptr(h_out),
                                       _ptr(ws), ws.numel(), _stream(stream)))

    def verify_step(self, R: int, last_token: torch.Tensor, pos: torch.Tensor, drafts: torch.Tensor,
                    temperature: float, top_k: int, top_p: float, seed: int, tokens: torch.Tensor,
                    accepted: torch.Tensor, ws: torch.Tensor, logits: torch.Tensor = None, stream=None):
        sp = SamplingC(temperature, top_k, top_p)
        _check(load().tf_verify_step(ctypes.byref(self._c), R, _ptr(last_token), _ptr(pos),
                                     _ptr(drafts) if R > 1 else None, ctypes.byref(sp),
                                     ctypes.c_uint64(seed & (2**64 - 1)), _ptr(tokens), _ptr(accepted),
                                     _ptr(logits), _ptr(ws), ws.numel(), _stream(stream)))
