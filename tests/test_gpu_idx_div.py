"""The lane GEMM's reciprocal quotient (tfk::idx_div) equals the integer division.

`tests/idx_div_check.cu` is built here (nvcc, sm_103a) and called through
ctypes.  idx_div takes n / d from the fp32 reciprocal below 2^21 and the
integer division above; the kernels use it for problem = item / Pv and
tile = k-slice / Kc.  Checked for every n < 2^21 with d <= 256, on strides
for larger divisors up to 2^21, for every n within 2^16 of the 2^21 switch
with d <= 1024, and on a stride far above it.
"""

import ctypes
import os
import subprocess
import tempfile

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def lib():
    out = os.path.join(tempfile.mkdtemp(prefix="idxdiv_"), "idx_div.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xcompiler",
                    "-fPIC", "-shared", "-o", out, os.path.join(HERE, "idx_div_check.cu")], check=True)
    so = ctypes.CDLL(out)
    so.idx_div_check.argtypes = [ctypes.c_uint] * 6 + [ctypes.c_void_p] * 2
    return so


@pytest.mark.parametrize("d_lo,d_hi,d_step,n_begin,n_end,n_step", [
    (1, 256, 1, 0, 1 << 21, 1),                               # every n below the switch, small divisors
    (257, 1 << 21, 997, 0, 1 << 21, 7),                       # larger divisors
    (1, 1024, 1, (1 << 21) - (1 << 16), (1 << 21) + (1 << 16), 1),   # across the switch
    (1, 1 << 21, 65521, 1 << 21, 0xFFFFFFF0, 65537),          # far above it (integer division)
])
def test_idx_div_is_exact(lib, d_lo, d_hi, d_step, n_begin, n_end, n_step):
    torch.cuda.set_device(0)
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    first = torch.zeros(2, dtype=torch.int32, device="cuda")
    rc = lib.idx_div_check(d_lo, d_hi, d_step, n_begin, n_end, n_step, bad.data_ptr(), first.data_ptr())
    assert rc == 0
    n_bad = int(bad.item())
    n, d = (int(v) & 0xFFFFFFFF for v in first.cpu().tolist())
    assert n_bad == 0, f"{n_bad} mismatches, first n={n} d={d}"
