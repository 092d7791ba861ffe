"""Tensor-core rate probe behind the lane GEMM's choice of mma.sync.

`tests/tcgen05_rate.cu` is built here (nvcc, sm_103a) and called through ctypes:

* the tcgen05 chain's accumulator must equal A·Bᵀ·n_mma for small-integer
  operands (exact in fp32), with A read from shared memory or from tensor
  memory, which checks the descriptors and layouts before any timing is
  trusted;
* then issue-to-completion cycles are recorded for chains of M = 128, K = 16
  `tcgen05.mma` at N = 16 … 256 (the lane GEMM's verify rows are N ≤ 16), on
  one CTA and on one CTA per SM, next to `mma.sync.m16n8k16` chains.

The measured rates are printed (``pytest -s``) and attached as test
properties; the test asserts only correctness and that every rate is positive.
"""

import ctypes
import json
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
M, K, MAXN = 128, 16, 256


@pytest.fixture(scope="module")
def probe():
    out = os.path.join(tempfile.mkdtemp(prefix="tc05_"), "tc05.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xcompiler",
                    "-fPIC", "-shared", "-o", out, os.path.join(HERE, "tcgen05_rate.cu")], check=True)
    lib = ctypes.CDLL(out)
    lib.tc05_rate.argtypes = [ctypes.c_int] * 7 + [ctypes.c_void_p] * 3
    lib.mma_sync_rate.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p] * 2
    return lib


def operands(n):
    r = np.arange(M)[:, None]
    k = np.arange(K)[None, :]
    a = ((7 * r + 3 * k) % 11 - 5).astype(np.float64)
    rb = np.arange(n)[:, None]
    b = ((5 * rb + 13 * k) % 9 - 4).astype(np.float64)
    return a, b


def run_tc05(lib, grid, n, n_mma, lbo, sbo, a_tmem=0, n_acc=1):
    cycles = torch.zeros(grid, dtype=torch.int64, device="cuda")
    dout = torch.zeros(M * MAXN, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.tc05_rate(grid, n, n_mma, n_acc, lbo, sbo, a_tmem, cycles.data_ptr(), dout.data_ptr(),
                       status.data_ptr())
    assert rc == 0, f"tc05_rate returned {rc}"
    assert int(status.item()) == 0, "a tcgen05 wait gave up"
    return cycles.cpu().numpy(), dout.view(M, MAXN)[:, :n].cpu().numpy().astype(np.float64)


def test_tcgen05_product_and_rates(probe, record_property):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    layout = (128, 256)   # (leading byte offset: K-adjacent core matrices, stride byte offset: 8-row groups)
    for a_tmem in (0, 1):
        for n in (16, 64, 256):
            a, b = operands(n)
            _, d = run_tc05(probe, 1, n, 3, *layout, a_tmem)
            np.testing.assert_array_equal(d, 3 * a @ b.T, err_msg=f"N={n} A in tensor memory: {a_tmem}")
    res = {"layout_lbo_sbo": layout, "tcgen05": {}, "tcgen05_a_tmem": {}, "tcgen05_4acc": {}, "mma_sync": {}}
    for a_tmem, key in ((0, "tcgen05"), (1, "tcgen05_a_tmem")):
        for n in (16, 32, 64, 128, 256):
            row = {}
            for grid in (1, sms):
                for n_mma in (1, 64, 512):
                    c, _ = run_tc05(probe, grid, n, n_mma, *layout, a_tmem)
                    row[f"grid{grid}_chain{n_mma}_cycles"] = int(np.median(c))
            c512 = row[f"grid{sms}_chain512_cycles"]
            row["cycles_per_mma_all_sms"] = c512 / 512
            row["flop_per_cycle_per_sm"] = 2 * M * n * K * 512 / c512
            res[key][f"N{n}"] = row
    # four independent accumulators in turn (is the floor a dependency or a rate?)
    for a_tmem in (0, 1):
        for n in (16, 64):
            c, _ = run_tc05(probe, sms, n, 512, *layout, a_tmem, 4)
            res["tcgen05_4acc"][f"N{n}_a_tmem{a_tmem}"] = {"cycles_per_mma_all_sms": float(np.median(c)) / 512}
    sink = torch.zeros(512, dtype=torch.float32, device="cuda")
    iters = 2048
    for warps in (4, 16):
        for chains in (1, 4, 8):
            cyc = torch.zeros(sms, dtype=torch.int64, device="cuda")
            rc = probe.mma_sync_rate(sms, warps, chains, iters, cyc.data_ptr(), sink.data_ptr())
            assert rc == 0
            c = float(np.median(cyc.cpu().numpy()))
            n_mma = warps * chains * iters
            res["mma_sync"][f"warps{warps}_chains{chains}"] = {
                "cycles": int(c), "mma_per_cycle_per_sm": n_mma / c,
                "flop_per_cycle_per_sm": 2 * 16 * 8 * 16 * n_mma / c}
    for v in list(res["tcgen05"].values()) + list(res["tcgen05_a_tmem"].values()) + list(res["tcgen05_4acc"].values()):
        assert v["cycles_per_mma_all_sms"] > 0
    for v in res["mma_sync"].values():
        assert v["mma_per_cycle_per_sm"] > 0
    record_property("tensor_core_rates", json.dumps(res))
    print("TC05 " + json.dumps(res))
