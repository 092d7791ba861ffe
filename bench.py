"""Benchmark of the W4 verify-pass GEMM (and the rest of the verify pass) on GB300.

Headline workload (one "step"): the 27B-class dense projections of the verify
pass, W4 group-64 5120->17408 and 17408->5120, each launched once at every
verify width R in {1, 2, 4, 8, 16} -- ten launches that each stream 47,349,760
bytes of codes + scales.  ``value`` = algorithmic weight bytes of the step /
device time (GB/s); inputs are resident in HBM.  Weights rotate over copies
totalling > 3x L2 so every launch reads HBM.

Also reported on the same JSON line (``extra``): per-R GB/s, the LM head +
keyed sampler + acceptance verify pass (steps/s, rows/s), the MoE layer, and
the synthetic decoder's verify steps/s; plus the CPU oracle timed on a bounded
sample (``cpu_baseline``), the end-to-end number through the C ABI with host
buffers (``e2e``), the roofline of the dominant kernel and the SM clocks.

``--impl reference`` times the CPU oracle (the reference arm) on
the same metric and workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "W4 verify-GEMM HBM GB/s & % of peak at R=1..16; verify steps/s"
SHAPES = ((5120, 17408), (17408, 5120))
ROWS = (1, 2, 4, 8, 16)
GROUP = 64
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def bytes_per_launch(K, N, G=GROUP):
    return K * N // 2 + 2 * N * (K // G)


STEP_BYTES = sum(bytes_per_launch(K, N) for K, N in SHAPES) * len(ROWS)
WORKLOAD = ("27B-class dense verify projections: W4 g64 5120->17408 and 17408->5120, "
            "one launch each at R=1,2,4,8,16 (10 launches/step)")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            for key in ("hbm_gbs", "hbm_GBs", "hbm"):
                if key in d:
                    return float(d[key]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("w4_gemm.cu", "w4_gemm.cuh", "tf_ptx.cuh"):
        h.update(open(os.path.join(ROOT, "w4_gemm_keyed_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch from a committed ncu summary, if it was taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", "w4_lane_gemm_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
    except Exception:
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ----------------------------------------------------------------------------- GPU arm
def setup_dense(tf, torch, rank):
    from w4_gemm_keyed_gb300 import inputs
    mats = {}
    for K, N in SHAPES:
        rng = inputs.rng_for(2, K, N)
        codes, scales = inputs.w4_weights(rng, K, N, GROUP)
        dc = torch.from_numpy(codes).cuda()
        ds = torch.from_numpy(scales.view(np.int16)).cuda()
        n_copies = max(2, -(-3 * L2_BYTES // bytes_per_launch(K, N)))
        copies = [tf.pack_w4(dc, ds, GROUP) for _ in range(n_copies)]
        x = inputs.bf16_normal(rng, (16, K))
        mats[(K, N)] = dict(copies=copies, codes=codes, scales=scales, x_host=x,
                            x=torch.from_numpy(x.view(np.int16)).cuda(),
                            y=torch.empty((16, N), dtype=torch.float32, device="cuda"),
                            ws=tf.workspace(tf.lane_gemm_workspace_bytes(K, N, GROUP)))
        del dc, ds
    torch.cuda.synchronize()
    return mats


def dense_launches():
    return [(K, N, R) for R in ROWS for (K, N) in SHAPES]


def time_dense(tf, torch, mats, steps, warmup):
    """Timed region: exactly ``steps`` steps, as CUDA-graph replays of one
    weight-rotation cycle (n_copies steps) followed by one graph of the first
    ``steps % n_copies`` steps of the next cycle.

    Returns (seconds, steps timed, launches per step)."""
    n_copies = min(len(m["copies"]) for m in mats.values())

    def step(c):
        for K, N, R in dense_launches():
            m = mats[(K, N)]
            tf.lane_gemm_w4(m["copies"][c], m["x"][:R], y=m["y"][:R], ws=m["ws"])

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for c in range(n):
                step(c)
        return g

    for i in range(warmup):
        step(i % n_copies)
    torch.cuda.synchronize()
    full_reps, rem = divmod(steps, n_copies)
    full = capture(n_copies)
    tail = capture(rem) if rem else None
    full.replay()
    if tail is not None:
        tail.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(full_reps):
        full.replay()
    if tail is not None:
        tail.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / 1e3, steps, len(dense_launches())


def time_per_launch(tf, torch, mats, reps=20):
    """Latency view: GPU time of each (shape, R) launch issued alone with events
    around it (rotating copies) -- includes launch latency and the pipeline ramp."""
    per = {}
    n_copies = min(len(m["copies"]) for m in mats.values())
    c = 0
    for _ in range(reps):
        for K, N, R in dense_launches():
            m = mats[(K, N)]
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            tf.lane_gemm_w4(m["copies"][c % n_copies], m["x"][:R], y=m["y"][:R], ws=m["ws"])
            b.record()
            c += 1
            per.setdefault((K, N, R), []).append((a, b))
    torch.cuda.synchronize()
    return {k: [a.elapsed_time(b) for a, b in v] for k, v in per.items()}


def time_per_r_graph(tf, torch, mats, reps=20):
    """Device rate of each (shape, R): one CUDA graph of back-to-back launches of
    that shape and R over every weight copy (> 3x L2 in total, so each launch
    reads HBM), replayed ``reps`` times; microseconds per launch."""
    out = {}
    for K, N, R in dense_launches():
        m = mats[(K, N)]
        xv, yv = m["x"][:R], m["y"][:R]

        def cycle():
            for W in m["copies"]:
                tf.lane_gemm_w4(W, xv, y=yv, ws=m["ws"])
        cycle()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cycle()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        out[(K, N, R)] = a.elapsed_time(b) * 1e3 / (reps * len(m["copies"]))
        del g
    return out


def time_dense_e2e(tf, torch, mats, steps, warmup):
    """Same step through the C ABI with host buffers.  Every step copies all of
    its inputs host->device in one pinned copy, runs the ten launches on slices
    of the device buffers (leading dimensions through the ABI) and reads all
    outputs back device->host in one copy.  Two buffer sets alternate: the
    host->device copy of step i + 1 and the device->host copy of step i - 1 run
    on their own streams while step i computes (events order each buffer's
    reuse); the timed region ends when the last step's outputs are on the host."""
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    launches = dense_launches()
    x_off, y_off, xo, yo = [], [], 0, 0
    for K, N, R in launches:
        x_off.append(xo)
        y_off.append(yo)
        xo += R * K
        yo += R * N
    hx = torch.empty(xo, dtype=torch.int16).pin_memory()
    for (K, N, R), o in zip(launches, x_off):
        hx[o:o + R * K] = torch.from_numpy(mats[(K, N)]["x_host"][:R].reshape(-1).view(np.int16))
    hy = [torch.empty(yo, dtype=torch.float32).pin_memory() for _ in range(2)]
    dx = [torch.empty(xo, dtype=torch.int16, device="cuda") for _ in range(2)]
    dy = [torch.empty(yo, dtype=torch.float32, device="cuda") for _ in range(2)]
    h2d, d2h = xo * 2, yo * 4
    # per buffer set and launch: the weight copies it rotates over and its slices of the device buffers
    plans = [[(mats[(K, N)]["copies"], dx[b][xo_:xo_ + R * K].view(R, K), dy[b][yo_:yo_ + R * N].view(R, N),
               mats[(K, N)]["ws"]) for (K, N, R), xo_, yo_ in zip(launches, x_off, y_off)] for b in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs of the set are on the device
    ev_out = [torch.cuda.Event() for _ in range(2)]     # outputs of the set are computed
    ev_back = [torch.cuda.Event() for _ in range(2)]    # outputs of the set are on the host
    counter = [0]

    def step():
        i = counter[0]
        counter[0] += 1
        b = i % 2
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(ev_out[b])                # step i - 2 has finished reading dx[b]
            dx[b].copy_(hx, non_blocking=True)
            ev_in[b].record(up)
        comp.wait_event(ev_in[b])
        if i >= 2:
            comp.wait_event(ev_back[b])                 # step i - 2's outputs have left dy[b]
        for copies, xv, yv, ws in plans[b]:
            tf.lane_gemm_w4(copies[i % len(copies)], xv, y=yv, ws=ws)
        ev_out[b].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(ev_out[b])
            hy[b].copy_(dy[b], non_blocking=True)
            ev_back[b].record(down)

    def drain():
        for b in range(2):
            if counter[0] > b:
                comp.wait_event(ev_back[(counter[0] - 1 - b) % 2])

    for _ in range(warmup):
        step()
    drain()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    up.wait_event(t0)
    down.wait_event(t0)
    for _ in range(steps):
        step()
    drain()
    t1.record(comp)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / 1e3, h2d, d2h


def extra_lmhead(tf, torch, steps=30):
    """LM head (5120 -> 151936) + keyed sampler + acceptance at R = 1, 2, 4, 8, 16: the fused
    call, the unfused sequence and the GEMM alone, each timed back to back."""
    from w4_gemm_keyed_gb300 import inputs
    K, V = 5120, 151936
    rng = inputs.rng_for(3)
    codes, scales = inputs.w4_weights(rng, K, V, GROUP)
    W = tf.pack_w4(torch.from_numpy(codes).cuda(), torch.from_numpy(scales.view(np.int16)).cuda(), GROUP)
    x = torch.from_numpy(inputs.bf16_normal(rng, (16, K)).view(np.int16)).cuda()
    logits = torch.empty((16, V), device="cuda")
    ws_g = tf.workspace(tf.lane_gemm_workspace_bytes(K, V, GROUP))
    ws_s = tf.workspace(tf.keyed_sample_workspace_bytes(16, V))
    pos = torch.arange(16, dtype=torch.int64, device="cuda")
    toks = torch.empty(16, dtype=torch.int32, device="cuda")
    drafts = torch.zeros(15, dtype=torch.int32, device="cuda")
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    bonus = torch.empty(1, dtype=torch.int32, device="cuda")
    ws_f = tf.workspace(tf.lmhead_sample_workspace_bytes(W, 16))
    out = {"step": "tf_lmhead_sample (LM head with candidate epilogue, finaliser with acceptance)",
           "unfused_step": "tf_lane_gemm_w4 + tf_keyed_sample + tf_accept"}
    by = bytes_per_launch(K, V)
    for R in ROWS:
        def one():
            tf.lmhead_sample(W, x[:R], 0.6, 20, 0.95, 1234, pos[:R], tokens=toks[:R], drafts=drafts[:max(R - 1, 1)],
                             accepted=acc, bonus=bonus, ws=ws_f)

        def one_unfused():
            tf.lane_gemm_w4(W, x[:R], y=logits[:R], ws=ws_g)
            tf.keyed_sample(logits[:R], 0.6, 20, 0.95, 1234, pos[:R], tokens=toks[:R], ws=ws_s)
            tf.accept(drafts[:max(R - 1, 1)], toks[:R], accepted=acc, bonus=bonus)

        def gemm():
            tf.lane_gemm_w4(W, x[:R], y=logits[:R], ws=ws_g)

        def timed(fn):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(steps):
                fn()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) / steps

        ms, ums, gms = timed(one), timed(one_unfused), timed(gemm)
        out[f"R{R}"] = {"verify_steps_per_s": 1e3 / ms, "rows_per_s": R * 1e3 / ms, "ms_per_step": ms,
                        "unfused_ms_per_step": ums, "lmhead_gemm_ms": gms, "step_over_gemm": ms / gms,
                        "lmhead_gbs": by / (gms * 1e-3) / 1e9,
                        "lmhead_frac_of_hbm_peak": by / (gms * 1e-3) / 1e9 / peaks()[0]}
    del W
    return out


def extra_sampler(tf, torch, steps=20):
    """tf_keyed_sample alone on V = 151936 fp32 logits (N(0, 2)), R = 1 and 16:
    greedy, the fast candidate path (top-k 20, top-p 0.95) and the general one
    (top-k <= 0 with top-p 0.95 and 1.0); CUDA-graph replays of 10 calls."""
    from w4_gemm_keyed_gb300 import inputs
    V = 151936
    out = {}
    rng = inputs.rng_for(12)
    for R in (1, 16):
        lg = torch.from_numpy(inputs.logits_normal(rng, R, V, std=2.0)).cuda()
        pos = torch.arange(R, dtype=torch.int64, device="cuda")
        toks = torch.empty(R, dtype=torch.int32, device="cuda")
        ws = tf.workspace(tf.keyed_sample_workspace_bytes(R, V))
        for name, (T, k, p) in {"greedy": (0.0, 0, 1.0), "k20_p0.95": (0.6, 20, 0.95),
                                "k0_p0.95": (0.7, 0, 0.95), "k0_p1": (0.7, 0, 1.0)}.items():
            def call():
                tf.keyed_sample(lg, T, k, p, 1234, pos, tokens=toks, ws=ws)
            call()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(10):
                    call()
            g.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(steps):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            out[f"R{R}_{name}_us"] = a.elapsed_time(b) * 1e3 / (10 * steps)
    return out


def extra_affine(tf, torch, steps=30):
    """MLX-style affine W4 (bf16 scale and bias per group) on the 5120 -> 17408
    projection, G = 64, R = 1 / 8 / 16: GB/s over codes + scales + biases, weights
    rotating over copies larger than L2, CUDA-graph replay of one rotation."""
    K, N, G = 5120, 17408, GROUP
    gen = torch.Generator(device="cuda")
    gen.manual_seed(9)
    nbytes = K * N // 2 + 4 * N * (K // G)
    n_copies = max(3, -(-3 * L2_BYTES // nbytes))
    copies = []
    for _ in range(n_copies):
        codes = torch.randint(-2**31, 2**31 - 1, (N, K // 8), dtype=torch.int32, device="cuda", generator=gen)
        sc = (torch.rand((N, K // G), device="cuda", generator=gen) * 0.02 + 1e-3).bfloat16()
        bi = (-sc.float() * 7.5).bfloat16()
        copies.append(tf.pack_w4_affine(codes, sc.view(torch.int16), bi.view(torch.int16), G))
    x = (torch.randn((16, K), device="cuda", generator=gen)).bfloat16().view(torch.int16)
    y = torch.empty((16, N), device="cuda")
    ws = tf.workspace(tf.lane_gemm_workspace_bytes(K, N, G))
    out = {"bytes_per_launch": nbytes}
    for R in (1, 8, 16):
        xv, yv = x[:R], y[:R]
        for c in copies:
            tf.lane_gemm_w4(c, xv, y=yv, ws=ws)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for c in copies:
                tf.lane_gemm_w4(c, xv, y=yv, ws=ws)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / (steps * n_copies)
        out[f"R{R}"] = {"us_per_launch": us, "gbs": nbytes / us / 1e3, "frac_of_hbm_peak": nbytes / us / 1e3 / peaks()[0]}
    return out


def extra_nvfp4(tf, torch, steps=30):
    """NVFP4 weights (E2M1 codes, E4M3 scale per 16 features, fp32 tensor scale)
    on the 5120 -> 17408 projection, R = 1 / 8 / 16: GB/s over codes + scale
    bytes, weights rotating over copies larger than L2, CUDA-graph replay."""
    from w4_gemm_keyed_gb300 import inputs
    K, N = 5120, 17408
    nbytes = K * N // 2 + K * N // 16
    n_copies = max(3, -(-3 * L2_BYTES // nbytes))
    rng = inputs.rng_for(10)
    codes, scales, gs = inputs.nvfp4_weights(rng, K, N)
    dc, ds = torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda()
    copies = [tf.pack_nvfp4(dc, ds, gs) for _ in range(n_copies)]
    x = torch.from_numpy(inputs.bf16_normal(rng, (16, K)).view(np.int16)).cuda()
    y = torch.empty((16, N), device="cuda")
    ws = tf.workspace(int(tf.load().tf_lane_gemm_nvfp4_workspace_bytes(K, N)))
    out = {"bytes_per_launch": nbytes}
    for R in (1, 8, 16):
        xv, yv = x[:R], y[:R]
        for c in copies:
            tf.lane_gemm_nvfp4(c, xv, y=yv, ws=ws)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for c in copies:
                tf.lane_gemm_nvfp4(c, xv, y=yv, ws=ws)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / (steps * n_copies)
        out[f"R{R}"] = {"us_per_launch": us, "gbs": nbytes / us / 1e3, "frac_of_hbm_peak": nbytes / us / 1e3 / peaks()[0]}
    return out


def attention_bytes(ctx, R, n_kv=8, group=8):
    """Algorithmic bytes of one verify attention call over ctx cached positions:
    K and V entries 0..ctx-1 (bf16), the bf16 queries and the fp32 outputs."""
    n_q = n_kv * group
    return ctx * n_kv * 128 * 2 * 2 + R * n_q * 128 * 2 + R * n_q * 128 * 4


def extra_attention(tf, torch, steps=30, ctxs=(8192, 32768), rows=(1, 8, 16)):
    """Verify attention over a KV cache (8 KV heads, group 8, head dim 128) at
    8192 and 32768 cached positions, R = 1 / 8 / 16: partial + combine kernels,
    caches rotating over copies larger than L2, CUDA-graph replay."""
    n_kv, group = 8, 8
    out = {}
    gen = torch.Generator(device="cuda")
    gen.manual_seed(11)
    for ctx in ctxs:
        cache_bytes = ctx * n_kv * 128 * 2 * 2
        n_copies = max(3, -(-3 * L2_BYTES // cache_bytes))
        caches = []
        for _ in range(n_copies):
            c = tf.KVCache(n_kv, ctx)
            c.k.copy_((torch.randn(c.k.shape, device="cuda", generator=gen)).bfloat16().view(torch.int16))
            c.v.copy_((torch.randn(c.v.shape, device="cuda", generator=gen)).bfloat16().view(torch.int16))
            caches.append(c)
        q = torch.randn((16, n_kv * group * 128), device="cuda", generator=gen).bfloat16().view(torch.int16)
        y = torch.empty((16, n_kv * group * 128), device="cuda")
        ws = tf.workspace(caches[0].workspace_bytes(group, 16))
        for R in rows:
            pos = torch.tensor([ctx - R], dtype=torch.int64, device="cuda")
            for c in caches:
                c.attention(q[:R], group, pos, out=y[:R], ws=ws)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for c in caches:
                    c.attention(q[:R], group, pos, out=y[:R], ws=ws)
            g.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(steps):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / (steps * n_copies)
            nbytes = attention_bytes(ctx, R, n_kv, group)
            out[f"ctx{ctx}_R{R}"] = {"us_per_call": us, "gbs": nbytes / us / 1e3, "bytes_per_call": nbytes,
                                     "frac_of_hbm_peak": nbytes / us / 1e3 / peaks()[0]}
        assert tf.workspace_status(ws) == tf.TF_DEV_OK
        del caches
        torch.cuda.empty_cache()
    return out


def extra_moe(tf, torch, steps=32, n_router=8):
    """30B-A3B-class MoE layer at R = 1, 4, 8, 16.  L2 is defeated twice over:
    two full copies of the 128 experts (2 x 340 MB) alternate, and every call
    draws one of n_router seeded router-logit sets, so the touched set changes
    from call to call.  GB/s counts the touched experts' weight bytes of each call."""
    from w4_gemm_keyed_gb300 import inputs
    E, H, F, G, k = 128, 2048, 768, 32, 8
    rng = inputs.rng_for(4, 99)
    sz_gu, sz_d = tf.packed_bytes(H, 2 * F, G), tf.packed_bytes(F, H, G)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(4)
    layers = []
    for _ in range(2):
        gu = torch.empty(E * sz_gu, dtype=torch.uint8, device="cuda")
        dn = torch.empty(E * sz_d, dtype=torch.uint8, device="cuda")
        for e in range(E):
            c = torch.randint(0, 256, (2 * F, H // 2), dtype=torch.uint8, device="cuda", generator=gen)
            s = (torch.randn((2 * F, H // G), device="cuda", generator=gen).abs() * 0.02 + 1e-3).half().view(torch.int16)
            tf.pack_w4(c, s, G, gate_up=True, out=gu[e * sz_gu:(e + 1) * sz_gu])
            c = torch.randint(0, 256, (H, F // 2), dtype=torch.uint8, device="cuda", generator=gen)
            s = (torch.randn((H, F // G), device="cuda", generator=gen).abs() * 0.02 + 1e-3).half().view(torch.int16)
            tf.pack_w4(c, s, G, out=dn[e * sz_d:(e + 1) * sz_d])
        layers.append(tf.MoeLayer(gu, dn, H, F, E, k, G))
    expert_bytes = (2 * F * H // 2 + 2 * 2 * F * (H // G)) + (H * F // 2 + 2 * H * (F // G))
    out = {"expert_bytes": expert_bytes, "l2": "two expert sets alternate; router logits rotate over 8 draws"}
    for R in (1, 4, 8, 16):
        x = torch.from_numpy(inputs.bf16_normal(rng, (R, H)).view(np.int16)).cuda()
        zs = [inputs.router_logits(rng, R, E) for _ in range(n_router)]
        touched = [len(np.unique(np.argsort(-z, axis=1, kind="stable")[:, :k])) for z in zs]
        zd = [torch.from_numpy(z).cuda() for z in zs]
        ws = tf.workspace(tf.moe_workspace_bytes(layers[0], R))
        y = torch.empty((R, H), device="cuda")

        def call(i):
            tf.moe_w4(layers[i % 2], x, zd[i % n_router], out=y, ws=ws)
        for i in range(4):
            call(i)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(steps):
            call(i)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        mean_touched = sum(touched[i % n_router] for i in range(steps)) / steps
        gbs = mean_touched * expert_bytes / (ms * 1e-3) / 1e9
        out[f"R{R}"] = {"touched_experts_mean": mean_touched, "touched_bytes_mean": mean_touched * expert_bytes,
                        "gbs": gbs, "frac_of_hbm_peak": gbs / peaks()[0], "us_per_layer": ms * 1e3}
    assert tf.workspace_status(ws) == tf.TF_DEV_OK
    del layers
    return out


def extra_decoder(tf, torch, steps=10):
    """Synthetic 27B-class decoder (8 blocks + LM head): verify steps/s at R = 1, 2, 4, 8, 16."""
    from w4_gemm_keyed_gb300 import decode
    V, H, F, L, G = 151936, 5120, 17408, 8, 64
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)

    def mat(K, N, gate_up=False):
        c = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda", generator=gen)
        s = (torch.randn((N, K // G), device="cuda", generator=gen).abs() * 0.02 + 1e-3).half().view(torch.int16)
        return tf.pack_w4(c, s, G, gate_up=gate_up)

    emb = (torch.randn((V, H), device="cuda", generator=gen) * 0.02).bfloat16().view(torch.int16)
    gu = [mat(H, 2 * F, True) for _ in range(L)]
    dn = [mat(F, H) for _ in range(L)]
    lm = mat(H, V)
    model = tf.Model(emb, gu, dn, lm, V, H, F, G)
    dec = decode.Decoder(model)
    step_bytes = L * (bytes_per_launch(H, 2 * F) + bytes_per_launch(F, H)) + bytes_per_launch(H, V)
    out = {"weight_bytes_per_step": step_bytes}
    for R in ROWS:
        dec.reset(1, 1)
        d = torch.zeros(16, dtype=torch.int32, device="cuda")
        for _ in range(2):
            model.verify_step(R, dec.last, dec.pos, d, 0.7, 20, 0.95, 1234, dec.tokens, dec.accepted, dec.ws)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            model.verify_step(R, dec.last, dec.pos, d, 0.7, 20, 0.95, 1234, dec.tokens, dec.accepted, dec.ws)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        out[f"R{R}"] = {"verify_steps_per_s": 1e3 / ms, "rows_per_s": R * 1e3 / ms, "ms_per_step": ms,
                        "gbs": step_bytes / (ms * 1e-3) / 1e9,
                        "frac_of_hbm_peak": step_bytes / (ms * 1e-3) / 1e9 / peaks()[0]}
    out["decode"] = decode_loop(tf, torch, dec, V)
    return out


def decode_loop(tf, torch, dec, V, n_tokens=64, R=8, p_match=0.75, seeds=(1234, 1235, 1236, 1237, 1238)):
    """Synthetic decoder, decode loop on the device (CUDA-graph replays of 8 passes):
    64 tokens serially (R = 1) and with R = 8 drafts that copy the serial token
    with probability 0.75, T = 0.7 / top-k 20 / top-p 0.95, per seed; tokens/s,
    mean tokens committed per drafted pass, and whether the token_sha agree."""
    from w4_gemm_keyed_gb300 import decode, inputs
    T, k, p, prompt = 0.7, 20, 0.95, 11
    ser_s = dr_s = 0.0
    committed = passes_needed = 0
    same = True
    for seed in seeds:
        loop1 = decode.GraphLoop(dec, n_tokens + 2 * R, 1, T, k, p, seed, prompt_token=prompt)
        loop1.run(prompt)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        serial, _ = loop1.run(prompt)
        b.record()
        torch.cuda.synchronize()
        ser_s += a.elapsed_time(b) / 1e3 * n_tokens / (n_tokens + 2 * R)
        rng = inputs.rng_for(701, seed)
        truth = np.zeros(n_tokens + 12 * R, dtype=np.int64)
        truth[1:1 + len(serial)] = serial[: len(truth) - 1]
        table = torch.from_numpy(inputs.noisy_drafts(rng, truth, p_match, V)).cuda()
        loop8 = decode.GraphLoop(dec, n_tokens, R, T, k, p, seed, table, prompt_token=prompt)
        loop8.run(prompt)
        a.record()
        drafted, _ = loop8.run(prompt)
        b.record()
        torch.cuda.synchronize()
        dr_s += a.elapsed_time(b) / 1e3
        same &= decode.token_sha(drafted) == decode.token_sha(serial[:n_tokens])
        host_table = table.cpu().numpy()
        _, lens = decode.drafted_decode(dec, prompt, n_tokens, R, T, k, p, seed,
                                        lambda pos0, m: host_table[pos0: pos0 + m])
        committed += sum(x + 1 for x in lens)
        passes_needed += len(lens)
    n = len(seeds)
    return {"tokens": n_tokens, "seeds": n, "serial_tokens_per_s": n * n_tokens / ser_s,
            "drafted_tokens_per_s": n * n_tokens / dr_s, "drafted_R": R,
            "mean_tokens_per_pass": committed / passes_needed, "token_sha_equal": bool(same),
            "note": "graph replays of 8 passes; a run ends at the first replay that reaches the token count"}


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample_rate(mats_host, budget_s):
    """Run the oracle on a column sample of the headline step; return (GB/s, cores, sample text)."""
    import oracle
    cores = oracle.num_threads()
    # calibrate on a small sample, then size the sample to the budget
    cols_per = 64
    t0 = time.perf_counter()
    done_bytes = 0
    rounds = 0
    while True:
        for K, N in SHAPES:
            codes, scales, x = mats_host[(K, N)]
            cols = np.linspace(0, N - 1, cols_per).astype(np.int64)
            for R in ROWS:
                oracle.w4_linear(codes, scales, x[:R], GROUP, cols=cols)
                done_bytes += cols_per * (K // 2 + 2 * (K // GROUP))
        rounds += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
        if el < budget_s / 8:
            cols_per *= 2
    gbs = done_bytes / el / 1e9
    return gbs, cores, (f"{rounds} passes of the step over evenly spaced column samples "
                        f"(final {cols_per} columns per shape), {done_bytes / 1e6:.1f} MB of weights in {el:.1f} s")


def host_mats():
    from w4_gemm_keyed_gb300 import inputs
    out = {}
    for K, N in SHAPES:
        rng = inputs.rng_for(2, K, N)
        codes, scales = inputs.w4_weights(rng, K, N, GROUP)
        x = inputs.bf16_normal(rng, (16, K))
        out[(K, N)] = (codes, scales, x)
    return out


# ----------------------------------------------------------------------------- main
def max_over_ranks(value: float, world: int, device: str) -> float:
    """The largest value over all ranks: the whole job's time is its slowest rank's."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step: int, steps: int, world: int, secs: float) -> float:
    """Replicas (weak scaling): every rank streams its own copy of the step's bytes."""
    return bytes_per_step * steps * world / secs / 1e9


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    budget_total = float(os.environ.get("TF_REFERENCE_BUDGET_S", "120"))
    per_step = max(0.05, budget_total / max(1, args.steps + args.warmup))
    mats = host_mats()
    import oracle
    cores = oracle.num_threads()
    cols_per = max(1, int(per_step * 2e4))  # rough first guess, refined by the warm-up
    # warm-up steps also calibrate the per-step sample size
    for _ in range(max(1, args.warmup)):
        t0 = time.perf_counter()
        for K, N in SHAPES:
            codes, scales, x = mats[(K, N)]
            cols = np.linspace(0, N - 1, cols_per).astype(np.int64)
            for R in ROWS:
                oracle.w4_linear(codes, scales, x[:R], GROUP, cols=cols)
        el = time.perf_counter() - t0
        cols_per = max(1, min(5120, int(cols_per * per_step / max(el, 1e-6))))
    step_bytes = sum(cols_per * (K // 2 + 2 * (K // GROUP)) for K, _ in SHAPES) * len(ROWS)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for K, N in SHAPES:
            codes, scales, x = mats[(K, N)]
            cols = np.linspace(0, N - 1, cols_per).astype(np.int64)
            for R in ROWS:
                oracle.w4_linear(codes, scales, x[:R], GROUP, cols=cols)
    el = time.perf_counter() - t0
    gbs = step_bytes * args.steps / el / 1e9
    sample = f"each step: {cols_per} evenly spaced output columns per shape at every R (of 17408 / 5120)"
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD + " (CPU oracle, column sample)", "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="tf", choices=["tf", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the LM-head / MoE / decoder side measurements")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--only", choices=["lmhead", "dense", "moe", "decoder", "affine", "attention", "nvfp4", "sampler"],
                    help="run one workload briefly and print its timings (for profiler captures)")
    ap.add_argument("--ctx", type=int, nargs="*", help="with --only attention: cached positions to time")
    ap.add_argument("--rows", type=int, nargs="*", help="with --only attention: verify rows R to time")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    world, rank, local = dist_env()
    import torch
    torch.cuda.set_device(local)
    if args.only:
        from w4_gemm_keyed_gb300 import tf
        tf.load()
        if args.only == "dense":
            mats = setup_dense(tf, torch, rank)
            secs, steps, lps = time_dense(tf, torch, mats, args.steps, args.warmup)
            out = {"dense_gbs": STEP_BYTES * steps / secs / 1e9}
        else:
            fn = {"lmhead": extra_lmhead, "moe": extra_moe, "decoder": extra_decoder, "affine": extra_affine,
                  "attention": extra_attention, "nvfp4": extra_nvfp4, "sampler": extra_sampler}[args.only]
            kw = {}
            if args.only == "attention" and args.ctx:
                kw["ctxs"] = tuple(args.ctx)
            if args.only == "attention" and args.rows:
                kw["rows"] = tuple(args.rows)
            out = fn(tf, torch, steps=args.steps, **kw)
        print(json.dumps({"only": args.only, "result": out}))
        return 0
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from w4_gemm_keyed_gb300 import tf
    tf.load()

    mats = setup_dense(tf, torch, rank)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # ---- headline: device-resident inputs
    barrier()
    with ClockSampler(local) as clk:
        secs, steps, launches_per_step = time_dense(tf, torch, mats, args.steps, args.warmup)
    barrier()
    secs = max_over_ranks(secs, world, "cuda")
    value = whole_job_gbs(STEP_BYTES, steps, world, secs)
    peak, peak_kind = peaks()
    # every launch of the step streams the same number of bytes; the average
    # launch duration over the timed region includes the inter-kernel gaps
    avg_launch_ms = secs * 1e3 / (steps * launches_per_step)
    achieved = bytes_per_launch(*SHAPES[0]) / (avg_launch_ms * 1e-3) / 1e9
    per = time_per_launch(tf, torch, mats)
    per_R = {}
    for (K, N, R), v in sorted(per.items()):
        ms = sum(v) / len(v)
        per_R[f"{K}x{N}_R{R}"] = {"us": ms * 1e3, "gbs": bytes_per_launch(K, N) / (ms * 1e-3) / 1e9,
                                  "frac": bytes_per_launch(K, N) / (ms * 1e-3) / 1e9 / peak}
    per_graph = {}
    for (K, N, R), us in sorted(time_per_r_graph(tf, torch, mats).items()):
        gbs = bytes_per_launch(K, N) / us / 1e3
        per_graph[f"{K}x{N}_R{R}"] = {"us": us, "gbs": gbs, "frac": gbs / peak}

    # ---- end to end through the C ABI with host buffers
    e2e_steps = max(10, args.steps // 4)
    barrier()
    e2e_secs, h2d, d2h = time_dense_e2e(tf, torch, mats, e2e_steps, args.warmup)
    barrier()
    e2e_secs = max_over_ranks(e2e_secs, world, "cuda")
    e2e_value = whole_job_gbs(STEP_BYTES, e2e_steps, world, e2e_secs)

    extra = {}
    if rank == 0 and not args.no_extra:
        for name, fn in (("lmhead_sampler", extra_lmhead), ("moe30b", extra_moe), ("decoder", extra_decoder),
                         ("affine_5120x17408", extra_affine), ("nvfp4_5120x17408", extra_nvfp4),
                         ("attention_kv", extra_attention), ("sampler_151936", extra_sampler)):
            try:
                extra[name] = fn(tf, torch)
            except Exception as exc:  # a side measurement must not hide the headline line
                extra[name] = {"error": repr(exc)}
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1:
        gbs, cores, sample = oracle_sample_rate(host_mats(), args.cpu_budget)
        cpu = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": secs / steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int4 codes x bf16 -> fp32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "bytes_per_step": STEP_BYTES,
                       "l2": "weights rotate over copies > 3x L2 (evict-first loads)",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "traffic": recorded_traffic(), "kernel": "w4_lane_gemm_kernel<64,HI>"},
            "per_r_device": per_graph,
            "per_r_device_note": ("each (shape, R) as a CUDA graph of back-to-back launches over weight "
                                  "copies > 3x L2; frac of the HBM peak above"),
            "per_launch": per_R,
            "per_launch_note": "each launch timed alone with events: includes launch latency",
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": steps * launches_per_step,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
            "extra": extra,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
