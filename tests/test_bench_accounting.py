"""The measurement arithmetic of bench.py, on CPU: algorithmic bytes per launch
and per step (the roofline numerators), the step's launch list, and that the
committed DRAM-traffic record is reported only for the kernel sources it was
taken on."""

import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    import sys
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench as b
    return b


def test_algorithmic_bytes_per_launch(bench):
    # codes K*N/2 + fp16 scales 2*N*K/64
    assert bench.bytes_per_launch(5120, 17408) == 44_564_480 + 2_785_280 == 47_349_760
    assert bench.bytes_per_launch(17408, 5120) == 47_349_760
    assert bench.bytes_per_launch(5120, 151936) == 413_265_920
    assert bench.bytes_per_launch(2048, 768, 32) == 2048 * 768 // 2 + 2 * 768 * 2048 // 32


def test_the_step_is_ten_launches_of_the_two_projections(bench):
    launches = bench.dense_launches()
    assert len(launches) == 10
    assert sorted({(K, N) for K, N, _ in launches}) == [(5120, 17408), (17408, 5120)]
    assert sorted(R for K, N, R in launches if (K, N) == (5120, 17408)) == [1, 2, 4, 8, 16]
    assert bench.STEP_BYTES == 10 * 47_349_760 == 473_497_600


def test_attention_bytes(bench):
    # K and V of every cached position (bf16) + bf16 queries + fp32 outputs
    assert bench.attention_bytes(32768, 1) == 32768 * 8 * 128 * 2 * 2 + 64 * 128 * 2 + 64 * 128 * 4 == 134_266_880
    assert bench.attention_bytes(8192, 16) == 8192 * 8 * 512 + 16 * 64 * 256 + 16 * 64 * 512


def test_traffic_record_is_used_only_for_the_sources_it_was_taken_on(bench):
    rec = json.load(open(os.path.join(ROOT, "profiles", "w4_lane_gemm_traffic.json")))
    if rec["kernel_source_hash"] == bench.kernel_source_hash():
        assert bench.recorded_traffic() == rec["dram_bytes_per_launch"]
    else:
        assert bench.recorded_traffic() is None     # the kernel changed since the counters were taken
    # the recorded traffic is within a few per cent of the algorithmic bytes: no re-reads
    assert 1.0 <= rec["dram_bytes_per_launch"] / 47_349_760 < 1.05


class _Counter:
    n = 0


class _FakeGraph:
    def __init__(self):
        self.calls = 0

    def replay(self):
        _Counter.n += self.calls


class _FakeEvent:
    def record(self, stream=None):
        self.at = _Counter.n

    def elapsed_time(self, end):
        return float(end.at - self.at)      # "milliseconds" = launches executed in between


class _FakeCuda:
    capturing = None

    def synchronize(self):
        pass

    def CUDAGraph(self):
        return _FakeGraph()

    def graph(self, g):
        import contextlib

        @contextlib.contextmanager
        def cm():
            _FakeCuda.capturing = g
            try:
                yield
            finally:
                _FakeCuda.capturing = None
        return cm()

    def current_stream(self):
        return None

    def Event(self, enable_timing=False):
        return _FakeEvent()


class _FakeTorch:
    cuda = _FakeCuda()


class _FakeTf:
    @staticmethod
    def lane_gemm_w4(W, x, y=None, ws=None):
        if _FakeCuda.capturing is not None:
            _FakeCuda.capturing.calls += 1  # recorded into the graph
        else:
            _Counter.n += 1


@pytest.mark.parametrize("steps", [1, 8, 9, 10, 2000, 2007])
def test_time_dense_times_exactly_the_requested_steps(bench, steps):
    """The device-timed region runs exactly ``steps`` steps of the ten launches,
    whatever the length of the weight-rotation cycle (9 copies here)."""
    mats = {(K, N): {"copies": list(range(9)), "x": [0] * 16, "y": [0] * 16, "ws": None}
            for K, N in {(K, N) for K, N, _ in bench.dense_launches()}}
    secs, timed, per_step = bench.time_dense(_FakeTf, _FakeTorch, mats, steps, warmup=3)
    assert timed == steps and per_step == 10
    assert secs * 1e3 == steps * 10           # launches executed between the two events
