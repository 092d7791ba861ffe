import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


@pytest.fixture(scope="session")
def tf():
    """The CUDA library's Python binding; fails loudly if it cannot be loaded."""
    if not gpu_available():
        pytest.skip("no CUDA device")
    from w4_gemm_keyed_gb300 import tf as binding
    binding.load()
    return binding


# Near-ties of the keyed sampler: a GPU token that differs from the oracle's is
# accepted only when the oracle's top-2 score gap is below 1e-9 (fp64 log/exp
# of the two sides may round differently).  Every such case is recorded on the
# test (JUnit property) and counted in the terminal summary, which prints even
# when the count is zero.
NEAR_TIES = []


@pytest.fixture
def near_tie(record_property):
    def log(where: str, gap: float):
        NEAR_TIES.append((where, float(gap)))
        record_property(f"near_tie_{len(NEAR_TIES)}", f"{where} gap={gap:.3e}")
    return log


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    if NEAR_TIES:
        worst = max(g for _, g in NEAR_TIES)
        terminalreporter.write_line(f"keyed-sampler near-ties accepted: {len(NEAR_TIES)} (largest oracle gap {worst:.3e})")
        for where, gap in NEAR_TIES[:20]:
            terminalreporter.write_line(f"  near-tie {where}: gap {gap:.3e}")
    else:
        terminalreporter.write_line("keyed-sampler near-ties accepted: 0")
