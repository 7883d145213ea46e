import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long CPU-side oracle runs")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library on a GPU; fails loudly if it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from serving_sparse_mla_gb300 import binding
    return binding.load()


def pytest_terminal_summary(terminalreporter):
    """Per-workload parity statistics recorded by the GPU tests (worst
    |out - oracle|, |lse - oracle| and the tight-check ratio), beside the
    pages' own maximum differences (1.22e-4 and 2.44e-4 on H200)."""
    from tests.parity import RECORD
    if not RECORD:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity statistics (pages' H200 max |diff|: 1.22e-4, 2.44e-4)")
    for name, st in RECORD.items():
        tr.write_line(f"{name}: " + ", ".join(
            f"{k}={v:.3e}" if isinstance(v, float) else f"{k}={v}" for k, v in st.items()))
