import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes of oracle CPU time)")


@pytest.fixture(scope="session")
def rng():
    import numpy as np

    return np.random.default_rng(1234)


def pytest_sessionfinish(session, exitstatus):
    """Write the parity margins the full-size GPU tests recorded (nothing when none ran)."""
    import gdr_testlib

    if not gdr_testlib._MARGINS:
        return
    try:
        import torch

        name = torch.cuda.get_device_name(0)
    except Exception:  # noqa: BLE001 - the name is only a label
        name = "unknown GPU"
    path = os.environ.get("GDR_PARITY_MARGINS", os.path.join(ROOT, "profiles", "parity_margins.md"))
    gdr_testlib.write_margins(path, name)
