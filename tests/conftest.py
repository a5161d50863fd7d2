import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# Every buffer the binding allocates for a test gets a guard tail that is
# checked after the test (memory-safety stand-in for a sanitizer run).
os.environ.setdefault("H3LIN_CANARY", "1")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


@pytest.fixture(autouse=True)
def _canaries():
    """After each test: no kernel wrote past the end of a workspace or output
    the binding allocated (the guard tails still hold their fill byte), and,
    under the bounds build, no workspace recorded H3LIN_E_BOUNDS."""
    yield
    h3lin = sys.modules.get("nvfp4_linear_lora_gb300.h3lin")
    torch = sys.modules.get("torch")
    if h3lin is None or torch is None or not torch.cuda.is_available():
        return
    h3lin.check_canaries()
    h3lin.check_bounds_status()   # bounds build: no kernel index left its buffer
