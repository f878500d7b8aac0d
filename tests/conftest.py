import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: larger CPU case")


@pytest.fixture(scope="session")
def golden():
    """Parse tests/golden/page_examples.txt into {name: value}."""
    path = os.path.join(ROOT, "tests", "golden", "page_examples.txt")
    vals = {}
    with open(path, encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (x.strip() for x in line.split("=", 1))
            vals[key] = eval(val, {"__builtins__": {}}, {"range": range, "list": list})  # literals only
    return vals


@pytest.fixture(scope="session")
def kvc_lib():
    """Build (if needed) and load the CUDA library; GPU tests fail loudly without it."""
    import torch

    import paged_kv_cache_135_gb300 as kvc
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    kvc.build()
    kvc.lib()
    return kvc
