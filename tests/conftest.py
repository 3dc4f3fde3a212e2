import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name):
    """Parse a `key = value` golden fixture; '#' starts a comment."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = v
    return out


@pytest.fixture(scope="session")
def cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _no_out_of_extent_access(request):
    """After every GPU test: no bounded device wait gave up, and under the
    bounds-checked library (ZERO_CHECKED=1) the kernels' out-of-extent
    record is empty."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    import zero_sharded_optimizer_device_gb300 as Z
    assert Z.zero_async_status(reset=True) == 0, "a bounded device wait gave up"
    if os.environ.get("ZERO_CHECKED") != "1":
        return
    r = Z.zero_bounds_report(reset=True)
    assert r["checked"] == 1, "ZERO_CHECKED=1 but the release library is loaded"
    assert r["count"] == 0, f"kernel accesses outside their buffer's extent: {r}"
