"""The bounds-checked build (libzero_checked.so): every kernel access is
tested against the extent the C ABI gives its buffer and recorded when
outside.  The GPU suite runs once more against it in a child process, where
an autouse fixture requires an empty record after every test."""
import os
import re
import subprocess
import sys

import pytest

import zero_sharded_optimizer_device_gb300 as Z

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CHECKED = os.environ.get("ZERO_CHECKED") == "1"


def test_probe_record_reaches_the_host(cuda):
    import torch
    Z.zero_bounds_report(reset=True)
    Z.zero_bounds_probe()
    r = Z.zero_bounds_report(reset=True)
    if CHECKED:
        assert r == dict(checked=1, site=Z.ZERO_SITE_PROBE, count=1, index=1, lo=0, hi=1)
    else:
        assert r == dict(checked=0, site=0, count=0, index=0, lo=0, hi=0)
    assert Z.zero_bounds_report()["count"] == 0
    torch.cuda.synchronize()


@pytest.mark.skipif(CHECKED, reason="already running under the checked build")
def test_gpu_suite_under_the_checked_build(cuda):
    import torch
    if not os.path.exists(os.path.join(ROOT, "zero_sharded_optimizer_device_gb300",
                                       "libzero_checked.so")):
        pytest.fail("libzero_checked.so is missing: run __graft_entry__.build()")
    torch.cuda.empty_cache()
    env = dict(os.environ, ZERO_CHECKED="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "tests", "-m", "gpu", "-q", "-x",
                        "-p", "no:cacheprovider", "-k", "not test_gpu_suite_under_the_checked"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-30:])
    assert r.returncode == 0, tail
    m = re.search(r"(\d+) passed", tail)
    assert m and int(m.group(1)) >= 60 and "failed" not in tail, tail
