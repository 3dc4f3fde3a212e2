"""Failure detection without a GPU fault: a bounded device wait on a flag
that a peer (here: the host) sets, or never sets.  The wait always ends and
reports ZERO_ETIMEOUT through a status word; the context stays usable."""
import threading
import time

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_wait_times_out_when_nothing_signals(cuda):
    import torch
    import zero_sharded_optimizer_device_gb300 as Z
    flag = torch.zeros(1, dtype=torch.int32, device=cuda)
    status = torch.full((1,), 99, dtype=torch.int32, device=cuda)
    t0 = time.time()
    Z.zero_wait_flag(flag, 1, 2000, status)
    torch.cuda.synchronize()
    assert status.item() == Z.ZERO_ETIMEOUT
    assert time.time() - t0 < 5.0
    # the context is still usable
    x = torch.arange(1024, device=cuda, dtype=torch.float32)
    y = torch.empty_like(x)
    Z.zero_copy(y, x, x.numel() * 4)
    torch.cuda.synchronize()
    assert torch.equal(x, y)


def test_wait_succeeds_on_a_preset_flag(cuda):
    import torch
    import zero_sharded_optimizer_device_gb300 as Z
    flag = torch.full((1,), 7, dtype=torch.int32, device=cuda)
    status = torch.full((1,), 99, dtype=torch.int32, device=cuda)
    Z.zero_wait_flag(flag, 7, 1000, status)
    torch.cuda.synchronize()
    assert status.item() == Z.ZERO_OK


def test_wait_sees_a_flag_the_host_sets_while_it_polls(cuda):
    """The flag lives in mapped pinned host memory; a host thread sets it
    ~50 ms after the launch, well inside the ~5 s bound."""
    import torch
    import bench
    import zero_sharded_optimizer_device_gb300 as Z
    flag = torch.zeros(1, dtype=torch.int32, pin_memory=True)
    if not bench.host_mapped(flag):
        pytest.skip("pinned host memory is not mapped into the device address space")
    status = torch.full((1,), 99, dtype=torch.int32, device=cuda)
    view = flag.numpy()
    Z.zero_wait_flag(flag, 1, 5_000_000, status)
    timer = threading.Timer(0.05, lambda: view.__setitem__(0, np.int32(1)))
    timer.start()
    torch.cuda.synchronize()
    timer.join()
    assert status.item() == Z.ZERO_OK
