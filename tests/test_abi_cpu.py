"""CPU-only checks of the C ABI: the library loads and exports every function
include/zero.h declares; the host planner matches the oracle's plan exactly;
argument checks return their error codes before any device work; host-side
fault injection; the benchmark's multi-rank aggregation over gloo."""
import os
import subprocess
import sys

import pytest

from oracle import zero_oracle as O
from synth import workloads as W

Z = pytest.importorskip("zero_sharded_optimizer_device_gb300")


def test_library_exports_every_declared_function():
    lib = Z.binding._lib()
    declared = Z.header_functions()
    assert len(declared) >= 20
    for name in declared:
        assert hasattr(lib, name), name
    # and the binding wraps each of them under the same name
    for name in declared:
        assert callable(getattr(Z, name)), name


def test_checked_build_exports_the_same_functions():
    import ctypes
    path = os.path.join(os.path.dirname(Z.binding.LIB_PATH), "libzero_checked.so")
    if not os.path.exists(path):
        pytest.skip("libzero_checked.so not built")
    lib = ctypes.CDLL(path)
    for name in Z.header_functions():
        assert hasattr(lib, name), name


def test_release_bounds_report_is_empty_without_a_device():
    """The release library has no checks: its report needs no device and says
    so; its probe is a no-op."""
    if os.environ.get("ZERO_CHECKED") == "1":
        pytest.skip("checked build loaded")
    assert Z.zero_bounds_report() == dict(checked=0, site=0, count=0, index=0, lo=0, hi=0)
    Z.zero_bounds_probe(0)
    with pytest.raises(Z.ZeroError) as e:
        Z.binding._check(Z.binding._lib().zero_bounds_report(None, 0), "zero_bounds_report")
    assert e.value.status == Z.ZERO_EINVAL


def test_strerror_covers_every_status():
    for code in range(0, -8, -1):
        assert Z.zero_strerror(code) and Z.zero_strerror(code) != "unknown status"
    assert Z.zero_strerror(-99) == "unknown status"


def _compare_plans(numels, n, align, groups=None):
    p = Z.zero_plan(numels, n, align, groups)
    o = O.plan(numels, n, align, groups)
    info = Z.zero_plan_info(p)
    assert (info["psi"], info["psi_pad"], info["shard_total"]) == (o.psi, o.psi_pad, o.shard_total)
    assert info["n_groups"] == len(o.groups)
    for gi, g in enumerate(o.groups):
        zg = Z.zero_plan_group(p, gi)
        assert (zg["psi"], zg["psi_pad"], zg["shard"], zg["flat_off"], zg["rank_off"]) == \
            (g.psi, g.psi_pad, g.shard, g.flat_off, g.rank_off)
        for r in range(n):
            assert Z.zero_plan_shard(p, gi, r) == o.shard_range(gi, r)
    for t in range(len(numels)):
        assert Z.zero_plan_tensor(p, t) == (o.tensor_flat_off(t), *o.owner_span(t))
    for r in range(n):
        assert Z.zero_plan_segments(p, r) == o.segments(r)
    for stage in range(4):
        assert Z.zero_plan_memory(p, stage) == o.memory(stage)
    assert Z.zero_plan_volume(p) == O.volume(o)


@pytest.mark.parametrize("w", list(W.ALL.values()), ids=lambda w: w.name)
def test_planner_matches_oracle_on_workloads(w):
    _compare_plans(w.numels, w.n_ranks, w.align, w.groups)


@pytest.mark.parametrize("numels,n,align,groups", [
    ([], 4, 16, None), ([0, 5, 0], 2, 1, None), ([7], 1, 1, None), ([1], 64, 1, None),
    ([3, 1, 4, 1, 5, 9, 2, 6], 3, 5, [0, 0, 1, 1, 1, 2, 3, 3]), ([10**12, 7], 64, 128, None),
])
def test_planner_matches_oracle_on_edge_cases(numels, n, align, groups):
    _compare_plans(numels, n, align, groups)


def test_planner_matches_oracle_on_random_plans():
    """300 seeded random plans: tensor counts 1-40 (empty tensors included),
    sizes over six decades, N = 1..64, align 1..128, random layer groups."""
    import numpy as np
    rng = np.random.default_rng(2024)
    for _ in range(300):
        T = int(rng.integers(1, 41))
        numels = [0 if rng.random() < 0.05 else int(10 ** rng.uniform(0, 6)) for _ in range(T)]
        n = int(rng.integers(1, 65))
        align = int(rng.choice([1, 2, 3, 4, 8, 16, 32, 128]))
        groups = None
        if rng.random() < 0.5:
            g = np.cumsum(rng.random(T) < 0.3)
            groups = [int(x) for x in (g - g[0])]
        _compare_plans(numels, n, align, groups)


def test_binding_rejects_pageable_cpu_tensors():
    """A CPU tensor in pageable memory never reaches the library (its address
    would mean nothing to a kernel); the check runs before any call."""
    import torch
    p = Z.zero_plan([100], 2, 16)
    cpu = torch.zeros(112, dtype=torch.float32)
    if Z.binding._host_memory_reachable(cpu.data_ptr()):
        pytest.skip("this system's GPU reads pageable host memory")
    with pytest.raises(ValueError):
        Z.zero_all_gather(p, 0, cpu, cpu, Z.ZERO_F32, 0)
    with pytest.raises(ValueError):
        Z.zero_gather_layer(p, 0, [cpu, cpu], Z.ZERO_F32, None, 0)


def test_planner_from_several_host_threads():
    """Plans are built and queried from 8 host threads at once (the library
    keeps no shared mutable planner state); every thread sees the oracle's map."""
    import threading
    w = W.GPT2_SMALL
    o = O.plan(w.numels, w.n_ranks, w.align)
    errors = []

    def worker():
        try:
            for _ in range(20):
                p = Z.zero_plan(w.numels, w.n_ranks, w.align)
                info = Z.zero_plan_info(p)
                assert (info["psi_pad"], info["shard_total"]) == (o.psi_pad, o.shard_total)
                for r in (0, w.n_ranks - 1):
                    assert Z.zero_plan_segments(p, r) == o.segments(r)
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker) for _ in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[0]


def test_random_calls_return_a_status_and_never_crash():
    """2 000 seeded random calls of the device entry points with random
    groups, windows, sizes, dtypes and (never dereferenced) addresses: each
    returns a known status code.  Host-only: with no GPU present any call
    that passes its checks fails at the launch with ZERO_ECUDA; it is skipped
    where a GPU is present, since there it could launch on bogus addresses."""
    import numpy as np
    import torch
    if torch.cuda.is_available():
        pytest.skip("would launch kernels on fake addresses")
    lib = Z.binding._lib()
    codes = {Z.ZERO_OK, Z.ZERO_EINVAL, Z.ZERO_EALIGN, Z.ZERO_ERANGE, Z.ZERO_EDTYPE,
             Z.ZERO_ENOMEM, Z.ZERO_ECUDA, Z.ZERO_ETIMEOUT}
    rng = np.random.default_rng(99)
    plans = [Z.zero_plan([int(x) for x in rng.integers(0, 5000, int(rng.integers(1, 8)))],
                         int(rng.integers(1, 17)), int(rng.choice([1, 8, 16])),
                         None) for _ in range(6)]
    addrs = [0, 1 << 40, (1 << 40) + 16, (1 << 40) + 4, (1 << 40) + 8]

    def addr():
        return int(rng.choice(addrs))

    def ptrs(n):
        return [addr() for _ in range(max(0, n))]

    hp = Z.adam_hp(int(rng.integers(0, 3)), 0.25)
    seen = set()
    for _ in range(2000):
        p = plans[int(rng.integers(0, len(plans)))]
        n = Z.zero_plan_info(p)["n_ranks"]
        g = int(rng.integers(-1, 3))
        a, b = (int(x) for x in rng.integers(-5, 12000, 2))
        dt = int(rng.integers(-1, 3))
        which = int(rng.integers(0, 8))
        B = Z.binding
        if which == 0:
            st = lib.zero_reduce_scatter(p, g, B._ptr_array(ptrs(n)), dt, addr(), a, b, 0.5,
                                         addr(), None)
        elif which == 1:
            st = lib.zero_step(p, g, B._ptr_array(ptrs(n)), dt, addr(), addr(), addr(),
                               B.ctypes.byref(hp), addr(), addr(), dt, None)
        elif which == 2:
            st = lib.zero_adam_shard(p, g, addr(), addr(), addr(), addr(), B.ctypes.byref(hp),
                                     addr(), a, b, addr(), dt, None)
        elif which == 3:
            st = lib.zero_all_gather(p, g, addr(), addr(), dt, None)
        elif which == 4:
            f = lib.zero_gather_layer if rng.integers(0, 2) else lib.zero_broadcast_layer
            st = f(p, g, B._ptr_array(ptrs(n)), dt, addr(), None)
        elif which == 5:
            k = int(rng.integers(0, 4))
            grp = (B.c_i32 * max(1, k))(*[int(x) for x in rng.integers(-1, 3, k)])
            st = lib.zero_gather_groups(p, grp, k, B._ptr_array(ptrs(n)), dt,
                                        B._ptr_array(ptrs(k)), None)
        elif which == 6:
            st = lib.zero_grad_norm(addr(), a, float(rng.choice([1.0, 0.0, -1.0])), addr(),
                                    addr(), None)
        else:
            st = lib.zero_copy(addr(), addr(), a, None)
        assert st in codes, (which, st)
        seen.add(st)
    # the random arguments reach every kind of check and, past them, the launch
    assert {Z.ZERO_EINVAL, Z.ZERO_EALIGN, Z.ZERO_ERANGE, Z.ZERO_EDTYPE} <= seen, seen


def test_binding_refuses_pointer_lists_of_the_wrong_length():
    """The C side reads exactly N per-rank addresses (and one output per
    group, two layer buffers): a list of another length never reaches it."""
    p = Z.zero_plan([1000], 4, 16)
    A = 1 << 40
    with pytest.raises(ValueError):
        Z.zero_reduce_scatter(p, 0, [A, A, A], Z.ZERO_BF16, A, 0, 16, 0.25, None, 0)
    with pytest.raises(ValueError):
        Z.zero_gather_layer(p, 0, [A] * 5, Z.ZERO_BF16, A, 0)
    with pytest.raises(ValueError):
        Z.zero_broadcast_layer(p, 0, [A] * 3, Z.ZERO_BF16, A, 0)
    with pytest.raises(ValueError):
        Z.zero_gather_groups(p, [0, 0], [A] * 4, Z.ZERO_BF16, [A], 0)
    with pytest.raises(ValueError):
        Z.zero_stage3_gather_pass(p, [0], [A] * 4, [A], 16, A, 1, 1, 2)


def test_binding_refuses_tensors_too_small_or_strided():
    """A tensor argument smaller than what the call touches, or not
    contiguous, is refused before the call (a kernel would run past it)."""
    import torch
    p = Z.zero_plan([1000, 24], 4, 16)           # psi_pad 1024
    ok = torch.zeros(1024)
    small = torch.zeros(1000)
    strided = torch.zeros(2048)[::2]
    g = [torch.zeros(1024, dtype=torch.bfloat16) for _ in range(4)]
    hp = Z.adam_hp(1, 0.25)
    with pytest.raises(ValueError, match="master: holds 4000 bytes"):
        Z.zero_step(p, 0, g, Z.ZERO_BF16, small, ok, ok, hp, None, None, Z.ZERO_BF16, 0)
    with pytest.raises(ValueError, match="m: not contiguous"):
        Z.zero_step(p, 0, g, Z.ZERO_BF16, ok, strided, ok, hp, None, None, Z.ZERO_BF16, 0)
    with pytest.raises(ValueError, match=r"grads\[2\]: holds"):
        Z.zero_step(p, 0, g[:2] + [torch.zeros(10, dtype=torch.bfloat16), g[3]], Z.ZERO_BF16,
                    ok, ok, ok, hp, None, None, Z.ZERO_BF16, 0)
    with pytest.raises(ValueError, match="full_out: holds"):
        Z.zero_all_gather(p, 0, ok, torch.zeros(100, dtype=torch.bfloat16), Z.ZERO_BF16, 0)
    with pytest.raises(ValueError, match="reduced: holds"):
        Z.zero_reduce_scatter(p, 0, g, Z.ZERO_BF16, small, 0, 1024, 0.25, None, 0)
    # the prepared step checks the same buffers once, when prepared
    with pytest.raises(ValueError, match="master: holds 4000 bytes"):
        Z.prepare_zero_step(p, 0, g, Z.ZERO_BF16, small, ok, ok, None, None, Z.ZERO_BF16, 0)
    with pytest.raises(ValueError, match=r"grads: 3 given"):
        Z.prepare_zero_step(p, 0, g[:3], Z.ZERO_BF16, ok, ok, ok, None, None, Z.ZERO_BF16, 0)


def test_plan_argument_errors():
    for args in [([4], 0, 1), ([4], 65, 1), ([4], 2, 0), ([-1], 2, 1)]:
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_plan(*args)
        assert e.value.status == Z.ZERO_EINVAL
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_plan([4, 4], 2, 1, [0, 2])
    assert e.value.status == Z.ZERO_EINVAL
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_plan([2 ** 62, 2 ** 62], 2, 1)
    assert e.value.status == Z.ZERO_EINVAL
    with pytest.raises(Z.ZeroError) as e:          # a group at the kernels' 2^40 index limit
        Z.zero_plan([1 << 40], 4, 1)
    assert e.value.status == Z.ZERO_EINVAL
    Z.zero_plan([(1 << 40) - 64], 4, 16)          # just below it is fine
    p = Z.zero_plan([10], 2, 1)
    for f, a in [(Z.zero_plan_group, (1,)), (Z.zero_plan_shard, (0, 2)),
                 (Z.zero_plan_tensor, (1,)), (Z.zero_plan_memory, (4,))]:
        with pytest.raises(Z.ZeroError) as e:
            f(p, *a)
        assert e.value.status == Z.ZERO_ERANGE


def test_device_call_argument_errors_return_before_any_launch():
    """Rejected calls never reach the GPU: fake (never dereferenced)
    addresses suffice, and the status names the first bad argument."""
    p = Z.zero_plan([100], 4, 1)
    A = 0x10000                      # 16-byte aligned fake address
    good = [A] * 4
    hp = Z.adam_hp(1, 0.25)
    E = Z.ZeroError

    def status(fn, *a):
        with pytest.raises(E) as e:
            fn(*a, stream=0)
        return e.value.status

    assert status(Z.zero_reduce_scatter, p, 1, good, Z.ZERO_BF16, A, 0, 4, 1.0) == Z.ZERO_ERANGE
    assert status(Z.zero_reduce_scatter, p, 0, good, 7, A, 0, 4, 1.0) == Z.ZERO_EDTYPE
    assert status(Z.zero_reduce_scatter, p, 0, good, Z.ZERO_BF16, A, 5, 4, 1.0) == Z.ZERO_ERANGE
    assert status(Z.zero_reduce_scatter, p, 0, good, Z.ZERO_BF16, A, 0, 101, 1.0) == Z.ZERO_ERANGE
    assert status(Z.zero_reduce_scatter, p, 0, [A, A, A, A + 8], Z.ZERO_BF16, A, 0, 4,
                  1.0) == Z.ZERO_EALIGN
    assert status(Z.zero_reduce_scatter, p, 0, [A, A, 0, A], Z.ZERO_BF16, A, 0, 4,
                  1.0) == Z.ZERO_EINVAL
    assert status(Z.zero_reduce_scatter, p, 0, good, Z.ZERO_BF16, A + 4, 0, 4, 1.0) == Z.ZERO_EALIGN
    assert status(Z.zero_step, p, 0, good, Z.ZERO_BF16, A, A, A + 2, hp, None, A) == Z.ZERO_EALIGN
    assert status(Z.zero_step, p, 0, good, Z.ZERO_BF16, A, A, A, Z.adam_hp(0, 0.25), None,
                  A) == Z.ZERO_EINVAL
    assert status(Z.zero_step, p, 0, good, Z.ZERO_BF16, A, A, A,
                  Z.adam_hp(1, 0.25, beta1=1.0), None, A) == Z.ZERO_EINVAL
    assert status(Z.zero_step, p, 0, good, Z.ZERO_BF16, A, A, A,
                  Z.adam_hp(1, 0.25, lr=float("nan")), None, A) == Z.ZERO_EINVAL
    assert status(Z.zero_step, p, 0, good, Z.ZERO_BF16, A, A, A, hp, None, A, 9) == Z.ZERO_EDTYPE
    assert status(Z.zero_step_group, p, 0, good, Z.ZERO_BF16, A, A, A, hp, None,
                  [A, A, A, 0]) == Z.ZERO_EINVAL
    assert status(Z.zero_adam_shard, p, 0, A, A, A, A, hp, None, 0, 200, None) == Z.ZERO_ERANGE
    assert status(Z.zero_all_gather, p, 3, A, A) == Z.ZERO_ERANGE
    assert status(Z.zero_gather_layer, p, 0, good, Z.ZERO_BF16, A + 1) == Z.ZERO_EALIGN
    assert status(Z.zero_broadcast_layer, p, 0, good, Z.ZERO_BF16, A + 1) == Z.ZERO_EALIGN
    assert status(Z.zero_broadcast_layer, p, 1, good, Z.ZERO_BF16, A) == Z.ZERO_ERANGE
    assert status(Z.zero_broadcast_layer, p, 0, good, 3, A) == Z.ZERO_EDTYPE
    assert status(Z.zero_broadcast_layer, p, 0, [A, A, 0, A], Z.ZERO_BF16, A) == Z.ZERO_EINVAL
    assert status(Z.zero_step_acc, p, 0, good, Z.ZERO_BF16, A, A, A + 16, A + 32, hp, None,
                  A + 48) == Z.ZERO_EINVAL                  # accumulated is also the master
    assert status(Z.zero_step_acc, p, 0, good, Z.ZERO_BF16, A + 48, A, A + 16, A + 32, hp, None,
                  A + 48) == Z.ZERO_EINVAL                  # ... or the output
    assert status(Z.zero_step_group_acc, p, 0, good, Z.ZERO_BF16, A + 32, A, A + 16, A + 32, hp,
                  None, good) == Z.ZERO_EINVAL              # accumulated is also v
    assert status(Z.zero_step_group_acc, p, 0, good, Z.ZERO_BF16, A + 8, A, A + 16, A + 32, hp,
                  None, good) == Z.ZERO_EALIGN
    assert status(Z.zero_step_group_acc, p, 1, good, Z.ZERO_BF16, A + 48, A, A + 16, A + 32, hp,
                  None, good) == Z.ZERO_ERANGE
    assert status(Z.zero_gather_groups, p, [0], good, Z.ZERO_BF16, [A + 2]) == Z.ZERO_EALIGN
    assert status(Z.zero_gather_groups, p, [0, 1], good, Z.ZERO_BF16, [A, A]) == Z.ZERO_ERANGE
    assert status(Z.zero_gather_groups, p, [], good, Z.ZERO_BF16, []) == Z.ZERO_EINVAL
    assert status(Z.zero_gather_groups, p, [0] * 65, good, Z.ZERO_BF16, [A] * 65) == \
        Z.ZERO_EINVAL
    assert status(Z.zero_gather_groups, p, [0], good, 5, [A]) == Z.ZERO_EDTYPE
    assert status(Z.zero_gather_groups, p, [0], good, Z.ZERO_BF16, [0]) == Z.ZERO_EINVAL
    assert status(Z.zero_grad_norm, A, 4, 0.0, None, None) == Z.ZERO_EINVAL
    assert status(Z.zero_layer_checksum, A, 10, 1, A + 4) == Z.ZERO_EALIGN
    assert status(Z.zero_layer_checksum, A, 10, 0, A) == Z.ZERO_EINVAL
    assert status(Z.zero_layer_checksum, A, 10, Z.ZERO_MAX_CONSUMER_ROUNDS + 1, A) == \
        Z.ZERO_EINVAL
    assert status(Z.zero_copy, A, A, 15) == Z.ZERO_EINVAL
    assert status(Z.zero_wait_flag, A, 1, Z.ZERO_MAX_POLLS + 1, A) == Z.ZERO_EINVAL
    assert status(Z.zero_wait_flag, A + 2, 1, 10, A) == Z.ZERO_EALIGN
    assert status(Z.zero_wait_flag, 0, 1, 10, A) == Z.ZERO_EINVAL
    assert status(Z.zero_adam_state_init, hp, A + 4) == Z.ZERO_EALIGN
    assert status(Z.zero_adam_state_init, hp, 0) == Z.ZERO_EINVAL
    assert status(Z.zero_adam_state_init, Z.adam_hp(0, 0.25), A) == Z.ZERO_EINVAL
    assert status(Z.zero_adam_state_advance, Z.adam_hp(1, 0.25, beta2=1.5), A) == Z.ZERO_EINVAL
    assert status(Z.zero_step, p, 0, good, Z.ZERO_BF16, A, A, A,
                  Z.adam_hp(1, 0.25, d_state=A + 2), None, A) == Z.ZERO_EALIGN


def test_rs_partials_requires_known_dtype():
    p = Z.zero_plan([100], 4, 1)
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_rs_partials(p, 5, 100)
    assert e.value.status == Z.ZERO_EDTYPE


def test_host_fault_injection_reports_enomem():
    code = ("import os, zero_sharded_optimizer_device_gb300 as Z\n"
            "try:\n    Z.zero_plan([4], 2, 1)\nexcept Z.ZeroError as e:\n"
            "    print(e.status)\n")
    env = dict(os.environ, ZERO_FAULT_INJECT="plan_alloc",
               PYTHONPATH=os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True)
    assert out.stdout.strip() == str(Z.ZERO_ENOMEM), out.stderr


def _gloo_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    d = bench.Dist()
    d.barrier()
    got = d.max(float(10 + rank))
    d.close()
    q.put((rank, got))


def test_bench_max_over_ranks_with_gloo():
    """The replicas path: every rank's timing reduced with MAX over a 2-rank
    gloo group (the same code torchrun drives on GPUs)."""
    import multiprocessing as mp
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_gloo_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert res == {0: 11.0, 1: 11.0}


def test_set_occupancy_round_trip_and_limits():
    prev = Z.zero_set_occupancy(Z.ZERO_OCC_ADAM, 5)
    assert prev >= 1
    assert Z.zero_set_occupancy(Z.ZERO_OCC_ADAM, 0) == 5
    assert Z.zero_set_occupancy(Z.ZERO_OCC_ADAM, 0) == prev     # default restored
    assert Z.zero_set_occupancy(Z.ZERO_OCC_PREFETCH, 0) >= 1    # the last kind exists
    for kind, n in [(-1, 1), (Z.ZERO_OCC_PREFETCH + 1, 1), (Z.ZERO_OCC_RS, 33), (0, -1)]:
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_set_occupancy(kind, n)
        assert e.value.status == Z.ZERO_EINVAL


def test_header_compiles_as_c99_and_library_links(tmp_path):
    """A plain C99 program includes include/zero.h, links libzero.so and
    plans the tiny workload on the CPU."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    lib_dir = os.path.join(root, "zero_sharded_optimizer_device_gb300")
    exe = str(tmp_path / "c_abi_check")
    cc = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                         "-I", os.path.join(root, "include"),
                         os.path.join(root, "tests", "c_abi_check.c"),
                         "-L", lib_dir, "-lzero", f"-Wl,-rpath,{lib_dir}", "-o", exe],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    lines = out.stdout.splitlines()
    assert lines[0] == "psi 10000 psi_pad 10048 shard 2512"
    assert lines[2] == "rank 1: (0 2512 2512 1584) (1 0 4096 928)"
    assert lines[5] == "stage2 17584 55264 volume 7536 7536"
    assert lines[6] == f"bad {Z.ZERO_EINVAL} invalid argument"


def test_bias_corrections_match_the_oracle_for_any_step_order():
    """The library's host bias corrections (which continue the beta^t product
    from the thread's previous call) equal the oracle's full product for
    growing steps, repeats, jumps back and forth, other betas in between, and
    from several host threads at once."""
    import threading
    import numpy as np
    from oracle import zero_oracle as O
    rng = np.random.default_rng(5)
    seq = list(range(1, 1501)) + [1500, 3, 3, 7000, 6999, 41_000, 42_500, 2, 1]
    betas = [(0.9, 0.999)] * len(seq)
    for i in rng.integers(0, len(seq), 40):                  # other betas in between
        betas[i] = (0.8, 0.99)
    for step, (b1, b2) in zip(seq, betas):
        got = Z.zero_adam_bias_corrections(Z.adam_hp(step, 0.25, beta1=b1, beta2=b2))
        want = O.bias_corrections(b1, b2, step)
        assert np.float32(got[0]) == want[0] and np.float32(got[1]) == want[1], (step, b1, b2)
    errors = []

    def worker(b1, b2, steps):
        for s in steps:
            got = Z.zero_adam_bias_corrections(Z.adam_hp(s, 0.25, beta1=b1, beta2=b2))
            want = O.bias_corrections(b1, b2, s)
            if not (np.float32(got[0]) == want[0] and np.float32(got[1]) == want[1]):
                errors.append((b1, b2, s))
    ts = [threading.Thread(target=worker, args=(b1, b2, range(1, 400)))
          for b1, b2 in [(0.9, 0.999), (0.95, 0.98), (0.5, 0.9)]]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors[:5]
    for bad in (Z.adam_hp(0, 0.25), Z.adam_hp(1, 0.25, beta2=1.0)):
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_adam_bias_corrections(bad)
        assert e.value.status == Z.ZERO_EINVAL


def test_binding_refuses_tensors_of_another_device(monkeypatch):
    """The library launches on the current device, so a tensor that lives on
    another GPU is refused before any call (it would be an illegal address
    there).  Host-only: the current device and the tensor are stand-ins."""
    import torch

    class OtherGpuTensor:
        is_cuda = True
        device = torch.device("cuda", 1)

        def data_ptr(self):
            return 1 << 40

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    with pytest.raises(ValueError, match="cuda:1 passed while cuda:0"):
        Z.binding._ptr(OtherGpuTensor())
    OtherGpuTensor.device = torch.device("cuda", 0)
    assert Z.binding._ptr(OtherGpuTensor()) == 1 << 40
