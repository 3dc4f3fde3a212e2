"""Benchmark of the ZeRO sharded-optimizer hot path on one GB300 per rank.

Default workload: the Llama-7B stage-3 step -- 291 tensors, 6,738,415,616
parameters in 34 layer groups (embedding, 32 transformer blocks, final norm +
head), N = 16 emulated data-parallel ranks, bf16 gradients, fp32 master / m /
v; one step = per layer group, in reverse order, the fused ring-order
reduce-scatter + scale + Adam writing each owner's bf16 parameter shard
(zero_step_group), 58 bytes per parameter.  The line also carries the
per-layer gathers of the updated shards (alone, prefetched beside a consumer,
and in the broadcast form) and the step end to end from host memory.  Prints
one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload llama-7b-stage3|gpt2-small|gpt2-medium|llama-1.4b|tiny]

The other workloads: GPT-2-small (N = 8) and GPT-2-medium (N = 64, align 1)
through the fused zero_step; Llama-1.4B (N = 8) through the bucketed
reduce-scatter, global-norm clip and chunked Adam; tiny (N = 4).

Under torchrun every rank runs an independent replica on its own GPU (the
method shards nothing across GPUs here); value = all ranks' parameters
updated / max-over-ranks time.  --impl reference times the CPU oracle on a
bounded window of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused ZeRO step Gparams/s and achieved HBM GB/s (% of peak), 1 GB300"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0       # GB300 HBM3e, nominal
DEFAULT_WORKLOAD = "llama-7b-stage3"


# ------------------------------------------------------------ distributed --
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = torch.device("cuda", self.local_rank) if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def local_ranks() -> int:
    """Ranks on this host (each pins its own end-to-end buffers)."""
    return max(1, int(os.environ.get("LOCAL_WORLD_SIZE", "1")))


# ----------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self) -> dict:
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = [r.split(",") for r in self.out.strip().splitlines() if r.count(",") >= 8]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        top = max(sm)
        loaded = [s for s in sm if s >= 0.5 * top] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- helpers --
def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# Where each measured kernel lives and which occupancy cap launches it.
KERNEL_SOURCES = {"fused_kernel": ("zero_rs.cu", "ZERO_OCC_FUSED"),
                  "rs_kernel": ("zero_rs.cu", "ZERO_OCC_RS"),
                  "adam_kernel": ("zero_kernels.cu", "ZERO_OCC_ADAM"),
                  "gather_bulk_kernel": ("zero_kernels.cu", "ZERO_OCC_GATHER")}


def kernel_source_hash(kernel: str = "fused_kernel") -> str:
    """Hash of what decides a kernel's DRAM traffic: the device helpers, the
    kernel's own source text and its occupancy default (host code around it
    and the other kernels' defaults do not count)."""
    fname, occ = KERNEL_SOURCES[kernel]
    return _source_hash(_read_csrc("zero_device.cuh"), _read_csrc(fname), kernel,
                        _read_csrc("zero_rs.cu"), occ)


def _read_csrc(name: str) -> str:
    with open(os.path.join(ROOT, "zero_sharded_optimizer_device_gb300", "csrc", name)) as f:
        return f.read()


def _source_hash(device_h: str, src: str, kernel: str, rs_cu: str = None,
                 occ_kind: str = "ZERO_OCC_FUSED") -> str:
    h = hashlib.sha256()
    h.update(device_h.encode())
    start = src.index(f"    {kernel}(")
    start = src.rindex("template", 0, start)
    end = src.index("// ------", start)
    h.update(src[start:end].encode())
    rs_cu = src if rs_cu is None else rs_cu
    occ = rs_cu.index("constexpr int kOccDefault")
    block = rs_cu[occ:rs_cu.index("};", occ)]
    h.update(next(line for line in block.splitlines() if occ_kind in line).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str, key: str = None):
    """DRAM bytes per launch from a committed ncu summary, only while the
    kernel sources are unchanged since the capture.  key: the record's name
    under the workload (default: the kernel's)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(workload, {}).get(key or kernel)
    if not entry or entry.get("source_hash") != kernel_source_hash(kernel):
        return None
    return entry.get("bytes_per_launch")


def gpu_numa_node(dev_index: int):
    """The host memory node nearest this GPU: its PCI device's NUMA node as
    the kernel reports it (None when unknown or negative)."""
    import torch
    try:
        pr = torch.cuda.get_device_properties(dev_index)
        path = (f"/sys/bus/pci/devices/{pr.pci_domain_id:04x}:{pr.pci_bus_id:02x}:"
                f"{pr.pci_device_id:02x}.0/numa_node")
        node = int(open(path).read().strip())
    except (OSError, ValueError, AttributeError, RuntimeError, AssertionError):
        return None                 # no device, or the kernel reports no node
    return node if node >= 0 else None


def _set_mempolicy(node):
    """Bind this thread's future page allocations to one memory node (None:
    back to the default policy).  Returns True on success."""
    import ctypes
    import platform
    nr = {"aarch64": 237, "x86_64": 238}.get(platform.machine())
    if nr is None:
        return False
    libc = ctypes.CDLL(None, use_errno=True)
    if node is None:
        return libc.syscall(nr, 0, None, 0) == 0                      # MPOL_DEFAULT
    mask = (ctypes.c_ulong * 16)()
    mask[node // 64] = 1 << (node % 64)
    return libc.syscall(nr, 2, mask, 16 * 64) == 0                    # MPOL_BIND


def pinned_host_buffer(nbytes: int, near_gpu: bool = False):
    """One page-locked host byte buffer of exactly nbytes from cudaHostAlloc
    (torch's pinned allocator would round each tensor up to a power of two).
    With near_gpu the pages are taken from the memory node nearest the
    current GPU when the system reports one.  Returns (uint8 tensor over it,
    function that frees it, description of the placement)."""
    import ctypes
    import torch
    rt = ctypes.CDLL("libcudart.so.13")
    rt.cudaHostAlloc.restype = ctypes.c_int
    rt.cudaHostAlloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t, ctypes.c_uint]
    rt.cudaFreeHost.restype = ctypes.c_int
    rt.cudaFreeHost.argtypes = [ctypes.c_void_p]
    node = gpu_numa_node(torch.cuda.current_device()) if near_gpu else None
    bound = node is not None and _set_mempolicy(node)
    ptr = ctypes.c_void_p()
    try:
        rc = rt.cudaHostAlloc(ctypes.byref(ptr), nbytes, 0)
    finally:
        if bound:
            _set_mempolicy(None)
    if rc != 0:
        raise RuntimeError(f"cudaHostAlloc of {nbytes} bytes failed ({rc})")
    t = torch.frombuffer((ctypes.c_uint8 * nbytes).from_address(ptr.value), dtype=torch.uint8)
    where = (f"pages bound to memory node {node}, the GPU's PCI NUMA node" if bound else
             "default placement (the GPU reports no NUMA node)" if near_gpu and node is None else
             "default placement")
    return t, (lambda: rt.cudaFreeHost(ptr)), where


def host_mapped(t) -> bool:
    """True when a pinned host tensor is mapped into the device address space
    at the same address (so kernels may read and write it directly)."""
    import ctypes
    try:
        rt = ctypes.CDLL("libcudart.so.13")
    except OSError:
        return False
    f = rt.cudaHostGetDevicePointer
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p, ctypes.c_uint]
    dp = ctypes.c_void_p()
    return f(ctypes.byref(dp), ctypes.c_void_p(t.data_ptr()), 0) == 0 and dp.value == t.data_ptr()


def algorithmic_bytes(n_ranks: int, psi: int, grad_bytes: int) -> int:
    """Bytes one fused step must move: N gradient reads, 12 B of fp32
    master/m/v read and 12 B written, 2 B of bf16 parameters written."""
    return psi * (n_ranks * grad_bytes + 24 + 2)


# --------------------------------------------------------- our GPU arm ----
def bench_fused(w, steps: int, warmup: int, dist: Dist, kernel_only: bool = False,
                graph: bool = False, graph_steps: int = 1) -> dict:
    import torch
    import synth
    import zero_sharded_optimizer_device_gb300 as Z

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    plan = Z.zero_plan(w.numels, w.n_ranks, w.align)
    info = Z.zero_plan_info(plan)
    P, N = info["psi_pad"], w.n_ranks
    gdt = torch.bfloat16 if w.grad_dtype == "bf16" else torch.float32
    zg = Z.ZERO_BF16 if w.grad_dtype == "bf16" else Z.ZERO_F32
    gbytes = 2 if w.grad_dtype == "bf16" else 4
    grads = [torch.empty(P, dtype=gdt, device=dev) for _ in range(N)]
    for r in range(N):
        synth.fill_tensor(grads[r], w.seed, synth.GRAD, 1, r, 0, w.grad_sigma, w.psi,
                          w.heavy_tail)
    master = torch.empty(P, dtype=torch.float32, device=dev)
    synth.fill_tensor(master, w.seed, synth.MASTER, 0, 0, 0, w.master_sigma, w.psi)
    m = torch.zeros_like(master)
    v = torch.zeros_like(master)
    out = torch.empty(P, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    t = [0]
    prepared = Z.prepare_zero_step(plan, 0, grads, zg, master, m, v, None, out, Z.ZERO_BF16,
                                   stream)

    def step():
        t[0] += 1
        prepared(Z.adam_hp(t[0], 1.0 / N))

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()

    if graph:
        # graph_steps steps captured once -- each: advance the device-resident
        # Adam step state, then the fused kernel -- and replayed
        state = torch.zeros(4, dtype=torch.float64, device=dev)
        hp = Z.adam_hp(t[0] + 1, 1.0 / N, d_state=state)
        Z.zero_adam_state_init(hp, state, stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        per = max(1, min(graph_steps, steps))
        with torch.cuda.stream(side), torch.cuda.graph(g, stream=side):
            for _ in range(per):
                Z.zero_adam_state_advance(hp, state, side)
                Z.zero_step(plan, 0, grads, zg, master, m, v, hp, None, out, Z.ZERO_BF16, side)
        stream.wait_stream(side)
        for _ in range(3):
            g.replay()
        reps = max(1, steps // per)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(dev.index) as clocks:
            dist.barrier()
            torch.cuda.synchronize()
            t0.record(stream)
            for _ in range(reps):
                g.replay()
            t1.record(stream)
            torch.cuda.synchronize()
            dist.barrier()
        ms = t0.elapsed_time(t1) / (reps * per)
        return dict(local_ms=ms, launch_ms=ms, e2e_ms=None, psi=w.psi, psi_pad=P, n_ranks=N,
                    gbytes=gbytes, copy_gbs=None, clocks=clocks.summary(), h2d=0, d2h=0,
                    e2e_steps=0, e2e_transfer="not measured with --graph", graph=per)

    if kernel_only:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        return dict(local_ms=ms, launch_ms=ms, e2e_ms=ms, psi=w.psi, psi_pad=P, n_ranks=N,
                    gbytes=gbytes, copy_gbs=None, clocks={}, h2d=0, d2h=0, e2e_steps=0)

    # copy-kernel peak of this GPU (context for the roofline denominator)
    cbytes = 2 << 30
    a = torch.empty(cbytes // 4, dtype=torch.float32, device=dev)
    b = torch.empty_like(a)
    for _ in range(3):
        Z.zero_copy(b, a, cbytes, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(10):
        Z.zero_copy(b, a, cbytes, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    copy_gbs = 2 * cbytes * 10 / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del a, b

    # timed region: K steps, per-launch events on the launching stream
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clocks:
        dist.barrier()
        torch.cuda.synchronize()
        t0.record(stream)
        for i in range(steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
    local_ms = t0.elapsed_time(t1) / steps
    launch_ms = statistics.fmean(s.elapsed_time(e) for s, e in zip(starts, ends))

    # end to end through the public API: inputs from pinned host memory,
    # updated bf16 parameters back to pinned host memory, every step.  Two
    # ways: explicit copies around the step, or -- when the pinned buffers
    # are mapped into the device address space -- zero_step on the host
    # buffers themselves, so the kernel moves the data over the host link
    # while it streams the state (zero-copy).  Both are timed; the faster is
    # reported with its mode.
    host_bytes = N * P * gbytes + P * 2
    ram = os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")
    if host_bytes * local_ranks() > 0.4 * ram:  # too large to pin on this host: no e2e leg
        return dict(local_ms=local_ms, launch_ms=launch_ms, e2e_ms=None, psi=w.psi, psi_pad=P,
                    n_ranks=N, gbytes=gbytes, copy_gbs=copy_gbs, clocks=clocks.summary(),
                    h2d=N * P * gbytes, d2h=P * 2, e2e_steps=0,
                    e2e_transfer=f"skipped: {host_bytes / 1e9:.0f} GB of pinned host memory "
                                 f"x {local_ranks()} local ranks exceeds 40% of the host's "
                                 f"{ram / 1e9:.0f} GB")
    try:
        pinned, free_pinned, numa = pinned_host_buffer(host_bytes, near_gpu=True)
    except RuntimeError as err:       # the host could not pin that much: no e2e leg
        return dict(local_ms=local_ms, launch_ms=launch_ms, e2e_ms=None, psi=w.psi, psi_pad=P,
                    n_ranks=N, gbytes=gbytes, copy_gbs=copy_gbs, clocks=clocks.summary(),
                    h2d=N * P * gbytes, d2h=P * 2, e2e_steps=0, e2e_transfer=f"skipped: {err}")
    h_grads = [pinned[r * P * gbytes:(r + 1) * P * gbytes].view(gdt) for r in range(N)]
    for r in range(N):
        h_grads[r].copy_(grads[r])
    h_out = pinned[N * P * gbytes:].view(torch.bfloat16)
    e2e_steps = max(5, min(50, steps // 20))
    mapped = all(host_mapped(x) for x in h_grads + [h_out])

    def e2e_step(zero_copy):
        if zero_copy:
            t[0] += 1
            Z.zero_step(plan, 0, h_grads, zg, master, m, v, Z.adam_hp(t[0], 1.0 / N), None,
                        h_out, Z.ZERO_BF16, stream)
            return
        for r in range(N):
            grads[r].copy_(h_grads[r], non_blocking=True)
        step()
        h_out.copy_(out, non_blocking=True)

    def e2e_time(zero_copy):
        for _ in range(2):
            e2e_step(zero_copy)
        torch.cuda.synchronize()
        dist.barrier()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(e2e_steps):
            e2e_step(zero_copy)
        s1.record(stream)
        torch.cuda.synchronize()
        return s0.elapsed_time(s1) / e2e_steps

    # both ways a user can hand host buffers to the library; report the faster
    modes = {False: e2e_time(False)}
    if mapped:
        modes[True] = e2e_time(True)
    zero_copy = min(modes, key=modes.get)
    e2e_ms = modes[zero_copy]
    del h_grads, h_out, pinned
    free_pinned()

    return dict(local_ms=local_ms, launch_ms=launch_ms, e2e_ms=e2e_ms, psi=w.psi, psi_pad=P,
                n_ranks=N, gbytes=gbytes, copy_gbs=copy_gbs, clocks=clocks.summary(),
                h2d=N * P * gbytes, d2h=P * 2, e2e_steps=e2e_steps, numa=numa,
                e2e_transfer="zero-copy kernel access to mapped pinned host memory" if zero_copy
                else "cudaMemcpyAsync from/to pinned host memory")


# ----------------------------------------- bucketed pipeline with clipping --
def _timed_seq(stream, f) -> float:
    """Device milliseconds of everything f enqueues on `stream` (one event
    pair around the whole sequence, so back-to-back launches stay back to
    back)."""
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    f()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def bench_bucketed(w, steps: int, warmup: int, dist: Dist, kernel_only: bool = False) -> dict:
    """Reduce-scatter in fixed-size buckets with fp64 norm partials, global
    norm and clip coefficient on the device, Adam in chunks writing the bf16
    gathered parameters (the Llama-1.4B workload)."""
    import torch
    import synth
    import zero_sharded_optimizer_device_gb300 as Z

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    plan = Z.zero_plan(w.numels, w.n_ranks, w.align)
    P, N = Z.zero_plan_info(plan)["psi_pad"], w.n_ranks
    bucket, chunk = w.extra["bucket"], w.extra["chunk"]
    gdt = torch.bfloat16 if w.grad_dtype == "bf16" else torch.float32
    zg = Z.ZERO_BF16 if w.grad_dtype == "bf16" else Z.ZERO_F32
    grads = [torch.empty(P, dtype=gdt, device=dev) for _ in range(N)]
    for r in range(N):
        synth.fill_tensor(grads[r], w.seed, synth.GRAD, 1, r, 0, w.grad_sigma, w.psi, w.heavy_tail)
    master = torch.empty(P, dtype=torch.float32, device=dev)
    synth.fill_tensor(master, w.seed, synth.MASTER, 0, 0, 0, w.master_sigma, w.psi)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    reduced = torch.empty(P, dtype=torch.float32, device=dev)
    out = torch.empty(P, dtype=torch.bfloat16, device=dev)
    windows = [(a, min(P, a + bucket)) for a in range(0, P, bucket)]
    chunks = [(a, min(P, a + chunk)) for a in range(0, P, chunk)]
    npart = [Z.zero_rs_partials(plan, zg, b - a) for a, b in windows]
    offs = [sum(npart[:i]) for i in range(len(npart))]
    partials = torch.zeros(sum(npart), dtype=torch.float64, device=dev)
    norm = torch.zeros(1, dtype=torch.float32, device=dev)
    coef = torch.zeros(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    t = [0]

    def calls(grads=grads, out=out):
        t[0] += 1
        hp = Z.adam_hp(t[0], 1.0 / N)
        cs = []
        for (a, b), o, k in zip(windows, offs, npart):
            cs.append(lambda a=a, b=b, o=o, k=k: Z.zero_reduce_scatter(
                plan, 0, grads, zg, reduced, a, b, 1.0 / N, partials[o:o + k], stream))
        cs.append(lambda: Z.zero_grad_norm(partials, partials.numel(), w.extra["max_norm"], norm,
                                           coef, stream))
        for a, b in chunks:
            cs.append(lambda a=a, b=b: Z.zero_adam_shard(plan, 0, master, m, v, reduced, hp, coef,
                                                         a, b, out, Z.ZERO_BF16, stream))
        return cs

    for _ in range(warmup):
        for f in calls():
            f()
    torch.cuda.synchronize()
    nl = len(windows) + 1 + len(chunks)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nl + 1)] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clocks:
        dist.barrier()
        torch.cuda.synchronize()
        t0.record(stream)
        for i in range(steps):
            for j, f in enumerate(calls()):
                evs[i][j].record(stream)
                f()
            evs[i][nl].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
    ms = [[e[j].elapsed_time(e[j + 1]) for j in range(nl)] for e in evs]
    nw = len(windows)
    res = dict(local_ms=t0.elapsed_time(t1) / steps,
               rs_ms=statistics.fmean(sum(x[:nw]) for x in ms),
               norm_ms=statistics.fmean(x[nw] for x in ms),
               adam_ms=statistics.fmean(sum(x[nw + 1:]) for x in ms),
               P=P, N=N, n_launches=nl, clocks=clocks.summary(), norm=float(norm.item()),
               coef=float(coef.item()))

    # end to end: gradients read from, and gathered parameters written to,
    # page-locked host memory (zero-copy when mapped, else explicit copies)
    gb = 2 if w.grad_dtype == "bf16" else 4
    host_bytes = N * P * gb + P * 2
    res.update(h2d=N * P * gb, d2h=P * 2, e2e_ms=None, e2e_steps=0)
    if kernel_only:
        return res
    ram = os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")
    if host_bytes * local_ranks() > 0.4 * ram:
        res["e2e_transfer"] = (f"skipped: {host_bytes / 1e9:.0f} GB of pinned host memory "
                               f"x {local_ranks()} local ranks exceeds 40% of the host's "
                               f"{ram / 1e9:.0f} GB")
        return res
    try:
        pinned, free_pinned, numa = pinned_host_buffer(host_bytes, near_gpu=True)
    except RuntimeError as err:       # the host could not pin that much: no e2e leg
        res["e2e_transfer"] = f"skipped: {err}"
        return res
    h_grads = [pinned[r * P * gb:(r + 1) * P * gb].view(gdt) for r in range(N)]
    h_out = pinned[N * P * gb:].view(torch.bfloat16)
    for r in range(N):
        h_grads[r].copy_(grads[r])
    mapped = all(host_mapped(x) for x in h_grads + [h_out])

    def e2e_step():
        if mapped:
            for f in calls(h_grads, h_out):
                f()
            return
        for r in range(N):
            grads[r].copy_(h_grads[r], non_blocking=True)
        for f in calls():
            f()
        h_out.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e2e_steps = 3
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    s1.record(stream)
    torch.cuda.synchronize()
    res.update(e2e_ms=s0.elapsed_time(s1) / e2e_steps, e2e_steps=e2e_steps, numa=numa,
               e2e_transfer="zero-copy kernel access to mapped pinned host memory" if mapped
               else "cudaMemcpyAsync from/to pinned host memory")
    del h_grads, h_out, pinned
    free_pinned()
    return res


# ------------------------------------------- stage 3: step + per-layer gathers --
# Rounds of the arithmetic-bound stand-in consumer (zero_layer_checksum): at 64
# its 68 launches over the Llama-7B groups take about 3.5x the gathers.
ARITH_ROUNDS = 64
# Tokens of the tensor-core consumer's activation batch: at 2048 its 68 bf16
# GEMMs over the Llama-7B layers (1.8 PFLOP/s) take about 4x the gathers.
GEMM_TOKENS = 2048


def _hidden(gathers_ms: float, consumers_ms: float, schedule_ms: float) -> float:
    """Fraction of the shorter of the two kernel streams that the two-stream
    schedule hides behind the other: 1 = fully overlapped, 0 = serial."""
    return (gathers_ms + consumers_ms - schedule_ms) / min(gathers_ms, consumers_ms)


def bench_stage3(w, steps: int, warmup: int, dist: Dist, use_graph: bool = False,
                 kernel_only: bool = False) -> dict:
    """Stage 3 (the Llama-7B workload).  One step = per layer group, in
    reverse order (the order backward produces them), the fused
    reduce-scatter + scale + Adam writing each owner's bf16 shard
    (zero_step_group).  Every group's N gradient buffers are prefixes of one
    resident slot of N x (largest group) bf16 elements, filled once before
    the clock starts (the full model's gradients, 216 GB at N = 16, do not
    fit beside the state).  Then, untimed by the step: every group gathered
    into a contiguous layer buffer in forward and then reverse order, alone,
    in the two-stream prefetch schedule beside a consumer, and in the
    broadcast form; and the step end to end from host memory."""
    import torch
    import synth
    import zero_sharded_optimizer_device_gb300 as Z

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    N = w.n_ranks
    plan = Z.zero_plan(w.numels, N, w.align, w.groups)
    info = Z.zero_plan_info(plan)
    groups = [Z.zero_plan_group(plan, g) for g in range(info["n_groups"])]
    G = len(groups)
    P, ST = info["psi_pad"], info["shard_total"]
    big = max(range(G), key=lambda i: groups[i]["psi_pad"])
    gmax = groups[big]["psi_pad"]
    master = torch.empty(P, dtype=torch.float32, device=dev)
    for g in groups:
        synth.fill_tensor(master[g["flat_off"]:g["flat_off"] + g["psi_pad"]], w.seed, synth.MASTER,
                          0, 0, g["flat_off"], w.master_sigma, g["flat_off"] + g["psi"])
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    shards = [torch.zeros(ST, dtype=torch.bfloat16, device=dev) for _ in range(N)]
    gdt = torch.bfloat16 if w.grad_dtype == "bf16" else torch.float32
    zg = Z.ZERO_BF16 if w.grad_dtype == "bf16" else Z.ZERO_F32
    slot = [torch.empty(gmax, dtype=gdt, device=dev) for _ in range(N)]
    gb = groups[big]
    for r in range(N):
        synth.fill_tensor(slot[r], w.seed, synth.GRAD, 1, r, gb["flat_off"], w.grad_sigma,
                          gb["flat_off"] + gb["psi"])
    views = [[t[:g["psi_pad"]] for t in slot] for g in groups]
    sa = torch.cuda.current_stream(dev)
    rs_order = list(reversed(range(G)))
    t = [0]

    def step(grads=views, out=shards, stream=sa, events=None):
        t[0] += 1
        hp = Z.adam_hp(t[0], 1.0 / N)
        for j, gi in enumerate(rs_order):
            if events is not None:
                events[j].record(stream)
            Z.zero_step_group(plan, gi, grads[gi], zg, master, m, v, hp, None, out, stream)
        if events is not None:
            events[G].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()

    # timed region: K steps; events between launches give each launch's time
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(G + 1)] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clocks:
        dist.barrier()
        torch.cuda.synchronize()
        t0.record(sa)
        for i in range(steps):
            step(events=evs[i])
        t1.record(sa)
        torch.cuda.synchronize()
        dist.barrier()
    local_ms = t0.elapsed_time(t1) / steps
    per_launch = [[e[j].elapsed_time(e[j + 1]) for j in range(G)] for e in evs]
    launch_sum_ms = statistics.fmean(sum(x) for x in per_launch)
    block = [j for j, gi in enumerate(rs_order) if 0 < gi < G - 1]     # transformer blocks
    block_ms = statistics.fmean(x[j] for x in per_launch for j in block)
    res = dict(local_ms=local_ms, launch_sum_ms=launch_sum_ms, block_ms=block_ms,
               block_psi_pad=groups[1]["psi_pad"], P=P, N=N, groups=G, clocks=clocks.summary(),
               launches_per_step=G, gbytes=2 if w.grad_dtype == "bf16" else 4)
    if kernel_only:
        return res

    # copy-kernel peak of this GPU (context for the roofline denominator)
    cbytes = 2 << 30
    a = torch.empty(cbytes // 4, dtype=torch.float32, device=dev)
    b = torch.empty_like(a)
    for _ in range(3):
        Z.zero_copy(b, a, cbytes, sa)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(sa)
    for _ in range(10):
        Z.zero_copy(b, a, cbytes, sa)
    c1.record(sa)
    torch.cuda.synchronize()
    res["copy_gbs"] = 2 * cbytes * 10 / (c0.elapsed_time(c1) * 1e-3) / 1e9
    del a, b

    res.update(_stage3_gathers(Z, plan, groups, shards, dev, sa, steps, use_graph))
    res.update(_stage3_e2e(Z, plan, groups, N, ST, slot, zg, master, m, v, sa, t))
    return res


def _stage3_gathers(Z, plan, groups, shards, dev, sa, steps, use_graph) -> dict:
    """Forward + reverse per-group gathers of the updated bf16 shards: alone,
    in the two-stream prefetch schedule beside the stand-in consumer (one
    round: memory-bound; ARITH_ROUNDS: compute-bound), replayed from a CUDA
    graph, and in the broadcast form (zero_broadcast_layer)."""
    import torch
    G = len(groups)
    gmax = max(g["psi_pad"] for g in groups)
    bufs = [torch.empty(gmax, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    sums = torch.zeros(2 * G, dtype=torch.int64, device=dev)
    sb = torch.cuda.Stream(dev)
    order = list(range(G)) + list(reversed(range(G)))

    def timed(f):
        return _timed_seq(sa, f)

    def schedule(rounds):
        return lambda: Z.zero_stage3_gather_pass(plan, order, shards, bufs, gmax, sums, rounds,
                                                 sa, sb)

    def consumers(rounds):
        def f():
            for j, gi in enumerate(order):
                Z.zero_layer_checksum(bufs[j % 2], groups[gi]["psi_pad"], rounds, sums[j:j + 1],
                                      sa)
        return f

    def gathers():
        for j, gi in enumerate(order):
            Z.zero_gather_layer(plan, gi, shards, Z.ZERO_BF16, bufs[j % 2], sa)

    def broadcasts():
        for j, gi in enumerate(order):
            Z.zero_broadcast_layer(plan, gi, shards, Z.ZERO_BF16, bufs[j % 2], sa)

    runs = {"gathers_only_ms": gathers, "schedule_ms": schedule(1),
            "schedule_arith_ms": schedule(ARITH_ROUNDS), "consumers_only_ms": consumers(1),
            "consumers_arith_ms": consumers(ARITH_ROUNDS), "broadcast_ms": broadcasts}
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        gs, gsb = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        gs.wait_stream(sa)
        with torch.cuda.stream(gs):
            with torch.cuda.graph(graph, stream=gs):
                Z.zero_stage3_gather_pass(plan, order, shards, bufs, gmax, sums, 1, gs, gsb)
        sa.wait_stream(gs)
        torch.cuda.synchronize()
        runs["schedule_graph_ms"] = graph.replay
    # a tensor-core consumer: each gathered layer used as a [d, cols] bf16
    # weight matrix (cols = psi_pad/d rounded down to a multiple of 64, so its
    # rows stay 16-byte aligned and cuBLAS runs at full speed) against
    # GEMM_TOKENS activations (a cuBLAS GEMM through torch.matmul) -- the
    # matrix products prefetching is meant to hide -- in the same two-stream
    # schedule as zero_stage3_gather_pass
    d = 4096 if min(g["psi_pad"] for g in groups) >= 4096 * 256 else 256
    x = torch.randn(GEMM_TOKENS, d, device=dev).to(torch.bfloat16)
    y = torch.empty(GEMM_TOKENS * (gmax // d), dtype=torch.bfloat16, device=dev)
    cols = [groups[gi]["psi_pad"] // d // 64 * 64 for gi in order]    # 16-byte aligned rows
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def gemm(j):
        w = bufs[j % 2][:d * cols[j]].view(d, cols[j])
        torch.matmul(x, w, out=y[:GEMM_TOKENS * cols[j]].view(GEMM_TOKENS, cols[j]))

    def gemms():
        with torch.cuda.stream(sa):
            for j in range(len(order)):
                gemm(j)

    def gemm_schedule():
        start = torch.cuda.Event()
        start.record(sa)
        sb.wait_event(start)

        def issue(j):
            if j >= 2:
                sb.wait_event(done[j % 2])
            Z.zero_gather_layer(plan, order[j], shards, Z.ZERO_BF16, bufs[j % 2], sb)
            ready[j % 2].record(sb)

        issue(0)
        with torch.cuda.stream(sa):
            for j in range(len(order)):
                if j + 1 < len(order):
                    issue(j + 1)
                sa.wait_event(ready[j % 2])
                gemm(j)
                done[j % 2].record(sa)

    runs["gemm_consumers_only_ms"] = gemms
    runs["gemm_schedule_ms"] = gemm_schedule
    for f in runs.values():           # warm-up
        timed(f)
    out = {k: statistics.fmean(timed(f) for _ in range(max(1, min(steps, 10))))
           for k, f in runs.items()}
    out["gather_elems"] = 2 * sum(g["psi_pad"] for g in groups)
    out["gather_launches"] = len(order)
    out["gemm_flops"] = 2 * GEMM_TOKENS * d * sum(cols)
    out["gemm_shape"] = f"[{GEMM_TOKENS}, {d}] x [{d}, psi_pad/{d} to a multiple of 64] per layer"
    return out


def _stage3_e2e(Z, plan, groups, N, ST, slot, zg, master, m, v, sa, t) -> dict:
    """The step end to end through the public API from host memory: the N
    gradient buffers of each group in one page-locked host slot (N x largest
    group, reused for every group, as the device slot is) and the owners'
    bf16 shards written back to page-locked host buffers.  Mapped into the
    device address space, zero_step_group reads and writes them over the host
    link itself; otherwise explicit copies surround each group's step."""
    import torch
    G = len(groups)
    gmax, gb = slot[0].numel(), slot[0].element_size()
    h2d = N * sum(g["psi_pad"] for g in groups) * gb
    d2h = N * ST * 2
    host_bytes = N * gmax * gb + N * ST * 2
    ram = os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")
    base = dict(e2e_ms=None, h2d=h2d, d2h=d2h, e2e_steps=0)
    if host_bytes * local_ranks() > 0.4 * ram:
        return dict(base, e2e_transfer=f"skipped: {host_bytes / 1e9:.0f} GB of pinned host memory "
                                       f"x {local_ranks()} local ranks exceeds 40% of the "
                                       f"host's {ram / 1e9:.0f} GB")
    try:
        pinned, free_pinned, numa = pinned_host_buffer(host_bytes, near_gpu=True)
    except RuntimeError as err:       # the host could not pin that much: no e2e leg
        return dict(base, e2e_transfer=f"skipped: {err}")
    h_slot = [pinned[r * gmax * gb:(r + 1) * gmax * gb].view(slot[0].dtype) for r in range(N)]
    off = N * gmax * gb
    h_shards = [pinned[off + r * ST * 2:off + (r + 1) * ST * 2].view(torch.bfloat16)
                for r in range(N)]
    for r in range(N):
        h_slot[r].copy_(slot[r])
    mapped = all(host_mapped(x) for x in h_slot + h_shards)
    h_views = [[x[:g["psi_pad"]] for x in h_slot] for g in groups]
    d_views = [[x[:g["psi_pad"]] for x in slot] for g in groups]
    dshards = None if mapped else [torch.empty(ST, dtype=torch.bfloat16, device=master.device)
                                   for _ in range(N)]

    def e2e_step():
        t[0] += 1
        hp = Z.adam_hp(t[0], 1.0 / N)
        for gi in reversed(range(G)):
            if mapped:
                Z.zero_step_group(plan, gi, h_views[gi], zg, master, m, v, hp, None,
                                  h_shards, sa)
            else:
                for r in range(N):
                    d_views[gi][r].copy_(h_views[gi][r], non_blocking=True)
                Z.zero_step_group(plan, gi, d_views[gi], zg, master, m, v, hp, None,
                                  dshards, sa)
        if not mapped:
            for r in range(N):
                h_shards[r].copy_(dshards[r], non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    steps = 3
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(sa)
    for _ in range(steps):
        e2e_step()
    s1.record(sa)
    torch.cuda.synchronize()
    ms = s0.elapsed_time(s1) / steps
    del h_slot, h_shards, h_views, pinned
    free_pinned()
    return dict(base, e2e_ms=ms, e2e_steps=steps, numa=numa,
                e2e_transfer="zero-copy kernel access to mapped pinned host memory" if mapped
                else "cudaMemcpyAsync from/to pinned host memory")


# ------------------------------------------- stage-3 gather granularity sweep --
def regroup(w, per: str):
    """Layer-group list of the stage-3 workload at another granularity:
    'tensor' (per-parameter partitioning: every tensor its own group; also
    'tensor-coalesced', the same plan gathered one layer's tensors per
    launch), 'layer' (the workload's groups) or 'k-layers' (k consecutive
    groups)."""
    if per.startswith("tensor"):
        return list(range(len(w.numels)))
    if per == "layer":
        return list(w.groups)
    k = int(per.split("-")[0])
    return [g // k for g in w.groups]


def bench_gather_sweep(w, steps: int, dist: Dist, only=None) -> dict:
    """Forward + reverse per-group gathers of the stage-3 workload's bf16
    shards at several partition granularities (the shards are generated
    directly; no optimizer step is needed to time the gathers)."""
    import torch
    import synth
    import zero_sharded_optimizer_device_gb300 as Z

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    N = w.n_ranks
    sa = torch.cuda.current_stream(dev)
    res = {}
    for per in ("tensor", "tensor-coalesced", "layer", "2-layers", "4-layers"):
        if only and per != only:
            continue
        groups_of = regroup(w, per)
        plan = Z.zero_plan(w.numels, N, w.align, groups_of)
        info = Z.zero_plan_info(plan)
        groups = [Z.zero_plan_group(plan, g) for g in range(info["n_groups"])]
        shards = [torch.empty(info["shard_total"], dtype=torch.bfloat16, device=dev)
                  for _ in range(N)]
        for r in range(N):
            synth.fill_tensor(shards[r], w.seed, synth.MASTER, 0, r, 0, w.master_sigma,
                              info["shard_total"])
        if per == "tensor-coalesced":
            # one launch per layer: that layer's tensors, each into its own
            # 16-byte-aligned slice of the layer's buffer
            layers = [[t for t, g in enumerate(w.groups) if g == L] for L in sorted(set(w.groups))]
            spans = []
            for ts in layers:
                offs, o = [], 0
                for t in ts:
                    offs.append(o)
                    o += -(-groups[t]["psi_pad"] // 8) * 8
                spans.append((ts, offs, o))
            gmax = max(o for _, _, o in spans)
            bufs = [torch.empty(gmax, dtype=torch.bfloat16, device=dev) for _ in range(2)]
            order = list(range(len(layers))) + list(reversed(range(len(layers))))
            calls = [lambda j=j, L=L: Z.zero_gather_groups(
                plan, spans[L][0], shards, Z.ZERO_BF16,
                [bufs[j % 2][o:] for o in spans[L][1]], sa)
                for j, L in enumerate(order)]
        else:
            gmax = max(g["psi_pad"] for g in groups)
            bufs = [torch.empty(gmax, dtype=torch.bfloat16, device=dev) for _ in range(2)]
            order = list(range(len(groups))) + list(reversed(range(len(groups))))
            calls = [lambda j=j, gi=gi: Z.zero_gather_layer(plan, gi, shards, Z.ZERO_BF16,
                                                            bufs[j % 2], sa)
                     for j, gi in enumerate(order)]
        def run_all():
            for f in calls:
                f()

        _timed_seq(sa, run_all)                          # warm-up
        ms = statistics.fmean(_timed_seq(sa, run_all) for _ in range(steps))
        elems = 2 * sum(g["psi_pad"] for g in groups)
        res[per] = {"groups": len(groups), "gathers": len(order), "ms": ms,
                    "gbs": 4 * elems / (ms * 1e-3) / 1e9,
                    "mean_gather_mb": 2 * elems / len(order) / 1e6}
        if per in ("tensor-coalesced", "layer"):
            # the two-stream pass (prefetch on stream B, one-round consumer on A)
            sums = torch.zeros(len(order), dtype=torch.int64, device=dev)
            sb = torch.cuda.Stream(dev)
            if per == "layer":
                run = lambda: Z.zero_stage3_gather_pass(plan, order, shards, bufs, gmax, sums,
                                                        1, sa, sb)
            else:
                step_groups = [spans[L][0] for L in order]
                run = lambda: Z.zero_stage3_gather_pass_steps(plan, step_groups, shards, bufs,
                                                              gmax, sums, 1, sa, sb)
            run()
            torch.cuda.synchronize()
            pass_ms = []
            for _ in range(steps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(sa)
                run()
                e1.record(sa)
                torch.cuda.synchronize()
                pass_ms.append(e0.elapsed_time(e1))
            res[per]["pass_ms"] = statistics.fmean(pass_ms)
        del shards, bufs
        torch.cuda.empty_cache()
    return res


# ------------------------------------------------- oracle on the host cores --
def workload_kind(w) -> str:
    if w.name.startswith("llama-1.4b"):
        return "bucketed"
    if w.groups is not None:
        return "stage3"
    return "fused"


def oracle_sample(w, target_s: float, max_steps: int | None = None, window: int | None = None):
    """Time the CPU oracle's step on a window of the workload that straddles
    the boundary between owners 0 and 1 (stage 3: of the first transformer
    block's group); inputs generated before the clock starts.  The bucketed
    workload's step adds the global norm of the window and its clip.
    Returns (params per second, description, steps, seconds)."""
    import numpy as np
    import synth
    from oracle import zero_oracle as O

    pin_to_one_core()
    kind = workload_kind(w)
    p = O.plan(w.numels, w.n_ranks, w.align, w.groups)
    gi = 1 if kind == "stage3" else 0
    g = p.groups[gi]
    S = g.shard
    win = min(g.psi_pad, window or (1 << 20))
    a = max(0, min(S - win // 2, g.psi_pad - win))
    b = a + win
    sdt = synth.DTYPE_BF16 if w.grad_dtype == "bf16" else synth.DTYPE_F32
    fo = g.flat_off
    local = []
    for r in range(w.n_ranks):
        x = synth.values(w.seed, synth.GRAD, 1, r, fo + a, fo + b, w.grad_sigma, fo + g.psi,
                         w.heavy_tail, sdt)
        local.append(O.bf16_to_f32(x) if sdt == synth.DTYPE_BF16 else x)
    master = synth.values(w.seed, synth.MASTER, 0, 0, fo + a, fo + b, w.master_sigma, fo + g.psi)
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    hp = O.AdamHP()
    inv_n = np.float32(1.0) / np.float32(w.n_ranks)
    steps = 0
    t0 = time.perf_counter()
    while True:
        steps += 1
        coef = None
        if kind == "bucketed":
            red, _, _ = O.ring_reduce_scatter(local, S, (a, b))
            _, coef = O.grad_norm(O.scale(red, inv_n), w.extra["max_norm"])
        r = O.zero_step(local, master, m, v, S, steps, hp, window=(a, b), clip_coef=coef)
        master, m, v = r["master"], r["m"], r["v"]
        el = time.perf_counter() - t0
        if (max_steps and steps >= max_steps) or (not max_steps and el >= target_s):
            break
    where = f"group {gi} " if kind == "stage3" else ""
    what = {"fused": "fused step", "bucketed": "step with global-norm clip",
            "stage3": "stage-3 group step"}[kind]
    desc = (f"oracle {what} on elements [{a},{b}) of {where}{w.name} (N={w.n_ranks}, owner 0/1 "
            f"boundary), {steps} steps, single-threaded numpy")
    return win * steps / el, desc, steps, el


def pin_to_one_core() -> None:
    """Run the oracle on one host core (the baseline is single-threaded)."""
    try:
        cores = sorted(os.sched_getaffinity(0))
        os.sched_setaffinity(0, {cores[-1]})
    except (AttributeError, OSError):
        pass


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def cpu_baseline(w) -> dict:
    """The oracle, as it stands, timed for about 12 s on one host core."""
    rate, desc, _, _ = oracle_sample(w, 12.0)
    return {"value": rate / 1e9, "unit": "Gparams/s", "cores": 1, "kind": "oracle",
            "sample": desc, "cpu": cpu_model(), "nproc": os.cpu_count()}


def bucketed_bytes(w):
    """(formula, path) bytes per step of the bucketed clipped workload: the
    fused formula N*g + 26 per parameter, and what the clipped path moves --
    the reduce-scatter's N*g + 4 (fp32 reduced gradient stored) and Adam's
    4 + 24 + 2."""
    gb = 2 if w.grad_dtype == "bf16" else 4
    return algorithmic_bytes(w.n_ranks, w.psi, gb), w.psi * ((gb * w.n_ranks + 4) + 30)


def fused_config(w, n_gpus: int) -> dict:
    """The `config` object both arms report for a fused-step workload."""
    abytes = algorithmic_bytes(w.n_ranks, w.psi, 2 if w.grad_dtype == "bf16" else 4)
    return {"workload": f"{w.name} fused zero_step", "psi": w.psi, "n_ranks": w.n_ranks,
            "align": w.align, "grad_dtype": w.grad_dtype, "state": "fp32 master/m/v",
            "gathered": "bf16",
            "parallelism": f"replicas x{n_gpus} (ranks emulated on each GPU)",
            "bytes_per_step": abytes,
            "l2": f"inputs {abytes / 1e9:.2f} GB per step > L2 129 MB, no flush"}


def workload_config(w, n_gpus: int) -> dict:
    """The `config` object both arms report for any workload."""
    kind = workload_kind(w)
    if kind == "fused":
        return fused_config(w, n_gpus)
    common = {"psi": w.psi, "n_ranks": w.n_ranks, "align": w.align, "grad_dtype": w.grad_dtype,
              "state": "fp32 master/m/v",
              "parallelism": f"replicas x{n_gpus} (ranks emulated on each GPU)"}
    if kind == "bucketed":
        formula, path = bucketed_bytes(w)
        return {"workload": f"{w.name} bucketed reduce-scatter (50M windows) + global-norm clip "
                            "1.0 + Adam (200M chunks) + bf16 all-gather", **common,
                "gathered": "bf16", "bytes_per_step": path, "bytes_per_step_formula": formula,
                "l2": f"inputs {path / 1e9:.1f} GB per step > L2 129 MB, no flush"}
    abytes = algorithmic_bytes(w.n_ranks, w.psi, 2 if w.grad_dtype == "bf16" else 4)
    return {"workload": f"{w.name}: one stage-3 step = per layer group (34, reverse order) "
                        "fused reduce-scatter + scale + Adam writing each owner's bf16 shard",
            **common, "groups": len(set(w.groups)), "gathered": "bf16 owner shards",
            "grads": f"each group's N buffers are prefixes of one resident N x 202M "
                     f"{w.grad_dtype} slot",
            "bytes_per_step": abytes,
            "l2": f"inputs {abytes / 1e9:.0f} GB per step > L2 129 MB, no flush"}


def _bf16_peak():
    """Measured dense bf16 TFLOP/s (burst) of this machine's GPUs, or None."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return None


def _peaks() -> dict:
    peak, kind = measured_hbm_peak()
    return {"peak": peak, "peak_kind": kind, "peak_nominal_gbs": NOMINAL_HBM_GBS}


# ------------------------------------------------------------------ lines --
def fused_line(w, args, dist) -> dict:
    res = bench_fused(w, args.steps, args.warmup, dist, args.kernel_only, args.graph,
                      args.graph_steps)
    ms = dist.max(res["local_ms"])
    e2e_ms = dist.max(res["e2e_ms"]) if res["e2e_ms"] is not None else None
    n_gpus = dist.world
    value = n_gpus * w.psi / (ms * 1e-3) / 1e9
    e2e_value = n_gpus * w.psi / (e2e_ms * 1e-3) / 1e9 if e2e_ms else None
    abytes = algorithmic_bytes(res["n_ranks"], res["psi_pad"], res["gbytes"])
    pk = _peaks()
    achieved = abytes / (res["launch_ms"] * 1e-3) / 1e9
    step_gbs = abytes / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "Gparams/s", "n_gpus": n_gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": fused_config(w, n_gpus),
        "hbm_gbs": step_gbs, "hbm_pct_of_peak": 100.0 * step_gbs / pk["peak"],
        "roofline": {"bound": "hbm", "achieved": achieved, "unit": "GB/s",
                     "frac": achieved / pk["peak"], **pk,
                     "kernel": f"fused_kernel<{res['n_ranks']},{w.grad_dtype}>",
                     "algorithmic_bytes_per_launch": abytes,
                     "traffic": profiled_traffic("fused_kernel", w.name)},
        "copy_peak_gbs": res["copy_gbs"],
        "clocks": res["clocks"],
        "e2e": {"value": e2e_value, "unit": "Gparams/s", "h2d_bytes_per_step": res["h2d"],
                "d2h_bytes_per_step": res["d2h"], "ms_per_step": e2e_ms,
                "steps": res["e2e_steps"], "transfer": res.get("e2e_transfer"),
                "host_memory": res.get("numa")},
        "gpu_launches": 2 * args.steps if res.get("graph") else args.steps,
    }
    if res.get("graph"):
        line["config"]["launch"] = (f"CUDA graph of {res['graph']} step(s), each an Adam state "
                                    "advance + the fused kernel")
    if args.kernel_only:
        return {"kernel_only": True, "workload": w.name, "psi": w.psi, "ms_per_step": ms,
                "value": value, "unit": "Gparams/s", "roofline": line["roofline"]}
    return line


def bucketed_line(w, args, dist) -> dict:
    """JSON line of the clipped bucketed workload (Llama-1.4B)."""
    r = bench_bucketed(w, args.steps, args.warmup, dist, args.kernel_only)
    ms = dist.max(r["local_ms"])
    P = r["P"]
    N = r["N"]
    gb = 2 if w.grad_dtype == "bf16" else 4
    formula, path = bucketed_bytes(w)
    pk = _peaks()
    rs_bytes, adam_bytes = P * (gb * N + 4), P * 30
    e2e_ms = dist.max(r["e2e_ms"]) if r["e2e_ms"] is not None else None
    n_gpus = dist.world
    line = {"metric": METRIC, "value": n_gpus * w.psi / (ms * 1e-3) / 1e9,
            "unit": "Gparams/s", "n_gpus": n_gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(workload_config(w, n_gpus), launches_per_step=r["n_launches"]),
            "hbm_gbs_formula": formula / (ms * 1e-3) / 1e9,
            "hbm_gbs_path": path / (ms * 1e-3) / 1e9,
            "roofline": {"bound": "hbm", **pk, "unit": "GB/s",
                         "kernel": "rs_kernel + norm_kernel + adam_kernel (the step)",
                         "achieved": path / (ms * 1e-3) / 1e9,
                         "frac": path / (ms * 1e-3) / 1e9 / pk["peak"],
                         "frac_formula_42B": formula / (ms * 1e-3) / 1e9 / pk["peak"],
                         "algorithmic_bytes_per_step": path,
                         "traffic": _sum_or_none(
                             profiled_traffic("rs_kernel", w.name, "rs_kernel_step"),
                             profiled_traffic("adam_kernel", w.name, "adam_kernel_step")),
                         "rs_gbs": rs_bytes / (r["rs_ms"] * 1e-3) / 1e9,
                         "adam_gbs": adam_bytes / (r["adam_ms"] * 1e-3) / 1e9,
                         "rs_ms": r["rs_ms"], "adam_ms": r["adam_ms"], "norm_ms": r["norm_ms"]},
            "norm": r["norm"], "clip_coef": r["coef"], "clocks": r["clocks"],
            "e2e": {"value": n_gpus * w.psi / (e2e_ms * 1e-3) / 1e9 if e2e_ms else None,
                    "unit": "Gparams/s", "h2d_bytes_per_step": r["h2d"],
                    "d2h_bytes_per_step": r["d2h"], "ms_per_step": e2e_ms,
                    "steps": r["e2e_steps"], "transfer": r.get("e2e_transfer"),
                    "host_memory": r.get("numa")},
            "gpu_launches": r["n_launches"] * args.steps}
    if args.kernel_only:
        return {"kernel_only": True, "workload": w.name, "psi": w.psi, "ms_per_step": ms,
                "value": line["value"], "unit": "Gparams/s", "roofline": line["roofline"]}
    return line


def _sum_or_none(*xs):
    return None if any(x is None for x in xs) else sum(xs)


def stage3_line(w, args, dist) -> dict:
    """JSON line of the stage-3 workload (Llama-7B): the step, its roofline
    on a transformer block's launch, the gathers, end to end."""
    r = bench_stage3(w, args.steps, args.warmup, dist, args.graph, args.kernel_only)
    P, N = r["P"], r["N"]
    ms = dist.max(r["local_ms"])
    n_gpus = dist.world
    pk = _peaks()
    step_bytes = algorithmic_bytes(N, P, r["gbytes"])
    block_bytes = algorithmic_bytes(N, r["block_psi_pad"], r["gbytes"])
    achieved = block_bytes / (r["block_ms"] * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "unit": "GB/s", "frac": achieved / pk["peak"],
            **pk, "kernel": f"fused_kernel<{N},{w.grad_dtype}> (zero_step_group), one "
                            "transformer block's group per launch",
            "algorithmic_bytes_per_launch": block_bytes,
            "traffic": profiled_traffic("fused_kernel", w.name, "fused_kernel_block"),
            "step_launches_gbs": step_bytes / (r["launch_sum_ms"] * 1e-3) / 1e9}
    if args.kernel_only:
        return {"kernel_only": True, "workload": w.name, "psi": w.psi, "ms_per_step": ms,
                "value": n_gpus * w.psi / (ms * 1e-3) / 1e9, "unit": "Gparams/s",
                "roofline": roof}
    ge = r["gather_elems"]
    gather = {"launches": r["gather_launches"],
              "gathers_only_ms": r["gathers_only_ms"],
              "gather_gbs": 4 * ge / (r["gathers_only_ms"] * 1e-3) / 1e9,
              "gather_frac": 4 * ge / (r["gathers_only_ms"] * 1e-3) / 1e9 / pk["peak"],
              "gather_traffic": profiled_traffic("gather_bulk_kernel", w.name,
                                                 "gather_bulk_kernel_block"),
              "broadcast_ms": r["broadcast_ms"],
              "broadcast_gbs": 4 * ge / (r["broadcast_ms"] * 1e-3) / 1e9,
              "schedule_ms": r["schedule_ms"],
              "schedule_gbs_incl_consumer": 6 * ge / (r["schedule_ms"] * 1e-3) / 1e9,
              "schedule_frac_incl_consumer": 6 * ge / (r["schedule_ms"] * 1e-3) / 1e9 / pk["peak"],
              "consumers_only_ms": r["consumers_only_ms"],
              "hidden": _hidden(r["gathers_only_ms"], r["consumers_only_ms"], r["schedule_ms"]),
              "arith_consumer": {
                  "rounds": ARITH_ROUNDS, "consumers_only_ms": r["consumers_arith_ms"],
                  "schedule_ms": r["schedule_arith_ms"],
                  "hidden": _hidden(r["gathers_only_ms"], r["consumers_arith_ms"],
                                    r["schedule_arith_ms"])}}
    if "schedule_graph_ms" in r:
        gather["schedule_graph_ms"] = r["schedule_graph_ms"]
    tf_peak = _bf16_peak()
    gather["gemm_consumer"] = {
        "shape": r["gemm_shape"], "consumers_only_ms": r["gemm_consumers_only_ms"],
        "consumer_tflops": r["gemm_flops"] / (r["gemm_consumers_only_ms"] * 1e-3) / 1e12,
        "consumer_frac_of_bf16_peak": (r["gemm_flops"] / (r["gemm_consumers_only_ms"] * 1e-3)
                                       / 1e12 / tf_peak) if tf_peak else None,
        "schedule_ms": r["gemm_schedule_ms"],
        "hidden": _hidden(r["gathers_only_ms"], r["gemm_consumers_only_ms"],
                          r["gemm_schedule_ms"])}
    e2e_ms = dist.max(r["e2e_ms"]) if r["e2e_ms"] is not None else None
    return {"metric": METRIC, "value": n_gpus * w.psi / (ms * 1e-3) / 1e9,
            "unit": "Gparams/s", "n_gpus": n_gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic", "config": workload_config(w, n_gpus),
            "hbm_gbs": step_bytes / (ms * 1e-3) / 1e9,
            "hbm_pct_of_peak": 100.0 * step_bytes / (ms * 1e-3) / 1e9 / pk["peak"],
            "roofline": roof, "copy_peak_gbs": r["copy_gbs"], "clocks": r["clocks"],
            "gather": gather,
            "e2e": {"value": n_gpus * w.psi / (e2e_ms * 1e-3) / 1e9 if e2e_ms else None,
                    "unit": "Gparams/s", "h2d_bytes_per_step": r["h2d"],
                    "d2h_bytes_per_step": r["d2h"], "ms_per_step": e2e_ms,
                    "steps": r["e2e_steps"], "transfer": r.get("e2e_transfer"),
                    "host_memory": r.get("numa")},
            "gpu_launches": r["launches_per_step"] * args.steps}


# -------------------------------------------------------------------- main --
def reference_line(w, args, dist) -> dict:
    """The reference arm: the CPU oracle, as it stands, on a bounded window
    of the same workload per step (rank 0 only)."""
    probe_rate, _, _, _ = oracle_sample(w, 0.0, max_steps=1, window=1 << 16)
    budget = 120.0 / max(1, args.steps + args.warmup)
    win = int(min(1 << 22, max(1 << 12, probe_rate * budget)))
    win -= win % 16
    if args.warmup:
        oracle_sample(w, 0.0, max_steps=args.warmup, window=win)
    rate, desc, steps, el = oracle_sample(w, 0.0, max_steps=args.steps, window=win)
    value = rate / 1e9
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "Gparams/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(w, args.gpus),
            "cpu_baseline": {"value": value, "unit": "Gparams/s", "cores": 1,
                             "kind": "oracle", "sample": desc, "cpu": cpu_model()},
            "e2e": {"value": value, "unit": "Gparams/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="llama-7b-stage3 (default), gpt2-small, gpt2-medium, llama-1.4b or tiny")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--scale", type=int, default=1,
                    help="shrink the workload's tensors by this factor (profiling cases)")
    ap.add_argument("--kernel-only", action="store_true",
                    help="time only the step kernels: no copy peak, gathers, e2e or CPU baseline")
    ap.add_argument("--graph", action="store_true",
                    help="fused workloads: time CUDA-graph replays of the step (device-resident "
                         "Adam step state); stage-3 workload: also time the gather pass "
                         "replayed from a graph")
    ap.add_argument("--graph-steps", type=int, default=1,
                    help="with --graph: steps captured in one graph (amortises the replay launch)")
    ap.add_argument("--grad-dtype", choices=["bf16", "f32"], default=None,
                    help="override the workload's gradient dtype (fp32 doubles the source bytes)")
    ap.add_argument("--gather-sweep", action="store_true",
                    help="stage-3 workload: gather bandwidth at several partition granularities")
    ap.add_argument("--gather-granularity", default=None,
                    choices=["tensor", "tensor-coalesced", "layer", "2-layers", "4-layers"],
                    help="with --gather-sweep: only this granularity")
    args = ap.parse_args(argv)
    from synth import workloads as W
    w = W.ALL[args.workload]
    if args.scale > 1:
        w = W.mini(w, scale=args.scale)
    if args.grad_dtype and args.grad_dtype != w.grad_dtype:
        import dataclasses
        w = dataclasses.replace(w, name=f"{w.name}-{args.grad_dtype}-grads",
                                grad_dtype=args.grad_dtype)
    dist = Dist()

    if args.impl == "reference":
        if dist.rank == 0:
            print(json.dumps(reference_line(w, args, dist)), flush=True)
        dist.close()
        return

    import torch
    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    import zero_sharded_optimizer_device_gb300  # noqa: F401  (fails loudly when unbuilt)

    if args.gather_sweep:
        res = bench_gather_sweep(w, max(1, args.steps), dist, args.gather_granularity)
        if dist.rank == 0:
            print(json.dumps({"workload": f"{w.name} stage-3 gathers, forward + reverse",
                              "n_ranks": w.n_ranks, "granularity": res}), flush=True)
        dist.close()
        return
    kind = workload_kind(w)
    line = {"fused": fused_line, "bucketed": bucketed_line, "stage3": stage3_line}[kind](
        w, args, dist)
    if (dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline
            and not line.get("kernel_only")):
        line["cpu_baseline"] = cpu_baseline(w)
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
