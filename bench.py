"""Benchmark of the ZeRO sharded-optimizer hot path on one GB300 per rank.

Default workload: the GPT-2-small parameter list (124,439,808 parameters, 148
tensors), N = 8 emulated data-parallel ranks, bf16 gradients, fp32 master /
m / v, bf16 gathered parameters; one step = one fused zero_step (ring-order
reduce-scatter + scale + Adam on every owner shard + all-gather).  Prints one
JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload gpt2-small|gpt2-medium|llama-1.4b|llama-7b-stage3|tiny]

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


def kernel_source_hash(kernel: str = "fused_kernel") -> str:
    """Hash of what decides a kernel's DRAM traffic: the device helpers, the
    kernel's own source text and its occupancy default (host code around it
    and the other kernels' defaults do not count)."""
    return _source_hash(_read_csrc("zero_device.cuh"), _read_csrc("zero_rs.cu"), kernel)


def _read_csrc(name: str) -> str:
    with open(os.path.join(ROOT, "zero_sharded_optimizer_device_gb300", "csrc", name)) as f:
        return f.read()


def _source_hash(device_h: str, rs_cu: str, kernel: str) -> str:
    h = hashlib.sha256()
    h.update(device_h.encode())
    start = rs_cu.index(f"    {kernel}(")
    start = rs_cu.rindex("template", 0, start)
    end = rs_cu.index("// ------", start)
    h.update(rs_cu[start:end].encode())
    occ = rs_cu.index("constexpr int kOccDefault")
    block = rs_cu[occ:rs_cu.index("};", occ)]
    h.update(next(line for line in block.splitlines() if "ZERO_OCC_FUSED" in line).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, only while the
    kernel sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(workload, {}).get(kernel)
    if not entry or entry.get("source_hash") != kernel_source_hash(kernel):
        return None
    return entry.get("bytes_per_launch")


def pinned_host_buffer(nbytes: int):
    """One page-locked host byte buffer of exactly nbytes from cudaHostAlloc
    (torch's pinned allocator would round each tensor up to a power of two).
    Returns (uint8 tensor over it, function that frees it)."""
    import ctypes
    import torch
    rt = ctypes.CDLL("libcudart.so.13")
    rt.cudaHostAlloc.restype = ctypes.c_int
    rt.cudaHostAlloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t, ctypes.c_uint]
    rt.cudaFreeHost.restype = ctypes.c_int
    rt.cudaFreeHost.argtypes = [ctypes.c_void_p]
    ptr = ctypes.c_void_p()
    rc = rt.cudaHostAlloc(ctypes.byref(ptr), nbytes, 0)
    if rc != 0:
        raise RuntimeError(f"cudaHostAlloc of {nbytes} bytes failed ({rc})")
    t = torch.frombuffer((ctypes.c_uint8 * nbytes).from_address(ptr.value), dtype=torch.uint8)
    return t, (lambda: rt.cudaFreeHost(ptr))


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

    def step():
        t[0] += 1
        Z.zero_step(plan, 0, grads, zg, master, m, v, Z.adam_hp(t[0], 1.0 / N), None, out,
                    Z.ZERO_BF16, stream)

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
    if host_bytes > 0.4 * ram:      # too large to pin on this host: no end-to-end leg
        return dict(local_ms=local_ms, launch_ms=launch_ms, e2e_ms=None, psi=w.psi, psi_pad=P,
                    n_ranks=N, gbytes=gbytes, copy_gbs=copy_gbs, clocks=clocks.summary(),
                    h2d=N * P * gbytes, d2h=P * 2, e2e_steps=0,
                    e2e_transfer=f"skipped: {host_bytes / 1e9:.0f} GB of pinned host memory "
                                 f"exceeds 40% of the host's {ram / 1e9:.0f} GB")
    pinned, free_pinned = pinned_host_buffer(host_bytes)
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
                h2d=N * P * gbytes, d2h=P * 2, e2e_steps=e2e_steps,
                e2e_transfer="zero-copy kernel access to mapped pinned host memory" if zero_copy
                else "cudaMemcpyAsync from/to pinned host memory")


# ----------------------------------------- bucketed pipeline with clipping --
def _timed_launches(stream, calls):
    """Run callables on `stream`, each bracketed by CUDA events; returns the
    per-call device milliseconds (after a synchronize)."""
    import torch
    evs = []
    for f in calls:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        f()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def bench_bucketed(w, steps: int, warmup: int, dist: Dist) -> dict:
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

    def calls():
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
    per_step, rs_ms, adam_ms, norm_ms = [], 0.0, 0.0, 0.0
    with ClockSampler(dev.index) as clocks:
        dist.barrier()
        for _ in range(steps):
            ms = _timed_launches(stream, calls())
            per_step.append(sum(ms))
            rs_ms += sum(ms[:len(windows)])
            norm_ms += ms[len(windows)]
            adam_ms += sum(ms[len(windows) + 1:])
        dist.barrier()
    return dict(local_ms=statistics.fmean(per_step), rs_ms=rs_ms / steps, norm_ms=norm_ms / steps,
                adam_ms=adam_ms / steps, P=P, N=N, n_launches=len(windows) + 1 + len(chunks),
                clocks=clocks.summary(), norm=float(norm.item()), coef=float(coef.item()))


# ------------------------------------------- stage 3: step + per-layer gathers --
# Rounds of the arithmetic-bound stand-in consumer (zero_layer_checksum): at 64
# its 68 launches over the Llama-7B groups take about 3.5x the gathers.
ARITH_ROUNDS = 64


def _hidden(gathers_ms: float, consumers_ms: float, schedule_ms: float) -> float:
    """Fraction of the shorter of the two kernel streams that the two-stream
    schedule hides behind the other: 1 = fully overlapped, 0 = serial."""
    return (gathers_ms + consumers_ms - schedule_ms) / min(gathers_ms, consumers_ms)


def bench_stage3(w, steps: int, warmup: int, dist: Dist, use_graph: bool = False) -> dict:
    """Stage 3 (the Llama-7B workload): per layer group, in reverse order, a
    fused reduce-scatter + Adam writing each owner's bf16 shard (gradients
    regenerated into one slot per group, untimed); then every group gathered
    into a contiguous layer buffer in forward and then reverse order, the
    next group prefetched on a second stream while a consumer reads the
    current one.  With ``use_graph`` the gather pass is also captured once in
    a CUDA graph and its replay timed."""
    import torch
    import synth
    import zero_sharded_optimizer_device_gb300 as Z

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    N = w.n_ranks
    plan = Z.zero_plan(w.numels, N, w.align, w.groups)
    info = Z.zero_plan_info(plan)
    groups = [Z.zero_plan_group(plan, g) for g in range(info["n_groups"])]
    P, ST = info["psi_pad"], info["shard_total"]
    gmax = max(g["psi_pad"] for g in groups)
    master = torch.empty(P, dtype=torch.float32, device=dev)
    for g in groups:
        synth.fill_tensor(master[g["flat_off"]:g["flat_off"] + g["psi_pad"]], w.seed, synth.MASTER,
                          0, 0, g["flat_off"], w.master_sigma, g["flat_off"] + g["psi"])
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    shards = [torch.zeros(ST, dtype=torch.bfloat16, device=dev) for _ in range(N)]
    slot = [torch.empty(gmax, dtype=torch.bfloat16, device=dev) for _ in range(N)]
    bufs = [torch.empty(gmax, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    sums = torch.zeros(2 * len(groups), dtype=torch.int64, device=dev)  # one per gather
    sa = torch.cuda.current_stream(dev)
    sb = torch.cuda.Stream(dev)

    def fill(gi, step):
        g = groups[gi]
        for r in range(N):
            synth.fill_tensor(slot[r][:g["psi_pad"]], w.seed, synth.GRAD, step, r, g["flat_off"],
                              w.grad_sigma, g["flat_off"] + g["psi"])

    def rs_adam_step(step):
        ms = 0.0
        for gi in reversed(range(len(groups))):
            fill(gi, step)
            ms += _timed_launches(sa, [lambda gi=gi: Z.zero_step_group(
                plan, gi, slot, Z.ZERO_BF16, master, m, v, Z.adam_hp(step, 1.0 / N), None,
                shards, sa)])[0]
        return ms

    order = list(range(len(groups))) + list(reversed(range(len(groups))))

    def gather_schedule(rounds):
        """Prefetch on stream B into the free buffer, consume on stream A
        (the library's native two-stream schedule)."""
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(sa)
        Z.zero_stage3_gather_pass(plan, order, shards, bufs, gmax, sums, rounds, sa, sb)
        e1.record(sa)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    def consumers_only(rounds):
        calls = [lambda j=j, gi=gi: Z.zero_layer_checksum(bufs[j % 2], groups[gi]["psi_pad"],
                                                          rounds, sums[j:j + 1], sa)
                 for j, gi in enumerate(order)]
        return sum(_timed_launches(sa, calls))

    def gathers_only():
        calls = [lambda j=j, gi=gi: Z.zero_gather_layer(plan, gi, shards, Z.ZERO_BF16,
                                                        bufs[j % 2], sa)
                 for j, gi in enumerate(order)]
        return sum(_timed_launches(sa, calls))

    def broadcasts_only():
        """The ZeRO paper's broadcast form of the same gather: each owner in
        turn sends its shard to every rank -- here one copy launch per owner
        into the shared layer buffer instead of one all-gather kernel."""
        calls = []
        for j, gi in enumerate(order):
            g = groups[gi]
            nbytes = g["shard"] * 2
            for k in range(N):
                src = shards[k].data_ptr() + g["rank_off"] * 2
                dst = bufs[j % 2].data_ptr() + k * nbytes
                calls.append(lambda s=src, d=dst, b=nbytes: Z.zero_copy(d, s, b, sa))
        return sum(_timed_launches(sa, calls))

    for s in range(1, warmup + 1):
        rs_adam_step(s)
        gather_schedule(1)
        gather_schedule(ARITH_ROUNDS)
    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        gs, gsb = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        gs.wait_stream(sa)
        with torch.cuda.stream(gs):
            with torch.cuda.graph(graph, stream=gs):
                Z.zero_stage3_gather_pass(plan, order, shards, bufs, gmax, sums, 1, gs, gsb)
        sa.wait_stream(gs)
        torch.cuda.synchronize()

    def gather_schedule_graph():
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(sa)
        graph.replay()
        e1.record(sa)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    if graph is not None:
        gather_schedule_graph()
    rs_ms, sched_ms, gonly_ms, bcast_ms, graph_ms = [], [], [], [], []
    cons_ms, sched_a_ms, cons_a_ms = [], [], []
    with ClockSampler(dev.index) as clocks:
        dist.barrier()
        for s in range(warmup + 1, warmup + steps + 1):
            rs_ms.append(rs_adam_step(s))
            sched_ms.append(gather_schedule(1))
            sched_a_ms.append(gather_schedule(ARITH_ROUNDS))
            if graph is not None:
                graph_ms.append(gather_schedule_graph())
            gonly_ms.append(gathers_only())
            cons_ms.append(consumers_only(1))
            cons_a_ms.append(consumers_only(ARITH_ROUNDS))
            bcast_ms.append(broadcasts_only())
        dist.barrier()
    gather_elems = 2 * sum(g["psi_pad"] for g in groups)
    return dict(rs_ms=statistics.fmean(rs_ms), sched_ms=statistics.fmean(sched_ms),
                gonly_ms=statistics.fmean(gonly_ms), bcast_ms=statistics.fmean(bcast_ms),
                graph_ms=statistics.fmean(graph_ms) if graph_ms else None,
                cons_ms=statistics.fmean(cons_ms), sched_a_ms=statistics.fmean(sched_a_ms),
                cons_a_ms=statistics.fmean(cons_a_ms),
                P=P, N=N, groups=len(groups),
                gather_elems=gather_elems, clocks=clocks.summary())


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
        _timed_launches(sa, calls)                     # warm-up
        ms = statistics.fmean(sum(_timed_launches(sa, calls)) for _ in range(steps))
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
def oracle_sample(w, target_s: float, max_steps: int | None = None, window: int | None = None):
    """Time the CPU oracle's fused step on a window of the workload that
    straddles the boundary between owners 0 and 1; inputs generated before
    the clock starts.  Returns (params per second, description, steps)."""
    import numpy as np
    import synth
    from oracle import zero_oracle as O

    pin_to_one_core()
    p = O.plan(w.numels, w.n_ranks, w.align)
    S = p.groups[0].shard
    win = window or min(p.psi_pad, 1 << 20)
    a = max(0, min(S - win // 2, p.psi_pad - win))
    b = a + win
    sdt = synth.DTYPE_BF16 if w.grad_dtype == "bf16" else synth.DTYPE_F32
    local = []
    for r in range(w.n_ranks):
        x = synth.values(w.seed, synth.GRAD, 1, r, a, b, w.grad_sigma, w.psi, w.heavy_tail, sdt)
        local.append(O.bf16_to_f32(x) if sdt == synth.DTYPE_BF16 else x)
    master = synth.values(w.seed, synth.MASTER, 0, 0, a, b, w.master_sigma, w.psi)
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    hp = O.AdamHP()
    steps = 0
    t0 = time.perf_counter()
    while True:
        steps += 1
        r = O.zero_step(local, master, m, v, S, steps, hp, window=(a, b))
        master, m, v = r["master"], r["m"], r["v"]
        el = time.perf_counter() - t0
        if (max_steps and steps >= max_steps) or (not max_steps and el >= target_s):
            break
    desc = (f"oracle fused step on elements [{a},{b}) of {w.name} (N={w.n_ranks}, owner 0/1 "
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


def fused_config(w, n_gpus: int) -> dict:
    """The `config` object both arms report for a fused-step workload."""
    abytes = algorithmic_bytes(w.n_ranks, w.psi, 2 if w.grad_dtype == "bf16" else 4)
    return {"workload": f"{w.name} fused zero_step", "psi": w.psi, "n_ranks": w.n_ranks,
            "align": w.align, "grad_dtype": w.grad_dtype, "state": "fp32 master/m/v",
            "gathered": "bf16",
            "parallelism": f"replicas x{n_gpus} (ranks emulated on each GPU)",
            "bytes_per_step": abytes,
            "l2": f"inputs {abytes / 1e9:.2f} GB per step > L2 129 MB, no flush"}


def secondary_line(w, args, dist) -> dict:
    """JSON line for the bucketed and stage-3 workloads (not the headline)."""
    peak, peak_kind = measured_hbm_peak()
    n_gpus = dist.world
    if w.name.startswith("llama-1.4b"):
        r = bench_bucketed(w, args.steps, args.warmup, dist)
        ms = dist.max(r["local_ms"])
        P, N = r["P"], r["N"]
        gb = 2 if w.grad_dtype == "bf16" else 4
        formula = algorithmic_bytes(N, P, gb)             # N*gb + 26 B/param
        path = P * ((gb * N + 4) + (4 + 24 + 2))          # RS N*gb+4, Adam 30
        return {"metric": METRIC, "value": n_gpus * w.psi / (ms * 1e-3) / 1e9,
                "unit": "Gparams/s", "n_gpus": n_gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "dtype": "f32", "data": "synthetic",
                "config": {"workload": f"{w.name} bucketed RS (50M) + clip 1.0 + Adam (200M chunks)",
                           "psi": w.psi, "n_ranks": N, "launches_per_step": r["n_launches"]},
                "hbm_gbs_formula": formula / (ms * 1e-3) / 1e9,
                "hbm_gbs_path": path / (ms * 1e-3) / 1e9,
                "roofline": {"bound": "hbm", "peak": peak, "peak_kind": peak_kind,
                             "unit": "GB/s", "kernel": "rs_kernel + adam_kernel (the step)",
                             "achieved": path / (ms * 1e-3) / 1e9,
                             "frac": path / (ms * 1e-3) / 1e9 / peak,
                             "traffic": None,
                             "rs_gbs": P * (gb * N + 4) / (r["rs_ms"] * 1e-3) / 1e9,
                             "adam_gbs": P * 30 / (r["adam_ms"] * 1e-3) / 1e9,
                             "rs_ms": r["rs_ms"], "adam_ms": r["adam_ms"], "norm_ms": r["norm_ms"]},
                "norm": r["norm"], "clip_coef": r["coef"], "clocks": r["clocks"],
                "gpu_launches": r["n_launches"] * args.steps}
    r = bench_stage3(w, args.steps, args.warmup, dist, args.graph)
    P, N = r["P"], r["N"]
    rs_ms = dist.max(r["rs_ms"])
    return {"metric": METRIC, "value": n_gpus * w.psi / (rs_ms * 1e-3) / 1e9,
            "unit": "Gparams/s", "n_gpus": n_gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": rs_ms, "higher_is_better": True, "scaling": "weak", "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": f"{w.name}: per-group fused RS+Adam to owner shards, then "
                                   "forward+reverse per-layer gathers prefetched on stream B",
                       "psi": w.psi, "n_ranks": N, "groups": r["groups"]},
            "rs_adam_gbs": algorithmic_bytes(N, P, 2) / (rs_ms * 1e-3) / 1e9,
            "gather": {"schedule_ms": r["sched_ms"], "gathers_only_ms": r["gonly_ms"],
                       "gather_gbs": 4 * r["gather_elems"] / (r["gonly_ms"] * 1e-3) / 1e9,
                       "broadcast_ms": r["bcast_ms"],
                       "broadcast_gbs": 4 * r["gather_elems"] / (r["bcast_ms"] * 1e-3) / 1e9,
                       "schedule_gbs_incl_consumer": 6 * r["gather_elems"] /
                       (r["sched_ms"] * 1e-3) / 1e9,
                       "consumers_only_ms": r["cons_ms"],
                       "hidden": _hidden(r["gonly_ms"], r["cons_ms"], r["sched_ms"]),
                       "arith_consumer": {
                           "rounds": ARITH_ROUNDS, "consumers_only_ms": r["cons_a_ms"],
                           "schedule_ms": r["sched_a_ms"],
                           "hidden": _hidden(r["gonly_ms"], r["cons_a_ms"], r["sched_a_ms"])},
                       **({"schedule_graph_ms": r["graph_ms"],
                           "schedule_graph_gbs_incl_consumer": 6 * r["gather_elems"] /
                           (r["graph_ms"] * 1e-3) / 1e9} if r["graph_ms"] else {})},
            "roofline": {"bound": "hbm", "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "kernel": "fused_kernel<16,bf16> (zero_step_group, 34 groups)",
                         "achieved": algorithmic_bytes(N, P, 2) / (rs_ms * 1e-3) / 1e9,
                         "frac": algorithmic_bytes(N, P, 2) / (rs_ms * 1e-3) / 1e9 / peak,
                         "traffic": None},
            "clocks": r["clocks"]}


# -------------------------------------------------------------------- main --
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gpt2-small")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--scale", type=int, default=1,
                    help="shrink the workload's tensors by this factor (profiling cases)")
    ap.add_argument("--kernel-only", action="store_true",
                    help="time only the step kernel: no copy peak, e2e or CPU baseline")
    ap.add_argument("--graph", action="store_true",
                    help="replay one CUDA-graph-captured step (device-resident Adam step state); "
                         "stage-3 workload: also time the gather pass replayed from a graph")
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
        if dist.rank != 0:
            dist.close()
            return
        # per step a bounded window, sized so warmup + steps stay ~2 minutes
        probe_rate, _, _, _ = oracle_sample(w, 0.0, max_steps=1, window=1 << 16)
        budget = 120.0 / max(1, args.steps + args.warmup)
        win = int(min(1 << 22, max(1 << 12, probe_rate * budget)))
        win -= win % 16
        if args.warmup:
            oracle_sample(w, 0.0, max_steps=args.warmup, window=win)
        rate, desc, steps, el = oracle_sample(w, 0.0, max_steps=args.steps, window=win)
        value = rate / 1e9
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "Gparams/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": el / steps * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": fused_config(w, args.gpus),
                "cpu_baseline": {"value": value, "unit": "Gparams/s", "cores": 1,
                                 "kind": "oracle", "sample": desc, "cpu": cpu_model()},
                "e2e": {"value": value, "unit": "Gparams/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
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
    if w.name.startswith("llama-1.4b") or w.name.startswith("llama-7b"):
        line = secondary_line(w, args, dist)
        if dist.rank == 0:
            print(json.dumps(line), flush=True)
        dist.close()
        return

    res = bench_fused(w, args.steps, args.warmup, dist, args.kernel_only, args.graph,
                      args.graph_steps)
    ms = dist.max(res["local_ms"])
    e2e_ms = dist.max(res["e2e_ms"]) if res["e2e_ms"] is not None else None
    n_gpus = dist.world
    value = n_gpus * w.psi / (ms * 1e-3) / 1e9
    e2e_value = n_gpus * w.psi / (e2e_ms * 1e-3) / 1e9 if e2e_ms else None
    abytes = algorithmic_bytes(res["n_ranks"], res["psi_pad"], res["gbytes"])
    peak, peak_kind = measured_hbm_peak()
    achieved = abytes / (res["launch_ms"] * 1e-3) / 1e9
    step_gbs = abytes / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "Gparams/s", "n_gpus": n_gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": fused_config(w, n_gpus),
        "hbm_gbs": step_gbs, "hbm_pct_of_peak": 100.0 * step_gbs / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "kernel": f"fused_kernel<{res['n_ranks']},{w.grad_dtype}>",
                     "algorithmic_bytes_per_launch": abytes,
                     "traffic": profiled_traffic("fused_kernel", w.name)},
        "copy_peak_gbs": res["copy_gbs"],
        "clocks": res["clocks"],
        "e2e": {"value": e2e_value, "unit": "Gparams/s", "h2d_bytes_per_step": res["h2d"],
                "d2h_bytes_per_step": res["d2h"], "ms_per_step": e2e_ms,
                "steps": res["e2e_steps"], "transfer": res.get("e2e_transfer")},
        "gpu_launches": 2 * args.steps if res.get("graph") else args.steps,
    }
    if res.get("graph"):
        line["config"]["launch"] = (f"CUDA graph of {res['graph']} step(s), each an Adam state "
                                    "advance + the fused kernel")
    if args.kernel_only:
        line = {"kernel_only": True, "workload": w.name, "psi": w.psi, "ms_per_step": ms,
                "value": value, "unit": "Gparams/s", "roofline": line["roofline"]}
    elif dist.rank == 0 and n_gpus == 1 and not args.no_cpu_baseline:
        rate, desc, steps, el = oracle_sample(w, 12.0)
        line["cpu_baseline"] = {"value": rate / 1e9, "unit": "Gparams/s", "cores": 1,
                                "kind": "oracle", "sample": desc, "cpu": cpu_model(),
                                "nproc": os.cpu_count()}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
