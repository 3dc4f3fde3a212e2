"""Parity of the CUDA path (through the C ABI) with the CPU oracle, element by
element, on seeded inputs: small workloads in full, edge cases, and the
GPT-2-small workload at full size on sampled windows."""
import numpy as np
import pytest

import synth
from synth import workloads as W
from oracle import zero_oracle as O

from harness import Case, assert_bf16, assert_close_f32, bits_of, boundary_windows

pytestmark = pytest.mark.gpu


def _fused_steps(case: Case, steps: int, out_dtype: str = "bf16", group: int = 0):
    import torch
    Z = case.Z
    g = case.groups[group]
    tdt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
    out = torch.zeros(case.info["psi_pad"], dtype=tdt, device=case.dev)
    zdt = Z.ZERO_BF16 if out_dtype == "bf16" else Z.ZERO_F32
    grads = None
    last = None
    for s in range(1, steps + 1):
        grads = case.grads_dev(group, s, grads)
        Z.zero_step(case.plan, group, grads, case.zdtype, case.master, case.m, case.v,
                    case.hp_dev(s), None, out, zdt)
        last = case.oracle_step(group, s, out_dtype=out_dtype)
    torch.cuda.synchronize()
    f0 = g["flat_off"]
    sl = slice(f0, f0 + g["psi_pad"])
    if out_dtype == "bf16":
        assert_bf16(bits_of(out[sl]), last["full"], "gathered bf16")
    else:
        assert_close_f32(out[sl].cpu().numpy(), last["full"], "gathered fp32")
    return out


# ------------------------------------------------------------------- tiny --
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_tiny_fused_three_steps(cuda, out_dtype):
    w = W.TINY
    c = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed)
    _fused_steps(c, 3, out_dtype)
    c.check_state("tiny fused")
    # padding stays exactly zero
    assert not c.master[w.psi:].any().item()


def test_plain_c_program_drives_the_step(cuda, tmp_path):
    """A C99 program with its own cudaMalloc'd buffers (no Python framework
    between it and the ABI) runs three fused steps of the tiny workload; its
    master, m, v and gathered parameters equal the oracle's, bit for bit."""
    import os
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    lib_dir = os.path.join(root, "zero_sharded_optimizer_device_gb300")
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "c_abi_step")
    # C11 rather than pedantic C99: the CUDA runtime header uses anonymous unions
    cc = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror",
                         "-I", os.path.join(root, "include"), "-I", f"{cuda_home}/include",
                         os.path.join(root, "tests", "c_abi_step.c"), "-L", lib_dir, "-lzero",
                         "-L", f"{cuda_home}/lib64", "-lcudart", f"-Wl,-rpath,{lib_dir}",
                         f"-Wl,-rpath,{cuda_home}/lib64", "-o", exe],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    w = W.TINY
    c = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed)
    P, N, steps = c.info["psi_pad"], w.n_ranks, 3
    grads = c.grads_host(0, 1)                 # the same gradients every step
    header = (np.array([N, steps], np.int32).tobytes() + np.array([P], np.int64).tobytes() +
              np.array([len(w.numels)], np.int32).tobytes() +
              np.array(w.numels, np.int64).tobytes())
    inp = tmp_path / "in.bin"
    inp.write_bytes(header + b"".join(g.astype(np.float32).tobytes() for g in grads) +
                    c.h_master.astype(np.float32).tobytes())
    outp = tmp_path / "out.bin"
    run = subprocess.run([exe, str(inp), str(outp)], capture_output=True, text=True)
    assert run.returncode == 0, (run.returncode, run.stderr)
    raw = outp.read_bytes()
    got = [np.frombuffer(raw[i * 4 * P:(i + 1) * 4 * P], np.float32) for i in range(3)]
    got_out = np.frombuffer(raw[12 * P:], np.uint16)
    master, m, v = c.h_master.copy(), c.h_m.copy(), c.h_v.copy()
    for s in range(1, steps + 1):
        r = O.zero_step(grads, master, m, v, c.groups[0]["shard"], s, c.hp)
        master, m, v = r["master"], r["m"], r["v"]
    for g, want, what in zip(got, (master, m, v), ("master", "m", "v")):
        assert_close_f32(g, want, f"C program {what}")
    assert_bf16(got_out, r["full"], "C program gathered")


def test_plain_c_program_drives_a_stage3_step(cuda, tmp_path):
    """A C11 program with its own cudaMalloc'd buffers and streams runs one
    stage-3 step (per-group fused steps writing owner shards), gathers every
    layer directly and by the two-stream prefetch pass; its master weights,
    layers and the pass's checksums equal the oracle's, bit for bit."""
    import os
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    lib_dir = os.path.join(root, "zero_sharded_optimizer_device_gb300")
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "c_abi_stage3")
    cc = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror",
                         "-I", os.path.join(root, "include"), "-I", f"{cuda_home}/include",
                         os.path.join(root, "tests", "c_abi_stage3.c"), "-L", lib_dir, "-lzero",
                         "-L", f"{cuda_home}/lib64", "-lcudart", f"-Wl,-rpath,{lib_dir}",
                         f"-Wl,-rpath,{cuda_home}/lib64", "-o", exe],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    d, ffn, vocab = 48, 130, 301
    blocks = [[d * d] * 4 + [d * ffn] * 2 + [ffn * d, d, d] for _ in range(2)]
    numels = [vocab * d] + [x for b in blocks for x in b] + [d, vocab * d]
    groups = [0] + [1 + i // 9 for i in range(18)] + [3, 3]
    N = 8
    c = Case(numels, N, 16, "f32", grad_sigma=1e-2, seed=97, groups=groups)
    G, P = len(c.groups), c.info["psi_pad"]
    parts = [np.array([N, len(numels)], np.int32).tobytes(), np.array(numels, np.int64).tobytes(),
             np.array(groups, np.int32).tobytes()]
    for gi in range(G):
        parts += [x.astype(np.float32).tobytes() for x in c.grads_host(gi, 1)]
    parts.append(c.h_master.astype(np.float32).tobytes())
    inp = tmp_path / "in.bin"
    inp.write_bytes(b"".join(parts))
    outp = tmp_path / "out.bin"
    run = subprocess.run([exe, str(inp), str(outp)], capture_output=True, text=True)
    assert run.returncode == 0, (run.returncode, run.stderr)
    raw = outp.read_bytes()
    for gi in reversed(range(G)):
        c.oracle_step(gi, 1)
    assert_close_f32(np.frombuffer(raw[:4 * P], np.float32), c.h_master, "C program master")
    off = 4 * P
    layers = []
    for gi, g in enumerate(c.groups):
        f0, S = g["flat_off"], g["shard"]
        own = [O.f32_to_bf16(c.h_master[f0 + k * S:f0 + (k + 1) * S]) for k in range(N)]
        layers.append(O.gather_layer(own)[0])
        got = np.frombuffer(raw[off:off + 2 * g["psi_pad"]], np.uint16)
        off += 2 * g["psi_pad"]
        assert np.array_equal(got, layers[gi]), gi
    sums = np.frombuffer(raw[off:], np.uint64)
    order = list(range(G)) + list(reversed(range(G)))
    assert len(sums) == len(order)
    for j, gi in enumerate(order):
        assert int(sums[j]) == O.layer_checksum(layers[gi], 1), (j, gi)


def test_tiny_unfused_chain(cuda):
    import torch
    w = W.TINY
    c = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed)
    Z = c.Z
    P = c.info["psi_pad"]
    reduced = torch.empty(P, dtype=torch.float32, device=cuda)
    out32 = torch.empty(P, dtype=torch.float32, device=cuda)
    out16 = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    for s in range(1, 4):
        grads = c.grads_dev(0, s)
        Z.zero_reduce_scatter(c.plan, 0, grads, Z.ZERO_F32, reduced, 0, P, 1.0 / w.n_ranks)
        Z.zero_adam_shard(c.plan, 0, c.master, c.m, c.v, reduced, c.hp_dev(s), None, 0, P,
                          None)
        Z.zero_all_gather(c.plan, 0, c.master, out32, Z.ZERO_F32)
        Z.zero_all_gather(c.plan, -1, c.master, out16, Z.ZERO_BF16)
        r = c.oracle_step(0, s, out_dtype="f32")
        torch.cuda.synchronize()
        assert_close_f32(reduced.cpu().numpy(), np.concatenate(r["reduced"]), f"reduced s{s}")
    c.check_state("tiny unfused")
    assert_close_f32(out32.cpu().numpy(), r["full"], "fp32 gather")
    assert_bf16(bits_of(out16), O.f32_to_bf16(r["full"]), "bf16 gather")


# ------------------------------------------------------ minis of workloads --
@pytest.mark.parametrize("name,scale,steps", [("gpt2-small", 256, 2), ("gpt2-medium", 1024, 2)])
def test_mini_fused(cuda, name, scale, steps):
    w = W.mini(W.ALL[name], scale=scale)
    c = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed)
    _fused_steps(c, steps)
    c.check_state(w.name)


def test_llama_mini_bucketed_with_clip(cuda):
    import torch
    w = W.mini(W.LLAMA_1_4B, scale=1024)
    c = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed,
             heavy_tail=True)
    Z = c.Z
    P = c.info["psi_pad"]
    bucket, chunk = 100_003, 400_001       # ragged windows on purpose
    windows = [(a, min(P, a + bucket)) for a in range(0, P, bucket)]
    npart = [Z.zero_rs_partials(c.plan, Z.ZERO_BF16, b - a) for a, b in windows]
    partials = torch.zeros(sum(npart), dtype=torch.float64, device=cuda)
    reduced = torch.empty(P, dtype=torch.float32, device=cuda)
    norm = torch.zeros(1, dtype=torch.float32, device=cuda)
    coef = torch.zeros(1, dtype=torch.float32, device=cuda)
    out = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    for s in (1, 2):
        grads = c.grads_dev(0, s)
        off = 0
        for (a, b), k in zip(windows, npart):
            Z.zero_reduce_scatter(c.plan, 0, grads, Z.ZERO_BF16, reduced, a, b, 1.0 / w.n_ranks,
                                  partials[off:off + k])
            off += k
        Z.zero_grad_norm(partials, off, 1.0, norm, coef)
        for a in range(0, P, chunk):
            Z.zero_adam_shard(c.plan, 0, c.master, c.m, c.v, reduced, c.hp_dev(s), coef, a,
                              min(P, a + chunk), out, Z.ZERO_BF16)
        # oracle: reduce-scatter, global norm, clip coefficient, step
        local = c.grads_host(0, s)
        red, _, _ = O.ring_reduce_scatter(local, c.groups[0]["shard"])
        onorm, ocoef = O.grad_norm(O.scale(red, np.float32(1.0) / np.float32(w.n_ranks)), 1.0)
        r = c.oracle_step(0, s, clip_coef=ocoef)
        torch.cuda.synchronize()
        assert abs(norm.item() - onorm) <= 1e-6 * onorm, (norm.item(), onorm)
        assert abs(coef.item() - float(ocoef)) <= 1e-6 * float(ocoef)
        assert float(ocoef) < 1.0      # heavy tails: the clip is active
        assert_close_f32(reduced.cpu().numpy(), np.concatenate(red), "reduced")
        # the coefficient may differ in its last bit (fp64 sums in another order)
        exact = coef.item() == float(ocoef)
        c.check_state(f"llama mini step {s}", exact=exact)
        assert_bf16(bits_of(out), r["full"], "gathered", exact=exact)


def test_stage3_mini_step_gather_checksum(cuda):
    import torch
    # Llama-shaped stage-3 list, scaled down: embedding, two blocks, head
    d, ffn, vocab = 64, 172, 500
    blocks = [[d * d] * 4 + [d * ffn] * 2 + [ffn * d, d, d] for _ in range(2)]
    numels = [vocab * d] + blocks[0] + blocks[1] + [d, vocab * d]
    groups = [0] + [1] * 9 + [2] * 9 + [3, 3]
    c = Case(numels, 16, 16, "bf16", seed=77, groups=groups)
    Z = c.Z
    N = 16
    shards = [torch.zeros(c.info["shard_total"], dtype=torch.bfloat16, device=cuda)
              for _ in range(N)]
    for gi in reversed(range(len(c.groups))):
        grads = c.grads_dev(gi, 1)
        Z.zero_step_group(c.plan, gi, grads, Z.ZERO_BF16, c.master, c.m, c.v, c.hp_dev(1), None,
                          shards)
        c.oracle_step(gi, 1)
    torch.cuda.synchronize()
    c.check_state("stage3")
    sums = torch.zeros(len(c.groups), dtype=torch.int64, device=cuda)
    for gi, g in enumerate(c.groups):
        layer = torch.empty(g["psi_pad"], dtype=torch.bfloat16, device=cuda)
        Z.zero_gather_layer(c.plan, gi, shards, Z.ZERO_BF16, layer)
        Z.zero_layer_checksum(layer, g["psi_pad"], 1, sums[gi:gi + 1])
        torch.cuda.synchronize()
        # oracle: each owner's shard is the bf16 cast of its updated master
        f0, S = g["flat_off"], g["shard"]
        own = [O.f32_to_bf16(c.h_master[f0 + k * S:f0 + (k + 1) * S]) for k in range(N)]
        want, sent, recv = O.gather_layer(own)
        assert_bf16(bits_of(layer), want, f"layer {gi}")
        for k in range(N):
            ro = g["rank_off"]
            assert_bf16(bits_of(shards[k][ro:ro + S]), own[k], f"shard {k} group {gi}")
        assert sums[gi].item() % (1 << 64) == O.layer_checksum(want) % (1 << 64) or \
            (sums[gi].item() + (1 << 64)) == O.layer_checksum(want)


# ------------------------------------------------------------- edge cases --
@pytest.mark.parametrize("numels,n,align,gd", [
    ([37], 1, 1, "f32"),                 # one rank: the reduce is a copy
    ([1000, 333, 17], 3, 1, "bf16"),     # generic-N kernel, ragged shards
    ([5, 7, 11, 2001], 5, 3, "f32"),     # shards cut every vector
    ([4096 * 3 + 5], 64, 1, "bf16"),     # N = 64, S not a multiple of 8
    ([8, 8], 2, 8, "bf16"),              # tiny, exactly one vector per shard
    ([10_000, 77], 16, 16, "bf16"),
])
def test_edge_shapes_fused_and_unfused(cuda, numels, n, align, gd):
    import torch
    c = Case(numels, n, align, gd, seed=sum(numels) + n)
    Z = c.Z
    P = c.info["psi_pad"]
    out = torch.zeros(P, dtype=torch.bfloat16, device=cuda)
    grads = c.grads_dev(0, 1)
    Z.zero_step(c.plan, 0, grads, c.zdtype, c.master, c.m, c.v, c.hp_dev(1), None, out,
                Z.ZERO_BF16)
    r = c.oracle_step(0, 1)
    torch.cuda.synchronize()
    c.check_state(f"edge {numels} N={n}")
    assert_bf16(bits_of(out), r["full"], "edge gather")
    # unfused over odd windows reproduces the fused state bit for bit
    master2, m2, v2 = (torch.empty_like(c.master) for _ in range(3))
    master2.copy_(c.master)
    m2.copy_(c.m)
    v2.copy_(c.v)
    reduced = torch.zeros(P, dtype=torch.float32, device=cuda)
    grads = c.grads_dev(0, 2)
    cuts = sorted({0, P, P // 3 + 1, (2 * P) // 3 - 3, min(P, 9)})
    for a, b in zip(cuts, cuts[1:]):
        Z.zero_reduce_scatter(c.plan, 0, grads, c.zdtype, reduced, a, b, 1.0 / n)
        Z.zero_adam_shard(c.plan, 0, master2, m2, v2, reduced, c.hp_dev(2), None, a, b, None)
    Z.zero_step(c.plan, 0, grads, c.zdtype, c.master, c.m, c.v, c.hp_dev(2), None, out,
                Z.ZERO_BF16)
    c.oracle_step(0, 2)
    torch.cuda.synchronize()
    c.check_state("edge step 2")
    assert torch.equal(master2, c.master) and torch.equal(m2, c.m) and torch.equal(v2, c.v)


def test_weight_decay_and_fp32_grads_n8(cuda):
    hp = O.AdamHP(lr=3e-3, weight_decay=0.05)
    c = Case([20_000, 3_003], 8, 16, "f32", grad_sigma=1e-2, seed=5, hp=hp)
    _fused_steps(c, 3)
    c.check_state("wd fp32")


def test_multi_group_unaligned_group_offsets(cuda):
    # N*align = 3: group offsets are not multiples of 8 elements, so the
    # flat-array vectors fall back to element accesses
    import torch
    c = Case([50, 61, 70, 9], 3, 1, "bf16", seed=9, groups=[0, 1, 1, 2])
    assert any(g["flat_off"] % 8 for g in c.groups)
    out = torch.zeros(c.info["psi_pad"], dtype=torch.bfloat16, device=cuda)
    Z = c.Z
    for gi in range(len(c.groups)):
        Z.zero_step(c.plan, gi, c.grads_dev(gi, 1), Z.ZERO_BF16, c.master, c.m, c.v,
                    c.hp_dev(1), None, out, Z.ZERO_BF16)
        c.oracle_step(gi, 1)
    torch.cuda.synchronize()
    c.check_state("multi-group")
    assert_bf16(bits_of(out), O.f32_to_bf16(c.h_master), "multi-group gather")


def test_empty_plan_and_empty_window_are_noops(cuda):
    import torch
    import zero_sharded_optimizer_device_gb300 as Z
    p = Z.zero_plan([], 4, 16)
    x = torch.zeros(16, device=cuda)
    grads = [torch.zeros(16, device=cuda) for _ in range(4)]
    Z.zero_step(p, 0, grads, Z.ZERO_F32, x, x, x, Z.adam_hp(1, 0.25), None, None)
    # an empty stage-3 group (its tensors have no elements): gathers write nothing
    pe = Z.zero_plan([64, 0, 64], 4, 16, [0, 1, 2])
    assert Z.zero_plan_group(pe, 1)["psi_pad"] == 0
    sh = [torch.zeros(64, dtype=torch.bfloat16, device=cuda) for _ in range(4)]
    canary = torch.full((16,), 3.0, dtype=torch.bfloat16, device=cuda)
    Z.zero_gather_layer(pe, 1, sh, Z.ZERO_BF16, canary)
    Z.zero_broadcast_layer(pe, 1, sh, Z.ZERO_BF16, canary)
    torch.cuda.synchronize()
    assert bool((canary == 3.0).all())
    c = Case([100], 4, 1, "f32", seed=3)
    before = c.master.clone()
    red = torch.full((c.info["psi_pad"],), 7.0, device=cuda)
    Z.zero_reduce_scatter(c.plan, 0, c.grads_dev(0, 1), Z.ZERO_F32, red, 50, 50, 0.25)
    Z.zero_adam_shard(c.plan, 0, c.master, c.m, c.v, red, c.hp_dev(1), None, 10, 10, None)
    torch.cuda.synchronize()
    assert torch.equal(before, c.master) and bool((red == 7.0).all())


def test_outputs_stay_inside_their_buffers(cuda):
    """Guard bands: 256 canary bytes before and after every output buffer
    stay untouched by every call."""
    import torch
    c = Case([1000, 337], 4, 1, "bf16", seed=21)
    Z = c.Z
    P = c.info["psi_pad"]
    G = 64  # canary floats on each side

    def guarded(n, dtype):
        words = (n * (2 if dtype == torch.bfloat16 else 4) + 3) // 4
        buf = torch.full((words + 2 * G,), -12345.0, dtype=torch.float32, device=cuda)
        inner = buf[G:G + words].view(dtype)[:n]
        return buf, inner

    bufs = {}
    bufs["master"], master = guarded(P, torch.float32)
    bufs["m"], m = guarded(P, torch.float32)
    bufs["v"], v = guarded(P, torch.float32)
    bufs["red"], red = guarded(P, torch.float32)
    bufs["out"], out = guarded(P, torch.bfloat16)
    master.copy_(c.master)
    m.zero_()
    v.zero_()
    grads = c.grads_dev(0, 1)
    Z.zero_reduce_scatter(c.plan, 0, grads, Z.ZERO_BF16, red, 3, P - 5, 0.25)
    Z.zero_step(c.plan, 0, grads, Z.ZERO_BF16, master, m, v, c.hp_dev(1), None, out, Z.ZERO_BF16)
    Z.zero_adam_shard(c.plan, 0, master, m, v, red, c.hp_dev(2), None, 1, P - 1, out, Z.ZERO_BF16)
    Z.zero_all_gather(c.plan, 0, master, out, Z.ZERO_BF16)
    torch.cuda.synchronize()
    for name, b in bufs.items():
        assert bool((b[:G] == -12345.0).all()) and bool((b[-G:] == -12345.0).all()), name


def test_windowed_calls_write_only_their_window(cuda):
    """Reduce-scatter (store and accumulate), Adam and the fused step on a
    window [a, b) leave every element of their flat outputs outside it as it
    was; norm partials are written only in [0, zero_rs_partials)."""
    import torch
    c = Case([5000, 1337, 21], 4, 1, "bf16", seed=23, host_state=False)
    Z = c.Z
    P = c.info["psi_pad"]
    a, b = 1003, P - 997                      # ragged: cuts 8-element vectors on both ends
    grads = c.grads_dev(0, 1)
    mark = -12345.0

    def flat(dtype=torch.float32):
        return torch.full((P,), mark, dtype=dtype, device=cuda)

    def untouched(t, what):
        fill = torch.tensor(mark, dtype=t.dtype, device=cuda)   # the mark in t's dtype
        outside = torch.cat([t[:a], t[b:]])
        assert bool((outside == fill).all()), what
        assert not bool((t[a:b] == fill).any()), what + " (window not written)"

    red = flat()
    k = Z.zero_rs_partials(c.plan, Z.ZERO_BF16, b - a)
    part = torch.full((k + 64,), mark, dtype=torch.float64, device=cuda)
    Z.zero_reduce_scatter(c.plan, 0, grads, Z.ZERO_BF16, red, a, b, 0.25, part)
    torch.cuda.synchronize()
    untouched(red, "reduce-scatter")
    assert bool((part[k:] == mark).all()) and not bool((part[:k] == mark).any())
    Z.zero_reduce_scatter_acc(c.plan, 0, grads, Z.ZERO_BF16, red, a, b, 0.25)
    torch.cuda.synchronize()
    untouched(red, "accumulate")
    master, m, v = flat(), flat(), flat()
    master[a:b] = 0.5
    m[a:b] = 0.0
    v[a:b] = 0.0
    out = flat(torch.bfloat16)
    Z.zero_adam_shard(c.plan, 0, master, m, v, red, c.hp_dev(1), None, a, b, out, Z.ZERO_BF16)
    torch.cuda.synchronize()
    for t, name in ((master, "adam master"), (m, "adam m"), (v, "adam v"), (out, "adam out")):
        untouched(t, name)
    out32 = flat()
    Z.zero_all_gather(c.plan, 0, master, out32, Z.ZERO_F32)
    torch.cuda.synchronize()
    assert torch.equal(out32[a:b], master[a:b])


def test_stage3_outputs_stay_inside_their_buffers(cuda):
    """Guard bands around every rank's shard buffer, the layer buffer, the
    checksum word and the norm outputs: untouched by the stage-3 step, the
    gather, the consumer and the norm."""
    import torch
    numels = [700, 33, 1200, 5, 810]
    c = Case(numels, 5, 1, "bf16", seed=29, groups=[0, 0, 1, 1, 2], host_state=False)
    Z = c.Z
    G = 64

    def guarded(n, dtype):
        words = (n * (2 if dtype == torch.bfloat16 else (8 if dtype == torch.int64 else 4)) + 3) // 4
        buf = torch.full((words + 2 * G,), -12345.0, dtype=torch.float32, device=cuda)
        return buf, buf[G:G + words].view(dtype)[:n]

    sh = [guarded(c.info["shard_total"], torch.bfloat16) for _ in range(5)]
    shards = [x[1] for x in sh]
    for x in shards:
        x.zero_()
    for gi in reversed(range(len(c.groups))):
        Z.zero_step_group(c.plan, gi, c.grads_dev(gi, 1), Z.ZERO_BF16, c.master, c.m, c.v,
                          c.hp_dev(1), None, shards)
    gmax = max(g["psi_pad"] for g in c.groups)
    lb, layer = guarded(gmax, torch.bfloat16)
    sb, word = guarded(1, torch.int64)
    nb, norm = guarded(1, torch.float32)
    cb, coef = guarded(1, torch.float32)
    part = torch.ones(10, dtype=torch.float64, device=cuda)
    for gi, g in enumerate(c.groups):
        Z.zero_gather_layer(c.plan, gi, shards, Z.ZERO_BF16, layer[:g["psi_pad"]])
        Z.zero_layer_checksum(layer, g["psi_pad"], 3, word)
    Z.zero_grad_norm(part, 10, 1.0, norm, coef)
    torch.cuda.synchronize()
    for name, (b, _) in [("layer", (lb, None)), ("checksum", (sb, None)), ("norm", (nb, None)),
                         ("coef", (cb, None))] + [(f"shards {r}", sh[r]) for r in range(5)]:
        assert bool((b[:G] == -12345.0).all()) and bool((b[-G:] == -12345.0).all()), name


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n,align", [(16, 16), (4, 8), (5, 4), (3, 3), (7, 1)])
def test_gather_layer_every_path(cuda, dtype, n, align):
    """zero_gather_layer and its broadcast form zero_broadcast_layer on bf16
    and fp32 shard buffers, through the bulk-copy form (shard starts and
    lengths multiples of 16 bytes) and the element form (otherwise): the
    layer equals the oracle's all-gather and broadcast results (the
    concatenation of the owners' shards), bit for bit, with guard bands
    around it."""
    import torch
    rng = np.random.default_rng(1000 * n + align + (7 if dtype == "f32" else 0))
    numels = [int(x) for x in rng.integers(1, 40_000, 6)]
    groups = [0, 0, 1, 2, 2, 3]
    p = O.plan(numels, n, align, groups)
    Z = pytest.importorskip("zero_sharded_optimizer_device_gb300")
    zp = Z.zero_plan(numels, n, align, groups)
    tdt, ndt = (torch.int16, np.uint16) if dtype == "bf16" else (torch.int32, np.uint32)
    zdt = Z.ZERO_BF16 if dtype == "bf16" else Z.ZERO_F32
    host = [rng.integers(0, np.iinfo(ndt).max, p.shard_total, dtype=np.uint64).astype(ndt)
            for _ in range(n)]
    shards = [torch.from_numpy(h.view(np.int16 if dtype == "bf16" else np.int32)).to(cuda)
              for h in host]
    G = 64
    for gi, g in enumerate(p.groups):
        own = [h[g.rank_off:g.rank_off + g.shard] for h in host]
        want, _, _ = O.gather_layer(own)
        want_b, _, _, _ = O.broadcast_gather(own)
        for call, ref in ((Z.zero_gather_layer, want), (Z.zero_broadcast_layer, want_b)):
            buf = torch.full((g.psi_pad + 2 * G,), -7, dtype=tdt, device=cuda)
            call(zp, gi, shards, zdt, buf[G:G + g.psi_pad])
            torch.cuda.synchronize()
            got = buf.cpu().numpy().view(ndt)
            assert np.array_equal(got[G:G + g.psi_pad], ref), (call.__name__, gi, n, align, dtype)
            assert (buf[:G] == -7).all() and (buf[G + g.psi_pad:] == -7).all(), (gi, "guard")


@pytest.mark.parametrize("n,pieces", [(2, 1), (2, 150), (3, 304), (16, 305), (16, 1000),
                                      (5, 2999)])
@pytest.mark.parametrize("ctas", [1, 2, 8])
def test_bulk_gather_piece_walk(cuda, n, pieces, ctas):
    """The bulk-copy gather's CTAs walk their pieces (8 KiB, every G-th) with
    a cursor over owners and groups: per-owner piece counts below, at and
    above the grid (1 to 8 CTAs per SM), a ragged last piece per owner, and
    the broadcast form; every layer equals the plain concatenation of the
    owners' shards (torch.cat), bit for bit."""
    import torch
    Z = pytest.importorskip("zero_sharded_optimizer_device_gb300")
    S = pieces * 4096 - 8                        # bf16 elements per owner
    zp = Z.zero_plan([n * S - 3, 3], n, 8)
    assert Z.zero_plan_group(zp, 0)["shard"] == S
    gen = torch.Generator(device=cuda).manual_seed(n * 7919 + pieces)
    shards = [torch.randint(-32768, 32767, (S,), dtype=torch.int16, device=cuda, generator=gen)
              for _ in range(n)]
    want = torch.cat(shards)
    prev = Z.zero_set_occupancy(Z.ZERO_OCC_GATHER, ctas)
    try:
        for call in (Z.zero_gather_layer, Z.zero_broadcast_layer):
            out = torch.full((n * S + 64,), 5, dtype=torch.int16, device=cuda)
            call(zp, 0, shards, Z.ZERO_BF16, out)
            torch.cuda.synchronize()
            assert torch.equal(out[:n * S], want), call.__name__
            assert bool((out[n * S:] == 5).all())
    finally:
        Z.zero_set_occupancy(Z.ZERO_OCC_GATHER, prev)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n,align", [(16, 16), (8, 1), (5, 3)])
def test_gather_groups_per_parameter(cuda, dtype, n, align):
    """Per-parameter partitioning (every tensor its own group): zero_gather_groups
    over a module's tensors, in random subsets and orders with repeats,
    equals each tensor's own gather, bit for bit; mixed bulk-copy and
    element-wise groups in one call; guard bands around every output."""
    import torch
    rng = np.random.default_rng(77 * n + align + (5 if dtype == "f32" else 0))
    numels = [int(x) for x in rng.integers(1, 30_000, 12)] + [0, 7]
    groups = list(range(len(numels)))
    p = O.plan(numels, n, align, groups)
    Z = pytest.importorskip("zero_sharded_optimizer_device_gb300")
    zp = Z.zero_plan(numels, n, align, groups)
    tdt, ndt = (torch.int16, np.uint16) if dtype == "bf16" else (torch.int32, np.uint32)
    zdt = Z.ZERO_BF16 if dtype == "bf16" else Z.ZERO_F32
    host = [rng.integers(0, np.iinfo(ndt).max, p.shard_total, dtype=np.uint64).astype(ndt)
            for _ in range(n)]
    shards = [torch.from_numpy(h.view(np.int16 if dtype == "bf16" else np.int32)).to(cuda)
              for h in host]
    G = 64
    for trial in range(4):
        pick = [int(x) for x in rng.integers(0, len(groups), int(rng.integers(1, 20)))]
        bufs = [torch.full((p.groups[g].psi_pad + 2 * G,), -7, dtype=tdt, device=cuda)
                for g in pick]
        Z.zero_gather_groups(zp, pick, shards, zdt, [b[G:] for b in bufs])
        torch.cuda.synchronize()
        for g, b in zip(pick, bufs):
            gi = p.groups[g]
            got = b.cpu().numpy().view(ndt)
            want, _, _ = O.gather_layer([h[gi.rank_off:gi.rank_off + gi.shard] for h in host])
            assert np.array_equal(got[G:G + gi.psi_pad], want), (trial, g)
            assert (b[:G] == -7).all() and (b[G + gi.psi_pad:] == -7).all(), (trial, g)


def test_gather_groups_and_consumer_at_their_limits(cuda):
    """ZERO_MAX_COALESCE groups in one zero_gather_groups call, and the
    consumer at ZERO_MAX_CONSUMER_ROUNDS rounds, against the oracle."""
    import torch
    Z = pytest.importorskip("zero_sharded_optimizer_device_gb300")
    rng = np.random.default_rng(64)
    n, k = 4, Z.ZERO_MAX_COALESCE
    numels = [int(x) for x in rng.integers(1, 3000, k + 6)]
    groups = list(range(len(numels)))
    p = O.plan(numels, n, 16, groups)
    zp = Z.zero_plan(numels, n, 16, groups)
    host = [rng.integers(0, 1 << 16, p.shard_total, dtype=np.uint64).astype(np.uint16)
            for _ in range(n)]
    shards = [torch.from_numpy(h.view(np.int16)).to(cuda) for h in host]
    pick = [int(x) for x in rng.permutation(len(numels))[:k]]
    outs = [torch.empty(p.groups[g].psi_pad, dtype=torch.int16, device=cuda) for g in pick]
    Z.zero_gather_groups(zp, pick, shards, Z.ZERO_BF16, outs)
    sums = torch.zeros(1, dtype=torch.int64, device=cuda)
    Z.zero_layer_checksum(outs[0], p.groups[pick[0]].psi_pad, Z.ZERO_MAX_CONSUMER_ROUNDS, sums)
    torch.cuda.synchronize()
    for g, o in zip(pick, outs):
        gi = p.groups[g]
        want, _, _ = O.gather_layer([h[gi.rank_off:gi.rank_off + gi.shard] for h in host])
        assert np.array_equal(o.cpu().numpy().view(np.uint16), want), g
    want0, _, _ = O.gather_layer([h[p.groups[pick[0]].rank_off:p.groups[pick[0]].rank_off +
                                    p.groups[pick[0]].shard] for h in host])
    assert int(sums.item()) % (1 << 64) == O.layer_checksum(want0, Z.ZERO_MAX_CONSUMER_ROUNDS)


# ------------------------------------------------ full size, sampled windows --
def test_gpt2_small_full_size_sampled(cuda):
    """The workload the benchmark times (fused zero_step, N=8, bf16 grads),
    5 steps at full size; sampled windows across every owner boundary and a
    sample of tensor edges are recomputed by the oracle from generated
    inputs."""
    import torch
    w = W.GPT2_SMALL
    c = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed,
             host_state=False)
    Z = c.Z
    P, S = c.info["psi_pad"], c.groups[0]["shard"]
    assert P == 124_439_808 and S == 15_554_976
    out = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    grads = None
    for s in range(1, w.steps + 1):
        grads = c.grads_dev(0, s, grads)
        Z.zero_step(c.plan, 0, grads, Z.ZERO_BF16, c.master, c.m, c.v, c.hp_dev(s), None, out,
                    Z.ZERO_BF16)
    torch.cuda.synchronize()
    cuts = [k * S for k in range(1, w.n_ranks)] + np.cumsum(w.numels)[:-1].tolist()[::11]
    for a, b in boundary_windows(P, cuts, 4096):
        r = c.oracle_window(0, (a, b), range(1, w.steps + 1))
        c.check_window(0, (a, b), r, f"gpt2-small [{a},{b})")
        assert_bf16(bits_of(out[a:b]), r["full"], f"gathered [{a},{b})")


def test_gpt2_small_full_size_fp32_gradients_sampled(cuda):
    """The benchmark's fp32-gradient line (GPT-2-small, N=8, `--grad-dtype
    f32`: the 32-byte load path of the fused step), 3 steps at full size,
    sampled windows across every owner boundary and tensor edges."""
    import torch
    w = W.GPT2_SMALL
    c = Case(w.numels, w.n_ranks, w.align, "f32", w.grad_sigma, w.master_sigma, w.seed,
             host_state=False)
    Z = c.Z
    P, S = c.info["psi_pad"], c.groups[0]["shard"]
    out = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    grads = None
    for s in range(1, 4):
        grads = c.grads_dev(0, s, grads)
        Z.zero_step(c.plan, 0, grads, Z.ZERO_F32, c.master, c.m, c.v, c.hp_dev(s), None, out,
                    Z.ZERO_BF16)
    torch.cuda.synchronize()
    cuts = [k * S for k in range(1, w.n_ranks)] + np.cumsum(w.numels)[:-1].tolist()[::13]
    for a, b in boundary_windows(P, cuts, 2048):
        r = c.oracle_window(0, (a, b), range(1, 4))
        c.check_window(0, (a, b), r, f"gpt2-small fp32 grads [{a},{b})")
        assert_bf16(bits_of(out[a:b]), r["full"], f"gathered [{a},{b})")


def test_zero_copy_host_buffers_match_device_buffers(cuda):
    """Pinned host buffers mapped into the device address space may be
    passed straight to zero_step (the kernel then moves the data over the
    host link): same results, bit for bit, as device-resident buffers."""
    import torch
    import bench
    w = W.mini(W.GPT2_SMALL, scale=64)
    c = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed,
             host_state=False)
    Z = c.Z
    P = c.info["psi_pad"]
    grads = c.grads_dev(0, 1)
    h_grads = [torch.empty(P, dtype=torch.bfloat16, pin_memory=True) for _ in range(c.n)]
    for h, d in zip(h_grads, grads):
        h.copy_(d)
    h_out = torch.zeros(P, dtype=torch.bfloat16, pin_memory=True)
    if not all(bench.host_mapped(x) for x in h_grads + [h_out]):
        pytest.skip("pinned host memory is not mapped into the device address space")
    master2, m2, v2 = c.master.clone(), c.m.clone(), c.v.clone()
    out = torch.zeros(P, dtype=torch.bfloat16, device=cuda)
    Z.zero_step(c.plan, 0, grads, Z.ZERO_BF16, c.master, c.m, c.v, c.hp_dev(1), None, out,
                Z.ZERO_BF16)
    Z.zero_step(c.plan, 0, h_grads, Z.ZERO_BF16, master2, m2, v2, c.hp_dev(1), None, h_out,
                Z.ZERO_BF16)
    torch.cuda.synchronize()
    assert torch.equal(master2, c.master) and torch.equal(m2, c.m) and torch.equal(v2, c.v)
    assert torch.equal(h_out, out.cpu())


def test_zero_copy_stage3_slot_and_shards_match_device_buffers(cuda):
    """The end-to-end form of the stage-3 step: every group's N gradient
    buffers are prefixes of one mapped page-locked host slot, and the owners'
    bf16 shards are written to mapped host buffers over the link.  The state
    and shards equal, bit for bit, those of the same step from device
    buffers, and the oracle's."""
    import torch
    import bench
    w = W.mini(W.LLAMA_7B_STAGE3, scale=4096)
    c = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed,
             groups=w.groups)
    Z = c.Z
    N, G, ST = c.n, len(c.groups), c.info["shard_total"]
    gmax = max(g["psi_pad"] for g in c.groups)
    h_slot = [torch.zeros(gmax, dtype=torch.bfloat16, pin_memory=True) for _ in range(N)]
    h_shards = [torch.zeros(ST, dtype=torch.bfloat16, pin_memory=True) for _ in range(N)]
    if not all(bench.host_mapped(x) for x in h_slot + h_shards):
        pytest.skip("pinned host memory is not mapped into the device address space")
    d_slot = [torch.zeros(gmax, dtype=torch.bfloat16, device=cuda) for _ in range(N)]
    d_shards = [torch.zeros(ST, dtype=torch.bfloat16, device=cuda) for _ in range(N)]
    master2, m2, v2 = c.master.clone(), c.m.clone(), c.v.clone()
    for gi in reversed(range(G)):
        g = c.groups[gi]
        views = [t[:g["psi_pad"]] for t in d_slot]
        c.grads_dev(gi, 1, views)
        torch.cuda.synchronize()
        for h, d in zip(h_slot, d_slot):
            h.copy_(d)
        h_views = [t[:g["psi_pad"]] for t in h_slot]
        Z.zero_step_group(c.plan, gi, views, Z.ZERO_BF16, c.master, c.m, c.v, c.hp_dev(1), None,
                          d_shards)
        Z.zero_step_group(c.plan, gi, h_views, Z.ZERO_BF16, master2, m2, v2, c.hp_dev(1), None,
                          h_shards)
        torch.cuda.synchronize()
        c.oracle_step(gi, 1)
    assert torch.equal(master2, c.master) and torch.equal(m2, c.m) and torch.equal(v2, c.v)
    for h, d in zip(h_shards, d_shards):
        assert torch.equal(h, d.cpu())
    c.check_state("stage 3 from host buffers")


def test_large_step_numbers(cuda):
    """Step numbers where 1 - beta^t has reached 1 in fp32 (and beta1^t has
    underflowed): the bias corrections agree with the oracle's."""
    import torch
    c = Case([5_000, 333], 4, 16, "f32", grad_sigma=1e-2, seed=8)
    Z = c.Z
    out = torch.empty(c.info["psi_pad"], dtype=torch.bfloat16, device=cuda)
    for t in (10_000, 100_000, 1_000_001):
        Z.zero_step(c.plan, 0, c.grads_dev(0, t), Z.ZERO_F32, c.master, c.m, c.v, c.hp_dev(t),
                    None, out, Z.ZERO_BF16)
        r = c.oracle_step(0, t)
    torch.cuda.synchronize()
    c.check_state("large t")
    assert_bf16(bits_of(out), r["full"], "large t gathered")


def test_stage3_unaligned_shards(cuda):
    """align = 1 with N = 3: shard sizes and rank offsets are not multiples
    of 8, so the step writes owner shards element by element and the gather
    copies element by element."""
    import torch
    numels = [101, 57, 33, 1000, 7]
    groups = [0, 0, 1, 1, 2]
    c = Case(numels, 3, 1, "bf16", seed=13, groups=groups)
    Z = c.Z
    assert any(g["shard"] % 8 or g["rank_off"] % 8 for g in c.groups)
    shards = [torch.zeros(c.info["shard_total"], dtype=torch.bfloat16, device=cuda)
              for _ in range(3)]
    for gi in range(len(c.groups)):
        Z.zero_step_group(c.plan, gi, c.grads_dev(gi, 1), Z.ZERO_BF16, c.master, c.m, c.v,
                          c.hp_dev(1), None, shards)
        c.oracle_step(gi, 1)
    torch.cuda.synchronize()
    c.check_state("stage3 align 1")
    for gi, g in enumerate(c.groups):
        layer = torch.empty(g["psi_pad"], dtype=torch.bfloat16, device=cuda)
        Z.zero_gather_layer(c.plan, gi, shards, Z.ZERO_BF16, layer)
        torch.cuda.synchronize()
        f0 = g["flat_off"]
        assert_bf16(bits_of(layer), O.f32_to_bf16(c.h_master[f0:f0 + g["psi_pad"]]),
                    f"group {gi}")


@pytest.mark.parametrize("sigma", [1e-21, 1e-30, 3e18, 1e21])
def test_subnormal_and_overflowing_moments_match_the_oracle(cuda, sigma):
    """Gradient scales whose squares are subnormal (1e-21), underflow to zero
    (1e-30), stay large but finite (3e18) or overflow fp32 (1e21) take
    the same IEEE path on the GPU as in the oracle: no flush to zero, the
    same infinities, bit for bit over three steps."""
    import torch
    c = Case([5000, 123], 8, 16, "f32", grad_sigma=sigma, seed=23)
    Z = c.Z
    out = torch.empty(c.info["psi_pad"], dtype=torch.float32, device=cuda)
    r = None
    for s in range(1, 4):
        Z.zero_step(c.plan, 0, c.grads_dev(0, s), Z.ZERO_F32, c.master, c.m, c.v, c.hp_dev(s),
                    None, out, Z.ZERO_F32)
        with np.errstate(over="ignore", invalid="ignore"):
            r = c.oracle_step(0, s, out_dtype="f32")
    torch.cuda.synchronize()
    v = c.v.cpu().numpy()
    if sigma == 1e-21:
        assert ((v > 0) & (v < np.finfo(np.float32).tiny)).any()   # subnormals reached
    if sigma == 1e-30:
        assert (v == 0).all()                                    # g*g underflows to zero
    if sigma > 1e20:
        assert np.isinf(v).any()
    c.check_state(f"sigma {sigma}")
    got = out.cpu().numpy()
    same = (got.view(np.uint32) == r["full"].view(np.uint32)) | (np.isnan(got) & np.isnan(r["full"]))
    assert same.all()


@pytest.mark.parametrize("gd", ["f32", "bf16"])
def test_non_finite_gradients_propagate_like_the_oracle(cuda, gd):
    """A NaN or an infinity in one rank's gradient (fp32 or bf16) poisons
    exactly the elements it touches, on both sides; every other element stays
    bit-identical to the oracle."""
    import torch
    c = Case([4096], 4, 16, gd, grad_sigma=1e-2, seed=17)
    Z = c.Z
    grads = c.grads_dev(0, 1)
    bad = {10: float("nan"), 777: float("inf"), 2048: float("-inf")}
    for i, x in bad.items():
        grads[i % 4][i] = x
    out = torch.empty(c.info["psi_pad"], dtype=torch.bfloat16, device=cuda)
    Z.zero_step(c.plan, 0, grads, c.zdtype, c.master, c.m, c.v, c.hp_dev(1), None, out,
                Z.ZERO_BF16)
    local = c.grads_host(0, 1)
    for i, x in bad.items():
        local[i % 4][i] = np.float32(x)
    with np.errstate(invalid="ignore"):          # inf/inf on the poisoned elements
        r = O.zero_step(local, c.h_master, c.h_m, c.h_v, c.groups[0]["shard"], 1, c.hp)
    torch.cuda.synchronize()
    got = c.master.cpu().numpy()
    nan_g, nan_w = np.isnan(got), np.isnan(r["master"])
    assert np.array_equal(nan_g, nan_w) and nan_w[list(bad)].all()
    ok = ~nan_w
    assert_close_f32(got[ok], r["master"][ok], "finite master")
    assert_close_f32(c.m.cpu().numpy()[ok], r["m"][ok], "finite m")
    ob = bits_of(out)
    assert_bf16(ob[ok], r["full"][ok], "finite gathered")
    assert np.isnan(O.bf16_to_f32(ob[nan_w])).all()


def test_bf16_cast_of_special_values_on_the_gpu(cuda):
    """The GPU's fp32 -> bf16 casts (all-gather, and the fused step with zero
    gradients, which leaves the master unchanged) agree bit for bit with the
    oracle's round-to-nearest-even on ties, carries into the exponent,
    signed zeros, subnormals, infinities, the largest finite values and
    NaNs."""
    import torch
    rng = np.random.default_rng(5)
    hi = rng.integers(0, 1 << 16, 4096, dtype=np.uint64).astype(np.uint32) << 16
    special = np.array([0x00000000, 0x80000000, 0x00000001, 0x807FFFFF, 0x7F7FFFFF, 0xFF7FFFFF,
                        0x7F7F8000, 0x3F808000, 0x3F818000, 0x3FFF8000, 0x7F800000, 0xFF800000,
                        0x7FC00000, 0x7F800001, 0xFFC12345, 0x3F800001, 0x3F807FFF],
                       dtype=np.uint32)
    bits = np.concatenate([hi | 0x8000, hi | 0x7FFF, hi | 0x8001, special])   # ties, below, above
    c = Case([bits.size], 4, 16, "f32", seed=3, host_state=False)
    Z = c.Z
    P = c.info["psi_pad"]
    host = np.zeros(P, np.uint32)
    host[:bits.size] = bits
    c.master.copy_(torch.from_numpy(host.view(np.int32)).to(cuda).view(torch.float32))
    out = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    Z.zero_all_gather(c.plan, 0, c.master, out, Z.ZERO_BF16)
    torch.cuda.synchronize()
    want = O.f32_to_bf16(host.view(np.float32))
    got = bits_of(out)
    nan = np.isnan(host.view(np.float32))
    assert np.array_equal(got[~nan], want[~nan])
    assert np.isnan(O.bf16_to_f32(got[nan])).all()
    zeros = [torch.zeros(P, dtype=torch.float32, device=cuda) for _ in range(4)]
    out2 = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    Z.zero_step(c.plan, 0, zeros, Z.ZERO_F32, c.master, c.m, c.v, c.hp_dev(1), None, out2,
                Z.ZERO_BF16)
    torch.cuda.synchronize()
    mb = bits_of(c.master)                                  # zero gradients: master unchanged
    assert np.array_equal(mb[~nan], host[~nan]) and np.isnan(mb.view(np.float32)[nan]).all()
    got2 = bits_of(out2)
    assert np.array_equal(got2[~nan], want[~nan]) and np.isnan(O.bf16_to_f32(got2[nan])).all()


def test_zero_gradients_leave_parameters_unchanged(cuda):
    import torch
    c = Case([3000, 17], 8, 16, "bf16", seed=19, host_state=False)
    Z = c.Z
    grads = [torch.zeros(c.info["psi_pad"], dtype=torch.bfloat16, device=cuda) for _ in range(8)]
    before = c.master.clone()
    out = torch.empty(c.info["psi_pad"], dtype=torch.bfloat16, device=cuda)
    Z.zero_step(c.plan, 0, grads, Z.ZERO_BF16, c.master, c.m, c.v, c.hp_dev(1), None, out,
                Z.ZERO_BF16)
    torch.cuda.synchronize()
    assert torch.equal(before, c.master) and not c.m.any() and not c.v.any()
    assert torch.equal(out, before.to(torch.bfloat16))
