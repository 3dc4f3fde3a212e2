"""Seeded sweep over rank counts and gradient dtypes: every specialised kernel
instance (N = 1, 2, 4, 8, 16, 32, 64) and the generic one (N = 3, 5, 12, 33),
bf16 and fp32 gradients, random tensor lists, alignments, windows and buffer
offsets.  Each case runs a fused step, an unfused step (windowed
reduce-scatter with norm partials, device norm, chunked Adam) and a second
fused step, and compares every result with the oracle element by element."""
import numpy as np
import pytest

from oracle import zero_oracle as O

from harness import Case, assert_bf16, assert_close_f32, bits_of

pytestmark = pytest.mark.gpu

RANKS = [1, 2, 3, 4, 5, 8, 12, 16, 32, 33, 64]


def _windows(rng, P, k):
    """[a, b) windows covering [0, P), cut at k random interior points."""
    inner = [int(x) for x in rng.integers(1, P, size=k)] if P > 1 else []
    edges = sorted({0, P, *inner})
    return list(zip(edges[:-1], edges[1:]))


def _out(torch, P, out_f32, dev):
    return torch.zeros(P, dtype=torch.float32 if out_f32 else torch.bfloat16, device=dev)


def _check_out(out, r, out_f32, what):
    if out_f32:
        assert_close_f32(out.cpu().numpy(), r["full"], what)
    else:
        assert_bf16(bits_of(out), r["full"], what)


@pytest.mark.parametrize("gd", ["bf16", "f32"])
@pytest.mark.parametrize("n", RANKS)
def test_rank_count_sweep(cuda, n, gd):
    import torch
    rng = np.random.default_rng(7919 * n + (1 if gd == "f32" else 0))
    align = int(rng.choice([1, 2, 3, 4, 8, 16]))
    budget = max(4_000, 1_500_000 // n)          # oracle work grows with N * psi
    total = int(rng.integers(budget // 4, budget))
    weights = rng.dirichlet(np.full(int(rng.integers(1, 6)), 0.5))
    numels = [1 + int(total * x) for x in weights]  # several tiles, ragged, some tiny
    c = Case(numels, n, align, gd, grad_sigma=1e-2 if gd == "f32" else 1e-3,
             seed=int(rng.integers(1, 1 << 30)), heavy_tail=bool(rng.integers(0, 2)))
    Z = c.Z
    P = c.info["psi_pad"]
    out_f32 = bool(rng.integers(0, 2))
    zo, odt = (Z.ZERO_F32, "f32") if out_f32 else (Z.ZERO_BF16, "bf16")
    what = f"N={n} {gd} align={align} numels={numels} out={odt}"

    # gradient buffers, optionally starting 16 bytes into their allocation
    # (fp32: the two-load path instead of the 32-byte one)
    shift = 16 // (4 if gd == "f32" else 2) if rng.integers(0, 2) else 0
    bufs = [torch.empty(P + 8, dtype=c.tdtype, device=cuda) for _ in range(n)]
    grads = [b[shift:shift + P] for b in bufs]

    # step 1: fused
    out = _out(torch, P, out_f32, cuda)
    c.grads_dev(0, 1, grads)
    Z.zero_step(c.plan, 0, grads, c.zdtype, c.master, c.m, c.v, c.hp_dev(1), None, out, zo)
    r = c.oracle_step(0, 1, out_dtype=odt)
    torch.cuda.synchronize()
    c.check_state(what + " fused step 1")
    _check_out(out, r, out_f32, what + " fused step 1 gathered")

    # step 2: windowed reduce-scatter with norm partials, norm, chunked Adam
    c.grads_dev(0, 2, grads)
    windows = _windows(rng, P, 3)
    chunks = _windows(rng, P, 2)
    npart = [Z.zero_rs_partials(c.plan, c.zdtype, b - a) for a, b in windows]
    partials = torch.zeros(max(1, sum(npart)), dtype=torch.float64, device=cuda)
    reduced = torch.zeros(P, dtype=torch.float32, device=cuda)
    norm = torch.zeros(1, dtype=torch.float32, device=cuda)
    coef = torch.zeros(1, dtype=torch.float32, device=cuda)
    off = 0
    for (a, b), k in zip(windows, npart):
        Z.zero_reduce_scatter(c.plan, 0, grads, c.zdtype, reduced, a, b, 1.0 / n,
                              partials[off:off + k])
        off += k
    Z.zero_grad_norm(partials, off, 1e30, norm, coef)          # no clipping: coef = 1
    out = _out(torch, P, out_f32, cuda)
    for a, b in chunks:
        Z.zero_adam_shard(c.plan, 0, c.master, c.m, c.v, reduced, c.hp_dev(2), coef, a, b,
                          out, zo)
    r = c.oracle_step(0, 2, out_dtype=odt)
    onorm, ocoef = O.grad_norm(r["g"], 1e30)
    torch.cuda.synchronize()
    assert_close_f32(reduced.cpu().numpy(), np.concatenate(r["reduced"]), what + " reduced")
    assert abs(norm.item() - onorm) <= 1e-6 * onorm, (what, norm.item(), onorm)
    assert coef.item() == float(ocoef) == 1.0
    c.check_state(what + " unfused step 2")
    _check_out(out, r, out_f32, what + " unfused step 2 gathered")
    # the all-gather alone, in the other output dtype
    other = _out(torch, P, not out_f32, cuda)
    Z.zero_all_gather(c.plan, 0, c.master, other, Z.ZERO_BF16 if out_f32 else Z.ZERO_F32)
    torch.cuda.synchronize()
    if out_f32:
        assert_bf16(bits_of(other), O.f32_to_bf16(c.h_master), what + " all-gather bf16")
    else:
        assert_close_f32(other.cpu().numpy(), c.h_master, what + " all-gather fp32")

    # step 3: fused again, continuing from the unfused state
    out = _out(torch, P, out_f32, cuda)
    c.grads_dev(0, 3, grads)
    Z.zero_step(c.plan, 0, grads, c.zdtype, c.master, c.m, c.v, c.hp_dev(3), None, out, zo)
    r = c.oracle_step(0, 3, out_dtype=odt)
    torch.cuda.synchronize()
    c.check_state(what + " fused step 3")
    _check_out(out, r, out_f32, what + " fused step 3 gathered")


@pytest.mark.parametrize("n", [1, 2, 5, 8, 32, 64])
def test_stage3_rank_count_sweep(cuda, n):
    """Stage 3 at several rank counts: random tensor lists in random layer
    groups, a per-group fused step in reverse order writing the owners' bf16
    shards, then every group gathered (directly, in the broadcast form and by
    the two-stream pass) and compared with the oracle's gather and broadcast
    of the cast shards."""
    import torch
    rng = np.random.default_rng(104729 * n)
    align = int(rng.choice([1, 2, 4, 8, 16]))
    budget = max(6_000, 1_200_000 // n)
    T = int(rng.integers(3, 12))
    numels = [1 + int(budget * x) for x in rng.dirichlet(np.full(T, 0.7))]
    groups = np.cumsum(rng.integers(0, 2, size=T)).tolist()   # non-decreasing, gaps allowed
    groups = [int(g) for g in np.unique(groups, return_inverse=True)[1]]
    gd = "f32" if rng.integers(0, 2) else "bf16"
    c = Case(numels, n, align, gd, grad_sigma=1e-2 if gd == "f32" else 1e-3,
             seed=int(rng.integers(1, 1 << 30)), groups=groups)
    Z = c.Z
    what = f"stage3 N={n} {gd} align={align} numels={numels} groups={groups}"
    G = len(c.groups)
    shards = [torch.zeros(c.info["shard_total"], dtype=torch.bfloat16, device=cuda)
              for _ in range(n)]
    for gi in reversed(range(G)):
        Z.zero_step_group(c.plan, gi, c.grads_dev(gi, 1), c.zdtype, c.master, c.m, c.v,
                          c.hp_dev(1), None, shards)
        c.oracle_step(gi, 1)
    torch.cuda.synchronize()
    c.check_state(what)
    gmax = max(g["psi_pad"] for g in c.groups)
    want = []
    for gi, g in enumerate(c.groups):
        f0, S = g["flat_off"], g["shard"]
        own = [O.f32_to_bf16(c.h_master[f0 + k * S:f0 + (k + 1) * S]) for k in range(n)]
        want.append(O.gather_layer(own)[0])
        want_b = O.broadcast_gather(own)[0]
        layer = torch.empty(max(1, g["psi_pad"]), dtype=torch.bfloat16, device=cuda)
        Z.zero_gather_layer(c.plan, gi, shards, Z.ZERO_BF16, layer)
        torch.cuda.synchronize()
        assert_bf16(bits_of(layer[:g["psi_pad"]]), want[gi], f"{what} layer {gi}")
        layer.zero_()
        Z.zero_broadcast_layer(c.plan, gi, shards, Z.ZERO_BF16, layer)
        torch.cuda.synchronize()
        assert_bf16(bits_of(layer[:g["psi_pad"]]), want_b, f"{what} broadcast layer {gi}")
    bufs = [torch.empty(max(1, gmax), dtype=torch.bfloat16, device=cuda) for _ in range(2)]
    order = list(range(G)) + list(reversed(range(G)))
    sums = torch.zeros(len(order), dtype=torch.int64, device=cuda)
    rounds = int(rng.integers(1, 40))       # consumer from memory-bound to arithmetic-bound
    Z.zero_stage3_gather_pass(c.plan, order, shards, bufs, gmax, sums, rounds,
                              torch.cuda.current_stream(), torch.cuda.Stream())
    torch.cuda.synchronize()
    for j, gi in enumerate(order):
        assert int(sums[j].item()) % (1 << 64) == O.layer_checksum(want[gi], rounds), \
            (what, rounds, j, gi)
