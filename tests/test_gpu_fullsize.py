"""Full-size workloads in the launch configurations the benchmark uses,
checked on sampled windows the oracle recomputes from generated inputs (every
owner, bucket, chunk and group boundary), and by properties that hold at any
size where a value depends on the whole gradient (the global norm) or on the
whole layer (gathered buffers and their checksums)."""
import numpy as np
import pytest

from synth import workloads as W
from oracle import zero_oracle as O

from conftest import read_golden
from harness import Case, assert_bf16, bits_of, boundary_windows

pytestmark = pytest.mark.gpu


def test_gpt2_medium_full_size_n64_align1(cuda):
    """N = 64 ranks, shards not aligned to tensor edges (S = 5,544,112 is not
    a multiple of 8, so vectors straddle owners): fused zero_step, 3 steps."""
    import torch
    w = W.GPT2_MEDIUM
    c = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed,
             host_state=False)
    Z = c.Z
    P, S = c.info["psi_pad"], c.groups[0]["shard"]
    assert (P, S) == (354_823_168, 5_544_112)
    out = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    grads = None
    for s in range(1, w.steps + 1):
        grads = c.grads_dev(0, s, grads)
        Z.zero_step(c.plan, 0, grads, Z.ZERO_BF16, c.master, c.m, c.v, c.hp_dev(s), None, out,
                    Z.ZERO_BF16)
    torch.cuda.synchronize()
    tensor_edges = np.cumsum(w.numels)[:-1].tolist()
    cuts = [k * S for k in range(1, w.n_ranks)] + tensor_edges[::23]
    for win in boundary_windows(P, cuts, 512):
        r = c.oracle_window(0, win, range(1, w.steps + 1))
        c.check_window(0, win, r, f"gpt2-medium {win}")
        assert_bf16(bits_of(out[win[0]:win[1]]), r["full"], f"gathered {win}")


def test_llama_1_4b_full_size_bucketed_clip(cuda):
    """Bucketed reduce-scatter (50M-element windows) with fp64 norm
    partials, device-side norm and clip coefficient, Adam in 200M-element
    chunks writing the gathered bf16 parameters; 2 steps.  The global norm
    of each step is compared with the oracle's, computed over the whole
    gradient by tests/golden/make_llama_1_4b_norm.py, and the oracle windows
    use the oracle's own coefficients."""
    import torch
    w = W.LLAMA_1_4B
    gold = read_golden("llama_1_4b_norm.txt")
    c = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed,
             heavy_tail=True, host_state=False)
    Z = c.Z
    P, S = c.info["psi_pad"], c.groups[0]["shard"]
    assert int(gold["psi_pad"]) == P
    bucket, chunk = w.extra["bucket"], w.extra["chunk"]
    windows = [(a, min(P, a + bucket)) for a in range(0, P, bucket)]
    chunks = [(a, min(P, a + chunk)) for a in range(0, P, chunk)]
    assert len(windows) == 27 and len(chunks) == 7
    npart = [Z.zero_rs_partials(c.plan, Z.ZERO_BF16, b - a) for a, b in windows]
    partials = torch.zeros(sum(npart), dtype=torch.float64, device=cuda)
    reduced = torch.empty(P, dtype=torch.float32, device=cuda)
    out = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    norm = torch.zeros(1, dtype=torch.float32, device=cuda)
    coef = torch.zeros(1, dtype=torch.float32, device=cuda)
    gold_coefs, exact = [], True
    grads = None
    for s in (1, 2):
        grads = c.grads_dev(0, s, grads)
        off = 0
        for (a, b), k in zip(windows, npart):
            Z.zero_reduce_scatter(c.plan, 0, grads, Z.ZERO_BF16, reduced, a, b, 1.0 / w.n_ranks,
                                  partials[off:off + k])
            off += k
        Z.zero_grad_norm(partials, off, w.extra["max_norm"], norm, coef)
        for a, b in chunks:
            Z.zero_adam_shard(c.plan, 0, c.master, c.m, c.v, reduced, c.hp_dev(s), coef, a, b,
                              out, Z.ZERO_BF16)
        torch.cuda.synchronize()
        # the device norm is the fp32 rounding of an fp64 sum taken in another
        # order: within one fp32 rounding of the oracle's; the coefficient
        # likewise (equal unless the two norms straddle a rounding boundary)
        o_norm, o_coef = float(gold[f"norm_step{s}"]), float(gold[f"coef_step{s}"])
        assert abs(norm.item() - o_norm) <= 2.0 ** -23 * o_norm, (s, norm.item(), o_norm)
        assert abs(coef.item() - o_coef) <= 2.0 ** -23 * o_coef, (s, coef.item(), o_coef)
        assert o_coef < 1.0                             # heavy tails: the clip is active
        exact = exact and coef.item() == o_coef
        gold_coefs.append(np.float32(o_coef))
        if s == 1:
            # reduced gradients of step 1 on sampled windows (bit-exact ring order)
            for win in boundary_windows(P, [k * S for k in range(1, 8)] +
                                        [a for a, _ in windows[1:]], 2048)[::3]:
                red, _, _ = O.ring_reduce_scatter(c.grads_host(0, 1, *win), S, win)
                np.testing.assert_array_equal(reduced[win[0]:win[1]].cpu().numpy(),
                                              np.concatenate(red))
    # state after 2 steps with the oracle's own coefficients: bit-exact when the
    # device's coefficients equal them, within tolerance otherwise
    cuts = [k * S for k in range(1, 8)] + [a for a, _ in windows[1:]] + [a for a, _ in chunks[1:]]
    for win in boundary_windows(P, cuts, 2048):
        r = c.oracle_window(0, win, (1, 2), clip_coefs=gold_coefs)
        c.check_window(0, win, r, f"llama-1.4b {win}", exact=exact)
        assert_bf16(bits_of(out[win[0]:win[1]]), r["full"], f"gathered {win}", exact=exact)


def test_llama_7b_stage3_full_size(cuda):
    """Stage 3: two steps, each per layer group (reverse order) a fused
    reduce-scatter + Adam writing each owner's bf16 shard from a regenerated
    gradient slot; then
    forward and reverse per-layer gathers prefetched on a second stream while
    a consumer checksums the current layer.  Every gathered layer is compared
    element by element."""
    import torch
    w = W.LLAMA_7B_STAGE3
    c = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed,
             groups=w.groups, host_state=False)
    Z = c.Z
    N = w.n_ranks
    G = len(c.groups)
    assert G == 34 and c.info["psi"] == 6_738_415_616
    gmax = max(g["psi_pad"] for g in c.groups)
    slot = [torch.empty(gmax, dtype=torch.bfloat16, device=cuda) for _ in range(N)]
    shards = [torch.zeros(c.info["shard_total"], dtype=torch.bfloat16, device=cuda)
              for _ in range(N)]
    steps = (1, 2)                  # the second step starts from nonzero m and v
    for s in steps:
        for gi in reversed(range(G)):
            g = c.groups[gi]
            views = [t[:g["psi_pad"]] for t in slot]
            c.grads_dev(gi, s, views)
            Z.zero_step_group(c.plan, gi, views, Z.ZERO_BF16, c.master, c.m, c.v, c.hp_dev(s),
                              None, shards)
    torch.cuda.synchronize()
    # sampled windows of every group: state and each owner's shard
    for gi, g in enumerate(c.groups):
        S, ro = g["shard"], g["rank_off"]
        wins = boundary_windows(g["psi_pad"], [k * S for k in range(1, N)], 256)
        for win in (wins if gi in (0, 1, G - 1) else wins[::5]):
            r = c.oracle_window(gi, win, steps)
            c.check_window(gi, win, r, f"group {gi} {win}")
            full = O.f32_to_bf16(r["master"])
            for j in range(win[0], win[1], 64):
                k = j // S
                e = min(win[1], j + 64, (k + 1) * S)
                got = bits_of(shards[k][ro + j - k * S:ro + e - k * S])
                assert_bf16(got, full[j - win[0]:e - win[0]], f"shard {k} group {gi}")
    # every layer gathered (and three in the broadcast form) and compared
    # element by element with the plain concatenation of the owners' shards
    cats = []
    buf = torch.empty(gmax, dtype=torch.bfloat16, device=cuda)
    for gi, g in enumerate(c.groups):
        ro, S = g["rank_off"], g["shard"]
        cats.append(torch.cat([shards[k][ro:ro + S] for k in range(N)]))
        calls = [Z.zero_gather_layer] + ([Z.zero_broadcast_layer] if gi in (0, 1, G - 1) else [])
        for call in calls:
            buf.fill_(0)
            call(c.plan, gi, shards, Z.ZERO_BF16, buf)
            torch.cuda.synchronize()
            assert torch.equal(buf[:g["psi_pad"]], cats[gi]), (call.__name__, gi)
    # the native two-stream schedule the benchmark times
    sb = torch.cuda.Stream()
    bufs = [torch.empty(gmax, dtype=torch.bfloat16, device=cuda) for _ in range(2)]
    order = list(range(G)) + list(reversed(range(G)))
    sums = torch.zeros(len(order), dtype=torch.int64, device=cuda)
    Z.zero_stage3_gather_pass(c.plan, order, shards, bufs, gmax, sums, 1,
                              torch.cuda.current_stream(), sb)
    torch.cuda.synchronize()
    # its consumer's checksum of each gathered layer, recomputed by plain
    # PyTorch integer arithmetic
    got = sums.cpu().numpy().view(np.uint64)
    for j, gi in enumerate(order):
        bits = cats[gi].view(torch.int16).to(torch.int64) & 0xFFFF
        idx = torch.arange(cats[gi].numel(), device=cuda, dtype=torch.int64)
        ref = int(((bits * (1 + (idx & 0xFFFF))).sum()).item()) % (1 << 64)
        assert int(got[j]) == ref, (j, gi)
    # and every buffer the schedule fills, element by element: the pass over
    # each prefix of the order leaves gather j in buffer j % 2
    for j in range(len(order)):
        Z.zero_stage3_gather_pass(c.plan, order[:j + 1], shards, bufs, gmax, sums, 1,
                                  torch.cuda.current_stream(), sb)
        torch.cuda.synchronize()
        gi = order[j]
        assert torch.equal(bufs[j % 2][:c.groups[gi]["psi_pad"]], cats[gi]), (j, gi)


def test_one_group_beyond_2_31_elements(cuda):
    """Maximum-size edge: one group of 2^31 + 12,345 parameters (N = 2, so
    the owner boundary also lies above 2^30 and the flat indices pass 2^31);
    fused step, windows around 2^31, the owner boundary and the ragged end."""
    import torch
    psi = (1 << 31) + 12_345
    c = Case([psi - 1000, 1000], 2, 16, "bf16", seed=2024, host_state=False)
    Z = c.Z
    P, S = c.info["psi_pad"], c.groups[0]["shard"]
    assert P > (1 << 31) and P == 2 * S
    out = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    grads = c.grads_dev(0, 1)
    Z.zero_step(c.plan, 0, grads, Z.ZERO_BF16, c.master, c.m, c.v, c.hp_dev(1), None, out,
                Z.ZERO_BF16)
    torch.cuda.synchronize()
    for a, b in [(0, 64), (S - 40, S + 40), ((1 << 31) - 37, (1 << 31) + 51),
                 (psi - 1003, psi + 5), (P - 64, P)]:
        r = c.oracle_window(0, (a, b), (1,))
        c.check_window(0, (a, b), r, f"2^31 group [{a},{b})")
        assert_bf16(bits_of(out[a:b]), r["full"], f"gathered [{a},{b})")
    del grads
