"""Full-size workloads in the launch configurations the benchmark uses,
checked on sampled windows the oracle recomputes from generated inputs (every
owner, bucket, chunk and group boundary), and by properties that hold at any
size where a value depends on the whole gradient (the global norm) or on the
whole layer (gathered buffers and their checksums)."""
import numpy as np
import pytest

from synth import workloads as W
from oracle import zero_oracle as O

from harness import Case, assert_bf16, bits_of, boundary_windows

pytestmark = pytest.mark.gpu


def _torch_norm_fp64(grads, n_ranks, chunk=1 << 26):
    """Independent reference of the global norm (plain PyTorch, fp64): the
    sum over ranks of bf16 gradients is exact in fp64, then /N and squared."""
    import torch
    P = grads[0].numel()
    acc = 0.0
    for a in range(0, P, chunk):
        s = torch.zeros(min(P, a + chunk) - a, dtype=torch.float64, device=grads[0].device)
        for g in grads:
            s += g[a:a + chunk].double()
        s /= n_ranks
        acc += float((s * s).sum().item())
    return acc ** 0.5


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
    chunks writing the gathered bf16 parameters; 2 steps."""
    import torch
    w = W.LLAMA_1_4B
    c = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed,
             heavy_tail=True, host_state=False)
    Z = c.Z
    P, S = c.info["psi_pad"], c.groups[0]["shard"]
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
    ref_coefs = []
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
        ref = _torch_norm_fp64(grads, w.n_ranks)
        torch.cuda.synchronize()
        assert abs(norm.item() - ref) <= 1e-6 * ref, (norm.item(), ref)
        ref_coef = np.float32(min(1.0, w.extra["max_norm"] / (ref + 1e-6)))
        assert abs(coef.item() - float(ref_coef)) <= 1e-6 * float(ref_coef)
        assert ref_coef < 1.0
        ref_coefs.append(ref_coef)
        if s == 1:
            # reduced gradients of step 1 on sampled windows (bit-exact ring order)
            for win in boundary_windows(P, [k * S for k in range(1, 8)] +
                                        [a for a, _ in windows[1:]], 2048)[::3]:
                red, _, _ = O.ring_reduce_scatter(c.grads_host(0, 1, *win), S, win)
                np.testing.assert_array_equal(reduced[win[0]:win[1]].cpu().numpy(),
                                              np.concatenate(red))
    # state after 2 steps: the coefficients come from the fp64 reference, so
    # the last bit of the device's coefficient may differ -> tolerance
    cuts = [k * S for k in range(1, 8)] + [a for a, _ in windows[1:]] + [a for a, _ in chunks[1:]]
    for win in boundary_windows(P, cuts, 2048):
        r = c.oracle_window(0, win, (1, 2), clip_coefs=ref_coefs)
        c.check_window(0, win, r, f"llama-1.4b {win}", exact=False)
        assert_bf16(bits_of(out[win[0]:win[1]]), r["full"], f"gathered {win}", exact=False)


def test_llama_7b_stage3_full_size(cuda):
    """Stage 3: per layer group (reverse order) a fused reduce-scatter + Adam
    writing each owner's bf16 shard from a regenerated gradient slot; then
    forward and reverse per-layer gathers prefetched on a second stream while
    a consumer checksums the current layer."""
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
    for gi in reversed(range(G)):
        g = c.groups[gi]
        views = [t[:g["psi_pad"]] for t in slot]
        c.grads_dev(gi, 1, views)
        Z.zero_step_group(c.plan, gi, views, Z.ZERO_BF16, c.master, c.m, c.v, c.hp_dev(1), None,
                          shards)
    torch.cuda.synchronize()
    # sampled windows of every group: state and each owner's shard
    for gi, g in enumerate(c.groups):
        S, ro = g["shard"], g["rank_off"]
        wins = boundary_windows(g["psi_pad"], [k * S for k in range(1, N)], 256)
        for win in (wins if gi in (0, 1, G - 1) else wins[::5]):
            r = c.oracle_window(gi, win, (1,))
            c.check_window(gi, win, r, f"group {gi} {win}")
            full = O.f32_to_bf16(r["master"])
            for j in range(win[0], win[1], 64):
                k = j // S
                e = min(win[1], j + 64, (k + 1) * S)
                got = bits_of(shards[k][ro + j - k * S:ro + e - k * S])
                assert_bf16(got, full[j - win[0]:e - win[0]], f"shard {k} group {gi}")
    # gathers: the native two-stream schedule the benchmark times
    sb = torch.cuda.Stream()
    bufs = [torch.empty(gmax, dtype=torch.bfloat16, device=cuda) for _ in range(2)]
    order = list(range(G)) + list(reversed(range(G)))
    sums = torch.zeros(len(order), dtype=torch.int64, device=cuda)
    Z.zero_stage3_gather_pass(c.plan, order, shards, bufs, gmax, sums, 1,
                              torch.cuda.current_stream(), sb)
    torch.cuda.synchronize()
    # property at any size: each gathered layer is the concatenation of the
    # owners' shards, checksummed by plain PyTorch integer arithmetic
    got = sums.cpu().numpy().view(np.uint64)
    for j, gi in enumerate(order):
        g = c.groups[gi]
        ro, S = g["rank_off"], g["shard"]
        cat = torch.cat([shards[k][ro:ro + S] for k in range(N)])
        bits = cat.view(torch.int16).to(torch.int64) & 0xFFFF
        idx = torch.arange(cat.numel(), device=cuda, dtype=torch.int64)
        ref = int(((bits * (1 + (idx & 0xFFFF))).sum()).item()) % (1 << 64)
        assert int(got[j]) == ref, (j, gi)
    # and one full layer buffer compared element by element
    last = order[-1]
    Z.zero_gather_layer(c.plan, last, shards, Z.ZERO_BF16, bufs[0])
    torch.cuda.synchronize()
    g = c.groups[last]
    cat = torch.cat([shards[k][g["rank_off"]:g["rank_off"] + g["shard"]] for k in range(N)])
    assert torch.equal(bufs[0][:g["psi_pad"]], cat)


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
