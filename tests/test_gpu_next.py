"""Beyond the step itself: the norm-only reduce-scatter pass of a two-pass
fused clip, gradient accumulation into owner shards over micro-batches, and
checkpoint/resume of the flat optimizer state -- each against the oracle or
the single-pass path, element by element."""
import numpy as np
import pytest

from synth import workloads as W
from oracle import zero_oracle as O

from harness import Case, assert_bf16, assert_close_f32, bits_of

pytestmark = pytest.mark.gpu


def test_two_pass_fused_clip_matches_bucketed_clip(cuda):
    """Pass 1 re-reads the gradients for the norm only; pass 2 is the fused
    step with the device clip coefficient.  Same result, bit for bit, as the
    reduce-scatter -> norm -> Adam path that stores the reduced gradient."""
    import torch
    w = W.mini(W.LLAMA_1_4B, scale=2048)
    c = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed,
             heavy_tail=True)
    Z = c.Z
    P = c.info["psi_pad"]
    grads = c.grads_dev(0, 1)
    npart = Z.zero_rs_partials(c.plan, Z.ZERO_BF16, P)
    part_a = torch.zeros(npart, dtype=torch.float64, device=cuda)
    part_b = torch.zeros(npart, dtype=torch.float64, device=cuda)
    coef_a = torch.zeros(1, dtype=torch.float32, device=cuda)
    coef_b = torch.zeros(1, dtype=torch.float32, device=cuda)
    reduced = torch.empty(P, dtype=torch.float32, device=cuda)
    out_a = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    out_b = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    ma, va, pa = c.m.clone(), c.v.clone(), c.master.clone()
    # storing path
    Z.zero_reduce_scatter(c.plan, 0, grads, Z.ZERO_BF16, reduced, 0, P, 1.0 / c.n, part_a)
    Z.zero_grad_norm(part_a, npart, 1.0, None, coef_a)
    Z.zero_adam_shard(c.plan, 0, pa, ma, va, reduced, c.hp_dev(1), coef_a, 0, P, out_a)
    # two-pass fused path
    Z.zero_reduce_scatter(c.plan, 0, grads, Z.ZERO_BF16, None, 0, P, 1.0 / c.n, part_b)
    Z.zero_grad_norm(part_b, npart, 1.0, None, coef_b)
    Z.zero_step(c.plan, 0, grads, Z.ZERO_BF16, c.master, c.m, c.v, c.hp_dev(1), coef_b, out_b)
    torch.cuda.synchronize()
    assert torch.equal(part_a, part_b) and coef_a.item() == coef_b.item() < 1.0
    assert torch.equal(pa, c.master) and torch.equal(ma, c.m) and torch.equal(va, c.v)
    assert torch.equal(out_a, out_b)
    # and the oracle, given its own clip coefficient
    red, _, _ = O.ring_reduce_scatter(c.grads_host(0, 1), c.groups[0]["shard"])
    _, ocoef = O.grad_norm(O.scale(red, np.float32(1.0) / np.float32(c.n)), 1.0)
    r = c.oracle_step(0, 1, clip_coef=ocoef)
    exact = coef_b.item() == float(ocoef)
    c.check_state("two-pass clip", exact=exact)
    assert_bf16(bits_of(out_b), r["full"], "two-pass gathered", exact=exact)


def test_gradient_accumulation_over_micro_batches(cuda):
    import torch
    M = 3
    c = Case([70_001, 3_333, 17], 8, 16, "bf16", seed=31)
    Z = c.Z
    P, S, N = c.info["psi_pad"], c.groups[0]["shard"], c.n
    scale = 1.0 / (N * M)
    npart = Z.zero_rs_partials(c.plan, Z.ZERO_BF16, P)
    partials = torch.zeros(npart, dtype=torch.float64, device=cuda)
    norm = torch.zeros(1, dtype=torch.float32, device=cuda)
    acc = torch.empty(P, dtype=torch.float32, device=cuda)
    out = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    # micro-batch b uses generator step 10 + b
    Z.zero_reduce_scatter(c.plan, 0, c.grads_dev(0, 10), Z.ZERO_BF16, acc, 0, P, scale)
    for b in range(1, M):
        Z.zero_reduce_scatter_acc(c.plan, 0, c.grads_dev(0, 10 + b), Z.ZERO_BF16, acc, 0, P,
                                  scale, partials if b == M - 1 else None)
    Z.zero_grad_norm(partials, npart, 1e9, norm, None)
    hp = Z.adam_hp(step=1, grad_scale=scale)
    Z.zero_adam_shard(c.plan, 0, c.master, c.m, c.v, acc, hp, None, 0, P, out)
    torch.cuda.synchronize()
    # oracle
    red = O.ring_reduce_scatter(c.grads_host(0, 10), S)[0]
    for b in range(1, M):
        red = O.accumulate_reduced(red, O.ring_reduce_scatter(c.grads_host(0, 10 + b), S)[0])
    assert_close_f32(acc.cpu().numpy(), np.concatenate(red), "accumulated")
    g = O.scale(red, np.float32(scale))
    onorm, _ = O.grad_norm(g, 1e9)
    assert abs(norm.item() - onorm) <= 1e-6 * onorm
    p, m, v = O.adam_update(c.h_master, c.h_m, c.h_v, np.concatenate(g), 1e-3, 0.9, 0.999, 1e-8,
                            0.0, 1)
    assert_close_f32(c.master.cpu().numpy(), p, "master")
    assert_close_f32(c.m.cpu().numpy(), m, "m")
    assert_close_f32(c.v.cpu().numpy(), v, "v")
    assert_bf16(bits_of(out), O.f32_to_bf16(p), "gathered")


@pytest.mark.parametrize("gd", ["bf16", "f32"])
def test_fused_last_micro_batch_equals_accumulate_then_adam(cuda, gd):
    """zero_step_acc (the last micro-batch's ring sum added to the
    accumulated buffer inside the fused step) equals zero_reduce_scatter_acc
    followed by zero_adam_shard bit for bit, and the oracle's accumulation;
    the accumulated buffer is left as it was."""
    import torch
    M = 3
    a, b = (Case([70_001, 3_333, 17], 8, 16, gd, grad_sigma=1e-2 if gd == "f32" else 1e-3,
                 seed=37) for _ in range(2))
    Z = a.Z
    P, S, N = a.info["psi_pad"], a.groups[0]["shard"], a.n
    hp = Z.adam_hp(step=1, grad_scale=1.0 / (N * M))
    acc_a = torch.empty(P, dtype=torch.float32, device=cuda)
    grads = [a.grads_dev(0, 20 + k) for k in range(M)]
    Z.zero_reduce_scatter(a.plan, 0, grads[0], a.zdtype, acc_a, 0, P, 1.0)
    for k in range(1, M - 1):
        Z.zero_reduce_scatter_acc(a.plan, 0, grads[k], a.zdtype, acc_a, 0, P, 1.0)
    acc_b = acc_a.clone()
    out_a = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    out_b = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    Z.zero_reduce_scatter_acc(a.plan, 0, grads[M - 1], a.zdtype, acc_a, 0, P, 1.0)
    Z.zero_adam_shard(a.plan, 0, a.master, a.m, a.v, acc_a, hp, None, 0, P, out_a)
    before = acc_b.clone()
    Z.zero_step_acc(b.plan, 0, grads[M - 1], b.zdtype, acc_b, b.master, b.m, b.v, hp, None,
                    out_b)
    torch.cuda.synchronize()
    assert torch.equal(acc_b, before)
    for x, y, what in ((a.master, b.master, "master"), (a.m, b.m, "m"), (a.v, b.v, "v"),
                       (out_a, out_b, "out")):
        assert torch.equal(x, y), what
    red = O.ring_reduce_scatter(a.grads_host(0, 20), S)[0]
    for k in range(1, M):
        red = O.accumulate_reduced(red, O.ring_reduce_scatter(a.grads_host(0, 20 + k), S)[0])
    g = O.scale(red, np.float32(1.0 / (N * M)))
    p, m, v = O.adam_update(b.h_master, b.h_m, b.h_v, np.concatenate(g), 1e-3, 0.9, 0.999, 1e-8,
                            0.0, 1)
    assert_close_f32(b.master.cpu().numpy(), p, "master")
    assert_bf16(bits_of(out_b), O.f32_to_bf16(p), "gathered")


def test_checkpoint_resume_is_bit_exact(cuda):
    """The optimizer state is three flat fp32 arrays plus the step number:
    dumping them to host memory after 3 steps and resuming in fresh buffers
    reproduces 5 uninterrupted steps bit for bit."""
    import torch
    w = W.mini(W.GPT2_SMALL, scale=128)
    a = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed,
             host_state=False)
    Z = a.Z
    P = a.info["psi_pad"]
    out = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    for s in range(1, 6):
        Z.zero_step(a.plan, 0, a.grads_dev(0, s), Z.ZERO_BF16, a.master, a.m, a.v, a.hp_dev(s),
                    None, out, Z.ZERO_BF16)
    b = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed,
             host_state=False)
    for s in range(1, 4):
        Z.zero_step(b.plan, 0, b.grads_dev(0, s), Z.ZERO_BF16, b.master, b.m, b.v, b.hp_dev(s),
                    None, out, Z.ZERO_BF16)
    ckpt = {"master": b.master.cpu(), "m": b.m.cpu(), "v": b.v.cpu(), "step": 3}
    del b
    plan = Z.zero_plan(w.numels, w.n_ranks, w.align)
    master, m, v = (ckpt[k].to(cuda) for k in ("master", "m", "v"))
    for s in range(ckpt["step"] + 1, 6):
        Z.zero_step(plan, 0, a.grads_dev(0, s), Z.ZERO_BF16, master, m, v, a.hp_dev(s), None,
                    out, Z.ZERO_BF16)
    torch.cuda.synchronize()
    assert torch.equal(master, a.master) and torch.equal(m, a.m) and torch.equal(v, a.v)


def test_stage3_checkpoint_resume_is_bit_exact(cuda):
    """Stage 3: the checkpoint is the same three flat fp32 arrays and the step
    number (the owners' bf16 shards are outputs, rebuilt by the next step).
    Dumped after 2 steps and resumed in fresh buffers, steps 3 and 4 give
    the state and every owner's shards of 4 uninterrupted steps, bit for
    bit."""
    import torch
    w = W.mini(W.LLAMA_7B_STAGE3, scale=2048)
    a = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed,
             groups=w.groups, host_state=False)
    Z = a.Z
    N, G, ST = a.n, len(a.groups), a.info["shard_total"]

    def steps(case, state, shards, first, last, plan=None):
        master, m, v = state
        for s in range(first, last + 1):
            for gi in reversed(range(G)):
                Z.zero_step_group(plan or case.plan, gi, a.grads_dev(gi, s), Z.ZERO_BF16, master,
                                  m, v, a.hp_dev(s), None, shards)

    sh_a = [torch.zeros(ST, dtype=torch.bfloat16, device=cuda) for _ in range(N)]
    steps(a, (a.master, a.m, a.v), sh_a, 1, 4)
    b = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed,
             groups=w.groups, host_state=False)
    sh_b = [torch.zeros(ST, dtype=torch.bfloat16, device=cuda) for _ in range(N)]
    steps(b, (b.master, b.m, b.v), sh_b, 1, 2)
    ckpt = {"master": b.master.cpu(), "m": b.m.cpu(), "v": b.v.cpu(), "step": 2}
    del b, sh_b
    plan = Z.zero_plan(w.numels, w.n_ranks, w.align, w.groups)
    state = tuple(ckpt[k].to(cuda) for k in ("master", "m", "v"))
    sh_c = [torch.zeros(ST, dtype=torch.bfloat16, device=cuda) for _ in range(N)]
    steps(None, state, sh_c, ckpt["step"] + 1, 4, plan)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(state, (a.master, a.m, a.v)))
    assert all(torch.equal(x, y) for x, y in zip(sh_c, sh_a))


def test_stage3_step_with_gradient_clipping(cuda):
    """Stage 3 with clipping by the global norm over all layer groups: a
    norm-only reduce-scatter pass per group (partials into consecutive
    slices), one device norm, then the per-group fused step with the device
    coefficient writing the owners' shards.  Agrees with the oracle, which
    takes the same global norm over all groups' scaled reduced gradients."""
    import torch
    d, ffn, vocab = 64, 172, 500
    blocks = [[d * d] * 4 + [d * ffn] * 2 + [ffn * d, d, d] for _ in range(2)]
    numels = [vocab * d] + blocks[0] + blocks[1] + [d, vocab * d]
    groups = [0] + [1] * 9 + [2] * 9 + [3, 3]
    c = Case(numels, 8, 16, "bf16", grad_sigma=3e-3, seed=57, groups=groups, heavy_tail=True)
    Z = c.Z
    G = len(c.groups)
    counts = [Z.zero_rs_partials(c.plan, Z.ZERO_BF16, g["psi_pad"]) for g in c.groups]
    part = torch.zeros(sum(counts), dtype=torch.float64, device=cuda)
    coef = torch.zeros(1, dtype=torch.float32, device=cuda)
    norm = torch.zeros(1, dtype=torch.float32, device=cuda)
    shards = [torch.zeros(c.info["shard_total"], dtype=torch.bfloat16, device=cuda)
              for _ in range(8)]
    grads = [c.grads_dev(gi, 1) for gi in range(G)]
    off = 0
    for gi, k in zip(range(G), counts):
        Z.zero_reduce_scatter(c.plan, gi, grads[gi], Z.ZERO_BF16, None, 0,
                              c.groups[gi]["psi_pad"], 1.0 / 8, part[off:off + k])
        off += k
    Z.zero_grad_norm(part, off, 1.0, norm, coef)
    for gi in reversed(range(G)):
        Z.zero_step_group(c.plan, gi, grads[gi], Z.ZERO_BF16, c.master, c.m, c.v, c.hp_dev(1),
                          coef, shards)
    torch.cuda.synchronize()
    # oracle: the same global norm, then each group's step with that coefficient
    scaled = []
    for gi, g in enumerate(c.groups):
        red, _, _ = O.ring_reduce_scatter(c.grads_host(gi, 1), g["shard"])
        scaled += O.scale(red, np.float32(1.0) / np.float32(8))
    onorm, ocoef = O.grad_norm(scaled, 1.0)
    assert float(ocoef) < 1.0                           # the clip is active
    assert abs(norm.item() - onorm) <= 1e-6 * onorm
    exact = coef.item() == float(ocoef)
    for gi in reversed(range(G)):
        c.oracle_step(gi, 1, clip_coef=ocoef)
    c.check_state("stage 3 clipped", exact=exact)
    for gi, g in enumerate(c.groups):
        f0, S = g["flat_off"], g["shard"]
        for k in range(8):
            ro = g["rank_off"]
            assert_bf16(bits_of(shards[k][ro:ro + S]),
                        O.f32_to_bf16(c.h_master[f0 + k * S:f0 + (k + 1) * S]),
                        f"shard {k} group {gi}", exact=exact)


def test_occupancy_setting_does_not_change_results(cuda):
    """The resident-block cap only changes which thread handles which
    vector: element-wise outputs are bit-identical for every setting, and the
    norm (whose partial grouping follows the grid) agrees to rounding."""
    import torch
    c = Case([123_457, 999, 4_096], 8, 16, "bf16", seed=12, host_state=False)
    Z = c.Z
    P = c.info["psi_pad"]
    grads = c.grads_dev(0, 1)
    results = []
    for cap in (1, 4, 0):
        for kind in (Z.ZERO_OCC_FUSED, Z.ZERO_OCC_RS):
            Z.zero_set_occupancy(kind, cap)
        master, m, v = c.master.clone(), c.m.clone(), c.v.clone()
        out = torch.empty(P, dtype=torch.bfloat16, device=cuda)
        red = torch.empty(P, dtype=torch.float32, device=cuda)
        n = Z.zero_rs_partials(c.plan, Z.ZERO_BF16, P)
        part = torch.zeros(n, dtype=torch.float64, device=cuda)
        norm = torch.zeros(1, dtype=torch.float32, device=cuda)
        Z.zero_step(c.plan, 0, grads, Z.ZERO_BF16, master, m, v, c.hp_dev(1), None, out)
        Z.zero_reduce_scatter(c.plan, 0, grads, Z.ZERO_BF16, red, 0, P, 1.0 / c.n, part)
        Z.zero_grad_norm(part, n, 1.0, norm, None)
        torch.cuda.synchronize()
        results.append((master, m, v, out, red, norm.item()))
    base = results[-1]
    for r in results[:-1]:
        for a, b in zip(r[:5], base[:5]):
            assert torch.equal(a, b)
        assert abs(r[5] - base[5]) <= 1e-6 * base[5]


def test_gather_occupancy_settings_do_not_change_results(cuda):
    """The bulk gather's CTAs per SM (ZERO_OCC_GATHER, ZERO_OCC_PREFETCH)
    and the consumer's blocks (ZERO_OCC_CONSUMER) change only which CTA moves
    which piece: gathered layers and the pass's checksums are identical for
    every setting, including caps the shared memory cannot hold at once."""
    import torch
    d, ffn, vocab = 64, 172, 500
    blocks = [[d * d] * 4 + [d * ffn] * 2 + [ffn * d, d, d] for _ in range(3)]
    numels = [vocab * d] + [n for b in blocks for n in b] + [d, vocab * d]
    groups = [0] + [1 + i // 9 for i in range(27)] + [4, 4]
    c = Case(numels, 16, 16, "bf16", seed=8, groups=groups, host_state=False)
    Z = c.Z
    N, G = 16, len(c.groups)
    shards = [torch.randn(c.info["shard_total"], device=cuda).to(torch.bfloat16) for _ in range(N)]
    gmax = max(g["psi_pad"] for g in c.groups)
    order = list(range(G)) + list(reversed(range(G)))
    results = []
    for cap in (1, 3, 12, 0):
        for kind in (Z.ZERO_OCC_GATHER, Z.ZERO_OCC_PREFETCH, Z.ZERO_OCC_CONSUMER):
            Z.zero_set_occupancy(kind, cap)
        layers = [torch.empty(g["psi_pad"], dtype=torch.bfloat16, device=cuda) for g in c.groups]
        for gi in range(G):
            Z.zero_gather_layer(c.plan, gi, shards, Z.ZERO_BF16, layers[gi])
        bufs = [torch.empty(gmax, dtype=torch.bfloat16, device=cuda) for _ in range(2)]
        sums = torch.zeros(len(order), dtype=torch.int64, device=cuda)
        Z.zero_stage3_gather_pass(c.plan, order, shards, bufs, gmax, sums, 9,
                                  torch.cuda.current_stream(), torch.cuda.Stream())
        torch.cuda.synchronize()
        results.append((layers, sums))
    base = results[-1]
    for layers, sums in results[:-1]:
        assert all(torch.equal(x, y) for x, y in zip(layers, base[0]))
        assert torch.equal(sums, base[1])


def test_stage3_per_parameter_partitioning(cuda):
    """Per-parameter partitioning (each tensor its own group, sharded over
    the N ranks and padded on its own): step and gather of every tensor
    match the oracle."""
    import torch
    d, ffn, vocab = 48, 130, 301
    numels = [vocab * d] + [d * d] * 4 + [d * ffn] * 2 + [ffn * d, d, d] + [d, vocab * d]
    groups = list(range(len(numels)))
    c = Case(numels, 16, 8, "bf16", seed=91, groups=groups)
    Z = c.Z
    N = 16
    assert c.info["n_groups"] == len(numels)
    shards = [torch.zeros(c.info["shard_total"], dtype=torch.bfloat16, device=cuda)
              for _ in range(N)]
    for gi in reversed(range(len(c.groups))):
        Z.zero_step_group(c.plan, gi, c.grads_dev(gi, 1), Z.ZERO_BF16, c.master, c.m, c.v,
                          c.hp_dev(1), None, shards)
        c.oracle_step(gi, 1)
    torch.cuda.synchronize()
    c.check_state("per-parameter stage 3")
    for gi, g in enumerate(c.groups):
        layer = torch.empty(g["psi_pad"], dtype=torch.bfloat16, device=cuda)
        Z.zero_gather_layer(c.plan, gi, shards, Z.ZERO_BF16, layer)
        torch.cuda.synchronize()
        f0 = g["flat_off"]
        assert_bf16(bits_of(layer), O.f32_to_bf16(c.h_master[f0:f0 + g["psi_pad"]]),
                    f"tensor {gi}")


def test_native_gather_schedule_matches_direct_gathers(cuda):
    """zero_stage3_gather_pass (gathers on stream B, consumer on stream A,
    double-buffered): for every gather of a forward + reverse pass the
    consumer's checksum and the gathered buffer itself, element by element,
    equal the oracle's all-gather of that layer; bad input is rejected."""
    import torch
    d, ffn, vocab = 64, 172, 500
    blocks = [[d * d] * 4 + [d * ffn] * 2 + [ffn * d, d, d] for _ in range(3)]
    numels = [vocab * d] + [n for b in blocks for n in b] + [d, vocab * d]
    groups = [0] + [1 + i // 9 for i in range(27)] + [4, 4]
    c = Case(numels, 16, 16, "bf16", seed=5, groups=groups, host_state=False)
    Z = c.Z
    N, G = 16, len(c.groups)
    shards = [torch.empty(c.info["shard_total"], dtype=torch.bfloat16, device=cuda)
              for _ in range(N)]
    for r in range(N):
        shards[r].copy_(torch.randn(c.info["shard_total"], device=cuda).to(torch.bfloat16))
    gmax = max(g["psi_pad"] for g in c.groups)
    bufs = [torch.empty(gmax, dtype=torch.bfloat16, device=cuda) for _ in range(2)]
    order = list(range(G)) + list(reversed(range(G)))
    sums = torch.zeros(len(order), dtype=torch.int64, device=cuda)
    sb = torch.cuda.Stream()
    Z.zero_stage3_gather_pass(c.plan, order, shards, bufs, gmax, sums, 1,
                              torch.cuda.current_stream(), sb)
    torch.cuda.synchronize()
    host = [bits_of(t) for t in shards]
    want = []
    for gi in order:
        g = c.groups[gi]
        ro, S = g["rank_off"], g["shard"]
        want.append(O.gather_layer([h[ro:ro + S] for h in host])[0])
    for j, gi in enumerate(order):
        assert int(sums[j].item()) % (1 << 64) == O.layer_checksum(want[j]), (j, gi)
    # every gathered layer element by element: the pass over each prefix of
    # the order leaves gather j in buffer j % 2 and gather j - 1 in the other
    for j in range(len(order)):
        Z.zero_stage3_gather_pass(c.plan, order[:j + 1], shards, bufs, gmax, sums, 1,
                                  torch.cuda.current_stream(), sb)
        torch.cuda.synchronize()
        for i in (j, j - 1):
            if i >= 0:
                n_i = c.groups[order[i]]["psi_pad"]
                assert np.array_equal(bits_of(bufs[i % 2][:n_i]), want[i]), (j, i)
    E = Z.ZeroError
    for bad, status in [(dict(order=[G]), Z.ZERO_ERANGE), (dict(buf_elems=10), Z.ZERO_ERANGE),
                        (dict(stream_b=torch.cuda.current_stream()), Z.ZERO_EINVAL),
                        (dict(rounds=0), Z.ZERO_EINVAL),
                        (dict(rounds=Z.ZERO_MAX_CONSUMER_ROUNDS + 1), Z.ZERO_EINVAL)]:
        kw = dict(order=order, buf_elems=gmax, stream_b=sb, rounds=1)
        kw.update(bad)
        with pytest.raises(E) as e:
            Z.zero_stage3_gather_pass(c.plan, kw["order"], shards, bufs, kw["buf_elems"], sums,
                                      kw["rounds"], torch.cuda.current_stream(),
                                      kw["stream_b"])
        assert e.value.status == status


def test_gather_pass_with_coalesced_steps(cuda):
    """Per-parameter partitioning with the two-stream pass: each step fetches
    one module's tensor groups together (zero_stage3_gather_pass_steps); the
    consumer's checksum of every step, and the step's packed buffer element
    by element, equal the oracle's concatenated gathered tensors, forward and
    reverse."""
    import torch
    d, ffn, vocab = 64, 172, 500
    blocks = [[d * d] * 4 + [d * ffn] * 2 + [ffn * d, d, d] for _ in range(3)]
    numels = [vocab * d] + [n for b in blocks for n in b] + [d, vocab * d]
    layer_of = [0] + [1 + i // 9 for i in range(27)] + [4, 4]
    groups = list(range(len(numels)))                      # every tensor its own group
    c = Case(numels, 16, 16, "bf16", seed=13, groups=groups, host_state=False)
    Z = c.Z
    N = 16
    rng = np.random.default_rng(13)
    host = [rng.integers(0, 1 << 16, c.info["shard_total"], dtype=np.uint64).astype(np.uint16)
            for _ in range(N)]
    shards = [torch.from_numpy(h.view(np.int16)).to(cuda) for h in host]
    layers = [[t for t, L in enumerate(layer_of) if L == k] for k in range(5)]
    steps = layers + layers[::-1]
    elems = [sum(c.groups[g]["psi_pad"] for g in st) for st in steps]
    bufs = [torch.empty(max(elems), dtype=torch.bfloat16, device=cuda) for _ in range(2)]
    sums = torch.zeros(len(steps), dtype=torch.int64, device=cuda)
    sb = torch.cuda.Stream()
    Z.zero_stage3_gather_pass_steps(c.plan, steps, shards, bufs, max(elems), sums, 5,
                                    torch.cuda.current_stream(), sb)
    torch.cuda.synchronize()
    want = []
    for j, st in enumerate(steps):
        parts = []
        for g in st:
            gi = c.groups[g]
            layer, _, _ = O.gather_layer([h[gi["rank_off"]:gi["rank_off"] + gi["shard"]]
                                          for h in host])
            parts.append(layer)
        want.append(np.concatenate(parts))
        assert int(sums[j].item()) % (1 << 64) == O.layer_checksum(want[j], 5), j
    # every step's packed buffer element by element (pass over each prefix)
    for j in range(len(steps)):
        Z.zero_stage3_gather_pass_steps(c.plan, steps[:j + 1], shards, bufs, max(elems), sums, 1,
                                        torch.cuda.current_stream(), sb)
        torch.cuda.synchronize()
        for i in (j, j - 1):
            if i >= 0:
                assert np.array_equal(bits_of(bufs[i % 2][:elems[i]]), want[i]), (j, i)
    E = Z.ZeroError
    with pytest.raises(E) as e:                           # a step must fit the buffers
        Z.zero_stage3_gather_pass_steps(c.plan, steps, shards, bufs, max(elems) - 1, sums, 1,
                                        torch.cuda.current_stream(), torch.cuda.Stream())
    assert e.value.status == Z.ZERO_ERANGE
    odd = Case([5, 7, 9], 3, 1, "bf16", seed=1, groups=[0, 1, 2], host_state=False)
    osh = [torch.zeros(odd.info["shard_total"], dtype=torch.bfloat16, device=cuda)
           for _ in range(3)]
    with pytest.raises(E) as e:                           # packed outputs must stay aligned
        Z.zero_stage3_gather_pass_steps(odd.plan, [[0, 1]], osh, bufs, max(elems), sums, 1,
                                        torch.cuda.current_stream(), torch.cuda.Stream())
    assert e.value.status == Z.ZERO_EALIGN
    Z.zero_stage3_gather_pass_steps(odd.plan, [[0], [1], [2]], osh, bufs, max(elems), sums, 1,
                                    torch.cuda.current_stream(), torch.cuda.Stream())
    torch.cuda.synchronize()


def test_cuda_graph_of_the_stage3_gather_pass(cuda):
    """The two-stream gather schedule captured once in a CUDA graph (stream B
    forks from and joins the capturing stream through the pass's events);
    a replay after the shards changed gives the eager pass's checksums."""
    import torch
    d, ffn, vocab = 64, 172, 500
    blocks = [[d * d] * 4 + [d * ffn] * 2 + [ffn * d, d, d] for _ in range(3)]
    numels = [vocab * d] + [n for b in blocks for n in b] + [d, vocab * d]
    groups = [0] + [1 + i // 9 for i in range(27)] + [4, 4]
    c = Case(numels, 16, 16, "bf16", seed=6, groups=groups, host_state=False)
    Z = c.Z
    N, G = 16, len(c.groups)
    shards = [torch.randn(c.info["shard_total"], device=cuda).to(torch.bfloat16)
              for _ in range(N)]
    gmax = max(g["psi_pad"] for g in c.groups)
    bufs = [torch.empty(gmax, dtype=torch.bfloat16, device=cuda) for _ in range(2)]
    order = list(range(G)) + list(reversed(range(G)))
    eager = torch.zeros(len(order), dtype=torch.int64, device=cuda)
    replayed = torch.zeros(len(order), dtype=torch.int64, device=cuda)
    cur = torch.cuda.current_stream()
    Z.zero_stage3_gather_pass(c.plan, order, shards, bufs, gmax, eager, 5, cur,
                              torch.cuda.Stream())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s, sb = torch.cuda.Stream(), torch.cuda.Stream()
    s.wait_stream(cur)
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            Z.zero_stage3_gather_pass(c.plan, order, shards, bufs, gmax, replayed, 5, s, sb)
    cur.wait_stream(s)
    torch.cuda.synchronize()
    for r in range(N):
        shards[r].copy_(torch.randn(c.info["shard_total"], device=cuda).to(torch.bfloat16))
    Z.zero_stage3_gather_pass(c.plan, order, shards, bufs, gmax, eager, 5, cur,
                              torch.cuda.Stream())
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager, replayed)
    assert int(torch.count_nonzero(eager)) == len(order)


def _eager_and_state_cases(w, seed):
    a = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, seed,
             host_state=False)
    b = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, seed,
             host_state=False)
    return a, b


def test_device_adam_state_matches_step_numbers(cuda):
    import torch
    w = W.mini(W.GPT2_SMALL, scale=256)
    a, b = _eager_and_state_cases(w, 41)
    Z = a.Z
    P = a.info["psi_pad"]
    out_a = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    out_b = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    state = torch.zeros(Z.ZERO_ADAM_STATE_BYTES // 8, dtype=torch.float64, device=cuda)
    hp_dev = Z.adam_hp(step=5000, grad_scale=1.0 / a.n, d_state=state)
    Z.zero_adam_state_init(hp_dev, state)            # "before step 5000"
    for t in range(5000, 5003):
        g = a.grads_dev(0, t)
        Z.zero_step(a.plan, 0, g, Z.ZERO_BF16, a.master, a.m, a.v, a.hp_dev(t), None, out_a)
        Z.zero_adam_state_advance(hp_dev, state)
        Z.zero_step(b.plan, 0, g, Z.ZERO_BF16, b.master, b.m, b.v, hp_dev, None, out_b)
    torch.cuda.synchronize()
    assert torch.equal(a.master, b.master) and torch.equal(a.m, b.m) and torch.equal(a.v, b.v)
    assert torch.equal(out_a, out_b)


def test_cuda_graph_of_a_fused_step_replays_exactly(cuda):
    """One step (advance the device Adam state, fused zero_step) captured in a
    CUDA graph and replayed three times equals three eager steps."""
    import torch
    w = W.mini(W.GPT2_SMALL, scale=256)
    a, b = _eager_and_state_cases(w, 43)
    Z = a.Z
    P = a.info["psi_pad"]
    grads = a.grads_dev(0, 1)
    out_a = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    out_b = torch.empty(P, dtype=torch.bfloat16, device=cuda)
    for t in range(1, 4):
        Z.zero_step(a.plan, 0, grads, Z.ZERO_BF16, a.master, a.m, a.v, a.hp_dev(t), None, out_a)
    state = torch.zeros(4, dtype=torch.float64, device=cuda)
    hp = Z.adam_hp(step=1, grad_scale=1.0 / b.n, d_state=state)
    # warm-up on scratch copies so that every launch parameter is cached
    sm, smm, sv = b.master.clone(), b.m.clone(), b.v.clone()
    Z.zero_adam_state_init(hp, state)
    Z.zero_adam_state_advance(hp, state)
    Z.zero_step(b.plan, 0, grads, Z.ZERO_BF16, sm, smm, sv, hp, None, out_b)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            Z.zero_adam_state_advance(hp, state)
            Z.zero_step(b.plan, 0, grads, Z.ZERO_BF16, b.master, b.m, b.v, hp, None, out_b)
    torch.cuda.current_stream().wait_stream(s)
    Z.zero_adam_state_init(hp, state)                  # back to "before step 1"
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(a.master, b.master) and torch.equal(a.m, b.m) and torch.equal(a.v, b.v)
    assert torch.equal(out_a, out_b)


def test_cuda_graph_of_the_bucketed_clip_pipeline(cuda):
    """Reduce-scatter buckets with norm partials, device norm and clip,
    chunked Adam and the state advance captured once; two replays equal two
    eager steps bit for bit."""
    import torch
    w = W.mini(W.LLAMA_1_4B, scale=1024)
    a, b = (Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma,
                 w.seed, heavy_tail=True, host_state=False) for _ in range(2))
    Z = a.Z
    P = a.info["psi_pad"]
    grads = a.grads_dev(0, 1)
    bucket, chunk = 100_003, 400_001
    windows = [(x, min(P, x + bucket)) for x in range(0, P, bucket)]
    chunks = [(x, min(P, x + chunk)) for x in range(0, P, chunk)]
    npart = [Z.zero_rs_partials(a.plan, Z.ZERO_BF16, hi - lo) for lo, hi in windows]

    def buffers():
        return (torch.empty(P, dtype=torch.float32, device=cuda),
                torch.zeros(sum(npart), dtype=torch.float64, device=cuda),
                torch.zeros(1, dtype=torch.float32, device=cuda),
                torch.empty(P, dtype=torch.bfloat16, device=cuda))

    def step(c, red, part, coef, out, hp):
        off = 0
        for (lo, hi), k in zip(windows, npart):
            Z.zero_reduce_scatter(c.plan, 0, grads, Z.ZERO_BF16, red, lo, hi, 1.0 / c.n,
                                  part[off:off + k])
            off += k
        Z.zero_grad_norm(part, off, 1.0, None, coef)
        for lo, hi in chunks:
            Z.zero_adam_shard(c.plan, 0, c.master, c.m, c.v, red, hp, coef, lo, hi, out)

    ba = buffers()
    for t in (1, 2):
        step(a, *ba, a.hp_dev(t))
    bb = buffers()
    state = torch.zeros(4, dtype=torch.float64, device=cuda)
    hp = Z.adam_hp(step=1, grad_scale=1.0 / b.n, d_state=state)
    Z.zero_adam_state_init(hp, state)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            Z.zero_adam_state_advance(hp, state)
            step(b, *bb, hp)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(a.master, b.master) and torch.equal(a.m, b.m) and torch.equal(a.v, b.v)
    assert torch.equal(ba[3], bb[3]) and torch.equal(ba[2], bb[2])


def test_step_clipped_equals_the_calls_it_strings_together(cuda):
    """zero_step_clipped (bucketed reduce-scatter with norm partials, norm,
    clip, chunked Adam, cast in one call) equals the same calls made one by
    one, bit for bit, over two steps of the Llama-1.4B mini with heavy tails
    (clip active); its argument checks return their codes."""
    import torch
    w = W.mini(W.LLAMA_1_4B, scale=1024)
    a, b = (Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma,
                 w.seed, heavy_tail=True, host_state=False) for _ in range(2))
    Z = a.Z
    P = a.info["psi_pad"]
    bucket, chunk = 100_003, 400_001
    windows = [(x, min(P, x + bucket)) for x in range(0, P, bucket)]
    npart = [Z.zero_rs_partials(a.plan, Z.ZERO_BF16, hi - lo) for lo, hi in windows]
    total = Z.zero_step_clipped_partials(b.plan, 0, Z.ZERO_BF16, bucket)
    assert total == sum(npart)

    def bufs():
        return (torch.empty(P, dtype=torch.float32, device=cuda),
                torch.zeros(total, dtype=torch.float64, device=cuda),
                torch.zeros(1, dtype=torch.float32, device=cuda),
                torch.zeros(1, dtype=torch.float32, device=cuda),
                torch.empty(P, dtype=torch.bfloat16, device=cuda))

    ra, pa, na, ca, oa = bufs()
    rb, pb, nb, cb, ob = bufs()
    for s in (1, 2):
        grads = a.grads_dev(0, s)
        off = 0
        for (lo, hi), k in zip(windows, npart):
            Z.zero_reduce_scatter(a.plan, 0, grads, Z.ZERO_BF16, ra, lo, hi, 1.0 / a.n,
                                  pa[off:off + k])
            off += k
        Z.zero_grad_norm(pa, off, 1.0, na, ca)
        for lo in range(0, P, chunk):
            Z.zero_adam_shard(a.plan, 0, a.master, a.m, a.v, ra, a.hp_dev(s), ca, lo,
                              min(P, lo + chunk), oa, Z.ZERO_BF16)
        Z.zero_step_clipped(b.plan, 0, grads, Z.ZERO_BF16, rb, b.master, b.m, b.v, b.hp_dev(s),
                            1.0, bucket, chunk, pb, total, nb, cb, ob, Z.ZERO_BF16)
        torch.cuda.synchronize()
        assert float(ca.item()) < 1.0                      # the clip is active
        for x, y, what in ((a.master, b.master, "master"), (a.m, b.m, "m"), (a.v, b.v, "v"),
                           (oa, ob, "out"), (ra, rb, "reduced"), (na, nb, "norm"),
                           (ca, cb, "coef")):
            assert torch.equal(x, y), (s, what)
    E = Z.ZeroError
    g = b.grads_dev(0, 3)
    for kw, status in [(dict(n_partials=total - 1), Z.ZERO_ERANGE), (dict(bucket=0), Z.ZERO_EINVAL),
                       (dict(d_coef=None), Z.ZERO_EINVAL), (dict(max_norm=0.0), Z.ZERO_EINVAL)]:
        args = dict(n_partials=total, bucket=bucket, d_coef=cb, max_norm=1.0)
        args.update(kw)
        with pytest.raises(E) as e:
            Z.zero_step_clipped(b.plan, 0, g, Z.ZERO_BF16, rb, b.master, b.m, b.v, b.hp_dev(3),
                                args["max_norm"], args["bucket"], chunk, pb, args["n_partials"],
                                nb, args["d_coef"], ob, Z.ZERO_BF16)
        assert e.value.status == status


def test_fp32_gradient_load_paths_agree(cuda):
    """fp32 gradient buffers that are all 32-byte aligned take one 32-byte
    load per thread, others two 16-byte loads: identical results, device and
    mapped pinned host memory alike."""
    import torch
    import bench
    c = Case([40_000, 1_234], 8, 16, "f32", grad_sigma=1e-2, seed=61, host_state=False)
    Z = c.Z
    P = c.info["psi_pad"]
    aligned = c.grads_dev(0, 1)
    offset = []                                   # same values at a 16-byte (not 32) offset
    for g in aligned:
        buf = torch.empty(P + 4, dtype=torch.float32, device=cuda)
        buf[4:].copy_(g)
        assert (buf[4:].data_ptr() % 32) == 16
        offset.append(buf[4:])
    results = []
    for grads in (aligned, offset):
        master, m, v = c.master.clone(), c.m.clone(), c.v.clone()
        out = torch.empty(P, dtype=torch.bfloat16, device=cuda)
        Z.zero_step(c.plan, 0, grads, Z.ZERO_F32, master, m, v, c.hp_dev(1), None, out)
        results.append((master, m, v, out))
    h = [torch.empty(P, dtype=torch.float32, pin_memory=True) for _ in range(8)]
    for x, g in zip(h, aligned):
        x.copy_(g)
    if all(bench.host_mapped(x) for x in h):
        master, m, v = c.master.clone(), c.m.clone(), c.v.clone()
        out = torch.empty(P, dtype=torch.bfloat16, device=cuda)
        Z.zero_step(c.plan, 0, h, Z.ZERO_F32, master, m, v, c.hp_dev(1), None, out)
        results.append((master, m, v, out))
    torch.cuda.synchronize()
    for r in results[1:]:
        for a, b in zip(r, results[0]):
            assert torch.equal(a, b)


def test_prepared_step_equals_zero_step(cuda):
    """prepare_zero_step (buffers checked and marshalled once) launches the
    same call as zero_step: three tiny steps through each give bit-identical
    state and gathered parameters, equal to the oracle's."""
    import torch
    w = W.TINY
    outs = []
    for prepared in (False, True):
        c = Case(w.numels, w.n_ranks, w.align, w.grad_dtype, w.grad_sigma, w.master_sigma, w.seed)
        Z = c.Z
        out = torch.empty(c.info["psi_pad"], dtype=torch.bfloat16, device=cuda)
        grads = c.grads_dev(0, 1)
        step = Z.prepare_zero_step(c.plan, 0, grads, c.zdtype, c.master, c.m, c.v, None, out)
        for s in range(1, 4):
            c.grads_dev(0, s, grads)
            if prepared:
                step(c.hp_dev(s))
            else:
                Z.zero_step(c.plan, 0, grads, c.zdtype, c.master, c.m, c.v, c.hp_dev(s), None,
                            out)
            r = c.oracle_step(0, s)
        torch.cuda.synchronize()
        c.check_state(f"prepared={prepared}")
        assert_bf16(bits_of(out), r["full"], "gathered")
        outs.append((c.master.clone(), out.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_gathers_queued_right_after_the_step_that_writes_their_shards(cuda):
    """The standalone bulk gather uses programmatic dependent launch: its CTAs
    may become resident before the kernel ahead of it on the stream has
    finished, and they copy only after griddepcontrol.wait.  Here each
    group's fused step writes the owners' shards and the group's gather, then
    its broadcast form, are queued right behind it with no synchronisation
    in between; every layer equals the oracle's gather of the owners' bf16
    shards, cast from the oracle's updated master."""
    import torch
    d, ffn, vocab = 64, 172, 500
    blocks = [[d * d] * 4 + [d * ffn] * 2 + [ffn * d, d, d] for _ in range(3)]
    numels = [vocab * d] + [n for b in blocks for n in b] + [d, vocab * d]
    groups = [0] + [1 + i // 9 for i in range(27)] + [4, 4]
    c = Case(numels, 16, 16, "bf16", seed=23, groups=groups)
    Z = c.Z
    N, G = 16, len(c.groups)
    shards = [torch.full((c.info["shard_total"],), 7.0, dtype=torch.bfloat16, device=cuda)
              for _ in range(N)]
    lay_a = [torch.zeros(g["psi_pad"], dtype=torch.bfloat16, device=cuda) for g in c.groups]
    lay_b = [torch.zeros(g["psi_pad"], dtype=torch.bfloat16, device=cuda) for g in c.groups]
    grads = [c.grads_dev(gi, 1) for gi in range(G)]
    torch.cuda.synchronize()
    for gi in reversed(range(G)):
        Z.zero_step_group(c.plan, gi, grads[gi], Z.ZERO_BF16, c.master, c.m, c.v, c.hp_dev(1),
                          None, shards)
        Z.zero_gather_layer(c.plan, gi, shards, Z.ZERO_BF16, lay_a[gi])
        Z.zero_broadcast_layer(c.plan, gi, shards, Z.ZERO_BF16, lay_b[gi])
    torch.cuda.synchronize()
    for gi in reversed(range(G)):
        c.oracle_step(gi, 1)
    c.check_state("stage 3, gathers queued behind the step")
    for gi, g in enumerate(c.groups):
        f0, S = g["flat_off"], g["shard"]
        own = [O.f32_to_bf16(c.h_master[f0 + k * S:f0 + (k + 1) * S]) for k in range(N)]
        want, _, _ = O.gather_layer(own)
        want_b, _, _, _ = O.broadcast_gather(own)
        assert np.array_equal(bits_of(lay_a[gi]), want), gi
        assert np.array_equal(bits_of(lay_b[gi]), want_b), gi
    # the same gathers captured once in a CUDA graph (programmatic launches
    # become graph edges) and replayed into cleared buffers
    for t in lay_a + lay_b:
        t.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s), torch.cuda.graph(g, stream=s):
        for gi in range(G):
            Z.zero_gather_layer(c.plan, gi, shards, Z.ZERO_BF16, lay_a[gi], s)
            Z.zero_broadcast_layer(c.plan, gi, shards, Z.ZERO_BF16, lay_b[gi], s)
    torch.cuda.current_stream().wait_stream(s)
    for t in lay_a + lay_b:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    for gi, gg in enumerate(c.groups):
        f0, S = gg["flat_off"], gg["shard"]
        own = [O.f32_to_bf16(c.h_master[f0 + k * S:f0 + (k + 1) * S]) for k in range(N)]
        assert np.array_equal(bits_of(lay_a[gi]), O.gather_layer(own)[0]), ("graph", gi)
        assert np.array_equal(bits_of(lay_b[gi]), O.broadcast_gather(own)[0]), ("graph", gi)


@pytest.mark.parametrize("gd", ["bf16", "f32"])
def test_stage3_last_micro_batch_fused_into_the_group_step(cuda, gd):
    """Stage 3 with gradient accumulation: per layer group the first micro-
    batches go through zero_reduce_scatter / zero_reduce_scatter_acc into the
    flat accumulation buffer, and the last one through zero_step_group_acc
    (its ring sum added to the accumulated buffer inside the fused step,
    owners' bf16 parameters into their shard buffers).  State and shards
    equal the oracle's accumulation + Adam; the accumulated buffer is left as
    it was."""
    import torch
    M = 3
    d, ffn, vocab = 48, 130, 301
    blocks = [[d * d] * 4 + [d * ffn] * 2 + [ffn * d, d, d] for _ in range(2)]
    numels = [vocab * d] + [n for b in blocks for n in b] + [d, vocab * d]
    groups = [0] + [1 + i // 9 for i in range(18)] + [3, 3]
    c = Case(numels, 8, 8, gd, grad_sigma=1e-2 if gd == "f32" else 1e-3, seed=41, groups=groups)
    Z = c.Z
    N, G = c.n, len(c.groups)
    scale = 1.0 / (N * M)
    acc = torch.full((c.info["psi_pad"],), 5.0, dtype=torch.float32, device=cuda)
    shards = [torch.zeros(c.info["shard_total"], dtype=torch.bfloat16, device=cuda)
              for _ in range(N)]
    for gi in reversed(range(G)):
        P = c.groups[gi]["psi_pad"]
        Z.zero_reduce_scatter(c.plan, gi, c.grads_dev(gi, 50), c.zdtype, acc, 0, P, 1.0)
        for k in range(1, M - 1):
            Z.zero_reduce_scatter_acc(c.plan, gi, c.grads_dev(gi, 50 + k), c.zdtype, acc, 0, P,
                                      1.0)
    before = acc.clone()
    hp = Z.adam_hp(step=1, grad_scale=scale)
    for gi in reversed(range(G)):
        Z.zero_step_group_acc(c.plan, gi, c.grads_dev(gi, 50 + M - 1), c.zdtype, acc, c.master,
                              c.m, c.v, hp, None, shards)
    torch.cuda.synchronize()
    assert torch.equal(acc, before)
    for gi, g in enumerate(c.groups):
        f0, S, ro = g["flat_off"], g["shard"], g["rank_off"]
        red = O.ring_reduce_scatter(c.grads_host(gi, 50), S)[0]
        for k in range(1, M):
            red = O.accumulate_reduced(red, O.ring_reduce_scatter(c.grads_host(gi, 50 + k), S)[0])
        gs = O.scale(red, np.float32(scale))
        sl = slice(f0, f0 + g["psi_pad"])
        p, m, v = O.adam_update(c.h_master[sl], c.h_m[sl], c.h_v[sl], np.concatenate(gs), 1e-3,
                                0.9, 0.999, 1e-8, 0.0, 1)
        c.h_master[sl], c.h_m[sl], c.h_v[sl] = p, m, v
        for k in range(N):
            assert_bf16(bits_of(shards[k][ro:ro + S]), O.f32_to_bf16(p[k * S:(k + 1) * S]),
                        f"group {gi} shard {k}")
    c.check_state(f"stage 3 accumulation ({gd})")
