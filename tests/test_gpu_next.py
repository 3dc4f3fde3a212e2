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
