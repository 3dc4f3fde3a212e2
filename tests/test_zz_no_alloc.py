"""The allocation-free reduce-scatter + norm entry point.

zero_reduce_scatter_norm_static serves callers that cannot allocate device
memory where they clip (code under another framework's allocator or memory
budget, loops that must not take cudaMalloc's device-wide synchronisation):
its fp64 partial sums live in the library's own static device array.  This
test calls it through the C ABI twice in a row, on different windows and
gradients, and checks each result against the existing zero_reduce_scatter +
zero_grad_norm pair run with a caller-allocated partials buffer and against
the CPU oracle; an empty window after a non-empty call reads no stale slot.
The file is named to be collected last.
"""
import numpy as np
import pytest

from harness import Case, assert_close_f32

pytestmark = pytest.mark.gpu


def _reference(c, grads, begin, end, max_norm):
    """The existing entry points, partials in a torch-allocated buffer."""
    import torch
    Z = c.Z
    n = Z.zero_rs_partials(c.plan, c.zdtype, end - begin)
    partials = torch.empty(n, dtype=torch.float64, device=c.dev)
    reduced = torch.full((c.info["psi_pad"],), -3.0, dtype=torch.float32, device=c.dev)
    norm = torch.zeros(1, dtype=torch.float32, device=c.dev)
    coef = torch.zeros(1, dtype=torch.float32, device=c.dev)
    Z.zero_reduce_scatter(c.plan, 0, grads, c.zdtype, reduced, begin, end, 1.0 / c.n, partials)
    Z.zero_grad_norm(partials, n, max_norm, norm, coef)
    torch.cuda.synchronize()
    return reduced.cpu().numpy(), float(norm.item()), float(coef.item())


def _oracle(c, step, begin, end, max_norm):
    """The CPU oracle on the window: ring reduce-scatter, 1/N scale, fp64
    norm and clip coefficient."""
    from oracle import zero_oracle as O
    red, _, _ = O.ring_reduce_scatter(c.grads_host(0, step, begin, end), c.groups[0]["shard"],
                                      (begin, end))
    norm, coef = O.grad_norm(O.scale(red, np.float32(1.0) / np.float32(c.n)), max_norm)
    return np.concatenate(red), norm, float(coef)


def test_static_partials_entry_matches_allocating_entries(cuda):
    import torch
    c = Case([300_000, 77_777, 4_099], 8, 16, "bf16", seed=4242, heavy_tail=True,
             host_state=False)
    Z = c.Z
    P = c.info["psi_pad"]
    calls = [(1, 0, P, 1.0),                 # whole group, clip active
             (2, 12_345, P - 999, 1e4)]      # ragged window, fresh gradients, no clip
    for step, begin, end, max_norm in calls:
        grads = c.grads_dev(0, step)
        reduced = torch.full((P,), -3.0, dtype=torch.float32, device=cuda)
        norm = torch.zeros(1, dtype=torch.float32, device=cuda)
        coef = torch.zeros(1, dtype=torch.float32, device=cuda)
        Z.zero_reduce_scatter_norm_static(c.plan, 0, grads, c.zdtype, reduced, begin, end,
                                          1.0 / c.n, max_norm, norm, coef)
        torch.cuda.synchronize()
        got_red = reduced.cpu().numpy()
        # against the existing entry points with a caller-allocated buffer
        want_red, want_norm, want_coef = _reference(c, grads, begin, end, max_norm)
        assert_close_f32(got_red, want_red, f"reduced, call at step {step}")
        assert abs(norm.item() - want_norm) <= 1e-6 * want_norm, (norm.item(), want_norm)
        assert abs(coef.item() - want_coef) <= 1e-6 * want_coef, (coef.item(), want_coef)
        assert want_norm > 0
        # and against the oracle: the reduced window bit for bit (ring
        # order), the norm and coefficient to the fp32 rounding of an fp64 sum
        o_red, o_norm, o_coef = _oracle(c, step, begin, end, max_norm)
        assert_close_f32(got_red[begin:end], o_red, f"reduced vs oracle, step {step}")
        assert abs(norm.item() - o_norm) <= 2.0 ** -23 * o_norm, (norm.item(), o_norm)
        assert abs(coef.item() - o_coef) <= 2.0 ** -23 * o_coef, (coef.item(), o_coef)
        assert (got_red[:begin] == -3.0).all() and (got_red[end:] == -3.0).all()
    # the first call clipped, the second did not
    assert want_coef == 1.0 and o_coef == 1.0


def test_static_partials_entry_empty_window_after_a_call(cuda):
    """An empty window right after a non-empty call: no reduce-scatter runs,
    and the norm is 0 with coefficient 1 -- not the slots the earlier call
    left behind."""
    import torch
    c = Case([50_000], 4, 16, "bf16", seed=99, host_state=False)
    Z = c.Z
    P = c.info["psi_pad"]
    grads = c.grads_dev(0, 1)
    reduced = torch.zeros(P, dtype=torch.float32, device=cuda)
    out = torch.full((2,), -1.0, dtype=torch.float32, device=cuda)
    Z.zero_reduce_scatter_norm_static(c.plan, 0, grads, c.zdtype, reduced, 0, P, 0.25, 1e-3,
                                      out[0:1], out[1:2])
    torch.cuda.synchronize()
    assert out[0].item() > 0 and out[1].item() < 1.0
    reduced.fill_(-3.0)
    Z.zero_reduce_scatter_norm_static(c.plan, 0, grads, c.zdtype, reduced, 777, 777, 0.25, 1e-3,
                                      out[0:1], out[1:2])
    torch.cuda.synchronize()
    assert out[0].item() == 0.0 and out[1].item() == 1.0
    assert bool((reduced == -3.0).all())


def test_static_partials_entry_rejects_bad_arguments(cuda):
    import torch
    c = Case([1000], 4, 16, "bf16", seed=1)
    Z = c.Z
    grads = c.grads_dev(0, 1)
    red = torch.zeros(c.info["psi_pad"], dtype=torch.float32, device=cuda)
    out = torch.zeros(2, dtype=torch.float32, device=cuda)
    for args, status in [((0, 10, 1.0, out[0:1]), None),
                         ((0, 10, 0.0, out[0:1]), Z.ZERO_EINVAL),
                         ((10, 5, 1.0, out[0:1]), Z.ZERO_ERANGE),
                         ((0, 10**9, 1.0, out[0:1]), Z.ZERO_ERANGE)]:
        begin, end, max_norm, norm = args
        if status is None:
            Z.zero_reduce_scatter_norm_static(c.plan, 0, grads, c.zdtype, red, begin, end, 0.25,
                                              max_norm, norm, out[1:2])
            continue
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_reduce_scatter_norm_static(c.plan, 0, grads, c.zdtype, red, begin, end, 0.25,
                                              max_norm, norm, out[1:2])
        assert e.value.status == status
    torch.cuda.synchronize()
    assert np.isfinite(out.cpu().numpy()).all()
