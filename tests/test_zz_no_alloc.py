"""The allocation-free reduce-scatter + norm entry point.

zero_reduce_scatter_norm_static serves callers that cannot allocate device
memory where they clip (code under another framework's allocator or memory
budget, loops that must not take cudaMalloc's device-wide synchronisation):
its fp64 partial sums live in the library's own static device array.  This
test calls it through the C ABI twice in a row, on different windows and
gradients, and checks each result against the existing zero_reduce_scatter +
zero_grad_norm pair run with a caller-allocated partials buffer.  The file is
named to be collected last.
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


def test_static_partials_entry_matches_allocating_entries(cuda):
    import torch
    c = Case([300_000, 77_777, 4_099], 8, 16, "bf16", seed=4242, heavy_tail=True)
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
        want_red, want_norm, want_coef = _reference(c, grads, begin, end, max_norm)
        assert_close_f32(reduced.cpu().numpy(), want_red, f"reduced, call at step {step}")
        assert abs(norm.item() - want_norm) <= 1e-6 * want_norm, (norm.item(), want_norm)
        assert abs(coef.item() - want_coef) <= 1e-6 * want_coef, (coef.item(), want_coef)
        assert want_norm > 0
    # the first call clipped, the second did not
    assert want_coef == 1.0


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
