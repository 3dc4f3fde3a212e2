"""Shared set-up for parity tests: one workload planned on both sides, device
buffers filled by the CUDA generator, host inputs by the numpy generator (the
same definition), and the CPU oracle's state advanced beside the device's.
Nothing the device computes is ever fed to the oracle."""
from __future__ import annotations

import numpy as np

import synth
from oracle import zero_oracle as O

F32 = np.float32


def bits_of(t) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor, or uint32 of an fp32 tensor."""
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy().view(np.uint32)


def assert_close_f32(got: np.ndarray, want: np.ndarray, what: str, exact: bool = True):
    """The contract: rel 1e-5 / abs 1e-7 on fp32; also bit-exact when the
    device follows the oracle's operation order (it does on every path)."""
    got = np.asarray(got, dtype=np.float32)
    want = np.asarray(want, dtype=np.float32)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    with np.errstate(invalid="ignore"):
        bad = ~(np.abs(got.astype(np.float64) - want) <= 1e-7 + 1e-5 * np.abs(want.astype(np.float64)))
    bad &= ~(got == want)                          # equal infinities
    bad &= ~(np.isnan(got) & np.isnan(want))
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside rel 1e-5/abs 1e-7, "
                             f"first at {i}: got {got[i]!r} want {want[i]!r}")
    if exact:
        diff = got.view(np.uint32) != want.view(np.uint32)
        if diff.any():
            i = int(np.flatnonzero(diff)[0])
            raise AssertionError(f"{what}: {int(diff.sum())} elements differ in bits, first at "
                                 f"{i}: got {got[i]!r} want {want[i]!r}")


def assert_bf16(got_bits: np.ndarray, want_bits: np.ndarray, what: str, exact: bool = True):
    """bf16 gathered parameters: within 1 bf16 ulp (the contract), and
    bit-exact when exact."""
    g = got_bits.astype(np.int32)
    w = want_bits.astype(np.int32)
    # ordered integer view of bf16 patterns for ulp distance
    def ordered(x):
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + (x & 0x7FFF))
    ulp = np.abs(ordered(g) - ordered(w))
    assert ulp.max(initial=0) <= 1, f"{what}: {int((ulp > 1).sum())} elements beyond 1 bf16 ulp"
    if exact:
        diff = got_bits != want_bits
        assert not diff.any(), f"{what}: {int(diff.sum())} bf16 elements differ in bits"


class Case:
    """A workload planned on both sides with its device and host state."""

    def __init__(self, numels, n_ranks, align, gdtype, grad_sigma=1e-3, master_sigma=0.02,
                 seed=1234, heavy_tail=False, groups=None, dev=None, hp=None, host_state=True):
        import torch
        import zero_sharded_optimizer_device_gb300 as Z
        self.Z = Z
        self.torch = torch
        self.numels = list(numels)
        self.n = n_ranks
        self.gdtype = gdtype
        self.tdtype = torch.bfloat16 if gdtype == "bf16" else torch.float32
        self.zdtype = Z.ZERO_BF16 if gdtype == "bf16" else Z.ZERO_F32
        self.sdtype = synth.DTYPE_BF16 if gdtype == "bf16" else synth.DTYPE_F32
        self.grad_sigma, self.master_sigma, self.seed = grad_sigma, master_sigma, seed
        self.heavy = heavy_tail
        self.hp = hp or O.AdamHP()
        self.dev = dev or torch.device("cuda:0")
        self.plan = Z.zero_plan(self.numels, n_ranks, align, groups)
        self.oplan = O.plan(self.numels, n_ranks, align, groups)
        self.info = Z.zero_plan_info(self.plan)
        self.groups = [Z.zero_plan_group(self.plan, g) for g in range(self.info["n_groups"])]
        P = self.info["psi_pad"]
        self.master = torch.zeros(P, dtype=torch.float32, device=self.dev)
        for g in self.groups:
            if g["psi_pad"]:
                synth.fill_tensor(self.master[g["flat_off"]:g["flat_off"] + g["psi_pad"]],
                                  seed, synth.MASTER, 0, 0, g["flat_off"], master_sigma,
                                  g["flat_off"] + g["psi"])
        self.m = torch.zeros_like(self.master)
        self.v = torch.zeros_like(self.master)
        if not host_state:          # full-size cases: the oracle works on windows only
            return
        # host (oracle) state, same generator definition
        self.h_master = np.zeros(P, F32)
        for g in self.groups:
            a = g["flat_off"]
            self.h_master[a:a + g["psi_pad"]] = synth.values(
                seed, synth.MASTER, 0, 0, a, a + g["psi_pad"], master_sigma, a + g["psi"])
        self.h_m = np.zeros(P, F32)
        self.h_v = np.zeros(P, F32)

    # ------------------------------------------------------------- inputs --
    def grads_dev(self, group: int, step: int, out=None):
        g = self.groups[group]
        ts = out or [self.torch.empty(g["psi_pad"], dtype=self.tdtype, device=self.dev)
                     for _ in range(self.n)]
        for r in range(self.n):
            synth.fill_tensor(ts[r][:g["psi_pad"]], self.seed, synth.GRAD, step, r, g["flat_off"],
                              self.grad_sigma, g["flat_off"] + g["psi"], self.heavy)
        return ts

    def grads_host(self, group: int, step: int, a: int = 0, b: int | None = None):
        g = self.groups[group]
        b = g["psi_pad"] if b is None else b
        out = []
        for r in range(self.n):
            x = synth.values(self.seed, synth.GRAD, step, r, g["flat_off"] + a, g["flat_off"] + b,
                             self.grad_sigma, g["flat_off"] + g["psi"], self.heavy, self.sdtype)
            out.append(O.bf16_to_f32(x) if self.gdtype == "bf16" else x)
        return out

    def hp_dev(self, step: int):
        return self.Z.adam_hp(step=step, grad_scale=1.0 / self.n, lr=self.hp.lr,
                              beta1=self.hp.beta1, beta2=self.hp.beta2, eps=self.hp.eps,
                              weight_decay=self.hp.weight_decay)

    # ------------------------------------------------------------- oracle --
    def oracle_step(self, group: int, step: int, clip_coef=None, out_dtype="bf16",
                    window=None):
        """Advance the host state of one group (or a window of it)."""
        g = self.groups[group]
        a, b = (0, g["psi_pad"]) if window is None else window
        f0 = g["flat_off"]
        local = self.grads_host(group, step, a, b)
        r = O.zero_step(local, self.h_master[f0 + a:f0 + b], self.h_m[f0 + a:f0 + b],
                        self.h_v[f0 + a:f0 + b], g["shard"], step, self.hp,
                        window=(a, b), clip_coef=clip_coef, out_dtype=out_dtype)
        self.h_master[f0 + a:f0 + b] = r["master"]
        self.h_m[f0 + a:f0 + b] = r["m"]
        self.h_v[f0 + a:f0 + b] = r["v"]
        return r

    def check_state(self, what: str, exact: bool = True, sl=None):
        sl = sl if sl is not None else slice(None)
        assert_close_f32(self.master[sl].cpu().numpy(), self.h_master[sl], what + " master", exact)
        assert_close_f32(self.m[sl].cpu().numpy(), self.h_m[sl], what + " m", exact)
        assert_close_f32(self.v[sl].cpu().numpy(), self.h_v[sl], what + " v", exact)

    def oracle_window(self, group: int, window, steps, clip_coefs=None, out_dtype="bf16"):
        """Run the oracle for `steps` (an iterable of step numbers) on one
        window of a group, from freshly generated master weights and m = v =
        0; returns the last step's result dict."""
        g = self.groups[group]
        a, b = window
        f0 = g["flat_off"]
        master = synth.values(self.seed, synth.MASTER, 0, 0, f0 + a, f0 + b, self.master_sigma,
                              f0 + g["psi"])
        m = np.zeros_like(master)
        v = np.zeros_like(master)
        r = None
        for i, s in enumerate(steps):
            local = self.grads_host(group, s, a, b)
            coef = None if clip_coefs is None else clip_coefs[i]
            r = O.zero_step(local, master, m, v, g["shard"], s, self.hp, window=(a, b),
                            clip_coef=coef, out_dtype=out_dtype)
            master, m, v = r["master"], r["m"], r["v"]
        return r

    def check_window(self, group: int, window, r, what: str, exact: bool = True):
        g = self.groups[group]
        f0 = g["flat_off"]
        sl = slice(f0 + window[0], f0 + window[1])
        assert_close_f32(self.master[sl].cpu().numpy(), r["master"], what + " master", exact)
        assert_close_f32(self.m[sl].cpu().numpy(), r["m"], what + " m", exact)
        assert_close_f32(self.v[sl].cpu().numpy(), r["v"], what + " v", exact)


def boundary_windows(P: int, cuts, half: int):
    """Windows of +-half elements around every cut (clipped to [0, P)),
    merged where they overlap, plus the first and last elements."""
    ws = [(0, min(P, 2 * half)), (max(0, P - 2 * half), P)]
    for c in cuts:
        ws.append((max(0, c - half), min(P, c + half)))
    ws.sort()
    out = []
    for a, b in ws:
        if out and a <= out[-1][1]:
            out[-1] = (out[-1][0], max(out[-1][1], b))
        else:
            out.append((a, b))
    return out
