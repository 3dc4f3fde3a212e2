"""Thin Python binding of libzero (argument marshalling only).

Every function has the name and argument order of its C entry point in
``include/zero.h``; device buffers may be given as torch tensors, raw
integer device addresses or None (NULL).  Streams default to torch's current
CUDA stream.  A non-zero status raises ``ZeroError``.  All computation happens
in the library's CUDA kernels; nothing here falls back to another path, and
importing this module fails loudly when the library is not built.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
# ZERO_CHECKED=1 in the environment loads the bounds-checked build of the same
# ABI instead (every kernel access tested against its buffer's extent).
LIB_PATH = os.path.join(_HERE, "libzero_checked.so" if os.environ.get("ZERO_CHECKED") == "1"
                        else "libzero.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "zero.h")

ZERO_OK = 0
ZERO_EINVAL = -1
ZERO_EALIGN = -2
ZERO_ERANGE = -3
ZERO_EDTYPE = -4
ZERO_ENOMEM = -5
ZERO_ECUDA = -6
ZERO_ETIMEOUT = -7
ZERO_F32 = 0
ZERO_BF16 = 1
ZERO_MAX_RANKS = 64
ZERO_MAX_POLLS = 10_000_000
ZERO_OCC_FUSED, ZERO_OCC_RS, ZERO_OCC_ADAM, ZERO_OCC_GATHER, ZERO_OCC_STREAM, \
    ZERO_OCC_CONSUMER, ZERO_OCC_PREFETCH = range(7)
ZERO_MAX_CONSUMER_ROUNDS = 4096
ZERO_MAX_COALESCE = 64

_NAMES = {0: "ZERO_OK", -1: "ZERO_EINVAL", -2: "ZERO_EALIGN", -3: "ZERO_ERANGE",
          -4: "ZERO_EDTYPE", -5: "ZERO_ENOMEM", -6: "ZERO_ECUDA", -7: "ZERO_ETIMEOUT"}

c_i64 = ctypes.c_int64
c_i32 = ctypes.c_int32
c_vp = ctypes.c_void_p
P = ctypes.POINTER


class ZeroError(RuntimeError):
    def __init__(self, status: int, func: str, cuda_error: int = 0):
        self.status = status
        self.name = _NAMES.get(status, str(status))
        self.cuda_error = cuda_error
        text = _lib().zero_strerror(status).decode()
        extra = f" (cudaError {cuda_error})" if status == ZERO_ECUDA else ""
        super().__init__(f"{func}: {self.name}: {text}{extra}")


class zero_plan_info_t(ctypes.Structure):
    _fields_ = [("psi", c_i64), ("psi_pad", c_i64), ("shard_total", c_i64),
                ("n_tensors", c_i64), ("n_ranks", c_i32), ("align", c_i32),
                ("n_groups", c_i32), ("reserved", c_i32)]


class zero_group_info_t(ctypes.Structure):
    _fields_ = [("psi", c_i64), ("psi_pad", c_i64), ("shard", c_i64), ("flat_off", c_i64),
                ("rank_off", c_i64), ("first_tensor", c_i64), ("n_tensors", c_i64)]


class zero_seg_t(ctypes.Structure):
    _fields_ = [("tensor", c_i64), ("tensor_off", c_i64), ("flat_off", c_i64), ("len", c_i64)]


class zero_mem_t(ctypes.Structure):
    _fields_ = [("values", c_i64), ("bytes", c_i64)]


class zero_adam_t(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("grad_scale", ctypes.c_float), ("step", c_i64), ("d_state", c_vp)]


ZERO_ADAM_STATE_BYTES = 32


class zero_bounds_t(ctypes.Structure):
    _fields_ = [("checked", c_i32), ("site", c_i32), ("count", c_i64), ("index", c_i64),
                ("lo", c_i64), ("hi", c_i64)]


ZERO_SITE_PROBE = 1


def adam_hp(step: int, grad_scale: float, lr: float = 1e-3, beta1: float = 0.9,
            beta2: float = 0.999, eps: float = 1e-8, weight_decay: float = 0.0,
            d_state=None) -> zero_adam_t:
    return zero_adam_t(lr, beta1, beta2, eps, weight_decay, grad_scale, step, _ptr(d_state))


_SIGS = {
    "zero_version": (c_i32, []),
    "zero_strerror": (ctypes.c_char_p, [c_i32]),
    "zero_last_cuda_error": (c_i32, []),
    "zero_plan": (c_i32, [P(c_i64), c_i64, c_i32, c_i32, P(c_i32), P(c_vp)]),
    "zero_plan_destroy": (c_i32, [c_vp]),
    "zero_plan_info": (c_i32, [c_vp, P(zero_plan_info_t)]),
    "zero_plan_group": (c_i32, [c_vp, c_i32, P(zero_group_info_t)]),
    "zero_plan_tensor": (c_i32, [c_vp, c_i64, P(c_i64), P(c_i32), P(c_i32)]),
    "zero_plan_shard": (c_i32, [c_vp, c_i32, c_i32, P(c_i64), P(c_i64), P(c_i64)]),
    "zero_plan_segments": (c_i32, [c_vp, c_i32, P(zero_seg_t), c_i64, P(c_i64)]),
    "zero_plan_memory": (c_i32, [c_vp, c_i32, P(zero_mem_t)]),
    "zero_plan_volume": (c_i32, [c_vp, P(c_i64), P(c_i64)]),
    "zero_rs_partials": (c_i32, [c_vp, c_i32, c_i64, P(c_i64)]),
    "zero_reduce_scatter": (c_i32, [c_vp, c_i32, P(c_vp), c_i32, c_vp, c_i64, c_i64,
                                    ctypes.c_float, c_vp, c_vp]),
    "zero_reduce_scatter_acc": (c_i32, [c_vp, c_i32, P(c_vp), c_i32, c_vp, c_i64, c_i64,
                                        ctypes.c_float, c_vp, c_vp]),
    "zero_grad_norm": (c_i32, [c_vp, c_i64, ctypes.c_float, c_vp, c_vp, c_vp]),
    "zero_adam_shard": (c_i32, [c_vp, c_i32, c_vp, c_vp, c_vp, c_vp, P(zero_adam_t), c_vp,
                                c_i64, c_i64, c_vp, c_i32, c_vp]),
    "zero_all_gather": (c_i32, [c_vp, c_i32, c_vp, c_vp, c_i32, c_vp]),
    "zero_step_clipped_partials": (c_i32, [c_vp, c_i32, c_i32, c_i64, P(c_i64)]),
    "zero_step_clipped": (c_i32, [c_vp, c_i32, P(c_vp), c_i32, c_vp, c_vp, c_vp, c_vp,
                                  P(zero_adam_t), ctypes.c_float, c_i64, c_i64, c_vp, c_i64,
                                  c_vp, c_vp, c_vp, c_i32, c_vp]),
    "zero_step": (c_i32, [c_vp, c_i32, P(c_vp), c_i32, c_vp, c_vp, c_vp, P(zero_adam_t), c_vp,
                          c_vp, c_i32, c_vp]),
    "zero_step_acc": (c_i32, [c_vp, c_i32, P(c_vp), c_i32, c_vp, c_vp, c_vp, c_vp,
                              P(zero_adam_t), c_vp, c_vp, c_i32, c_vp]),
    "zero_step_group": (c_i32, [c_vp, c_i32, P(c_vp), c_i32, c_vp, c_vp, c_vp,
                                P(zero_adam_t), c_vp, P(c_vp), c_vp]),
    "zero_step_group_acc": (c_i32, [c_vp, c_i32, P(c_vp), c_i32, c_vp, c_vp, c_vp, c_vp,
                                    P(zero_adam_t), c_vp, P(c_vp), c_vp]),
    "zero_gather_layer": (c_i32, [c_vp, c_i32, P(c_vp), c_i32, c_vp, c_vp]),
    "zero_broadcast_layer": (c_i32, [c_vp, c_i32, P(c_vp), c_i32, c_vp, c_vp]),
    "zero_gather_groups": (c_i32, [c_vp, P(c_i32), c_i32, P(c_vp), c_i32, P(c_vp), c_vp]),
    "zero_layer_checksum": (c_i32, [c_vp, c_i64, c_i32, c_vp, c_vp]),
    "zero_stage3_gather_pass": (c_i32, [c_vp, P(c_i32), c_i32, P(c_vp), P(c_vp), c_i64, c_vp,
                                        c_i32, c_vp, c_vp]),
    "zero_stage3_gather_pass_steps": (c_i32, [c_vp, P(c_i32), P(c_i32), c_i32, P(c_vp),
                                              P(c_vp), c_i64, c_vp, c_i32, c_vp, c_vp]),
    "zero_copy": (c_i32, [c_vp, c_vp, c_i64, c_vp]),
    "zero_adam_bias_corrections": (c_i32, [P(zero_adam_t), P(ctypes.c_float),
                                           P(ctypes.c_float)]),
    "zero_adam_state_init": (c_i32, [P(zero_adam_t), c_vp, c_vp]),
    "zero_adam_state_advance": (c_i32, [P(zero_adam_t), c_vp, c_vp]),
    "zero_set_occupancy": (c_i32, [c_i32, c_i32, P(c_i32)]),
    "zero_wait_flag": (c_i32, [c_vp, ctypes.c_uint32, c_i64, c_vp, c_vp]),
    "zero_reduce_scatter_norm_static": (c_i32, [c_vp, c_i32, P(c_vp), c_i32, c_vp, c_i64, c_i64,
                                                ctypes.c_float, ctypes.c_float, c_vp, c_vp,
                                                c_vp]),
    "zero_bounds_report": (c_i32, [P(zero_bounds_t), c_i32]),
    "zero_async_status": (c_i32, [P(c_i64), c_i32]),
    "zero_bounds_probe": (c_i32, [c_vp]),
}

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _LIB = lib
    return _LIB


def header_functions() -> list[str]:
    """Names of the functions include/zero.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(zero_\w+)\s*\(", text, re.M)))


# -------------------------------------------------------------- marshalling --
class _PointerAttributes(ctypes.Structure):
    """cudaPointerAttributes as the CUDA 13 runtime lays it out (with its
    trailing reserved words, which the runtime writes too)."""
    _fields_ = [("type", ctypes.c_int), ("device", ctypes.c_int),
                ("devicePointer", c_vp), ("hostPointer", c_vp),
                ("reserved", ctypes.c_long * 8)]


_CUDART = None


def _cudart():
    """The CUDA runtime libzero links against (None when it cannot load)."""
    global _CUDART
    if _CUDART is None:
        try:
            rt = ctypes.CDLL("libcudart.so.13")
            rt.cudaPointerGetAttributes.restype = ctypes.c_int
            rt.cudaPointerGetAttributes.argtypes = [P(_PointerAttributes), c_vp]
            rt.cudaGetDevice.restype = ctypes.c_int
            rt.cudaGetDevice.argtypes = [P(ctypes.c_int)]
            rt.cudaDeviceGetAttribute.restype = ctypes.c_int
            rt.cudaDeviceGetAttribute.argtypes = [P(ctypes.c_int), ctypes.c_int, ctypes.c_int]
            _CUDART = rt
        except OSError:
            _CUDART = False
    return _CUDART or None


def _host_memory_reachable(addr: int) -> bool:
    """True when the current device can dereference this host address:
    page-locked memory mapped at the same address, managed memory, or any
    host memory on a system whose GPU reads pageable memory directly."""
    rt = _cudart()
    if rt is None:
        return False
    a = _PointerAttributes()
    if rt.cudaPointerGetAttributes(ctypes.byref(a), c_vp(addr)) == 0:
        if a.type == 3 or (a.type == 1 and a.devicePointer == addr):   # managed / mapped host
            return True
    dev, flag = ctypes.c_int(), ctypes.c_int()
    pageable_access = 88                                           # cudaDevAttrPageableMemoryAccess
    return (rt.cudaGetDevice(ctypes.byref(dev)) == 0 and
            rt.cudaDeviceGetAttribute(ctypes.byref(flag), pageable_access, dev.value) == 0 and
            flag.value == 1)


def _ptr(x) -> int | None:
    """Address of a tensor the GPU can reach (a CUDA tensor on the current
    device, or a CPU tensor in host memory the device can dereference); raw
    integer addresses pass as they are."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    addr = x.data_ptr()
    if x.is_cuda:
        # the library launches on the current device: another device's memory
        # would be an illegal address there
        import torch
        if x.device.index != torch.cuda.current_device():
            raise ValueError(f"a tensor on {x.device} passed while cuda:"
                             f"{torch.cuda.current_device()} is the current device")
    elif not (x.is_pinned() or _host_memory_reachable(addr)):
        raise ValueError("a CPU tensor in pageable host memory is not device-accessible here: "
                         "use a CUDA tensor or page-locked (pinned) host memory")
    return addr


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _ptr_array(xs, n: int | None = None, what: str = "buffers"):
    """A host array of addresses; with n, the C side reads exactly n of them,
    so a list of another length is refused here."""
    if n is not None and len(xs) != n:
        raise ValueError(f"{what}: {len(xs)} given, the call reads {n}")
    arr = (c_vp * max(1, len(xs)))()
    for i, x in enumerate(xs):
        arr[i] = _ptr(x)
    return arr


def _ranks(plan, xs, what: str = "per-rank buffers", nbytes: int = 0):
    """The plan's N per-rank buffers (gradients or shards) as a host array,
    each tensor checked to hold nbytes."""
    if len(xs) == plan.n_ranks:
        for i, x in enumerate(xs):
            _need(x, nbytes, f"{what}[{i}]")
    return _ptr_array(xs, plan.n_ranks, what)


_ESIZE = {ZERO_F32: 4, ZERO_BF16: 2}


def _need(x, nbytes: int, what: str):
    """A tensor argument must be contiguous and hold the nbytes the call
    touches (a kernel would otherwise run past its end); raw integer
    addresses are the caller's responsibility, as in the C ABI."""
    if x is None or isinstance(x, int):
        return
    if not x.is_contiguous():
        raise ValueError(f"{what}: not contiguous")
    have = x.nbytes
    if have < nbytes:
        raise ValueError(f"{what}: holds {have} bytes, the call touches {nbytes}")


def _group(plan, group: int):
    """(flat_off, psi_pad) of a group, or None for an index the library will
    refuse (it reports the error)."""
    geo = plan.geometry()
    if 0 <= group < len(geo["groups"]):
        return geo["groups"][group]
    return None


def _check(status: int, func: str) -> None:
    if status != ZERO_OK:
        raise ZeroError(status, func, _lib().zero_last_cuda_error() if status == ZERO_ECUDA else 0)


class Plan:
    """Owns a zero_plan_t*; destroyed with the object."""

    def __init__(self, handle: int, n_ranks: int = 0):
        self.handle = handle
        self.n_ranks = n_ranks
        self._geometry = None

    def geometry(self) -> dict:
        """Group offsets and sizes (queried once), for the binding's buffer
        size checks."""
        if self._geometry is None:
            info = zero_plan_info(self)
            groups = []
            for g in range(info["n_groups"]):
                gi = zero_plan_group(self, g)
                groups.append((gi["flat_off"], gi["psi_pad"]))
            self._geometry = {"groups": groups, "psi_pad": info["psi_pad"],
                              "shard_total": info["shard_total"]}
        return self._geometry

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h and _LIB is not None:
            _LIB.zero_plan_destroy(h)

    @property
    def _as_parameter_(self):
        return c_vp(self.handle)


# ------------------------------------------------------------ entry points --
def zero_version() -> int:
    return _lib().zero_version()


def zero_strerror(status: int) -> str:
    return _lib().zero_strerror(status).decode()


def zero_last_cuda_error() -> int:
    return _lib().zero_last_cuda_error()


def zero_plan(numels, n_ranks: int, align: int = 16, group_of_tensor=None) -> Plan:
    n = len(numels)
    arr = (c_i64 * max(n, 1))(*[int(v) for v in numels])
    groups = None
    if group_of_tensor is not None:
        groups = (c_i32 * max(n, 1))(*[int(g) for g in group_of_tensor])
    out = c_vp()
    _check(_lib().zero_plan(arr, n, n_ranks, align, groups, ctypes.byref(out)), "zero_plan")
    return Plan(out.value, n_ranks)


def zero_plan_destroy(plan: Plan) -> None:
    """Free the plan now (otherwise it is freed with the Plan object)."""
    h, plan.handle = plan.handle, None
    if h:
        _check(_lib().zero_plan_destroy(h), "zero_plan_destroy")


def zero_plan_info(plan: Plan) -> dict:
    info = zero_plan_info_t()
    _check(_lib().zero_plan_info(plan, ctypes.byref(info)), "zero_plan_info")
    return {k: getattr(info, k) for k, _ in info._fields_ if k != "reserved"}


def zero_plan_group(plan: Plan, group: int) -> dict:
    g = zero_group_info_t()
    _check(_lib().zero_plan_group(plan, group, ctypes.byref(g)), "zero_plan_group")
    return {k: getattr(g, k) for k, _ in g._fields_}


def zero_plan_tensor(plan: Plan, t: int):
    off, a, b = c_i64(), c_i32(), c_i32()
    _check(_lib().zero_plan_tensor(plan, t, ctypes.byref(off), ctypes.byref(a), ctypes.byref(b)),
           "zero_plan_tensor")
    return off.value, a.value, b.value


def zero_plan_shard(plan: Plan, group: int, rank: int):
    b, n, v = c_i64(), c_i64(), c_i64()
    _check(_lib().zero_plan_shard(plan, group, rank, ctypes.byref(b), ctypes.byref(n),
                                  ctypes.byref(v)), "zero_plan_shard")
    return b.value, n.value, v.value


def zero_plan_segments(plan: Plan, rank: int):
    n = c_i64()
    _check(_lib().zero_plan_segments(plan, rank, None, 0, ctypes.byref(n)), "zero_plan_segments")
    buf = (zero_seg_t * max(n.value, 1))()
    _check(_lib().zero_plan_segments(plan, rank, buf, n.value, ctypes.byref(n)),
           "zero_plan_segments")
    return [(s.tensor, s.tensor_off, s.flat_off, s.len) for s in buf[:n.value]]


def zero_plan_memory(plan: Plan, stage: int):
    m = zero_mem_t()
    _check(_lib().zero_plan_memory(plan, stage, ctypes.byref(m)), "zero_plan_memory")
    return m.values, m.bytes


def zero_plan_volume(plan: Plan):
    s, r = c_i64(), c_i64()
    _check(_lib().zero_plan_volume(plan, ctypes.byref(s), ctypes.byref(r)), "zero_plan_volume")
    return s.value, r.value


def zero_rs_partials(plan: Plan, gdtype: int, n_elements: int) -> int:
    n = c_i64()
    _check(_lib().zero_rs_partials(plan, gdtype, n_elements, ctypes.byref(n)), "zero_rs_partials")
    return n.value


def zero_reduce_scatter(plan, group, grads, gdtype, reduced, begin, end, grad_scale,
                        sumsq_partials=None, stream=None) -> None:
    g, es = _group(plan, group), _ESIZE.get(gdtype, 0)
    if g is not None and 0 <= begin <= end <= g[1]:
        _need(reduced, (g[0] + end) * 4, "reduced")
        if sumsq_partials is not None and es:
            _need(sumsq_partials, zero_rs_partials(plan, gdtype, end - begin) * 8, "partials")
    grad_ptrs = _ranks(plan, grads, "grads", g[1] * es if g else 0)
    _check(_lib().zero_reduce_scatter(plan, group, grad_ptrs, gdtype, _ptr(reduced),
                                      begin, end, grad_scale, _ptr(sumsq_partials),
                                      _stream(stream)), "zero_reduce_scatter")


def zero_reduce_scatter_acc(plan, group, grads, gdtype, reduced, begin, end, grad_scale,
                            sumsq_partials=None, stream=None) -> None:
    g, es = _group(plan, group), _ESIZE.get(gdtype, 0)
    if g is not None and 0 <= begin <= end <= g[1]:
        _need(reduced, (g[0] + end) * 4, "reduced")
        if sumsq_partials is not None and es:
            _need(sumsq_partials, zero_rs_partials(plan, gdtype, end - begin) * 8, "partials")
    grad_ptrs = _ranks(plan, grads, "grads", g[1] * es if g else 0)
    _check(_lib().zero_reduce_scatter_acc(plan, group, grad_ptrs, gdtype, _ptr(reduced),
                                          begin, end, grad_scale, _ptr(sumsq_partials),
                                          _stream(stream)), "zero_reduce_scatter_acc")


def zero_grad_norm(partials, n, max_norm, d_norm, d_coef, stream=None) -> None:
    _need(partials, max(0, n) * 8, "partials")
    _need(d_norm, 4, "d_norm")
    _need(d_coef, 4, "d_coef")
    _check(_lib().zero_grad_norm(_ptr(partials), n, max_norm, _ptr(d_norm), _ptr(d_coef),
                                 _stream(stream)), "zero_grad_norm")


def zero_adam_shard(plan, group, master, m, v, reduced, hp, d_coef, begin, end, out,
                    out_dtype=ZERO_BF16, stream=None) -> None:
    g = _group(plan, group)
    if g is not None and 0 <= begin <= end <= g[1]:
        for x, what in ((master, "master"), (m, "m"), (v, "v"), (reduced, "reduced")):
            _need(x, (g[0] + end) * 4, what)
        _need(out, (g[0] + end) * _ESIZE.get(out_dtype, 0), "out")
    _need(d_coef, 4, "d_coef")
    _check(_lib().zero_adam_shard(plan, group, _ptr(master), _ptr(m), _ptr(v), _ptr(reduced),
                                  ctypes.byref(hp), _ptr(d_coef), begin, end, _ptr(out),
                                  out_dtype, _stream(stream)), "zero_adam_shard")


def zero_step_clipped_partials(plan, group, gdtype, bucket) -> int:
    n = c_i64()
    _check(_lib().zero_step_clipped_partials(plan, group, gdtype, bucket, ctypes.byref(n)),
           "zero_step_clipped_partials")
    return n.value


def zero_step_clipped(plan, group, grads, gdtype, reduced, master, m, v, hp, max_norm, bucket,
                      chunk, partials, n_partials, d_norm, d_coef, full_out,
                      out_dtype=ZERO_BF16, stream=None) -> None:
    g, es = _group(plan, group), _ESIZE.get(gdtype, 0)
    if g is not None:
        for x, what in ((reduced, "reduced"), (master, "master"), (m, "m"), (v, "v")):
            _need(x, (g[0] + g[1]) * 4, what)
        _need(full_out, (g[0] + g[1]) * _ESIZE.get(out_dtype, 0), "full_out")
    _need(partials, max(0, n_partials) * 8, "partials")
    _need(d_norm, 4, "d_norm")
    _need(d_coef, 4, "d_coef")
    grad_ptrs = _ranks(plan, grads, "grads", g[1] * es if g else 0)
    _check(_lib().zero_step_clipped(plan, group, grad_ptrs, gdtype, _ptr(reduced),
                                    _ptr(master), _ptr(m), _ptr(v), ctypes.byref(hp), max_norm,
                                    bucket, chunk, _ptr(partials), n_partials, _ptr(d_norm),
                                    _ptr(d_coef), _ptr(full_out), out_dtype, _stream(stream)),
           "zero_step_clipped")


def zero_all_gather(plan, group, master, full_out, out_dtype=ZERO_BF16, stream=None) -> None:
    g = _group(plan, group) if group != -1 else (0, plan.geometry()["psi_pad"])
    if g is not None:
        _need(master, (g[0] + g[1]) * 4, "master")
        _need(full_out, (g[0] + g[1]) * _ESIZE.get(out_dtype, 0), "full_out")
    _check(_lib().zero_all_gather(plan, group, _ptr(master), _ptr(full_out), out_dtype,
                                  _stream(stream)), "zero_all_gather")


def zero_step(plan, group, grads, gdtype, master, m, v, hp, d_coef, full_out,
              out_dtype=ZERO_BF16, stream=None) -> None:
    g, es = _group(plan, group), _ESIZE.get(gdtype, 0)
    if g is not None:
        for x, what in ((master, "master"), (m, "m"), (v, "v")):
            _need(x, (g[0] + g[1]) * 4, what)
        _need(full_out, (g[0] + g[1]) * _ESIZE.get(out_dtype, 0), "full_out")
    _need(d_coef, 4, "d_coef")
    grad_ptrs = _ranks(plan, grads, "grads", g[1] * es if g else 0)
    _check(_lib().zero_step(plan, group, grad_ptrs, gdtype, _ptr(master), _ptr(m),
                            _ptr(v), ctypes.byref(hp), _ptr(d_coef), _ptr(full_out), out_dtype,
                            _stream(stream)), "zero_step")


def prepare_zero_step(plan, group, grads, gdtype, master, m, v, d_coef, full_out,
                      out_dtype=ZERO_BF16, stream=None):
    """zero_step with its buffers checked and marshalled once: returns a
    function step(hp) that launches the same call with this step's Adam
    hyperparameters.  For small, host-bound workloads, where the binding's
    per-call checks cost more than the kernel.  The caller keeps every buffer
    alive, in place and at its size while the function is used."""
    g, es = _group(plan, group), _ESIZE.get(gdtype, 0)
    if g is not None:
        for x, what in ((master, "master"), (m, "m"), (v, "v")):
            _need(x, (g[0] + g[1]) * 4, what)
        _need(full_out, (g[0] + g[1]) * _ESIZE.get(out_dtype, 0), "full_out")
    _need(d_coef, 4, "d_coef")
    grad_ptrs = _ranks(plan, grads, "grads", g[1] * es if g else 0)
    head = (plan, group, grad_ptrs, gdtype, _ptr(master), _ptr(m), _ptr(v))
    tail = (_ptr(d_coef), _ptr(full_out), out_dtype, _stream(stream))
    f = _lib().zero_step

    def step(hp) -> None:
        _check(f(*head, ctypes.byref(hp), *tail), "zero_step")

    step.keep = (grads, master, m, v, d_coef, full_out)   # the buffers stay referenced
    return step


def zero_step_acc(plan, group, grads, gdtype, accumulated, master, m, v, hp, d_coef, full_out,
                  out_dtype=ZERO_BF16, stream=None) -> None:
    g, es = _group(plan, group), _ESIZE.get(gdtype, 0)
    if g is not None:
        for x, what in ((accumulated, "accumulated"), (master, "master"), (m, "m"), (v, "v")):
            _need(x, (g[0] + g[1]) * 4, what)
        _need(full_out, (g[0] + g[1]) * _ESIZE.get(out_dtype, 0), "full_out")
    _need(d_coef, 4, "d_coef")
    grad_ptrs = _ranks(plan, grads, "grads", g[1] * es if g else 0)
    _check(_lib().zero_step_acc(plan, group, grad_ptrs, gdtype, _ptr(accumulated), _ptr(master),
                                _ptr(m), _ptr(v), ctypes.byref(hp), _ptr(d_coef),
                                _ptr(full_out), out_dtype, _stream(stream)), "zero_step_acc")


def zero_step_group(plan, group, grads, gdtype, master, m, v, hp, d_coef, shards,
                    stream=None) -> None:
    g, es = _group(plan, group), _ESIZE.get(gdtype, 0)
    if g is not None:
        for x, what in ((master, "master"), (m, "m"), (v, "v")):
            _need(x, (g[0] + g[1]) * 4, what)
    _need(d_coef, 4, "d_coef")
    grad_ptrs = _ranks(plan, grads, "grads", g[1] * es if g else 0)
    shard_ptrs = _ranks(plan, shards, "shards", plan.geometry()["shard_total"] * 2)
    _check(_lib().zero_step_group(plan, group, grad_ptrs, gdtype, _ptr(master), _ptr(m),
                                  _ptr(v), ctypes.byref(hp), _ptr(d_coef), shard_ptrs,
                                  _stream(stream)), "zero_step_group")


def zero_step_group_acc(plan, group, grads, gdtype, accumulated, master, m, v, hp, d_coef,
                        shards, stream=None) -> None:
    g, es = _group(plan, group), _ESIZE.get(gdtype, 0)
    if g is not None:
        for x, what in ((accumulated, "accumulated"), (master, "master"), (m, "m"), (v, "v")):
            _need(x, (g[0] + g[1]) * 4, what)
    _need(d_coef, 4, "d_coef")
    grad_ptrs = _ranks(plan, grads, "grads", g[1] * es if g else 0)
    shard_ptrs = _ranks(plan, shards, "shards", plan.geometry()["shard_total"] * 2)
    _check(_lib().zero_step_group_acc(plan, group, grad_ptrs, gdtype, _ptr(accumulated),
                                      _ptr(master), _ptr(m), _ptr(v), ctypes.byref(hp),
                                      _ptr(d_coef), shard_ptrs, _stream(stream)),
           "zero_step_group_acc")


def zero_gather_layer(plan, group, shards, dtype, layer_out, stream=None) -> None:
    g, es = _group(plan, group), _ESIZE.get(dtype, 0)
    if g is not None:
        _need(layer_out, g[1] * es, "layer_out")
    shard_ptrs = _ranks(plan, shards, "shards", plan.geometry()["shard_total"] * es)
    _check(_lib().zero_gather_layer(plan, group, shard_ptrs, dtype, _ptr(layer_out),
                                    _stream(stream)), "zero_gather_layer")


def zero_broadcast_layer(plan, group, shards, dtype, layer_out, stream=None) -> None:
    g, es = _group(plan, group), _ESIZE.get(dtype, 0)
    if g is not None:
        _need(layer_out, g[1] * es, "layer_out")
    shard_ptrs = _ranks(plan, shards, "shards", plan.geometry()["shard_total"] * es)
    _check(_lib().zero_broadcast_layer(plan, group, shard_ptrs, dtype, _ptr(layer_out),
                                       _stream(stream)), "zero_broadcast_layer")


def zero_gather_groups(plan, groups, shards, dtype, layer_outs, stream=None) -> None:
    es = _ESIZE.get(dtype, 0)
    if len(layer_outs) == len(groups):
        for i, (gid, out) in enumerate(zip(groups, layer_outs)):
            g = _group(plan, int(gid))
            if g is not None:
                _need(out, g[1] * es, f"layer_outs[{i}]")
    shard_ptrs = _ranks(plan, shards, "shards", plan.geometry()["shard_total"] * es)
    out_ptrs = _ptr_array(layer_outs, len(groups), "layer_outs")
    arr = (c_i32 * max(1, len(groups)))(*[int(g) for g in groups])
    _check(_lib().zero_gather_groups(plan, arr, len(groups), shard_ptrs, dtype,
                                     out_ptrs, _stream(stream)),
           "zero_gather_groups")


def zero_stage3_gather_pass(plan, order, shards, layer_bufs, buf_elems, d_sums,
                            consumer_rounds, stream_a, stream_b) -> None:
    shard_ptrs = _ranks(plan, shards, "shards", plan.geometry()["shard_total"] * 2)
    if len(layer_bufs) == 2:
        for i, b in enumerate(layer_bufs):
            _need(b, max(0, buf_elems) * 2, f"layer_bufs[{i}]")
    _need(d_sums, len(order) * 8, "d_sums")
    buf_ptrs = _ptr_array(layer_bufs, 2, "layer_bufs")
    arr = (c_i32 * max(1, len(order)))(*[int(g) for g in order])
    _check(_lib().zero_stage3_gather_pass(plan, arr, len(order), shard_ptrs,
                                          buf_ptrs, buf_elems, _ptr(d_sums),
                                          consumer_rounds, _stream(stream_a), _stream(stream_b)),
           "zero_stage3_gather_pass")


def zero_stage3_gather_pass_steps(plan, steps, shards, layer_bufs, buf_elems, d_sums,
                                  consumer_rounds, stream_a, stream_b) -> None:
    """steps: a list of group lists, one per step (the C call's step_first
    and step_groups are built from it)."""
    shard_ptrs = _ranks(plan, shards, "shards", plan.geometry()["shard_total"] * 2)
    if len(layer_bufs) == 2:
        for i, b in enumerate(layer_bufs):
            _need(b, max(0, buf_elems) * 2, f"layer_bufs[{i}]")
    _need(d_sums, len(steps) * 8, "d_sums")
    buf_ptrs = _ptr_array(layer_bufs, 2, "layer_bufs")
    first = [0]
    for st in steps:
        first.append(first[-1] + len(st))
    flat = [int(g) for st in steps for g in st]
    fa = (c_i32 * len(first))(*first)
    ga = (c_i32 * max(1, len(flat)))(*flat)
    _check(_lib().zero_stage3_gather_pass_steps(plan, fa, ga, len(steps), shard_ptrs,
                                                buf_ptrs, buf_elems, _ptr(d_sums),
                                                consumer_rounds, _stream(stream_a),
                                                _stream(stream_b)),
           "zero_stage3_gather_pass_steps")


def zero_layer_checksum(layer, n, rounds, d_out, stream=None) -> None:
    _need(layer, max(0, n) * 2, "layer")
    _need(d_out, 8, "d_out")
    _check(_lib().zero_layer_checksum(_ptr(layer), n, rounds, _ptr(d_out), _stream(stream)),
           "zero_layer_checksum")


def zero_adam_bias_corrections(hp):
    """(bc1, bc2): the fp32 bias corrections the device calls use for
    hp.step (host only)."""
    a, b = ctypes.c_float(), ctypes.c_float()
    _check(_lib().zero_adam_bias_corrections(ctypes.byref(hp), ctypes.byref(a), ctypes.byref(b)),
           "zero_adam_bias_corrections")
    return a.value, b.value


def zero_adam_state_init(hp, d_state, stream=None) -> None:
    _need(d_state, ZERO_ADAM_STATE_BYTES, "d_state")
    _check(_lib().zero_adam_state_init(ctypes.byref(hp), _ptr(d_state), _stream(stream)),
           "zero_adam_state_init")


def zero_adam_state_advance(hp, d_state, stream=None) -> None:
    _need(d_state, ZERO_ADAM_STATE_BYTES, "d_state")
    _check(_lib().zero_adam_state_advance(ctypes.byref(hp), _ptr(d_state), _stream(stream)),
           "zero_adam_state_advance")


def zero_set_occupancy(kind: int, blocks_per_sm: int) -> int:
    """Set a kernel family's resident blocks per SM (0 = default); returns
    the previous value."""
    prev = c_i32()
    _check(_lib().zero_set_occupancy(kind, blocks_per_sm, ctypes.byref(prev)),
           "zero_set_occupancy")
    return prev.value


def zero_wait_flag(flag, expected, max_polls, d_status, stream=None) -> None:
    _need(flag, 4, "flag")
    _need(d_status, 4, "d_status")
    _check(_lib().zero_wait_flag(_ptr(flag), expected, max_polls, _ptr(d_status),
                                 _stream(stream)), "zero_wait_flag")


def zero_copy(dst, src, nbytes, stream=None) -> None:
    _need(dst, max(0, nbytes), "dst")
    _need(src, max(0, nbytes), "src")
    _check(_lib().zero_copy(_ptr(dst), _ptr(src), nbytes, _stream(stream)), "zero_copy")


def zero_reduce_scatter_norm_static(plan, group, grads, gdtype, reduced, begin, end, grad_scale,
                                    max_norm, d_norm, d_coef, stream=None) -> None:
    """zero_reduce_scatter + zero_grad_norm for one window with the fp64
    partials in the library's static device array: for callers that cannot
    allocate device memory where they clip (see include/zero.h)."""
    g, es = _group(plan, group), _ESIZE.get(gdtype, 0)
    if g is not None and 0 <= begin <= end <= g[1]:
        _need(reduced, (g[0] + end) * 4, "reduced")
    _need(d_norm, 4, "d_norm")
    _need(d_coef, 4, "d_coef")
    grad_ptrs = _ranks(plan, grads, "grads", g[1] * es if g else 0)
    _check(_lib().zero_reduce_scatter_norm_static(
        plan, group, grad_ptrs, gdtype, _ptr(reduced), begin, end, grad_scale, max_norm,
        _ptr(d_norm), _ptr(d_coef), _stream(stream)), "zero_reduce_scatter_norm_static")


def zero_bounds_report(reset: bool = False) -> dict:
    """The checked build's record of out-of-extent kernel accesses on the
    current device (synchronizes it); the release build reports checked = 0."""
    b = zero_bounds_t()
    _check(_lib().zero_bounds_report(ctypes.byref(b), 1 if reset else 0), "zero_bounds_report")
    return {k: getattr(b, k) for k, _ in zero_bounds_t._fields_}


def zero_bounds_probe(stream=None) -> None:
    _check(_lib().zero_bounds_probe(_stream(stream)), "zero_bounds_probe")


def zero_async_status(reset: bool = False) -> int:
    """Bounded device waits that gave up since the last reset (synchronizes)."""
    n = c_i64()
    _check(_lib().zero_async_status(ctypes.byref(n), 1 if reset else 0), "zero_async_status")
    return n.value
