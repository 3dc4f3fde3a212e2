"""Seeded synthetic inputs for the ZeRO sharded-optimizer hot path.

This module generates the inputs that both sides of every comparison consume:
per-rank gradients, the initial fp32 master parameters and the per-rank
heavy-tail masks.  It holds none of the method's arithmetic (no reduction, no
optimizer, no cast of results); it only turns a key and an element index into
a value.  The same definition is implemented twice, once here in numpy (used
for the CPU side and for windows of the large workloads) and once as a CUDA
kernel in ``synth_gen.cu`` (used to fill device buffers of up to hundreds of
GB quickly).  A test checks that the two agree bit for bit.

Definition
----------
SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014): a stream seeded with ``s`` has j-th output
``fmix(s + j*GOLDEN)`` for j = 1, 2, ..., where ``fmix`` is the published
64-bit finalizer and GOLDEN = 0x9E3779B97F4A7C15 (all arithmetic mod 2**64).

Keys.  ``key(seed, stream, step, rank)`` chains first outputs:
    k = first(seed) ^ stream; k = first(k) ^ step; k = first(k) ^ rank;
    key = first(k)
where ``first(s) = fmix(s + GOLDEN)``.

Values.  Element i of a stream with key K draws outputs 2i+1 and 2i+2 of the
SplitMix64 stream seeded with K.  Their eight 16-bit slices u_0..u_7 are summed
(Irwin-Hall with 8 terms, exact in integers) and centred:
    z = float32(sum(u) - 262140) * C,   C = float32(1/sqrt(8*(65536**2-1)/12))
so z has mean 0 and unit variance and is bounded by |z| <= sqrt(24) ~ 4.90.  The value
is float32(z * sigma) (one fp32 rounding), optionally multiplied by 100.0f
when the element is a heavy-tail element (below), then rounded to the
storage dtype (bf16: round to nearest even on the fp32 bit pattern).

Heavy tails.  Element i of rank r is a heavy-tail element when the upper 32
bits of output i+1 of the stream keyed ``key(seed, TAIL, step, r)`` are below
floor(0.01 * 2**32) = 42949672.

Padding.  Elements at or beyond the unpadded parameter count are 0.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB

# stream identifiers
GRAD = 0
MASTER = 1
TAIL = 2

TAIL_THRESHOLD = 42949672  # floor(0.01 * 2**32)
IH_CENTRE = 262140  # 8 * 32767.5
IH_SCALE = np.float32(1.0 / math.sqrt(8.0 * (65536.0 ** 2 - 1.0) / 12.0))

DTYPE_F32 = 0
DTYPE_BF16 = 1


def fmix(z: int) -> int:
    """SplitMix64 finalizer on a Python int (mod 2**64)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def splitmix64_outputs(seed: int, count: int) -> list[int]:
    """First ``count`` outputs of the SplitMix64 stream seeded with ``seed``."""
    return [fmix(seed + (j + 1) * GOLDEN) for j in range(count)]


def key(seed: int, stream: int, step: int, rank: int) -> int:
    k = fmix(seed + GOLDEN) ^ (stream & MASK64)
    k = fmix(k + GOLDEN) ^ (step & MASK64)
    k = fmix(k + GOLDEN) ^ (rank & MASK64)
    return fmix(k + GOLDEN)


def _fmix_np(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
    return z ^ (z >> np.uint64(31))


def _outputs_np(k: int, counters: np.ndarray) -> np.ndarray:
    """Outputs number ``counters`` (uint64 array) of the stream keyed ``k``."""
    with np.errstate(over="ignore"):
        return _fmix_np(np.uint64(k) + counters * np.uint64(GOLDEN))


def _bf16_bits_rne(x: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 bit patterns (nearest, ties to even)."""
    u = x.view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def values(seed: int, stream: int, step: int, rank: int, begin: int, end: int,
           sigma: float, valid: int, heavy_tail: bool = False,
           dtype: int = DTYPE_F32, block: int = 1 << 21) -> np.ndarray:
    """Elements [begin, end) of one generated stream, on the CPU.

    Returns float32 values for ``DTYPE_F32`` or uint16 bf16 bit patterns for
    ``DTYPE_BF16``.  Elements with index >= ``valid`` are 0.
    """
    n = max(0, end - begin)
    out = np.zeros(n, dtype=np.float32 if dtype == DTYPE_F32 else np.uint16)
    k = key(seed, stream, step, rank)
    kt = key(seed, TAIL, step, rank) if heavy_tail else None
    sig = np.float32(sigma)
    hundred = np.float32(100.0)
    stop = min(end, valid)
    for a in range(begin, stop, block):
        b = min(stop, a + block)
        idx = np.arange(a, b, dtype=np.uint64)
        w0 = _outputs_np(k, np.uint64(2) * idx + np.uint64(1))
        w1 = _outputs_np(k, np.uint64(2) * idx + np.uint64(2))
        s = np.zeros(b - a, dtype=np.int64)
        for w in (w0, w1):
            for sh in (0, 16, 32, 48):
                s += ((w >> np.uint64(sh)) & np.uint64(0xFFFF)).astype(np.int64)
        z = (s - IH_CENTRE).astype(np.float32) * IH_SCALE
        val = z * sig
        if kt is not None:
            h = _outputs_np(kt, idx + np.uint64(1)) >> np.uint64(32)
            val = np.where(h < np.uint64(TAIL_THRESHOLD), val * hundred, val)
        if dtype == DTYPE_F32:
            out[a - begin:b - begin] = val
        else:
            out[a - begin:b - begin] = _bf16_bits_rne(val.astype(np.float32))
    return out


# --------------------------------------------------------------------------
# CUDA implementation of the same definition (device buffers)
# --------------------------------------------------------------------------
_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(verbose: bool = False) -> str:
    """Compile ``libsynth.so`` for sm_103a with nvcc."""
    import subprocess
    nvcc = os.environ.get("NVCC", "nvcc")
    src = os.path.join(_HERE, "synth_gen.cu")
    cmd = [nvcc, "-O3", "-shared", "-Xcompiler", "-fPIC", "-cudart", "shared",
           "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
           "-o", _LIB_PATH, src]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is not built; run synth.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        lib.synth_fill.restype = ctypes.c_int
        lib.synth_fill.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int,
            ctypes.c_float, ctypes.c_float, ctypes.c_void_p]
        _lib = lib
    return _lib


def fill_device(ptr: int, seed: int, stream: int, step: int, rank: int,
                begin: int, count: int, sigma: float, valid: int,
                heavy_tail: bool = False, dtype: int = DTYPE_F32,
                cuda_stream: int = 0) -> None:
    """Fill ``count`` elements at device address ``ptr`` with elements
    [begin, begin+count) of the stream, asynchronously on ``cuda_stream``."""
    lib = _load()
    k = key(seed, stream, step, rank)
    kt = key(seed, TAIL, step, rank) if heavy_tail else 0
    rc = lib.synth_fill(ctypes.c_void_p(ptr), dtype, begin, count, valid, k, kt,
                        1 if heavy_tail else 0, float(IH_SCALE), float(np.float32(sigma)),
                        ctypes.c_void_p(cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth_fill failed with CUDA error {rc}")


def fill_tensor(t, seed: int, stream: int, step: int, rank: int, begin: int,
                sigma: float, valid: int, heavy_tail: bool = False) -> None:
    """Fill a contiguous CUDA tensor (float32 or bfloat16) on torch's current
    stream with elements [begin, begin + t.numel()) of a stream."""
    import torch
    assert t.is_cuda and t.is_contiguous()
    dt = DTYPE_F32 if t.dtype == torch.float32 else DTYPE_BF16
    assert t.dtype in (torch.float32, torch.bfloat16)
    fill_device(t.data_ptr(), seed, stream, step, rank, begin, t.numel(), sigma,
                valid, heavy_tail, dt, torch.cuda.current_stream().cuda_stream)
