"""Parameter-list shapes of the synthetic workloads (shapes and seeds only).

Each workload is a list of per-tensor element counts in the order a
Hugging-Face-style state dict lists them, the number of emulated data-parallel
ranks N, the shard alignment in elements, the gradient dtype and spread, and
(for the stage-3 workload) the layer group of every tensor.  No method
arithmetic lives here.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    numels: tuple
    n_ranks: int
    align: int
    grad_dtype: str          # "f32" or "bf16"
    grad_sigma: float
    master_sigma: float
    seed: int
    steps: int
    heavy_tail: bool = False
    groups: tuple | None = None   # layer group of each tensor (stage 3)
    extra: dict = field(default_factory=dict)

    @property
    def psi(self) -> int:
        return sum(self.numels)


def _gpt2(d: int, layers: int, vocab: int = 50257, ctx: int = 1024) -> list[int]:
    out = [vocab * d, ctx * d]                      # wte, wpe
    for _ in range(layers):
        out += [d, d,                               # ln_1 weight, bias
                d * 3 * d, 3 * d,                   # attn.c_attn weight, bias
                d * d, d,                           # attn.c_proj weight, bias
                d, d,                               # ln_2 weight, bias
                d * 4 * d, 4 * d,                   # mlp.c_fc weight, bias
                4 * d * d, d]                       # mlp.c_proj weight, bias
    out += [d, d]                                   # ln_f weight, bias (lm_head tied)
    return out


def _llama_blocks(d: int, ffn: int, layers: int) -> list[list[int]]:
    blocks = []
    for _ in range(layers):
        blocks.append([d * d, d * d, d * d, d * d,  # q, k, v, o projections
                       d * ffn, d * ffn,            # gate, up
                       ffn * d,                     # down
                       d, d])                       # input / post-attention RMSNorm
    return blocks


def _llama(d: int, ffn: int, layers: int, vocab: int = 32000):
    emb = [vocab * d]
    blocks = _llama_blocks(d, ffn, layers)
    head = [d, vocab * d]                            # final norm, untied lm_head
    numels = emb + [n for b in blocks for n in b] + head
    groups = [0] + [1 + li for li, b in enumerate(blocks) for _ in b] + [layers + 1] * 2
    return numels, groups


TINY = Workload("tiny", (4096, 3000, 2904), n_ranks=4, align=16, grad_dtype="f32",
                grad_sigma=1e-2, master_sigma=0.02, seed=0x5EED0000, steps=3)

GPT2_SMALL = Workload("gpt2-small", tuple(_gpt2(768, 12)), n_ranks=8, align=16,
                      grad_dtype="bf16", grad_sigma=1e-3, master_sigma=0.02,
                      seed=0x5EED0001, steps=5)

_l14, _ = _llama(2048, 5504, 24)
LLAMA_1_4B = Workload("llama-1.4b", tuple(_l14), n_ranks=8, align=16, grad_dtype="bf16",
                      grad_sigma=1e-3, master_sigma=0.02, seed=0x5EED0002, steps=5,
                      heavy_tail=True,
                      extra={"bucket": 50_000_000, "chunk": 200_000_000, "max_norm": 1.0})

GPT2_MEDIUM = Workload("gpt2-medium", tuple(_gpt2(1024, 24)), n_ranks=64, align=1,
                       grad_dtype="bf16", grad_sigma=1e-3, master_sigma=0.02,
                       seed=0x5EED0003, steps=3)

_l7, _g7 = _llama(4096, 11008, 32)
LLAMA_7B_STAGE3 = Workload("llama-7b-stage3", tuple(_l7), n_ranks=16, align=16,
                           grad_dtype="bf16", grad_sigma=1e-3, master_sigma=0.02,
                           seed=0x5EED0004, steps=1, groups=tuple(_g7))

ALL = {w.name: w for w in (TINY, GPT2_SMALL, LLAMA_1_4B, GPT2_MEDIUM, LLAMA_7B_STAGE3)}


def mini(w: Workload, n_tensors: int = 0, scale: int = 256) -> Workload:
    """A small workload with the same N, align, dtype and a ragged tensor list:
    the workload's own tensor sizes divided by ``scale`` (at least 1), plus an
    odd-sized tensor so the padding path is exercised."""
    nums = [max(1, n // scale) + (i % 7) for i, n in enumerate(w.numels)]
    if n_tensors:
        nums = nums[:n_tensors]
    nums.append(1 + 3 * w.n_ranks)
    groups = None
    if w.groups is not None:
        g = list(w.groups[:len(nums) - 1])
        g.append(g[-1])
        groups = tuple(g)
    return Workload(w.name + "-mini", tuple(nums), w.n_ranks, w.align, w.grad_dtype,
                    w.grad_sigma, w.master_sigma, w.seed + 0x100, w.steps, w.heavy_tail,
                    groups, dict(w.extra))
