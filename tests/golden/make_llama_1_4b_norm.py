"""Writes llama_1_4b_norm.txt: the global gradient norm and clip coefficient of
the full-size Llama-1.4B workload at steps 1 and 2, computed by the CPU oracle
alone.

The workload (219 tensors, 1,345,423,360 parameters, N = 8 ranks, bf16
gradients with heavy tails, clip at max_norm 1.0) is too large to hold on the
host at once, so the script streams it in windows of the flat buffer: per
window it generates every rank's gradient with the seeded numpy generator,
runs the oracle's ring reduce-scatter over the window, scales by 1/N and adds
the window's sum of squares (fp64) to the total.  Windows are independent, so
they run in a pool of worker processes; their totals are added in window
order.  norm = sqrt(total); coef = the oracle's clip coefficient.

Nothing here reads a device result: the values are the oracle's.

    python tests/golden/make_llama_1_4b_norm.py [--workers K] [--window ELEMENTS]
"""
from __future__ import annotations

import argparse
import math
import multiprocessing as mp
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

OUT = os.path.join(HERE, "llama_1_4b_norm.txt")
STEPS = (1, 2)


def window_sum_squares(args):
    """fp64 sum of squares of the scaled reduced gradient over [a, b)."""
    step, a, b = args
    import numpy as np
    import synth
    from synth import workloads as W
    from oracle import zero_oracle as O
    w = W.LLAMA_1_4B
    p = O.plan(w.numels, w.n_ranks, w.align)
    S = p.groups[0].shard
    local = [O.bf16_to_f32(synth.values(w.seed, synth.GRAD, step, r, a, b, w.grad_sigma, w.psi,
                                        w.heavy_tail, synth.DTYPE_BF16))
             for r in range(w.n_ranks)]
    reduced, _, _ = O.ring_reduce_scatter(local, S, (a, b))
    g = O.scale(reduced, np.float32(1.0) / np.float32(w.n_ranks))
    return O.sum_squares(g)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workers", type=int, default=os.cpu_count() or 1)
    ap.add_argument("--window", type=int, default=1 << 24)
    args = ap.parse_args(argv)
    from synth import workloads as W
    from oracle import zero_oracle as O
    w = W.LLAMA_1_4B
    p = O.plan(w.numels, w.n_ranks, w.align)
    P = p.psi_pad
    lines = [
        "# Global gradient norm and clip coefficient of the full-size Llama-1.4B",
        "# workload (219 tensors, psi = 1,345,423,360, N = 8, bf16 gradients with",
        "# heavy tails, gradient scale 1/8, max_norm = 1.0) at steps 1 and 2,",
        "# computed by the CPU oracle alone, window by window, with",
        "# tests/golden/make_llama_1_4b_norm.py.  sumsq is the fp64 sum of",
        "# squares of the scaled reduced gradient (windows of "
        f"{args.window} elements added in order),",
        "# norm = sqrt(sumsq), coef = fp32(min(1, max_norm / (norm + 1e-6))).",
        "# The clip is the coefficient torch's clip_grad_norm_ applies; the pages",
        "# do not define it (the workload's 'global grad-norm clip at 1.0').",
        f"psi_pad = {P}",
    ]
    ctx = mp.get_context("spawn")
    with ctx.Pool(args.workers) as pool:
        for step in STEPS:
            t0 = time.time()
            jobs = [(step, a, min(P, a + args.window)) for a in range(0, P, args.window)]
            parts = pool.map(window_sum_squares, jobs, chunksize=1)
            total = 0.0
            for x in parts:
                total += x
            norm = math.sqrt(total)
            coef = O.clip_coef(norm, w.extra["max_norm"])
            lines += [f"sumsq_step{step} = {total!r}",
                      f"norm_step{step} = {norm!r}",
                      f"coef_step{step} = {float(coef)!r}"]
            print(f"step {step}: norm {norm!r} coef {float(coef)!r} "
                  f"({len(jobs)} windows, {time.time() - t0:.0f} s)", flush=True)
    with open(OUT, "w") as f:
        f.write("\n".join(lines) + "\n")
    print(f"wrote {OUT}")


if __name__ == "__main__":
    main()
