"""Pins of the CPU oracle to facts outside itself: hand-derived partition maps,
the pages' volume and memory formulas, worked examples, closed forms of Adam,
brute force on tiny inputs, and library routines (torch.optim.Adam,
clip_grad_norm_, torch's bf16 cast) on the special cases that reduce to them.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import zero_oracle as O
from synth import workloads as W
import synth

from conftest import read_golden

F32 = np.float32


def ints(s):
    return [int(x) for x in s.split()]


# ---------------------------------------------------------------- a1 plan --
def test_tiny_plan_matches_hand_derivation():
    gold = read_golden("tiny_plan.txt")
    p = O.plan(ints(gold["numels"]), int(gold["n_ranks"]), int(gold["align"]))
    assert p.psi == int(gold["psi"])
    assert p.psi_pad == int(gold["psi_pad"])
    assert p.groups[0].shard == int(gold["shard"])
    assert p.psi_pad - p.psi == int(gold["padding"])
    assert [p.tensor_flat_off(t) for t in range(3)] == ints(gold["tensor_flat_off"])
    for t in range(3):
        assert list(p.owner_span(t)) == ints(gold[f"owner_span_{t}"])
    for r in range(4):
        want = [tuple(ints(seg)) for seg in gold[f"segments_{r}"].split(";")]
        assert p.segments(r) == want
    assert [p.shard_range(0, r)[2] for r in range(4)] == ints(gold["valid_len"])


@pytest.mark.parametrize("w", list(W.ALL.values()), ids=lambda w: w.name)
def test_plan_of_each_workload(w):
    p = O.plan(w.numels, w.n_ranks, w.align, w.groups)
    assert len(w.numels) == {"tiny": 3, "gpt2-small": 148, "llama-1.4b": 219,
                             "gpt2-medium": 292, "llama-7b-stage3": 291}[w.name]
    shards = [g.shard for g in p.groups]
    expect = {"tiny": [2512], "gpt2-small": [15_554_976], "llama-1.4b": [168_177_920],
              "gpt2-medium": [5_544_112],
              "llama-7b-stage3": [8_192_000] + [12_648_960] * 32 + [8_192_256]}[w.name]
    assert shards == expect
    # every element of every tensor is owned exactly once; the rest is padding
    covered = 0
    for r in range(w.n_ranks):
        for t, toff, foff, n in p.segments(r):
            assert 0 <= toff and toff + n <= w.numels[t]
            assert foff == p.tensor_flat_off(t) + toff
            covered += n
    assert covered == w.psi
    for g in p.groups:
        assert g.psi_pad % (w.n_ranks * w.align) == 0
        assert 0 <= g.psi_pad - g.psi < w.n_ranks * w.align


def test_stage3_groups_are_independent_plans():
    w = W.LLAMA_7B_STAGE3
    p = O.plan(w.numels, w.n_ranks, w.align, w.groups)
    off = 0
    roff = 0
    for g in p.groups:
        sub = O.plan([w.numels[t] for t in g.tensors], w.n_ranks, w.align)
        assert (g.psi, g.psi_pad, g.shard) == (sub.psi, sub.psi_pad, sub.groups[0].shard)
        assert g.flat_off == off and g.rank_off == roff
        off += g.psi_pad
        roff += g.shard
    assert len(p.groups) == 34


def test_plan_rejects_bad_groups():
    with pytest.raises(ValueError):
        O.plan([4, 4, 4], 2, 1, [0, 2, 2])
    with pytest.raises(ValueError):
        O.plan([4, 4], 2, 1, [1, 1])
    with pytest.raises(ValueError):
        O.plan([4, 4], 0, 1)


def test_empty_and_degenerate_plans():
    p = O.plan([], 4, 16)
    assert p.psi == 0 and p.psi_pad == 0 and p.groups[0].shard == 0
    p = O.plan([0, 5, 0], 2, 1)
    assert p.owner_span(0) == (-1, -1) and p.owner_span(2) == (-1, -1)
    assert p.psi_pad == 6 and p.groups[0].shard == 3
    p = O.plan([7], 1, 1)
    assert p.groups[0].shard == 7 and p.segments(0) == [(0, 0, 0, 7)]


# ------------------------------------------------------- memory and volume --
def test_memory_formulas_from_the_wiki_page():
    gold = read_golden("memory_formulas.txt")
    P, N = int(gold["P"]), int(gold["N"])
    p = O.plan(W.GPT2_SMALL.numels, N, 16)
    assert p.psi == P and p.psi_pad == P
    for stage, key in [(0, "baseline"), (1, "stage1"), (2, "stage2"), (3, "stage3")]:
        assert p.memory(stage)[0] == int(gold[key])
    # the formulas themselves, for several N dividing P exactly
    for n in (1, 2, 4, 8, 16, 64):
        P2 = n * 1000
        q = O.plan([P2], n, 1)
        f = Fraction(P2)
        assert q.memory(1)[0] == 2 * f + 2 * f / n
        assert q.memory(2)[0] == f + 3 * f / n
        assert q.memory(3)[0] == 4 * f / n


def test_memory_reduction_limits_match_4x_and_8x_in_bytes():
    # "ZeRO Stages": stage 1 "4x", stage 2 "8x" reductions.  In bytes (bf16
    # params/grads, fp32 master+m+v) the ratio to plain DP tends to 4 and 8.
    P = 1 << 40
    for N, tol in [(1 << 20, 1e-4)]:
        p = O.plan([P], N, 1)
        base = p.memory(0)[1]
        assert abs(base / p.memory(1)[1] - 4.0) < tol
        assert abs(base / p.memory(2)[1] - 8.0) < tol
        assert p.memory(3)[1] * N == base


def test_ring_volume_counters_tiny():
    gold = read_golden("tiny_plan.txt")
    w = W.TINY
    p = O.plan(w.numels, w.n_ranks, w.align)
    S = p.groups[0].shard
    rng = np.random.default_rng(0)
    local = [rng.standard_normal(p.psi_pad).astype(F32) for _ in range(w.n_ranks)]
    red, sent, recv = O.ring_reduce_scatter(local, S)
    assert sent == recv == [int(gold["volume_per_rank"])] * 4
    assert O.volume(p) == (int(gold["volume_per_rank"]),) * 2
    _, s2, r2 = O.ring_all_gather(red, S)
    assert s2 == r2 == [int(gold["volume_per_rank"])] * 4
    # reduce-scatter + all-gather = all-reduce: 2 (N-1)/N Psi_pad per rank,
    # i.e. the "2 Psi" of standard data parallelism as N grows
    assert sent[0] + s2[0] == 2 * (w.n_ranks - 1) * p.psi_pad // w.n_ranks
    _, sn, rn = O.ring_reduce_scatter(local, S, narrated=True)
    assert sn == rn == [int(gold["narrated_volume_per_rank"])] * 4


# ----------------------------------------------------- a2 reduce-scatter --
def _brute_allreduce_chain_order(local, S):
    """Plain loop: element i of owner k's chunk = ((g[k+1] + g[k+2]) + ...) + g[k]."""
    n = len(local)
    out = np.empty_like(local[0])
    for i in range(local[0].size):
        k = i // S
        acc = F32(local[(k + 1) % n][i])
        for j in range(2, n + 1):
            acc = F32(acc + local[(k + j) % n][i])
        out[i] = acc
    return out


def test_rs_then_ag_equals_bruteforce_allreduce():
    # "Why DeepSpeed ZeRO paper says ...": all-reduce = reduce-scatter + all-gather
    rng = np.random.default_rng(1)
    for n, S in [(2, 5), (3, 7), (4, 16), (5, 3)]:
        local = [(rng.standard_normal(n * S) * 10.0 ** rng.integers(-3, 4, n * S)).astype(F32)
                 for _ in range(n)]
        red, _, _ = O.ring_reduce_scatter(local, S)
        fulls, _, _ = O.ring_all_gather(red, S)
        want = _brute_allreduce_chain_order(local, S)
        for f in fulls:
            assert np.array_equal(f.view(np.uint32), want.view(np.uint32))
        # against the exact sum: the classical error bound of recursive
        # summation, |fl - s| <= gamma_{n-1} * sum |g|
        exact = np.sum(np.stack([x.astype(np.float64) for x in local]), axis=0)
        absum = np.sum(np.abs(np.stack([x.astype(np.float64) for x in local])), axis=0)
        u = 2.0 ** -24
        gamma = (n - 1) * u / (1 - (n - 1) * u)
        assert np.all(np.abs(fulls[0].astype(np.float64) - exact) <= gamma * absum + 1e-45)


def test_ring_order_worked_example():
    gold = read_golden("ring_order_n3.txt")
    local = [np.array([float(x) for x in gold[f"g{r}"].split()], dtype=F32) for r in range(3)]
    red, _, _ = O.ring_reduce_scatter(local, 1)
    assert [float(x[0]) for x in red] == [float(x) for x in gold["reduced"].split()]
    red, _, _ = O.ring_reduce_scatter(local, 1, narrated=True)
    assert [float(x[0]) for x in red] == [float(x) for x in gold["narrated_reduced"].split()]


def test_window_matches_full_run():
    rng = np.random.default_rng(2)
    n, S = 4, 40
    local = [rng.standard_normal(n * S).astype(F32) for _ in range(n)]
    full, _, _ = O.ring_reduce_scatter(local, S)
    full = np.concatenate(full)
    for a, b in [(0, 160), (13, 97), (39, 41), (120, 160), (50, 50)]:
        part, _, _ = O.ring_reduce_scatter([x[a:b] for x in local], S, window=(a, b))
        got = np.concatenate(part) if part else np.zeros(0, F32)
        assert np.array_equal(got, full[a:b])


# ------------------------------------------------------------------ a4 Adam --
def test_adam_step1_closed_form():
    # From m = v = 0, step 1: mh = g and vh = g^2, so p1 = p0 - lr*g/(|g|+eps)
    rng = np.random.default_rng(3)
    g = (rng.standard_normal(1000) * 1e-2).astype(F32)
    p0 = (rng.standard_normal(1000) * 0.02).astype(F32)
    z = np.zeros_like(g)
    p1, m1, v1 = O.adam_update(p0, z, z, g, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1)
    g64 = g.astype(np.float64)
    want = p0.astype(np.float64) - 1e-3 * g64 / (np.abs(g64) + 1e-8)
    np.testing.assert_allclose(p1, want, rtol=0, atol=4e-9)
    # the method's betas are fp32 values: 1 - 0.9f and 1 - 0.999f
    omb1 = 1.0 - float(F32(0.9))
    omb2 = 1.0 - float(F32(0.999))
    np.testing.assert_allclose(m1, omb1 * g64, rtol=2e-7)
    np.testing.assert_allclose(v1, omb2 * g64 * g64, rtol=4e-7)


def test_adam_constant_gradient_moves_lr_per_step():
    # A constant g gives mh = g and vh = g^2 at every step, so each step moves
    # the parameter by lr*g/(|g|+eps)
    g = np.array([3e-3, -2e-2, 5e-5, -7e-4], dtype=F32)
    p = np.zeros(4, F32)
    m = np.zeros(4, F32)
    v = np.zeros(4, F32)
    for t in range(1, 11):
        p, m, v = O.adam_update(p, m, v, g, 1e-3, 0.9, 0.999, 1e-8, 0.0, t)
    g64 = g.astype(np.float64)
    np.testing.assert_allclose(p, -10 * 1e-3 * g64 / (np.abs(g64) + 1e-8), rtol=2e-5)


def test_adam_zero_gradient_leaves_parameters():
    p0 = np.array([0.5, -0.25, 1e-30, 0.0], dtype=F32)
    z = np.zeros(4, F32)
    p, m, v = O.adam_update(p0, z, z, z, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1)
    assert np.array_equal(p, p0) and not m.any() and not v.any()


def test_adam_decoupled_weight_decay_closed_form():
    p0 = np.array([0.5, -0.25, 2.0], dtype=F32)
    z = np.zeros(3, F32)
    p, _, _ = O.adam_update(p0, z, z, z, 1e-2, 0.9, 0.999, 1e-8, 0.1, 1)
    np.testing.assert_allclose(p, p0.astype(np.float64) * (1 - 1e-3), rtol=1e-7)


def test_bias_corrections():
    bc1, bc2 = O.bias_corrections(0.9, 0.999, 1)
    assert bc1 == F32(1 - float(F32(0.9))) and bc2 == F32(1 - float(F32(0.999)))
    bc1, bc2 = O.bias_corrections(0.9, 0.999, 20)
    b1, b2 = float(F32(0.9)), float(F32(0.999))
    np.testing.assert_allclose([bc1, bc2], [1 - b1 ** 20, 1 - b2 ** 20], rtol=1e-7)


def test_identical_ranks_match_torch_adam():
    torch = pytest.importorskip("torch")
    n, S = 4, 64
    rng = np.random.default_rng(4)
    p0 = (rng.standard_normal(n * S) * 0.02).astype(F32)
    master, m, v = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    # the method's hyperparameters are fp32 values; torch keeps betas as
    # doubles, so hand it the fp32 roundings of 0.9 and 0.999
    betas = (float(F32(0.9)), float(F32(0.999)))
    opt = torch.optim.Adam([tp], lr=1e-3, betas=betas, eps=1e-8, foreach=False)
    for t in range(1, 6):
        g = (rng.standard_normal(n * S) * 1e-2).astype(F32)
        r = O.zero_step([g.copy() for _ in range(n)], master, m, v, S, t, O.AdamHP())
        master, m, v = r["master"], r["m"], r["v"]
        tp.grad = torch.from_numpy(g.copy())
        opt.step()
        st = opt.state[tp]
        np.testing.assert_allclose(master, tp.detach().numpy(), rtol=1e-5, atol=1e-7)
        np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=1e-5,
                                   atol=1e-6 * np.abs(m).max())
        np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-5,
                                   atol=1e-6 * np.abs(v).max())


def test_clip_matches_torch_clip_grad_norm():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    chunks = [(rng.standard_normal(n) * 0.3).astype(F32) for n in (100, 37, 250)]
    norm, coef = O.grad_norm(chunks, 1.0)
    ts = [torch.nn.Parameter(torch.zeros(len(c))) for c in chunks]
    for t, c in zip(ts, chunks):
        t.grad = torch.from_numpy(c.copy())
    tn = torch.nn.utils.clip_grad_norm_(ts, max_norm=1.0)
    assert abs(norm - float(tn)) <= 1e-5 * norm
    for t, c in zip(ts, chunks):
        np.testing.assert_allclose((c * coef).astype(F32), t.grad.numpy(), rtol=1e-5, atol=1e-9)
    # below the threshold the coefficient is exactly 1
    _, coef = O.grad_norm([np.full(4, 0.1, F32)], 1.0)
    assert coef == F32(1.0)


# ------------------------------------------------------------- a5 bf16 cast --
def test_bf16_cast_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(6)
    x = np.concatenate([
        (rng.standard_normal(10000) * 10.0 ** rng.integers(-40, 38, 10000)).astype(F32),
        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0, -0.0, np.inf,
                  -np.inf, 3.4028235e38, 1e-45, -1e-45, 1.1754942e-38, 2 ** -133], dtype=F32)])
    got = O.f32_to_bf16(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    nan = O.f32_to_bf16(np.array([np.nan, -np.nan], dtype=F32))
    assert np.all(np.isnan(O.bf16_to_f32(nan)))


def test_bf16_roundtrip_is_exact():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    f = O.bf16_to_f32(bits)
    finite = np.isfinite(f)
    assert np.array_equal(O.f32_to_bf16(f[finite]), bits[finite])


# ----------------------------------------------------- stage-3 gather (a6) --
def test_gather_layer_is_concatenation_of_shards():
    rng = np.random.default_rng(7)
    shards = [rng.integers(0, 1 << 16, 24).astype(np.uint16) for _ in range(5)]
    layer, sent, recv = O.gather_layer(shards)
    assert np.array_equal(layer, np.concatenate(shards))
    assert sent == recv == [4 * 24] * 5


def test_broadcast_gather_pins():
    """Broadcast form of the stage-3 gather ("Why does not the stage 3
    implementation use broadcast and reduce-scatter?", answer 1: broadcast
    and all-gather move a similar volume): every rank ends with the
    concatenation of the shards (brute force); in broadcast k only the root k
    sends, (N - 1) * S elements, and every other rank receives S; summed over
    the N broadcasts each rank sends and receives (N - 1) * S, the ring
    all-gather's per-rank count."""
    rng = np.random.default_rng(17)
    for n, S in [(1, 7), (2, 5), (5, 24), (16, 3)]:
        shards = [rng.integers(0, 1 << 16, S).astype(np.uint16) for _ in range(n)]
        layer, fulls, sent, recv = O.broadcast_gather(shards)
        cat = np.concatenate(shards)
        assert np.array_equal(layer, cat)
        assert all(np.array_equal(f, cat) for f in fulls)
        for k in range(n):
            assert sent[k] == [(n - 1) * S if r == k else 0 for r in range(n)]
            assert recv[k] == [0 if r == k else S for r in range(n)]
        _, ag_sent, ag_recv = O.gather_layer(shards)
        assert [sum(sent[k][r] for k in range(n)) for r in range(n)] == ag_sent
        assert [sum(recv[k][r] for k in range(n)) for r in range(n)] == ag_recv
    # fp32 shards pass through bit for bit (NaN payloads included)
    x = [np.array([np.nan, -0.0, 1e-45], dtype=F32), np.array([np.inf, 2.5, -1.0], dtype=F32)]
    layer, _, _, _ = O.broadcast_gather(x)
    assert np.array_equal(layer.view(np.uint32), np.concatenate(x).view(np.uint32))


def test_sum_squares_is_the_exact_sum():
    """fp32 squares are exact in fp64; on values whose squares and partial
    sums are all exactly representable the sum is exact, and on random
    values it is within fp64 rounding of math.fsum's correctly rounded sum."""
    import math
    rng = np.random.default_rng(18)
    ints = [rng.integers(-1000, 1000, 300).astype(F32) for _ in range(3)]
    want = sum(int(v) ** 2 for c in ints for v in c)
    assert O.sum_squares(ints) == float(want)
    xs = [(rng.standard_normal(5000) * 10.0 ** rng.integers(-8, 4, 5000)).astype(F32)
          for _ in range(4)]
    exact = math.fsum(float(v) * float(v) for c in xs for v in c)
    assert abs(O.sum_squares(xs) - exact) <= 1e-13 * exact
    assert O.clip_coef(math.sqrt(exact), 1.0) == O.grad_norm(xs, 1.0)[1]


def test_layer_checksum_small_case():
    bits = np.array([1, 2, 3], dtype=np.uint16)
    assert O.layer_checksum(bits) == 1 * 1 + 2 * 2 + 3 * 3
    big = np.full(65537, 7, dtype=np.uint16)
    assert O.layer_checksum(big) == 7 * (sum(range(1, 65537)) + 1)


def test_consumer_rounds_match_the_iterated_multiply_add():
    """Brute force on small buffers: per 8-element vector (and per tail
    element) the consumer's term is rounds - 1 dependent steps t = t*K + c
    from t = c, mod 2**64; the oracle uses the geometric-sum form."""
    M = 1 << 64
    rng = np.random.default_rng(11)
    for n in (0, 5, 8, 21, 64):
        bits = rng.integers(0, 1 << 16, n).astype(np.uint16)
        for rounds in (1, 2, 3, 17):
            total = 0
            starts = list(range(0, n - n % 8, 8)) + list(range(n - n % 8, n))
            for a in starts:
                b = a + 8 if a < n - n % 8 else a + 1
                c = sum(int(bits[j]) * (1 + (j % 65536)) for j in range(a, b)) % M
                t = c
                for _ in range(rounds - 1):
                    t = (t * O.CONSUME_K + c) % M
                total = (total + t) % M
            assert O.layer_checksum(bits, rounds) == total, (n, rounds)
    # one element, two rounds: the term is c * (1 + K)
    one = np.array([3], dtype=np.uint16)
    assert O.layer_checksum(one, 2) == (3 * (1 + O.CONSUME_K)) % M


# ---------------------------------------- whole step: invariants and negatives --
def test_step_window_equals_full_step():
    w = W.TINY
    p = O.plan(w.numels, w.n_ranks, w.align)
    S = p.groups[0].shard
    local = [synth.values(w.seed, synth.GRAD, 1, r, 0, p.psi_pad, w.grad_sigma, p.psi)
             for r in range(w.n_ranks)]
    master = synth.values(w.seed, synth.MASTER, 0, 0, 0, p.psi_pad, w.master_sigma, p.psi)
    z = np.zeros_like(master)
    full = O.zero_step(local, master, z, z, S, 1, O.AdamHP())
    for a, b in [(0, 100), (2500, 2530), (7000, 10048), (5023, 5025)]:
        part = O.zero_step([x[a:b] for x in local], master[a:b], z[a:b], z[a:b], S, 1,
                           O.AdamHP(), window=(a, b))
        for k in ("master", "m", "v", "full"):
            assert np.array_equal(part[k], full[k][a:b])
    # padding stays exactly zero
    assert not full["master"][p.psi:].any() and not full["full"][p.psi:].any()


def test_copartition_without_reduce_scatter_is_wrong():
    # The proposal in "[REQUEST] Direct Correspondence ...", section "Thoughts
    # and viewpoints", skips the reduce-scatter: each owner would update from
    # its own local gradient only.  That differs from the all-reduced update.
    rng = np.random.default_rng(8)
    n, S = 4, 32
    local = [(rng.standard_normal(n * S) * 1e-2).astype(F32) for _ in range(n)]
    p0 = (rng.standard_normal(n * S) * 0.02).astype(F32)
    z = np.zeros_like(p0)
    right = O.zero_step(local, p0, z, z, S, 1, O.AdamHP())
    wrong_m = np.concatenate([
        O.adam_update(p0[k * S:(k + 1) * S], z[:S], z[:S], local[k][k * S:(k + 1) * S],
                      1e-3, 0.9, 0.999, 1e-8, 0.0, 1)[1] for k in range(n)])
    assert not np.allclose(wrong_m, right["m"], rtol=1e-3)


# ---------------------------------------------- planted mistakes must be caught --
def test_planted_mistakes_fail_a_pin(monkeypatch):
    """Plant plausible mistakes in the oracle (on the CPU) and check that the
    brute-force and library pins above would catch each."""
    rng = np.random.default_rng(9)
    n, S = 4, 8
    local = [(rng.standard_normal(n * S) * 10.0 ** rng.integers(-4, 4, n * S)).astype(F32)
             for _ in range(n)]
    want = _brute_allreduce_chain_order(local, S)

    # a dropped term: the owner forgets to add its own copy
    def rs_dropped(loc, S_, window=None, narrated=False):
        red, s, r = O.ring_reduce_scatter(loc, S_, window, narrated)
        return [(x - loc[k][k * S_:(k + 1) * S_]).astype(F32) for k, x in enumerate(red)], s, r
    got = np.concatenate(rs_dropped(local, S)[0])
    assert not np.array_equal(got, want)

    # a wrong chain start (plain rank order 0..N-1)
    plain = np.zeros(n * S, F32)
    for r in range(n):
        plain = (plain + local[r]).astype(F32)
    assert not np.array_equal(plain, want)

    # swapped betas in Adam are caught by the torch.optim.Adam pin
    g = (rng.standard_normal(64) * 1e-2).astype(F32)
    p0 = (rng.standard_normal(64) * 0.02).astype(F32)
    z = np.zeros_like(g)
    p1, m1, v1 = O.adam_update(p0, z, z, g, 1e-3, 0.999, 0.9, 1e-8, 0.0, 1)
    p2, m2, v2 = O.adam_update(p1, m1, v1, g * F32(-0.5), 1e-3, 0.999, 0.9, 1e-8, 0.0, 2)
    torch = pytest.importorskip("torch")
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    betas = (float(F32(0.9)), float(F32(0.999)))
    opt = torch.optim.Adam([tp], lr=1e-3, betas=betas, eps=1e-8, foreach=False)
    for gg in (g, g * F32(-0.5)):
        tp.grad = torch.from_numpy(gg.copy())
        opt.step()
    assert not np.allclose(p2, tp.detach().numpy(), rtol=1e-5, atol=1e-7)

    # a wrong sign of the update is caught by the step-1 closed form
    wrong = p0 + 1e-3 * g / (np.abs(g) + F32(1e-8))
    right = p0.astype(np.float64) - 1e-3 * g.astype(np.float64) / (np.abs(g) + 1e-8)
    assert not np.allclose(wrong, right, atol=4e-9)

    # bf16 by truncation instead of round-to-nearest-even: the torch cast pin
    x = (rng.standard_normal(4096) * 3).astype(F32)
    truncated = (x.view(np.uint32) >> 16).astype(np.uint16)
    rne = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert not np.array_equal(truncated, rne)
    assert np.array_equal(O.f32_to_bf16(x), rne)

    # a norm without the square root, or without the 1/N scale: the clip pin
    gs = [(rng.standard_normal(64) * 0.3).astype(F32) for _ in range(3)]
    tg = [torch.nn.Parameter(torch.zeros(64)) for _ in gs]
    for t_, g_ in zip(tg, gs):
        t_.grad = torch.from_numpy(g_.copy())
    tnorm = float(torch.nn.utils.clip_grad_norm_(tg, 1.0, foreach=False))
    norm, _ = O.grad_norm(gs, 1.0)
    no_sqrt = sum(float(np.dot(g_.astype(np.float64), g_)) for g_ in gs)
    assert abs(norm - tnorm) <= 1e-6 * tnorm and abs(no_sqrt - tnorm) > 1e-3 * tnorm

    # the padding rounded down instead of up: the hand-derived tiny plan
    numels, nr, al = [4096, 3000, 2904], 4, 16
    floor_pad = (sum(numels) // (nr * al)) * nr * al
    assert floor_pad != 10048 and O.plan(numels, nr, al).psi_pad == 10048

    # the consumer's rounds as K**(rounds-1) instead of the geometric sum:
    # the brute-force iteration pin
    bits = rng.integers(0, 1 << 16, 24).astype(np.uint16)
    M = 1 << 64
    base = O.layer_checksum(bits, 1)
    assert (base * pow(O.CONSUME_K, 2, M)) % M != O.layer_checksum(bits, 3)

    # shards gathered in reverse owner order: the concatenation pin
    shards = [rng.integers(0, 1 << 16, 5).astype(np.uint16) for _ in range(3)]
    layer, _, _ = O.gather_layer(shards)
    assert np.array_equal(layer, np.concatenate(shards))
    assert not np.array_equal(layer, np.concatenate(shards[::-1]))

    # a broadcast whose root also sends to itself: the per-broadcast counter
    # pin ((N - 1) * S from the root) and the all-gather total pin both fail
    _, _, sent, recv = O.broadcast_gather(shards)
    n_, S_ = len(shards), len(shards[0])
    self_send = [[n_ * S_ if r == k else 0 for r in range(n_)] for k in range(n_)]
    assert sent != self_send
    assert [sum(x[r] for x in self_send) for r in range(n_)] != O.gather_layer(shards)[1]
    assert [sum(x[r] for x in sent) for r in range(n_)] == O.gather_layer(shards)[1]

    # a norm that sums |g| instead of g*g, or squares in fp32 before the fp64
    # sum: the exact integer pin of sum_squares
    ints = [np.array([3, -4, 12], np.float32), np.array([4097], np.float32)]
    exact = 9.0 + 16.0 + 144.0 + 4097.0 ** 2
    assert O.sum_squares(ints) == exact
    assert sum(float(np.abs(x).sum()) for x in ints) != exact
    g1 = np.float32(1.0 + 2.0 ** -23)                           # (1 + 2^-23)^2 needs 47 bits
    assert float(np.float32(g1 * g1)) != (1.0 + 2.0 ** -23) ** 2
    assert O.sum_squares([np.array([g1], np.float32)]) == (1.0 + 2.0 ** -23) ** 2


def test_accumulation_over_micro_batches():
    # exact arithmetic: accumulating M micro-batches' reduce-scatters equals
    # one reduce-scatter of every rank's summed gradient; with small integer
    # values every fp32 sum is exact, so the two agree bit for bit
    rng = np.random.default_rng(10)
    n, S, M = 4, 6, 3
    mbs = [[rng.integers(-50, 50, n * S).astype(F32) for _ in range(n)] for _ in range(M)]
    acc = O.ring_reduce_scatter(mbs[0], S)[0]
    for mb in mbs[1:]:
        acc = O.accumulate_reduced(acc, O.ring_reduce_scatter(mb, S)[0])
    summed = [sum(mb[r] for mb in mbs).astype(F32) for r in range(n)]
    want = O.ring_reduce_scatter(summed, S)[0]
    for a, b in zip(acc, want):
        assert np.array_equal(a, b)
    # general values: within the recursive-summation bound of the exact sum
    mbs = [[(rng.standard_normal(n * S) * 1e-3).astype(F32) for _ in range(n)] for _ in range(M)]
    acc = O.ring_reduce_scatter(mbs[0], S)[0]
    for mb in mbs[1:]:
        acc = O.accumulate_reduced(acc, O.ring_reduce_scatter(mb, S)[0])
    terms = np.stack([x.astype(np.float64) for mb in mbs for x in mb])
    exact, absum = terms.sum(axis=0), np.abs(terms).sum(axis=0)
    k = n * M - 1
    gamma = k * 2.0 ** -24 / (1 - k * 2.0 ** -24)
    assert np.all(np.abs(np.concatenate(acc).astype(np.float64) - exact) <= gamma * absum)


def test_golden_norm_script_window_and_file():
    """The script that wrote tests/golden/llama_1_4b_norm.txt: its per-window
    sum of squares is the oracle's ring reduce-scatter, 1/N scale and fp64
    sum of squares over that window (a window across the owner 0/1 boundary),
    and the stored norms and coefficients agree with each other."""
    import importlib.util
    import math
    import os
    import synth
    from synth import workloads as W
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    spec = importlib.util.spec_from_file_location("make_norm",
                                                  os.path.join(here, "make_llama_1_4b_norm.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    w = W.LLAMA_1_4B
    p = O.plan(w.numels, w.n_ranks, w.align)
    S = p.groups[0].shard
    a, b = S - 700, S + 900
    local = [O.bf16_to_f32(synth.values(w.seed, synth.GRAD, 2, r, a, b, w.grad_sigma, w.psi,
                                        True, synth.DTYPE_BF16)) for r in range(w.n_ranks)]
    red, _, _ = O.ring_reduce_scatter(local, S, (a, b))
    want = O.sum_squares(O.scale(red, F32(1.0) / F32(w.n_ranks)))
    assert mod.window_sum_squares((2, a, b)) == want
    gold = read_golden("llama_1_4b_norm.txt")
    assert int(gold["psi_pad"]) == p.psi_pad
    for s in (1, 2):
        norm = float(gold[f"norm_step{s}"])
        assert norm == math.sqrt(float(gold[f"sumsq_step{s}"]))
        assert float(gold[f"coef_step{s}"]) == float(O.clip_coef(norm, w.extra["max_norm"]))
        assert 100.0 < norm < 200.0          # heavy tails: the clip at 1.0 is active
