"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print for a worked example (fixtures under tests/golden, each with its
citation), closed forms, hand-derived table lookups, library routines for
special cases (numpy's first-occurrence argmax, float32 accumulate) and brute
force over every prefix-respecting allocation on tiny inputs.
"""

import itertools
import math

import numpy as np
import pytest

from conftest import golden
from confidence_scheduled_speculative_gb300 import workloads as wl

EPS_MIN = 2.0 ** -14


# ----------------------------------------------------------------------- STS

def test_sts_closed_forms(orc):
    # sigmoid(0) = 1/2 for any temperature
    for T in (0.5, 1.0, 3.0):
        assert orc.sts(0.0, T) == 0.5
    ln3 = float(np.float32(math.log(3.0)))
    # sigmoid(ln 3) = 3/4; dividing by T (not multiplying) keeps 3/4 at z=2ln3, T=2
    assert abs(orc.sts(ln3, 1.0) - 0.75) < 1e-7
    assert abs(orc.sts(2 * ln3, 2.0) - 0.75) < 1e-7
    assert abs(orc.sts(ln3 / 2, 0.5) - 0.75) < 1e-7
    # sign: sigmoid(-ln 3) = 1/4
    assert abs(orc.sts(-ln3, 1.0) - 0.25) < 1e-7
    # saturation
    assert orc.sts(40.0, 1.0) == 1.0
    assert 0.0 <= orc.sts(-120.0, 1.0) < 1e-30


def test_sts_symmetry(orc):
    rng = np.random.default_rng(3)
    for z in rng.normal(0, 4, size=200).astype(np.float32):
        a, b = orc.sts(float(z), 1.0), orc.sts(float(-z), 1.0)
        assert abs((a + b) - 1.0) <= 2 * np.spacing(np.float32(1.0))


def test_survival_pages_example(orc):
    g = golden("planner_example.json")
    z = wl.confidence_logits_for(np.array(g["confidences"]))
    s_raw, s_out, st = orc.survival(z, np.ones(2, np.float32), 1e-4)
    assert st == 0
    np.testing.assert_allclose(s_raw, np.array(g["survivals"]), atol=1e-6, rtol=0)
    np.testing.assert_array_equal(s_raw, s_out)


def test_survival_table_of_tutorial(orc):
    g = golden("survival_table.json")
    c = np.array(g["c"])[None, :]
    s_raw, _, _ = orc.survival(wl.confidence_logits_for(c), np.ones(c.shape[1], np.float32), 1e-4)
    half = 0.5 * 10.0 ** -g["printed_decimals"]
    for k, printed in enumerate(g["S_printed"]):
        if k == g["slip_index"]:
            # the page prints 0.665; the exact product 0.92*0.88*0.82 = 0.663872
            assert abs(s_raw[0, k] - g["slip_exact"]) < 1e-6
            assert abs(s_raw[0, k] - printed) > half
        else:
            assert abs(s_raw[0, k] - printed) <= half + 1e-6, (k, s_raw[0, k], printed)


def test_survival_is_sequential_float32_product(orc):
    rng = np.random.default_rng(11)
    z = rng.normal(1.0, 1.5, size=(37, 9)).astype(np.float32)
    T = (1.0 + 0.07 * np.arange(9)).astype(np.float32)
    s_raw, _, _ = orc.survival(z, T, 1e-4)
    c = np.array([[orc.sts(float(z[r, k]), float(T[k])) for k in range(9)] for r in range(37)],
                 dtype=np.float32)
    ref = np.multiply.accumulate(c, axis=1, dtype=np.float32)
    np.testing.assert_array_equal(s_raw, ref)
    # non-increasing per request
    assert np.all(np.diff(s_raw, axis=1) <= 0)


def test_eps_drop(orc):
    z = np.full((3, 6), -2.0, np.float32)  # c ~ 0.119: survival falls below 1e-4 at depth 4
    s_raw, s_out, _ = orc.survival(z, np.ones(6, np.float32), 1e-4)
    keep = s_raw >= np.float32(1e-4)
    assert keep[:, 0].all() and not keep[:, -1].any()
    np.testing.assert_array_equal(s_out[keep], s_raw[keep])
    assert np.all(s_out[~keep] == 0.0)


def test_bad_temperature_is_flagged(orc):
    _, _, st = orc.survival(np.zeros((1, 2), np.float32), np.array([1.0, 0.0], np.float32), 1e-4)
    assert st & orc.ST_BAD_INPUT


# -------------------------------------------------------------- planner

def _f32(a):
    return np.array(a, dtype=np.float32)


def test_pages_example_allocation(orc):
    g = golden("planner_example.json")
    s = _f32(g["survivals"])
    r = orc.plan_from_survivals(s, EPS_MIN, 1, 3, g["extra_budget"], wl.COST_SPS_1D, [1], [1.0])
    assert r.budget == 2
    assert list(r.verify_lens) == g["verify_lens"]
    assert abs(r.tau - g["tau"]) < 1e-6
    assert abs(r.tau_curve[3] - g["tau_budget3"]) < 1e-6


def test_pages_example_budget_choice(orc):
    """3.62 / 1 ms = 3620 beats 4.22 / 1.4 ms ~ 3014, so the 2-row budget wins."""
    g = golden("planner_example.json")
    s = _f32(g["survivals"])
    B = 2
    # 1-D SPS table over M = B + b: 1 ms at b=2, 1.4 ms at b=3, slow elsewhere
    M = np.arange(B, B + 5, dtype=np.int32)
    sps = np.array([1.0, 1.0, 1000.0 / g["step_ms"]["2"], 1000.0 / g["step_ms"]["3"], 1.0])
    r = orc.plan_from_survivals(s, EPS_MIN, 1, 3, -1, wl.COST_SPS_1D, M, sps)
    assert r.budget == g["chosen_budget"]
    assert abs(r.theta - g["throughput"]["2"]) < 1e-6 * g["throughput"]["2"]
    assert abs(r.theta_curve[3] - g["throughput"]["3"]) < g["throughput_b3_tolerance"]
    assert list(r.verify_lens) == g["verify_lens"]


def test_tie_order_depth_then_request(orc):
    # two identical requests: ties go to the lower request id
    s = _f32([[0.5, 0.25], [0.5, 0.25]])
    lens = lambda b, s=s: list(orc.plan_from_survivals(s, EPS_MIN, 1, 3, b, 0, [1], [1.0]).verify_lens)
    assert lens(1) == [2, 1]
    assert lens(2) == [2, 2]
    assert lens(3) == [3, 2]
    # a depth-1 candidate of request 0 ties depth-0 candidates: earlier depth first
    s2 = _f32([[0.5, 0.5], [0.5, 0.1]])
    assert list(orc.plan_from_survivals(s2, EPS_MIN, 1, 3, 2, 0, [1], [1.0]).verify_lens) == [2, 2]
    # equal depth, three requests
    s3 = _f32([[0.3], [0.3], [0.3]])
    assert list(orc.plan_from_survivals(s3, EPS_MIN, 1, 2, 2, 0, [1], [1.0]).verify_lens) == [2, 2, 1]


def _best_sums_brute_force(s, eps, max_len):
    """max over prefix-respecting allocations of the survival sum, per total b."""
    B, g = s.shape
    kept = [int(np.sum((s[r] >= eps) & (np.arange(g) < max_len - 1))) for r in range(B)]
    best = {}
    for alloc in itertools.product(*[range(k + 1) for k in kept]):
        b = sum(alloc)
        tot = sum(float(s[r, k]) for r in range(B) for k in range(alloc[r]))
        if tot > best.get(b, -1.0):
            best[b] = tot
    return best, kept


@pytest.mark.parametrize("seed", range(120))
def test_brute_force_tiny(orc, seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 5))
    g = int(rng.integers(1, 5))
    # conditional confidences from a small set so that exact ties occur
    c = rng.choice(np.array([1.0, 0.8, 0.5, 0.25, 0.125, 0.9], np.float32), size=(B, g))
    s = np.multiply.accumulate(c, axis=1, dtype=np.float32)
    eps = float(np.float32(rng.choice([EPS_MIN, 0.05, 0.2])))
    max_len = int(rng.integers(1, g + 2))
    n_tab = int(rng.integers(1, 6))
    M = np.sort(rng.choice(np.arange(1, B + B * g + 3), size=n_tab, replace=False)).astype(np.int32)
    sps = rng.uniform(0.5, 3.0, size=n_tab)
    r = orc.plan_from_survivals(s, eps, 1, max_len, -1, wl.COST_SPS_1D, M, sps)
    best, kept = _best_sums_brute_force(s, eps, max_len)
    assert r.n_kept == sum(kept)
    # tau(b) - B is the best achievable survival sum with b extra rows, exactly
    for b in range(r.n_kept + 1):
        assert r.tau_curve[b] - B == best[b], (b, r.tau_curve[b], best[b])
    # the budget is the first maximiser of theta (numpy's first-occurrence argmax)
    th = np.where(r.feasible, r.theta_curve, -np.inf)
    assert r.budget == int(np.argmax(th))
    # the allocation at the budget is prefix-respecting and optimal
    alloc = r.verify_lens - 1
    assert alloc.sum() == r.budget
    assert all(0 <= alloc[q] <= kept[q] for q in range(B))
    got = sum(float(s[q, k]) for q in range(B) for k in range(alloc[q]))
    assert got == best[r.budget]


def test_cost_lookup_1d_floor(orc):
    s = _f32([[0.5, 0.25], [0.5, 0.25]])  # sorted 0.5 0.5 0.25 0.25 -> tau 2 2.5 3 3.25 3.5
    # samples at M=4 (100 steps/s) and M=6 (50 steps/s); M < 4 uses sample 0
    r = orc.plan_from_survivals(s, EPS_MIN, 1, 3, -1, wl.COST_SPS_1D, [4, 6], [100.0, 50.0])
    np.testing.assert_array_equal(r.tau_curve, [2.0, 2.5, 3.0, 3.25, 3.5])
    np.testing.assert_allclose(r.theta_curve, [200.0, 250.0, 300.0, 325.0, 175.0], rtol=1e-15)
    assert r.budget == 3
    assert list(r.verify_lens) == [3, 2]


def test_cost_lookup_additive_ceil_tier(orc):
    s = _f32([[0.5, 0.25], [0.5, 0.25]])
    # T = bias + alpha + cost(ceil_tier(M)): M<=3 -> 0.5+0.5+1 = 2 ms; M in 4..5 -> 4 ms; M>5 infeasible
    r = orc.plan_from_survivals(s, EPS_MIN, 1, 3, -1, wl.COST_ADDITIVE, [3, 5], [1.0, 3.0],
                                bias=0.5, alpha=0.5)
    np.testing.assert_allclose(r.theta_curve[:4], [1.0, 1.25, 0.75, 0.8125], rtol=1e-15)
    assert list(r.feasible) == [True, True, True, True, False]
    assert r.budget == 1 and abs(r.theta - 1.25) < 1e-15
    # a forced budget is clipped to the largest in-range budget (M <= 5 -> b <= 3)
    f = orc.plan_from_survivals(s, EPS_MIN, 1, 3, 4, wl.COST_ADDITIVE, [3, 5], [1.0, 3.0],
                                bias=0.5, alpha=0.5)
    assert f.budget == 3 and list(f.verify_lens) == [3, 2]


def test_cost_lookup_additive_interpolated(orc):
    """The additive table's runtime linear interpolation of theta(M): one
    request, survivals 0.875 0.5 0.25 0.0625 (tau 1, 1.875, 2.375, 2.625,
    2.6875), samples theta(1) = 0, theta(5) = 0.5 ms, bias + alpha = 1 ms:
    T(b) = 1 + b/8, so theta = 1, 1.667, 1.9, 1.909, 1.792 -> budget 3.
    The ceil-to-tier lookup of the same table gives T = 1, 1.5, 1.5, 1.5,
    1.5 -> budget 4: the two modes differ only between samples."""
    s = _f32([[0.875, 0.5, 0.25, 0.0625]])
    r = orc.plan_from_survivals(s, EPS_MIN, 1, 5, -1, wl.COST_ADDITIVE_INTERP, [1, 5], [0.0, 0.5],
                                bias=0.25, alpha=0.75)
    tau = [1.0, 1.875, 2.375, 2.625, 2.6875]
    np.testing.assert_array_equal(r.tau_curve, tau)
    np.testing.assert_allclose(r.theta_curve, [t / (1 + b / 8) for b, t in enumerate(tau)],
                               rtol=1e-15)
    assert r.budget == 3 and list(r.verify_lens) == [4]
    c = orc.plan_from_survivals(s, EPS_MIN, 1, 5, -1, wl.COST_ADDITIVE, [1, 5], [0.0, 0.5],
                                bias=0.25, alpha=0.75)
    assert c.budget == 4
    # at the samples themselves both lookups give the same T
    assert r.theta_curve[0] == c.theta_curve[0] and r.theta_curve[4] == c.theta_curve[4]


def test_cost_lookup_interpolated_edges(orc):
    s = _f32([[0.5, 0.25], [0.5, 0.25]])  # tau 2 2.5 3 3.25 3.5, M = 2 + b
    # samples at M = 3 and 4 only: M = 2 is below the first (val_0), M > 4 infeasible
    r = orc.plan_from_survivals(s, EPS_MIN, 1, 3, -1, wl.COST_ADDITIVE_INTERP, [3, 4], [1.0, 3.0],
                                bias=0.5, alpha=0.5)
    assert list(r.feasible) == [True, True, True, False, False]
    np.testing.assert_allclose(r.theta_curve[:3], [1.0, 1.25, 0.75], rtol=1e-15)
    # three samples, a midpoint: M = 4 between (3, 1 ms) and (5, 5 ms) -> 3 ms
    q = orc.plan_from_survivals(s, EPS_MIN, 1, 3, -1, wl.COST_ADDITIVE_INTERP, [3, 5, 9],
                                [1.0, 5.0, 6.0], bias=0.5, alpha=0.5)
    np.testing.assert_allclose(q.theta_curve, [2 / 2, 2.5 / 2, 3 / 4, 3.25 / 6, 3.5 / 6.25],
                               rtol=1e-15)
    assert q.budget == 1
    # a non-positive interpolated T is infeasible and flagged
    z = orc.plan_from_survivals(s, EPS_MIN, 1, 3, -1, wl.COST_ADDITIVE_INTERP, [2, 6],
                                [-1.0, 3.0], bias=0.0, alpha=0.0)
    assert z.status & orc.ST_BAD_COST and not z.feasible[0] and z.feasible[2]


def test_cost_lookup_interpolated_at_samples_is_exact(orc):
    """At a sample M = M_j the interpolated cost is val_j itself, even when
    the segment's slope is not exact in binary (0.6 / 3 here): the
    interpolation does not pass through the previous segment."""
    s = _f32([[0.5, 0.25, 0.125, 0.0625, 0.03125, 0.015625, 0.0078125, 0.00390625, 0.001953125]])
    M, val, bias, alpha = [1, 4, 7, 10], [0.1, 0.7, 0.3, 0.9], 0.2, 0.05
    r = orc.plan_from_survivals(s, EPS_MIN, 1, 10, -1, wl.COST_ADDITIVE_INTERP, M, val,
                                bias=bias, alpha=alpha)
    for j, Mj in enumerate(M):
        b = Mj - 1  # B = 1
        assert r.theta_curve[b] == r.tau_curve[b] / ((bias + alpha) + val[j]), j
    # between samples: val_j + (M - M_j) * slope_j in that order
    b = 5  # M = 6, segment [4, 7)
    slope = (val[2] - val[1]) / (M[2] - M[1])
    assert r.theta_curve[b] == r.tau_curve[b] / ((bias + alpha) + (val[1] + (6 - 4) * slope))


def test_invalid_cost_and_infeasible(orc):
    s = _f32([[0.5, 0.25]])
    r = orc.plan_from_survivals(s, EPS_MIN, 1, 3, -1, wl.COST_SPS_1D, [1, 2], [0.0, 5.0])
    assert r.status & orc.ST_BAD_COST
    assert not r.feasible[0] and r.feasible[1]
    # every budget above the largest tier: infeasible, budget 0
    q = orc.plan_from_survivals(_f32([[0.5], [0.5], [0.5]]), EPS_MIN, 1, 2, -1,
                                wl.COST_ADDITIVE, [2], [1.0], bias=1.0)
    assert q.status & orc.ST_INFEASIBLE and q.budget == 0 and list(q.verify_lens) == [1, 1, 1]


def test_min_verify_len_clamp(orc):
    s = _f32([[0.9, 0.8, 0.7], [0.1, 0.01, 0.001]])
    r = orc.plan_from_survivals(s, EPS_MIN, 2, 4, 2, 0, [1], [1.0])
    assert list(r.verify_lens) == [3, 2]  # request 1 raised to the minimum of 2
    # max_verify_len bounds both the candidates and the lens
    r2 = orc.plan_from_survivals(s, EPS_MIN, 1, 2, 3, 0, [1], [1.0])
    assert list(r2.verify_lens) == [2, 2] and r2.n_kept == 2


def test_plan_invariants_on_workloads(orc):
    for w in (wl.TINY, wl.QWEN, wl.DSV4, wl.MIXED):
        step = wl.make_step(w, seed=0)
        r = orc.plan_step(step)
        lens = r.verify_lens
        assert np.all(lens >= w.min_verify_len) and np.all(lens <= w.max_len)
        assert lens.sum() == w.B + r.budget  # min_verify_len = 1
        assert np.all(np.diff(r.survivals, axis=1) <= 0)
        assert r.status == 0


# ------------------------------------------------------------------ pack

def test_pack_cu_seqlens(orc):
    for ex in golden("pack_examples.json")["cu_seqlens"]:
        lens = np.array(ex["verify_lens"], np.int32)
        B, g = len(lens), int(lens.max())
        p = orc.pack(np.zeros(B), np.zeros((B, g)), np.zeros(B), lens, [], 64)
        assert list(p.cu_seqlens) == ex["cu_seqlens"]
        assert p.total == p.padded == ex["rows"]


def test_pack_layout_of_the_page(orc):
    ex = golden("pack_examples.json")["packed_layout"]
    lens = np.array(ex["verify_lens"], np.int32)
    gamma = 3
    # token of request q (letter) at chain position j is encoded 100*(q+1)+j
    anchor = np.array([100 * (q + 1) for q in range(3)], np.int32)
    draft = np.array([[100 * (q + 1) + j for j in range(1, gamma + 1)] for q in range(3)], np.int32)
    prefix = np.array([10, 20, 30], np.int32)
    p = orc.pack(anchor, draft, prefix, lens, [], 12)
    names = [f"{'ABC'[t // 100 - 1]}{t % 100}" for t in p.ids[:p.total]]
    assert names == ex["rows"]
    assert list(p.req[:7]) == [0, 0, 1, 2, 2, 2, 2]
    assert list(p.pos[:7]) == [10, 11, 20, 30, 31, 32, 33]
    assert list(p.src[:7]) == [0, 1, 4, 8, 9, 10, 11]
    assert np.all(p.ids[7:] == -7)  # rows past the packed total are not touched


def test_pack_tier_round_up(orc):
    for ex in golden("pack_examples.json")["tiers"]:
        for total, padded in ex["total_to_padded"]:
            lens = np.ones(total, np.int32)
            p = orc.pack(np.arange(total), np.zeros((total, 1)), np.zeros(total), lens,
                         ex["tiers"], 128)
            assert p.total == total and p.padded == padded
            assert np.all(p.req[total:padded] == -1) and np.all(p.src[total:padded] == -1)
            assert np.all(p.ids[total:padded] == 0) and np.all(p.pos[total:padded] == 0)
            assert np.all(p.req[padded:] == -7)
            if "padding" in ex:
                assert padded - total == ex["padding"]


def test_pack_capacity_and_bad_len(orc):
    p = orc.pack(np.zeros(2), np.zeros((2, 3)), np.zeros(2), [4, 4], [], 6)
    assert p.status & orc.ST_CAPACITY and p.total == 8
    q = orc.pack(np.zeros(2), np.zeros((2, 3)), np.zeros(2), [0, 9], [], 16)
    assert q.status & orc.ST_BAD_LEN and list(q.cu_seqlens) == [0, 1, 5]
    r = orc.pack(np.zeros(3), np.zeros((3, 3)), np.zeros(3), [4, 4, 4], [8], 16)
    assert r.status & orc.ST_CAPACITY and r.padded == 12


def test_dp_shared_tier_pads_every_rank_to_the_largest(orc):
    """[AVS] §六 (local verify tier -> DP gather -> DP-global max tier) and
    [SGL] "Ragged verify" (DP ranks share the largest tier any rank needs),
    with the tutorial's tiers {40, 64, 80}: a rank with 37 rows (local tier
    40) and one with 58 (local tier 64) both replay 64; the first rank's rows
    37..63 become pad rows (27, as in [AVS] §五's 37 real + 27 padding), its
    real rows stay as they were."""
    tiers = [40, 64, 80]
    ranks = []
    for total in (37, 58):
        lens = np.ones(total, np.int32)
        p = orc.pack(np.arange(1, total + 1), np.zeros((total, 1)), np.arange(total) + 100,
                     lens, tiers, 96)
        ranks.append(p)
    assert [p.padded for p in ranks] == [40, 64]
    shared = max(p.padded for p in ranks)
    a, b = (orc.pad_to_tier(p, shared, 96) for p in ranks)
    assert (a.total, a.padded, b.total, b.padded) == (37, 64, 58, 64)
    assert a.status == 0 and b.status == 0
    assert list(a.ids[:37]) == list(range(1, 38)) and list(a.pos[:37]) == list(range(100, 137))
    assert list(a.req[:37]) == list(range(37)) and list(a.src[:37]) == [2 * r for r in range(37)]
    for k, v in (("ids", 0), ("pos", 0), ("req", -1), ("src", -1)):
        assert np.all(a[k][37:64] == v), k
        assert np.all(a[k][64:] == -7), k  # past the shared tier: untouched
    for k in ("ids", "pos", "req", "src"):  # the rank that set the tier is unchanged
        np.testing.assert_array_equal(b[k], ranks[1][k])


def test_dp_shared_tier_edges(orc):
    """A shared tier below the rank's real rows changes nothing (BAD_TIER); a
    shared tier past the capacity writes pad rows up to the capacity and
    flags CAPACITY; a shared tier equal to the local one is a no-op."""
    lens = np.ones(37, np.int32)
    p = orc.pack(np.arange(37), np.zeros((37, 1)), np.zeros(37), lens, [40, 64], 50)
    low = orc.pad_to_tier(p, 30, 50)
    assert low.status == orc.ST_BAD_TIER and low.padded == 40
    for k in ("ids", "pos", "req", "src"):
        np.testing.assert_array_equal(low[k], p[k])
    over = orc.pad_to_tier(p, 64, 50)
    assert over.status == orc.ST_CAPACITY and over.padded == 64
    assert np.all(over.req[37:50] == -1)
    same = orc.pad_to_tier(p, 40, 50)
    assert same.status == 0 and same.padded == 40
    for k in ("ids", "pos", "req", "src"):
        np.testing.assert_array_equal(same[k], p[k])


# ---------------------------------------------------------------- scatter

def test_scatter_example_of_the_page(orc):
    """[ROUND] §三: lengths [2, 5, 3] at a stride of 5 -- 10 compact rows go
    back to their places among 15 strided rows; the other 5 stay untouched."""
    ex = golden("pack_examples.json")["scatter"]
    lens = np.array(ex["verify_lens"], np.int32)
    B, stride = len(lens), ex["stride"]
    p = orc.pack(np.zeros(B), np.zeros((B, stride - 1)), np.zeros(B), lens, [], 32)
    assert p.total == ex["compact_rows"]
    compact = np.arange(p.total * 3, dtype=np.uint16).reshape(p.total, 3) + 1
    strided = np.zeros((ex["strided_rows"], 3), np.uint16)
    out, st = orc.scatter_rows(compact, p.src, p.total, strided)
    assert st == 0
    # request r's row j lands at r*stride + j
    want = [r * stride + j for r in range(B) for j in range(int(lens[r]))]
    assert list(p.src[:p.total]) == want == [0, 1, 5, 6, 7, 8, 9, 10, 11, 12]
    for i, d in enumerate(want):
        assert np.array_equal(out[d], compact[i])
    untouched = sorted(set(range(ex["strided_rows"])) - set(want))
    assert untouched == [2, 3, 4, 13, 14] and not out[untouched].any()


def test_scatter_inverts_the_compact_gather(orc):
    """Gathering the selected strided rows into compact order and scattering
    them back restores exactly those rows; pad rows and rows past the total
    are not written; a destination outside the buffer is flagged."""
    rng = np.random.default_rng(11)
    for _ in range(20):
        B, g = int(rng.integers(1, 9)), int(rng.integers(1, 6))
        lens = rng.integers(1, g + 2, size=B).astype(np.int32)
        tiers = [int(lens.sum()) + int(rng.integers(0, 4))]
        p = orc.pack(np.zeros(B), np.zeros((B, g)), np.zeros(B), lens, tiers, 64)
        S = rng.integers(1, 60000, size=(B * (g + 1), 5)).astype(np.uint16)
        compact = np.zeros((64, 5), np.uint16)
        compact[:p.total] = S[p.src[:p.total]]
        compact[p.total:] = 9  # pad rows: never copied
        back, st = orc.scatter_rows(compact, p.src, p.total, np.zeros_like(S))
        sel = p.src[:p.total]
        assert st == 0 and np.array_equal(back[sel], S[sel])
        rest = np.setdiff1d(np.arange(B * (g + 1)), sel)
        assert not back[rest].any()
    src_of = np.array([0, 7, -1, 2], np.int32)
    out, st = orc.scatter_rows(np.ones((4, 2), np.float32), src_of, 4, np.zeros((3, 2), np.float32))
    assert st & orc.ST_BAD_INDEX and out[0].all() and out[2].all() and not out[1].any()
    out2, st2 = orc.scatter_rows(np.ones((4, 2), np.float32), [0, 1, 2, 0], 9,
                                 np.zeros((3, 2), np.float32), max_rows=2)
    assert st2 == 0 and out2[:2].all() and not out2[2].any()  # total clamped to max_rows


# ---------------------------------------------------------------- accept

_TOK = {"A": 11, "B": 12, "C": 13, "D": 14, "E": 15, "X": 5, "Y": 6, "Z": 7}


def _one_hot_rows(tokens, V, rng):
    x = rng.normal(0, 1, size=(len(tokens), V)).astype(np.float32)
    for i, t in enumerate(tokens):
        x[i, t] += 8.0
    return x


def test_greedy_accept_page_example(orc):
    ex = golden("accept_examples.json")
    rng = np.random.default_rng(5)
    for key in ("greedy", "all_accepted"):
        e = ex[key]
        draft = np.array([[_TOK[t] for t in e["drafts"]]], np.int32)
        logits = _one_hot_rows([_TOK[t] for t in e["target_chain"]], 32, rng)
        cu = np.array([0, 5], np.int32)
        fin = orc.greedy_accept(logits, 32, cu, draft, np.array([10], np.int32))
        assert fin.num_accepted[0] == e["correct_len"]
        assert fin.commit_lens[0] == e["commit_len"]
        assert fin.status == 0
        if "bonus" in e:
            assert fin.bonus[0] == _TOK[e["bonus"]]
            valid = fin.out_tokens[0, :fin.commit_lens[0]]
            assert [t for t in valid] == [_TOK[t] for t in e["valid_output"]]
    f = ex["finalize"]
    fin = orc.greedy_accept(_one_hot_rows([11, 12, 5], 32, rng), 32, np.array([0, 3], np.int32),
                            np.array([[11, 12, 13, 14]], np.int32),
                            np.array([f["prefix_len"]], np.int32))
    assert fin.commit_lens[0] == f["commit_len"] and fin.new_seq_lens[0] == f["new_seq_len"]


def test_no_recovery_after_first_mismatch(orc):
    rng = np.random.default_rng(6)
    draft = np.array([[11, 12, 13, 14]], np.int32)
    # the target matches drafts 0, 2 and 3 but not 1: only one draft is accepted
    logits = _one_hot_rows([11, 5, 13, 14, 15], 32, rng)
    fin = orc.greedy_accept(logits, 32, np.array([0, 5], np.int32), draft, np.zeros(1, np.int32))
    assert fin.num_accepted[0] == 1 and fin.bonus[0] == 5 and fin.commit_lens[0] == 2
    assert list(fin.out_tokens[0]) == [11, 5, 13, 14, -1]


def test_cap_accept_page_example(orc):
    e = golden("accept_examples.json")["cap_accept"]
    gamma = e["width"] - 1
    B = len(e["verify_lens"])
    rng = np.random.default_rng(7)
    draft = rng.integers(0, 32, size=(B, gamma)).astype(np.int32)
    chain = [int(draft[r, j]) if j < gamma else 3 for r in range(B) for j in range(gamma + 1)]
    logits = _one_hot_rows(chain, 32, rng)
    assert logits.shape[0] == e["target_rows"]
    cap = orc.cap_accept(logits, 32, np.array(e["verify_lens"], np.int32), draft,
                         np.zeros(B, np.int32))
    assert list(cap.num_accepted) == e["draft_caps"]
    assert list(cap.ceiling) == [gamma] * B
    assert list(cap.commit_lens) == [c + 1 for c in e["draft_caps"]]
    assert cap.sum_commit == sum(c + 1 for c in e["draft_caps"])
    assert cap.sum_ceiling == B * (gamma + 1)


def test_argmax_special_cases(orc):
    V = 64
    am, st = orc.argmax_rows(np.zeros((3, V), np.float32))
    assert list(am) == [0, 0, 0] and st == 0
    rng = np.random.default_rng(8)
    x = rng.normal(size=(50, V)).astype(np.float32)
    x[5, 7] = x[5, 40] = 9.0  # tie: lowest index
    am, _ = orc.argmax_rows(x)
    np.testing.assert_array_equal(am, np.argmax(x, axis=1))
    assert am[5] == 7
    # bf16 rows agree with numpy's argmax of the decoded values
    b = wl.to_bf16_bits(rng.normal(size=(40, 300)).astype(np.float32))
    am, _ = orc.argmax_rows(b)
    np.testing.assert_array_equal(am, np.argmax(wl.bf16_bits_to_f32(b), axis=1))
    # -0 equals +0; NaN is skipped and flagged; a row with nothing above -inf gives 0
    z = np.array([[-1.0, -0.0, 0.0, -2.0]], np.float32)
    assert orc.argmax_rows(z)[0][0] == 1
    n = np.array([[np.nan, 1.0, 2.0, np.nan]], np.float32)
    am, st = orc.argmax_rows(n)
    assert am[0] == 2 and st & orc.ST_NAN_LOGIT
    m = np.array([[np.nan, -np.inf, -np.inf]], np.float32)
    assert orc.argmax_rows(m)[0][0] == 0
    # ld > V: trailing columns are ignored
    y = np.zeros((2, 8), np.float32)
    y[:, 6] = 5.0
    y[:, 2] = 1.0
    assert list(orc.argmax_rows(y, V=5)[0]) == [2, 2]


def test_greedy_bad_ranges_and_tokens(orc):
    rng = np.random.default_rng(9)
    logits = _one_hot_rows([1, 2, 3], 16, rng)
    draft = np.array([[1, 2], [3, 99]], np.int32)
    fin = orc.greedy_accept(logits, 16, np.array([0, 3, 3], np.int32), draft,
                            np.array([4, 5], np.int32))
    assert fin.status & orc.ST_BAD_LEN and fin.status & orc.ST_TOKEN_RANGE
    assert fin.num_accepted[1] == 0 and fin.bonus[1] == -1 and fin.commit_lens[1] == 0
    assert fin.new_seq_lens[1] == 5
    # rows beyond max_rows: capacity flag, the request past them is a bad range
    fin2 = orc.greedy_accept(logits, 16, np.array([0, 2, 4], np.int32),
                             np.array([[1, 2], [3, 4]], np.int32), np.zeros(2, np.int32))
    assert fin2.status & orc.ST_CAPACITY and fin2.status & orc.ST_BAD_LEN


def test_compact_equals_cap_accept(orc):
    """Compact and cap-accept commit the same tokens (the review page's mode
    table); the compact window is the gather of the strided rows."""
    for seed in range(3):
        step = wl.make_step(wl.TINY, seed=seed)
        r = orc.plan_step(step)
        strided = wl.strided_logits(step)
        p = orc.pack(step.anchor, step.draft, step.prefix_lens, r.verify_lens, step.tiers,
                     step.capacity)
        compact = strided[p.src[:p.total]]
        g = orc.greedy_accept(compact, step.V, p.cu_seqlens, step.draft, step.prefix_lens)
        c = orc.cap_accept(strided, step.V, r.verify_lens, step.draft, step.prefix_lens)
        for key in ("num_accepted", "bonus", "commit_lens", "new_seq_lens", "out_tokens"):
            np.testing.assert_array_equal(g[key], c[key], err_msg=key)
        assert np.all(c.ceiling >= c.num_accepted)


def test_expected_commit_equals_tau(orc):
    """E[sum(commit_lens)] = B + sum of the selected survivals when the survival
    estimates are the true prefix probabilities (adaptive verify page, section
    三, expectation by linearity)."""
    B, gamma, V = 48, 6, 256
    c = np.array([0.95, 0.9, 0.85, 0.8, 0.7, 0.6])
    w = wl.Workload("expectation", B=B, gamma=gamma, V=V, logits_dtype="fp32")
    z = np.tile(wl.confidence_logits_for(c[None, :]), (B, 1))
    res = orc.plan(z, np.ones(gamma, np.float32), 1e-4, 1, gamma + 1, 150, 0, [1], [1.0])
    commits, n_steps = [], 160
    for seed in range(n_steps):
        rng = np.random.default_rng(seed)
        step = wl.StepInputs(workload=w, seed=seed, conf_logits=z,
                             sts_temps=np.ones(gamma, np.float32),
                             draft=rng.integers(0, V, size=(B, gamma)).astype(np.int32),
                             anchor=np.zeros(B, np.int32), prefix_lens=np.zeros(B, np.int32),
                             match_prob=np.tile(c, (B, 1)), cost=None, tiers=np.zeros(0, np.int32),
                             capacity=B * (gamma + 1))
        cap = orc.cap_accept(wl.strided_logits(step), V, res.verify_lens, step.draft,
                             step.prefix_lens)
        commits.append(cap.sum_commit)
    mean = float(np.mean(commits))
    sem = float(np.std(commits)) / math.sqrt(n_steps)
    assert abs(mean - res.tau) < 4.5 * sem + 1e-3, (mean, res.tau, sem)


def test_budget_theta_tie_goes_to_smaller_budget(orc):
    # tau = 2, 2.5, 2.75; SPS 5, 4, 3 -> theta = 10, 10, 8.25 (exact in fp64)
    s = _f32([[0.5], [0.25]])
    r = orc.plan_from_survivals(s, EPS_MIN, 1, 2, -1, wl.COST_SPS_1D, [2, 3, 4], [5.0, 4.0, 3.0])
    np.testing.assert_array_equal(r.theta_curve, [10.0, 10.0, 8.25])
    assert r.budget == int(np.argmax(r.theta_curve)) == 0
    assert list(r.verify_lens) == [1, 1]


# ------------------------------------------------- planner options ([AVS] §三)

def test_plan_ex_without_options_is_the_plan(orc):
    rng = np.random.default_rng(21)
    for _ in range(10):
        B, g = int(rng.integers(1, 7)), int(rng.integers(1, 8))
        z = rng.normal(1, 1.5, (B, g)).astype(np.float32)
        T = rng.uniform(0.5, 2, g).astype(np.float32)
        M = np.sort(rng.choice(np.arange(1, B * (g + 1) + 4), 3, replace=False)).astype(np.int32)
        val = rng.uniform(0.1, 2, 3)
        a = orc.plan(z, T, 1e-4, 1, g + 1, -1, 1, M, val, 0.5, 0.2)
        b = orc.plan_ex(z, T, 1e-4, 1, g + 1, -1, 1, M, val, 0.5, 0.2)
        assert a.budget == b.budget and a.tau == b.tau and a.theta == b.theta
        assert np.array_equal(a.verify_lens, b.verify_lens) and np.array_equal(a.survivals, b.survivals)
        # the same confidences as "lagged" change nothing either
        c = orc.plan_ex(z, T, 1e-4, 1, g + 1, -1, 1, M, val, 0.5, 0.2, lagged_z=z)
        assert c.budget == a.budget and np.array_equal(c.verify_lens, a.verify_lens)


def test_plan_ex_stale_generation_survives_with_one(orc):
    """A request whose confidences belong to another generation of its slot
    plans with survival 1 at every depth: its candidates come first (depth,
    then request order) and tau grows by exactly 1 per candidate taken."""
    z = np.full((3, 4), -3.0, np.float32)  # low confidence everywhere
    T = np.ones(4, np.float32)
    M = np.array([1, 100], np.int32)
    val = np.array([1.0, 1.0])  # 1-D SPS constant: theta = tau, largest budget wins
    res = orc.plan_ex(z, T, 0.5, 1, 5, 2, 0, M, val, conf_gen=[7, 8, 9], req_gen=[7, 1, 9])
    assert np.all(res.survivals[1] == 1.0) and np.all(res.survivals[[0, 2]] < 0.5)
    # eps 0.5 keeps only the stale request's candidates; a forced budget of 2
    # takes its two shallowest depths: tau = B + 2 exactly
    assert res.budget == 2 and list(res.verify_lens) == [1, 3, 1] and res.tau == 3 + 2
    fresh = orc.plan_ex(z, T, 0.5, 1, 5, 2, 0, M, val, conf_gen=[7, 8, 9], req_gen=[7, 8, 9])
    assert fresh.budget == 0 and list(fresh.verify_lens) == [1, 1, 1]


def test_plan_ex_lagged_budget_current_allocation(orc):
    """The budget comes from the lagged confidences, the allocation from the
    current ones: lens are the top-b of the current order, however the lagged
    survivals were ranked."""
    rng = np.random.default_rng(22)
    for _ in range(20):
        B, g = int(rng.integers(2, 7)), int(rng.integers(2, 8))
        z_now = rng.normal(1, 1.5, (B, g)).astype(np.float32)
        z_lag = rng.normal(0, 2, (B, g)).astype(np.float32)
        T = np.ones(g, np.float32)
        M = np.arange(1, B * (g + 1) + 2, dtype=np.int32)
        val = 1.0 / (1e-3 + rng.uniform(1e-5, 5e-4) * M)
        lag = orc.plan(z_lag, T, 1e-4, 1, g + 1, -1, 0, M, val)
        res = orc.plan_ex(z_now, T, 1e-4, 1, g + 1, -1, 0, M, val, lagged_z=z_lag)
        now = orc.plan(z_now, T, 1e-4, 1, g + 1, lag.budget, 0, M, val)
        assert res.budget == now.budget == min(lag.budget, now.n_kept)
        assert np.array_equal(res.verify_lens, now.verify_lens) and res.tau == now.tau
        # brute force: the top-b of the current order, survival desc, depth, request
        s = now.survivals
        cand = sorted(((-float(s[r, k]), k, r) for r in range(B) for k in range(g)
                       if s[r, k] >= np.float32(1e-4)))[:res.budget]
        cnt = np.zeros(B, int)
        for _, _, r in cand:
            cnt[r] += 1
        assert list(res.verify_lens) == list(1 + cnt)


def test_plan_ex_tier_alignment_paid_padding(orc):
    """[AVS] §五: 37 real rows replayed at a 64-row tier -- alignment fills
    the 27 padding rows with the next candidates by survival, never past the
    tier, and only as far as candidates remain."""
    B, g = 4, 31
    z = np.full((B, g), 6.0, np.float32)
    T = np.ones(g, np.float32)
    M = np.array([4, 38], np.int32)
    val = np.array([1000.0, 1.0])  # SPS drops past 37 rows: the plan takes 37
    tiers = [16, 32, 64, 128]
    plain = orc.plan_ex(z, T, 1e-4, 1, g + 1, -1, 0, M, val)
    assert plain.budget == 33 and plain.verify_lens.sum() == 37
    al = orc.plan_ex(z, T, 1e-4, 1, g + 1, -1, 0, M, val, align_tiers=tiers)
    assert al.budget == 60 and al.verify_lens.sum() == 64
    # the extra rows are the next candidates of the order: a superset of the plan
    assert np.all(al.verify_lens >= plain.verify_lens)
    # too few candidates left (eps keeps 40): filled as far as they go
    z2 = np.tile(np.concatenate([np.full(10, 6.0), np.full(g - 10, -20.0)]).astype(np.float32), (B, 1))
    few = orc.plan_ex(z2, T, 1e-4, 1, g + 1, -1, 0, M, val, align_tiers=tiers)
    assert few.n_kept == 40 and few.budget == 40 and few.verify_lens.sum() == 44
    # no tier holds the plan's rows: unchanged
    none = orc.plan_ex(z, T, 1e-4, 1, g + 1, -1, 0, M, val, align_tiers=[8, 16])
    assert none.budget == plain.budget and np.array_equal(none.verify_lens, plain.verify_lens)


# ------------------------------------------------ sampling accept ([ROUND] §五 AcceptSampling)

def _logp(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, np.float64)).astype(np.float32)


def test_sampling_accept_hand_case(orc):
    """p = [.5, .3, .2, 0], q uniform, draft token 3 (p = 0): rejected at
    any u; the residual max(0, p - q) = [.25, .05, 0, 0] (W = .3) gives token
    1 for u = .9 (.27 lies in (.25, .30]) and token 0 for u = .5."""
    tgt = np.stack([_logp([.5, .3, .2, 0]), _logp([.1, .2, .3, .4])])
    dft = np.zeros((1, 4), np.float32)  # uniform q
    for ub, tok in ((0.9, 1), (0.5, 0)):
        r = orc.sampling_accept(tgt, 4, [0, 2], dft, [[3]], [10], [[0.5]], [ub])
        assert r.num_accepted[0] == 0 and r.bonus[0] == tok and r.commit_lens[0] == 1
        assert list(r.out_tokens[0]) == [tok, -1] and r.new_seq_lens[0] == 11
    # accepted when u * q < p: draft 0 (p = .5, q = .25) always, then the
    # bonus comes from the last row's p: C = .1, .3, .6, 1.0 and u = .65 -> 3
    r = orc.sampling_accept(tgt, 4, [0, 2], dft, [[0]], [10], [[0.99]], [0.65])
    assert r.num_accepted[0] == 1 and r.bonus[0] == 3 and list(r.out_tokens[0]) == [0, 3]


def test_sampling_accept_equal_distributions_always_accept(orc):
    rng = np.random.default_rng(31)
    B, g, V = 50, 4, 16
    rows = rng.normal(0, 2, (B * g, V)).astype(np.float32)
    tgt = np.zeros((B * (g + 1), V), np.float32)
    for r in range(B):
        tgt[r * (g + 1):r * (g + 1) + g] = rows[r * g:(r + 1) * g]
    cu = np.arange(0, B * (g + 1) + 1, g + 1, dtype=np.int32)
    draft = rng.integers(0, V, (B, g)).astype(np.int32)
    res = orc.sampling_accept(tgt, V, cu, rows, draft, np.zeros(B), rng.random((B, g)), rng.random(B))
    assert np.all(res.num_accepted == g) and res.status == 0


def test_sampling_accept_rate_is_one_minus_tv(orc):
    """Drafts drawn from q are accepted with mean probability sum min(p, q)
    = 1 - TV(p, q) ([AVS] §一): Monte Carlo over 40000 requests."""
    rng = np.random.default_rng(32)
    V, n = 6, 40000
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    tgt = np.tile(_logp(p), (2 * n, 1))
    dft = np.tile(_logp(q), (n, 1))
    draft = rng.choice(V, size=(n, 1), p=q).astype(np.int32)
    cu = np.arange(0, 2 * n + 1, 2, dtype=np.int32)
    res = orc.sampling_accept(tgt, V, cu, dft, draft, np.zeros(n), rng.random((n, 1)), rng.random(n))
    rate = res.num_accepted.mean()
    want = np.minimum(p, q).sum()
    assert abs(rate - want) < 4 * np.sqrt(want * (1 - want) / n), (rate, want)


def test_sampling_accept_output_is_distributed_as_p(orc):
    """The point of the rule: with the draft drawn from q, the first token
    the request commits (the accepted draft, or the bonus drawn from the
    residual) is distributed exactly as p.  Chi-square over 60000 draws; a
    residual of max(0, q - p) or an unnormalised draw fails it."""
    rng = np.random.default_rng(33)
    V, n = 5, 60000
    p = np.array([0.35, 0.05, 0.3, 0.2, 0.1])
    q = np.array([0.1, 0.4, 0.1, 0.25, 0.15])
    tgt = np.tile(_logp(p), (2 * n, 1))
    dft = np.tile(_logp(q), (n, 1))
    draft = rng.choice(V, size=(n, 1), p=q).astype(np.int32)
    cu = np.arange(0, 2 * n + 1, 2, dtype=np.int32)
    res = orc.sampling_accept(tgt, V, cu, dft, draft, np.zeros(n), rng.random((n, 1)), rng.random(n))
    first = res.out_tokens[:, 0]
    counts = np.bincount(first, minlength=V)
    chi2 = float(((counts - n * p) ** 2 / (n * p)).sum())
    assert chi2 < 20.5, (chi2, counts / n)  # 4 degrees of freedom, p-value 4e-4


def test_sampling_accept_flags(orc):
    tgt = np.zeros((2, 4), np.float32)
    tgt[0, 2] = np.nan
    dft = np.zeros((1, 4), np.float32)
    r = orc.sampling_accept(tgt, 4, [0, 2], dft, [[7]], [0], [[0.1]], [0.5])
    assert r.status & orc.ST_NAN_LOGIT and r.status & orc.ST_TOKEN_RANGE
    assert r.num_accepted[0] == 0  # an out-of-range draft has p = q = 0: rejected
    bad = orc.sampling_accept(tgt, 4, [0, 3], dft, [[1]], [5], [[0.1]], [0.5])
    assert bad.status & orc.ST_BAD_LEN and bad.bonus[0] == -1 and bad.new_seq_lens[0] == 5


def _residual_threshold_case():
    """Two requests, V = 2, one draft each (token 1), target row p = (1/2,
    1/2) (logits 0, 0) and proposal q from logits (b, 0): with e = exp(b)
    (fp32, exact here: 1 - 2^-17 and 1 - 2^-19), q_0 = e / (1 + e) < 1/2 and
    the residual max(0, p - q) = (W, 0) with W = (1 - e) / (2 (1 + e)):
    W = 2^-19 / (1 - 2^-18) for request 0 (above 2^-20) and W = 2^-21 /
    (1 - 2^-20) for request 1 (below).  u_accept = 1 - 2^-24 rejects both
    drafts (accept iff u q_1 < p_1, and q_1 = 1/2 + W exceeds 1/2 by more
    than 2^-24 q_1)."""
    b = np.array([-(2.0 ** -17), -(2.0 ** -19)], np.float32)
    tgt = np.zeros((4, 2), np.float32)  # rows 0-1 request 0, rows 2-3 request 1
    dft = np.stack([[b[0], 0.0], [b[1], 0.0]]).astype(np.float32)
    cu = np.array([0, 2, 4], np.int32)
    draft = np.array([[1], [1]], np.int32)
    ua = np.full((2, 1), np.float32(1.0 - 2.0 ** -24), np.float32)
    return tgt, dft, cu, draft, ua


def test_sampling_residual_mass_threshold(orc):
    """Reading R23's cut-off, pinned on both sides by hand-derived masses
    ([AVS] §一: accept with probability min(1, p/q), else draw from the
    normalised residual max(0, p - q)).  A residual of mass W >= 2^-20 is
    drawn from: it holds token 0 only, so the bonus is 0 whatever u_bonus.
    A residual of mass W < 2^-20 is read as empty and the bonus is drawn
    from p = (1/2, 1/2) by inverse CDF: u_bonus = 0.75 gives token 1,
    u_bonus = 0.25 token 0.  Drawing from p there moves the committed
    token's distribution by at most W in total variation (the output is
    min(p, q) + W p instead of min(p, q) + (p - q)+, and both vectors have
    mass W)."""
    tgt, dft, cu, draft, ua = _residual_threshold_case()
    hi = orc.sampling_accept(tgt, 2, cu, dft, draft, np.zeros(2), ua, np.array([0.75, 0.75]))
    assert hi.num_accepted.tolist() == [0, 0]
    assert hi.bonus.tolist() == [0, 1]  # residual (token 0) / p (u = 0.75 -> token 1)
    assert hi.out_tokens.tolist() == [[0, -1], [1, -1]] and hi.status == 0
    lo = orc.sampling_accept(tgt, 2, cu, dft, draft, np.zeros(2), ua, np.array([0.25, 0.25]))
    assert lo.num_accepted.tolist() == [0, 0] and lo.bonus.tolist() == [0, 0]
    # the same masses one step further from the cut-off keep their sides
    ua_lo = np.full((2, 1), np.float32(0.5), np.float32)
    acc = orc.sampling_accept(tgt, 2, cu, dft, draft, np.zeros(2), ua_lo, np.array([0.75, 0.75]))
    assert acc.num_accepted.tolist() == [1, 1]  # u q_1 < p_1: accepted, bonus from row 1's p
    assert acc.bonus.tolist() == [1, 1]
