"""Pins of the oracle's calibration functions (STS recorder, reliability
statistics, sequential temperature fit) against what the pages print, hand
derivations, closed forms and properties that hold at any size.

The recovery test draws samples from a known temperature-miscalibrated head
(the seeded generator) and checks that the fit finds that temperature; the
cross-check tests compare the fitter with the statistics function, which is
pinned on its own by the hand-derived tables.
"""

import math

import numpy as np
import pytest

from conftest import golden
from confidence_scheduled_speculative_gb300 import workloads as wl

Q32 = 2.0 ** 32


def _z(rows):
    return np.array([[float(v) for v in r] for r in rows], np.float32)


# ------------------------------------------------------------------ recorder

def test_prefix_mask_page_example(orc):
    g = golden("calibration_examples.json")["prefix_mask"]
    gamma = g["gamma"]
    z = np.zeros((1, gamma), np.float32)
    rec_z = np.zeros((4, gamma), np.float32)
    rc = np.zeros(4, np.int32)
    rt = np.zeros(4, np.int32)
    cur, mask, st = orc.sts_record(z, [g["num_correct"]], None, None, rec_z, rc, rt, 0)
    assert st == 0 and cur == 1
    assert mask[0].tolist() == g["mask"]
    # a chance match after the first mismatch does not change the label: the
    # mask depends on num_correct alone
    assert mask[0, g["chance_match_after_mismatch_draft_row"]] == 0
    assert rc[0] == 3 and rt[0] == gamma


def test_record_censoring_example(orc):
    g = golden("calibration_examples.json")["censoring"]
    gamma = g["gamma"]
    z = np.zeros((1, gamma), np.float32)
    rec_z = np.zeros((1, gamma), np.float32)
    rc = np.zeros(1, np.int32)
    rt = np.zeros(1, np.int32)
    _, mask, st = orc.sts_record(z, [g["tested"]], [g["verify_len"]], None, rec_z, rc, rt, 0)
    assert st == 0 and rt[0] == g["tested"] and rc[0] == g["tested"]
    assert mask[0].tolist() == [1] * 4 + [0] * 4
    # depths past the window carry no label: the statistics leave them out
    res = orc.calib_stats(rec_z, rc, rt, np.ones(gamma, np.float32), 4)
    n = res.metrics[0, :, 0]
    assert [k for k in range(gamma) if n[k] > 0] == g["observed_depths"]


def test_record_ring_by_hand(orc):
    gamma = 3
    z = np.arange(4 * gamma, dtype=np.float32).reshape(4, gamma)
    cap = 5
    rec_z = np.full((cap, gamma), -1, np.float32)
    rc = np.full(cap, -1, np.int32)
    rt = np.full(cap, -1, np.int32)
    sel = np.array([1, 0, 1, 1], np.uint8)
    cur, mask, st = orc.sts_record(z, [0, 1, 2, 3], [4, 4, 3, 2], sel, rec_z, rc, rt, 3)
    assert st == orc.ST_BAD_LEN and cur == 6
    # rows 0, 2, 3 land at slots 3, 4, 0
    assert rec_z[3].tolist() == z[0].tolist() and rec_z[4].tolist() == z[2].tolist()
    assert rec_z[0].tolist() == z[3].tolist()
    assert rc.tolist() == [1, -1, -1, 0, 2] and rt.tolist() == [1, -1, -1, 3, 2]
    # request 3: verify_len 2 -> one tested draft; correct 3 is clamped to 1
    # (the flag above)
    assert mask.tolist() == [[0, 0, 0], [1, 0, 0], [1, 1, 0], [1, 0, 0]]


def test_record_clamps_and_capacity(orc):
    gamma = 4
    z = np.zeros((3, gamma), np.float32)
    rec_z = np.zeros((2, gamma), np.float32)
    rc = np.full(2, -1, np.int32)
    rt = np.full(2, -1, np.int32)
    # verify_len 0 and 9 are outside [1, gamma+1]; correct 5 > tested
    cur, _, st = orc.sts_record(z, [0, 5, 2], [0, 9, 3], None, rec_z, rc, rt, 7)
    assert cur == 10
    assert st & orc.ST_BAD_LEN and st & orc.ST_CAPACITY
    # three rows into two slots: rows 1 and 2 survive, at slots (7+1)%2, (7+2)%2
    assert rt.tolist() == [4, 2] and rc.tolist() == [4, 2]


# -------------------------------------------------------------- reliability

def test_reliability_by_hand(orc):
    g = golden("calibration_examples.json")["ece_by_hand"]
    hist, met, E = orc.reliability(g["p"], g["y"], g["n_bins"])
    assert hist.tolist() == g["hist"]
    assert met[0] == 4 and met[1] == g["ece"] and E == int(g["ece"] * 4 * Q32)
    assert met[2] == g["brier"]
    assert abs(met[3] - g["logloss"]) < 1e-15


def test_reliability_overconfident_page_example(orc):
    g = golden("calibration_examples.json")["overconfident_bin"]
    y = [1] * g["passing"] + [0] * (g["n"] - g["passing"])
    _, met, _ = orc.reliability([g["p"]] * g["n"], y, 10)
    assert abs(met[1] - g["ece"]) < 1e-15


@pytest.mark.parametrize("p0,k,n", [(0.625, 3, 8), (0.125, 0, 5), (1.0, 7, 7), (0.0, 2, 9),
                                    (0.5, 1, 3)])
def test_reliability_constant_prediction(orc, p0, k, n):
    """All predictions p0 (exact in binary), k of n labels 1: ECE = |k/n - p0|,
    Brier = (k (1-p0)^2 + (n-k) p0^2) / n, log loss with the 2^-24 clamp."""
    y = [1] * k + [0] * (n - k)
    hist, met, E = orc.reliability([p0] * n, y, 10)
    assert met[0] == n
    assert E == abs(k * int(Q32) - n * int(p0 * Q32))
    assert abs(met[1] - abs(k / n - p0)) < 1e-15
    assert abs(met[2] - (k * (1 - p0) ** 2 + (n - k) * p0 ** 2) / n) < 1e-15
    pc = min(max(p0, 2.0 ** -24), 1 - 2.0 ** -24)
    ll = (-k * math.log(pc) - (n - k) * math.log(1 - pc)) / n
    assert abs(met[3] - ll) < 1e-12 * max(1.0, ll)
    # one bin holds everything: the right one
    b = min(int(p0 * 10), 9)
    assert hist[b].tolist() == [n, k, n * int(p0 * Q32)]
    assert hist.sum(axis=0)[0] == n


def test_reliability_perfectly_calibrated_is_zero(orc):
    p = [0.375] * 8 + [0.875] * 8 + [0.0625] * 16
    y = [1] * 3 + [0] * 5 + [1] * 7 + [0] * 1 + [1] * 1 + [0] * 15
    _, met, E = orc.reliability(p, y, 10)
    assert E == 0 and met[1] == 0.0


def test_reliability_bin_edges(orc):
    # p = 0.5 with two bins goes up; p = 1 goes to the last bin; p = 0 to bin 0
    hist, _, _ = orc.reliability([0.5, 1.0, 0.0], [1, 1, 0], 2)
    assert hist[:, 0].tolist() == [1, 2]
    # fp32(0.1) is just above 0.1, so floor(p*10) = 1
    hist, _, _ = orc.reliability([0.1], [0], 10)
    assert hist[1, 0] == 1
    # the confidence sum floors to 2^-32 units
    hist, _, _ = orc.reliability([2.0 ** -40], [0], 1)
    assert hist[0, 2] == 0


def test_reliability_single_bin_is_calibration_in_the_large(orc):
    rng = np.random.default_rng(5)
    p = rng.random(1000).astype(np.float32)
    y = (rng.random(1000) < 0.4).astype(np.uint8)
    _, met, _ = orc.reliability(p, y, 1)
    q = np.floor(p.astype(np.float64) * Q32) / Q32
    assert abs(met[1] - abs(y.mean() - q.mean())) < 1e-12


def test_reliability_permutation_invariant(orc):
    rng = np.random.default_rng(6)
    p = rng.random(5000).astype(np.float32)
    y = (rng.random(5000) < p).astype(np.uint8)
    h1, m1, E1 = orc.reliability(p, y, 15)
    perm = rng.permutation(5000)
    h2, m2, E2 = orc.reliability(p[perm], y[perm], 15)
    assert E1 == E2 and (h1 == h2).all() and m1[1] == m2[1]
    assert abs(m1[2] - m2[2]) < 1e-13 and abs(m1[3] - m2[3]) < 1e-12


def test_reliability_empty(orc):
    hist, met, E = orc.reliability(np.zeros(0, np.float32), np.zeros(0, np.uint8), 4)
    assert E == 0 and met.tolist() == [0.0, 0.0, 0.0, 0.0] and hist.sum() == 0


# -------------------------------------------------------------------- stats

def test_calib_stats_by_hand(orc):
    g = golden("calibration_examples.json")["stats_by_hand"]
    res = orc.calib_stats(_z(g["z"]), g["correct"], g["tested"], np.ones(3, np.float32),
                          g["n_bins"])
    assert res.status == 0
    for f, key in ((0, "cumulative"), (1, "per_position")):
        m = res.metrics[f]
        assert m[:, 0].tolist() == g[key]["n"]
        assert m[:, 1].tolist() == g[key]["ece"]
        assert np.allclose(m[:, 2], g[key]["brier"], rtol=0, atol=1e-15)


def test_calib_stats_matches_survival(orc):
    """The cumulative flavour at depth k scores the planner's own survival
    S_k (the same fp32 product), on the samples whose window reached k."""
    cs = wl.calibration_samples(3000, 6, [1.0, 1.3, 0.8, 1.0, 2.0, 1.0], seed=3)
    T = np.array([1.0, 1.25, 0.75, 1.0, 1.5, 1.1], np.float32)
    res = orc.calib_stats(cs.conf_logits, cs.correct, cs.tested, T, 12)
    s_raw, _, _ = orc.survival(cs.conf_logits, T, 0.0)
    for k in range(6):
        take = cs.tested > k
        p = s_raw[take, k]
        y = (cs.correct[take] > k).astype(np.uint8)
        hist, met, _ = orc.reliability(p, y, 12)
        assert (res.hist[0, k] == hist).all()
        assert res.metrics[0, k, 1] == met[1]
        # per-position: c_k given the prefix survived through k-1
        c = np.array([orc.sts(float(zz), float(T[k])) for zz in cs.conf_logits[:, k]],
                     np.float32)
        take = (cs.tested > k) & (cs.correct >= k)
        hist, met, _ = orc.reliability(c[take], (cs.correct[take] > k).astype(np.uint8), 12)
        assert (res.hist[1, k] == hist).all()


def test_calib_stats_nan_and_bad_temperature(orc):
    z = np.array([[0.5, np.nan, 1.0], [1.0, 1.0, 1.0]], np.float32)
    res = orc.calib_stats(z, [3, 3], [3, 3], np.ones(3, np.float32), 4)
    assert res.status & orc.ST_BAD_INPUT
    # the NaN leaves sample 0 out of depth 1 (both flavours) and of the
    # cumulative flavour at depth 2; its c_2 is still scored
    assert res.metrics[0, :, 0].tolist() == [2, 1, 1]
    assert res.metrics[1, :, 0].tolist() == [2, 1, 2]
    res = orc.calib_stats(np.ones((1, 2), np.float32), [1], [2], np.array([1, 0], np.float32), 4)
    assert res.status & orc.ST_BAD_INPUT


def test_calib_stats_clamps_lengths(orc):
    z = np.zeros((2, 3), np.float32)
    res = orc.calib_stats(z, [5, -1], [2, 7], np.ones(3, np.float32), 2)
    assert res.status & orc.ST_BAD_LEN
    # sample 0: tested 2, correct clamped to 2; sample 1: tested 3, correct 0
    assert res.metrics[0, :, 0].tolist() == [2, 2, 1]


# ---------------------------------------------------------------------- fit

def test_fit_recovers_true_temperature(orc):
    """Samples from a head miscalibrated by known per-depth temperatures: the
    fit lands within a few grid steps of each one."""
    true_T = [1.0, 1.5, 0.7, 2.0, 1.0, 1.2, 0.8, 1.0]
    cs = wl.calibration_samples(100000, 8, true_T, seed=1)
    grid = wl.temperature_grid(32)
    res = orc.sts_fit(cs.conf_logits, cs.correct, cs.tested, grid, 10)
    assert res.status == 0
    step = math.log(grid[1] / grid[0])
    err = np.abs(np.log(res.T / np.array(true_T))) / step
    assert (err <= 3.0).all(), (res.T, true_T)
    # the fitted temperatures are no worse calibrated than the true ones by
    # more than sampling noise, and much better than T = 1 at the
    # miscalibrated depths
    fit = orc.calib_stats(cs.conf_logits, cs.correct, cs.tested, res.T, 10).metrics[0, :, 1]
    one = orc.calib_stats(cs.conf_logits, cs.correct, cs.tested, np.ones(8, np.float32),
                          10).metrics[0, :, 1]
    assert fit[3] < one[3] / 3 and fit[1] < one[1] / 2


def test_fit_closed_form_two_point(orc):
    """Logits +-a at depth 0 with label rates r and 1-r: with fine bins,
    ECE(T) = |r - sigmoid(a/T)|, minimised at T = a / logit(r)."""
    a = 2.0 * math.log(3.0)  # logit(3/4) = ln 3, so T* = 2
    n = 400
    z = np.zeros((2 * n, 1), np.float32)
    z[:n, 0] = a
    z[n:, 0] = -a
    correct = np.zeros(2 * n, np.int32)
    correct[: 3 * n // 4] = 1          # 3/4 of the +a samples pass
    correct[n: n + n // 4] = 1         # 1/4 of the -a samples pass
    tested = np.ones(2 * n, np.int32)
    grid = np.array([1.0, 1.5, 2.0, 2.5, 3.0], np.float32)
    res = orc.sts_fit(z, correct, tested, grid, 32)
    assert res.choice.tolist() == [2] and res.T.tolist() == [2.0]
    for j, T in enumerate(grid):
        s = 1.0 / (1.0 + math.exp(-float(np.float32(a)) / float(T)))
        assert abs(res.ece_curve[0, j] - abs(0.75 - s)) < 1e-6


def test_fit_matches_stats_brute_force(orc):
    """ece_curve[k][j] is the cumulative ECE at depth k under the temperatures
    already chosen for depths < k and grid[j] at k; choice is its first
    minimiser."""
    cs = wl.calibration_samples(4000, 5, [1.2, 0.8, 1.5, 1.0, 2.0], seed=9)
    grid = wl.temperature_grid(9, 0.5, 2.5)
    res = orc.sts_fit(cs.conf_logits, cs.correct, cs.tested, grid, 8)
    for k in range(5):
        eces = []
        for j in range(9):
            T = np.ones(5, np.float32)
            T[:k] = res.T[:k]
            T[k] = grid[j]
            m = orc.calib_stats(cs.conf_logits, cs.correct, cs.tested, T, 8).metrics[0, k]
            eces.append(m[1])
            assert m[0] == res.n_obs[k]
        assert res.ece_curve[k].tolist() == eces
        assert res.choice[k] == int(np.argmin(eces))
        assert res.T[k] == grid[res.choice[k]]


def test_fit_is_sequential(orc):
    """Changing the data of depths > k leaves the choices of depths <= k."""
    cs = wl.calibration_samples(3000, 6, 1.3, seed=4)
    grid = wl.temperature_grid(16)
    a = orc.sts_fit(cs.conf_logits, cs.correct, cs.tested, grid, 10)
    z = cs.conf_logits.copy()
    z[:, 3:] = -z[:, 3:] * 2.0
    b = orc.sts_fit(z, cs.correct, cs.tested, grid, 10)
    assert (a.choice[:3] == b.choice[:3]).all()
    assert (a.ece_curve[:3] == b.ece_curve[:3]).all()


def test_fit_degenerate_cases(orc):
    cs = wl.calibration_samples(500, 4, 1.0, seed=2)
    # nothing observed: T = 1, choice -1
    res = orc.sts_fit(cs.conf_logits, cs.correct * 0, np.zeros(500, np.int32),
                      wl.temperature_grid(8), 10)
    assert res.choice.tolist() == [-1] * 4 and res.T.tolist() == [1.0] * 4
    assert res.n_obs.tolist() == [0] * 4
    # one candidate: chosen wherever something is observed
    res = orc.sts_fit(cs.conf_logits, cs.correct, cs.tested, np.array([1.7], np.float32), 10)
    assert res.choice.tolist() == [0] * 4 and res.T.tolist() == [np.float32(1.7)] * 4
    # duplicate candidates tie: the lower index wins
    res = orc.sts_fit(cs.conf_logits, cs.correct, cs.tested,
                      np.array([2.0, 2.0, 0.5], np.float32), 10)
    assert set(res.choice.tolist()) <= {0, 2}
    # permuting the samples changes nothing
    perm = np.random.default_rng(0).permutation(500)
    a = orc.sts_fit(cs.conf_logits, cs.correct, cs.tested, wl.temperature_grid(8), 10)
    b = orc.sts_fit(cs.conf_logits[perm], cs.correct[perm], cs.tested[perm],
                    wl.temperature_grid(8), 10)
    assert (a.choice == b.choice).all() and (a.ece_curve == b.ece_curve).all()
