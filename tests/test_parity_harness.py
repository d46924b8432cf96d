"""CPU checks of the planner parity harness (tests/gpu_helpers.compare_plan).

The harness compares the GPU planner with the oracle bit for bit; when a
survival differs in its last bit it reruns the oracle's later steps on the
GPU's survivals and holds the GPU's outputs to that.  These tests feed it
GPU-like results built from the oracle itself, with survivals flipped by one
ulp and lens or budgets planted wrong, and check that it accepts exactly the
results that are correct for the survivals they come with."""

import warnings

import numpy as np
import pytest

from gpu_helpers import compare_plan, restage


def _problem():
    # two requests with equal confidences: equal survivals at every depth;
    # the forced budget of 1 takes the first candidate of the order, which
    # the tie sends to request 0 ([AVS] §一: equal survivals go to the
    # earlier position, then the lower request id)
    z = np.array([[2.0, 1.0], [2.0, 1.0], [0.5, -3.0]], np.float32)
    T = np.ones(2, np.float32)
    M = np.array([3, 4, 5, 6, 7, 8, 9], np.int32)
    val = np.full(M.size, 100.0)
    return dict(z=z, T=T, eps=1e-4, min_len=1, max_len=3, forced=1, kind=0, M=M, val=val,
                bias=0.0, alpha=0.0)


def _run(orc, P):
    args = (P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], P["forced"], P["kind"],
            P["M"], P["val"], P["bias"], P["alpha"])
    return orc.plan(*args), restage(orc, *args)


def _as_gpu(res, survivals=None):
    return {"survivals": np.array(res.survivals if survivals is None else survivals, np.float32),
            "verify_lens": np.array(res.verify_lens, np.int32),
            "budget": np.array([res.budget], np.int32),
            "tau_theta": np.array([res.tau, res.theta], np.float64)}


def _bump(s, r, k):
    """s with element (r, k) one ulp larger."""
    out = np.array(s, np.float32)
    out[r, k] = np.nextafter(out[r, k], np.float32(2.0))
    return out


def test_exact_results_pass(orc):
    P = _problem()
    ref, rs = _run(orc, P)
    assert ref.verify_lens.tolist() == [2, 1, 1]
    assert compare_plan("exact", _as_gpu(ref), ref, 3, 2, 1, rs) is ref


def test_wrong_lens_fail_when_survivals_agree(orc):
    P = _problem()
    ref, rs = _run(orc, P)
    g = _as_gpu(ref)
    g["verify_lens"] = np.array([1, 2, 1], np.int32)  # the tie sent the wrong way
    with pytest.raises(AssertionError):
        compare_plan("wrong lens", g, ref, 3, 2, 1, rs)


def test_flipped_survival_is_held_to_the_restaged_oracle(orc):
    """Request 1's first survival one ulp above request 0's: the candidate
    order, and so the lens, change.  Results planned on the bumped survivals
    pass; the unbumped oracle's lens, now wrong for those survivals, fail."""
    P = _problem()
    ref, rs = _run(orc, P)
    s1 = _bump(ref.survivals, 1, 0)
    alt = rs(s1)
    assert alt.verify_lens.tolist() == [1, 2, 1]
    assert alt.tau != ref.tau  # the selected survival is the bumped one
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")
        got = compare_plan("flip ok", _as_gpu(alt, s1), ref, 3, 2, 1, rs)
        assert got.verify_lens.tolist() == [1, 2, 1]
        stale = _as_gpu(ref, s1)  # lens, budget and tau of the other survivals
        with pytest.raises(AssertionError):
            compare_plan("flip stale", stale, ref, 3, 2, 1, rs)
        bad_tau = _as_gpu(alt, s1)
        bad_tau["tau_theta"][0] = ref.tau
        with pytest.raises(AssertionError):
            compare_plan("flip tau", bad_tau, ref, 3, 2, 1, rs)


def test_flipped_survival_with_wrong_budget_or_lens_fails(orc):
    """A flipped bit away from the boundary leaves the plan as it was; a
    planted lens or budget error is still caught."""
    P = dict(_problem(), forced=-1)
    ref, rs = _run(orc, P)
    s1 = _bump(ref.survivals, 2, 0)
    alt = rs(s1)
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")
        compare_plan("flip far", _as_gpu(alt, s1), ref, 3, 2, 1, rs)
        g = _as_gpu(alt, s1)
        g["verify_lens"] = g["verify_lens"].copy()
        g["verify_lens"][0] += 1
        g["verify_lens"][1] -= 1
        with pytest.raises(AssertionError):
            compare_plan("flip lens", g, ref, 3, 2, 1, rs)
        g = _as_gpu(alt, s1)
        g["budget"][0] += 1
        with pytest.raises(AssertionError):
            compare_plan("flip budget", g, ref, 3, 2, 1, rs)


def test_survivals_apart_by_more_than_the_tolerance_fail(orc):
    P = _problem()
    ref, rs = _run(orc, P)
    s = np.array(ref.survivals, np.float32)
    s[0, 0] += np.float32(3e-6)
    with pytest.raises(AssertionError):
        compare_plan("far", _as_gpu(rs(s), s), ref, 3, 2, 1, rs)


def test_restage_with_options_uses_the_given_survivals(orc):
    """With the plan_ex options (here tier alignment) the restaged plan is
    plan_ex's composition on the given survivals."""
    P = dict(_problem(), forced=-1)
    args = (P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], P["forced"], P["kind"],
            P["M"], P["val"], P["bias"], P["alpha"])
    ref = orc.plan_ex(*args, align_tiers=[5, 6])
    rs = restage(orc, *args, align_tiers=[5, 6])
    same = rs(ref.survivals)
    assert same.verify_lens.tolist() == ref.verify_lens.tolist() and same.tau == ref.tau
    assert compare_plan("options", _as_gpu(ref), ref, 3, 2, 1, rs) is ref
