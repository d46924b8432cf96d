"""GPU parity of the planner (dspark_plan) and the pack (dspark_pack_verify)
against the CPU oracle, element by element on the same seeded inputs,
through the C-ABI.  Discrete outputs are compared bit-exactly; survivals,
tau and theta too (the arithmetic is defined to give identical floats)."""

import zlib

import numpy as np
import pytest
import torch

from confidence_scheduled_speculative_gb300 import workloads as wl
from gpu_helpers import (compare_plan, oracle_plan, oracle_restage, require_gpu, restage,
                         run_plan_pack)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _pack_ref(orc, step, lens, sentinel):
    return orc.pack(step.anchor, step.draft, step.prefix_lens, lens, step.tiers, step.capacity,
                    sentinel=sentinel)


def _check_pack(tag, gpu, ref, cap):
    tot = ref.total
    np.testing.assert_array_equal(gpu["cu_seqlens"], ref.cu_seqlens, err_msg=f"{tag} cu")
    assert list(gpu["totals"]) == [ref.total, ref.padded], tag
    n = min(max(ref.padded, tot), cap)
    for k in ("ids", "pos", "req", "src"):
        np.testing.assert_array_equal(gpu["packed_" + k][:n], ref[k][:n], err_msg=f"{tag} {k}")


CASES = ([("tiny", s, None) for s in range(6)] + [("qwen_like", s, None) for s in range(3)]
         + [("dsv4_like", s, None) for s in range(3)] + [("mixed", s, None) for s in range(4)]
         + [("stress", 0, f) for f in (None, 0, 1024, 8192, 16384)])


@pytest.mark.parametrize("name,seed,forced", CASES)
def test_plan_and_pack_workloads(dev, orc, name, seed, forced):
    step = wl.make_step(wl.WORKLOADS[name], seed=seed)
    vs, g = run_plan_pack(dev, step, forced)
    ref = oracle_plan(orc, step, forced)
    exp = compare_plan(f"{name}/{seed}/{forced}", g, ref, step.B, step.gamma,
                       step.workload.min_verify_len, oracle_restage(orc, step, forced))
    assert int(g["status"][0]) == exp.status
    # the pack consumes the GPU's verify_lens, equal to the (restaged) oracle's
    p = _pack_ref(orc, step, exp.verify_lens, sentinel=0)
    _check_pack(name, g, p, step.capacity)


def _random_problem(rng):
    while True:
        gamma = int(rng.integers(1, 32))
        B = int(rng.integers(1, 48))
        if B * (gamma + 1) <= 65536:
            break
    mu, sd = rng.uniform(-1, 4), rng.uniform(0.1, 3)
    z = rng.normal(mu, sd, size=(B, gamma)).astype(np.float32)
    if rng.random() < 0.4:  # exact ties: repeat some requests
        k = int(rng.integers(1, B + 1))
        z[rng.integers(0, B, size=k)] = z[int(rng.integers(0, B))]
    if rng.random() < 0.2:  # saturated confidences: survivals of exactly 1.0
        z[:, : max(1, gamma // 2)] = 40.0
    T = rng.uniform(0.5, 2.0, size=gamma).astype(np.float32)
    if rng.random() < 0.3:
        T[:] = 1.0
    eps = float(np.float32(rng.choice([2.0 ** -14, 1e-4, 0.01, 0.2])))
    max_len = int(rng.integers(1, gamma + 2))
    min_len = int(rng.integers(1, max_len + 1)) if rng.random() < 0.3 else 1
    kind = int(rng.integers(0, 2))
    # tables up to 31 entries take the select path, longer ones the rank path
    n = int(rng.integers(1, 12)) if rng.random() < 0.6 else int(rng.integers(12, 40))
    hi = B + B * gamma + 6
    M = np.sort(rng.choice(np.arange(1, hi + 1), size=min(n, hi), replace=False)).astype(np.int32)
    val = (rng.uniform(100, 1000, M.size) if kind == 0 else rng.uniform(0.01, 3.0, M.size))
    if rng.random() < 0.1:
        val[int(rng.integers(0, M.size))] = 0.0 if kind == 0 else -100.0
    forced = -1 if rng.random() < 0.6 else int(rng.integers(0, B * gamma + 4))
    bias, alpha = float(rng.uniform(0, 2)), float(rng.uniform(0, 1))
    return dict(B=B, gamma=gamma, z=z, T=T, eps=eps, min_len=min_len, max_len=max_len,
                kind=kind, M=M, val=val, forced=forced, bias=bias, alpha=alpha)


def _restage(orc, P, **options):
    return restage(orc, P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], P["forced"],
                   P["kind"], P["M"], P["val"], P["bias"], P["alpha"], **options)


def _gpu_plan(dev, P):
    from confidence_scheduled_speculative_gb300 import api
    B, g = P["B"], P["gamma"]
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(survivals=torch.zeros((B, g), dtype=torch.float32, device=dev),
               verify_lens=torch.zeros(B, **i32), budget=torch.zeros(1, **i32),
               tau_theta=torch.zeros(2, dtype=torch.float64, device=dev),
               status=torch.zeros(1, **i32))
    ws = api.workspace(api.dspark_plan_workspace_bytes(B, g), dev)
    api.dspark_plan(torch.from_numpy(P["z"]).to(dev), torch.from_numpy(P["T"]).to(dev), B=B,
                    gamma=g, survival_eps=P["eps"], min_verify_len=P["min_len"],
                    max_verify_len=P["max_len"], forced_budget=P["forced"], cost_kind=P["kind"],
                    cost_M=torch.from_numpy(P["M"]).to(dev),
                    cost_val=torch.from_numpy(P["val"]).to(dev), bias_ms=P["bias"],
                    alpha_ms=P["alpha"], workspace=ws, **out)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


@pytest.mark.parametrize("seed", range(150))
def test_plan_random(dev, orc, seed):
    rng = np.random.default_rng(70000 + seed)
    P = _random_problem(rng)
    g = _gpu_plan(dev, P)
    ref = orc.plan(P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], P["forced"], P["kind"],
                   P["M"], P["val"], P["bias"], P["alpha"])
    exp = compare_plan(f"random/{seed}", g, ref, P["B"], P["gamma"], P["min_len"],
                       _restage(orc, P))
    assert int(g["status"][0]) == exp.status


@pytest.mark.parametrize("seed", range(80))
def test_plan_random_interpolated_table(dev, orc, seed):
    """The interpolated additive table (every budget its own cost; the
    single-CTA interp path), with few and many samples, forced budgets and
    invalid entries."""
    rng = np.random.default_rng(91000 + seed)
    P = _random_problem(rng)
    P["kind"] = 2
    B, g = P["B"], P["gamma"]
    n = int(rng.integers(1, 12)) if rng.random() < 0.5 else int(rng.integers(17, 200))
    hi = B + B * g + 6
    M = np.sort(rng.choice(np.arange(1, hi + 1), size=min(n, hi), replace=False)).astype(np.int32)
    val = np.sort(rng.uniform(0.0, 3.0, M.size))
    if rng.random() < 0.3:
        val = rng.uniform(-0.5, 3.0, M.size)  # not monotone; may go non-positive
    if rng.random() < 0.1:
        val[int(rng.integers(0, M.size))] = np.inf
    P["M"], P["val"] = M, val
    gres = _gpu_plan(dev, P)
    ref = orc.plan(P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], P["forced"], 2,
                   P["M"], P["val"], P["bias"], P["alpha"])
    exp = compare_plan(f"interp/{seed}", gres, ref, B, g, P["min_len"], _restage(orc, P))
    assert int(gres["status"][0]) == exp.status


@pytest.mark.parametrize("seed", range(4))
def test_plan_interpolated_table_on_the_rank_path(dev, orc, seed):
    """Interpolated tables of more than 2048 samples keep the multi-CTA rank
    path; against the oracle."""
    from confidence_scheduled_speculative_gb300 import api
    rng = np.random.default_rng(93000 + seed)
    B, g = 300, 16
    z = rng.normal(1.2, 1.4, (B, g)).astype(np.float32)
    hi = B + B * g + 6
    M = np.sort(rng.choice(np.arange(1, hi + 1), size=api.INTERP_MAX_SAMPLES + 1 + 300 * seed,
                           replace=False)).astype(np.int32)
    val = 0.002 * M + 0.2 * np.sin(M / 53.0) ** 2
    P = dict(B=B, gamma=g, z=z, T=np.ones(g, np.float32), eps=1e-4, min_len=1, max_len=g + 1,
             kind=2, M=M, val=val, forced=-1 if seed < 3 else 1500, bias=1.0, alpha=0.4)
    assert api.planner_path(B * g, 2, M.size) == "rank"
    gres = _gpu_plan(dev, P)
    ref = orc.plan(z, P["T"], 1e-4, 1, g + 1, P["forced"], 2, M, val, 1.0, 0.4)
    exp = compare_plan(f"interp_rank/{seed}", gres, ref, B, g, 1, _restage(orc, P))
    assert int(gres["status"][0]) == exp.status


def _dense_problem(rng, seed):
    """A cost table of more than 64 entries read as given (1-D floor lookup or
    additive ceil-to-tier): the single-CTA dense path up to 6143 entries,
    the rank path beyond."""
    if seed % 4 == 3:  # large: a table at every M can pass 6143 entries
        while True:
            B, g = int(rng.integers(200, 700)), int(rng.integers(8, 32))
            if B * g <= 16380 and B * (g + 1) <= 65536 and B * g > 4700:
                break
    else:
        while True:
            B, g = int(rng.integers(4, 300)), int(rng.integers(2, 32))
            if B * g <= 16380 and B * g >= 70:
                break
    z = rng.normal(rng.uniform(0, 3), rng.uniform(0.3, 2), (B, g)).astype(np.float32)
    if rng.random() < 0.3:
        z[rng.integers(0, B, size=B // 3)] = z[int(rng.integers(0, B))]
    T = np.ones(g, np.float32) if rng.random() < 0.5 else rng.uniform(0.7, 1.5, g).astype(np.float32)
    kind = int(rng.integers(0, 2))
    hi = B + B * g + 4
    if rng.random() < 0.5:  # every M in a range
        lo = int(rng.integers(1, B + 2))
        M = np.arange(lo, hi + 1, dtype=np.int32)
    else:
        n = int(rng.integers(65, hi + 1))
        M = np.sort(rng.choice(np.arange(1, hi + 1), size=min(n, hi), replace=False)).astype(np.int32)
    if kind == 0:
        a_, b_ = rng.uniform(1e-3, 4e-3), rng.uniform(1e-6, 1e-5)
        val = 1.0 / (a_ + b_ * M) if rng.random() < 0.7 else rng.uniform(100, 1000, M.size)
    else:
        val = rng.uniform(0.002, 0.004) * M if rng.random() < 0.7 else rng.uniform(0.01, 3, M.size)
    val = np.asarray(val, np.float64)
    if rng.random() < 0.15:  # an invalid value somewhere
        val[int(rng.integers(0, M.size))] = rng.choice([0.0, -5.0, np.inf, np.nan])
    forced = -1 if rng.random() < 0.7 else int(rng.integers(0, B * g + 3))
    eps = float(np.float32(rng.choice([2.0 ** -14, 1e-4, 0.01])))
    max_len = int(rng.integers(2, g + 2))
    min_len = int(rng.integers(1, max_len + 1)) if rng.random() < 0.25 else 1
    return dict(B=B, gamma=g, z=z, T=T, eps=eps, min_len=min_len, max_len=max_len, kind=kind, M=M,
                val=val, forced=forced, bias=float(rng.uniform(0, 2)),
                alpha=float(rng.uniform(0, 1)))


@pytest.mark.parametrize("seed", range(60))
def test_plan_random_dense_table(dev, orc, seed):
    """Dense tables (the single-CTA dense path up to 6143 entries, the rank
    path beyond): theta bounded in fp32 at every entry and evaluated in fp64
    where the bounds cannot exclude the maximum; the budget, lens, tau and
    theta must equal the oracle's, which evaluates every budget in fp64."""
    rng = np.random.default_rng(47000 + seed)
    P = _dense_problem(rng, seed)
    g = _gpu_plan(dev, P)
    ref = orc.plan(P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], P["forced"], P["kind"],
                   P["M"], P["val"], P["bias"], P["alpha"])
    exp = compare_plan(f"dense/{seed}", g, ref, P["B"], P["gamma"], P["min_len"],
                       _restage(orc, P))
    assert int(g["status"][0]) == exp.status


def _crowded_problem(B, g, p, kind, flat, forced=-1, eps=1e-4):
    """Every request with the same confidences: each depth's survival is
    shared by the whole batch, so one histogram bin holds B equal keys.  With
    B > 512 the bins of the entries left after the bounds hold more keys than
    the dense path gathers at once, and it takes the threshold slots 32
    entries at a time.  A flat table (theta proportional to tau) with
    survivals near eps leaves many entries within the fp32 margin of the
    maximum."""
    z = np.full((B, g), np.log(p / (1 - p)), np.float32)
    M = np.arange(B, B + B * g + 1, dtype=np.int32)
    if kind == 2:  # interpolated: a few samples, every budget a candidate
        M = np.unique(np.linspace(B, B + B * g, 9).astype(np.int32))
    if kind == 0:
        val = np.full(M.size, 500.0) if flat else 1.0 / (2e-3 + 3e-6 * M)
    else:
        val = 1e-9 * M if flat else 0.002 * M
    return dict(B=B, gamma=g, z=z, T=np.ones(g, np.float32), eps=eps, min_len=1,
                max_len=g + 1, kind=kind, M=M, val=val, forced=forced, bias=1.0, alpha=0.5)


@pytest.mark.parametrize("case", [
    dict(B=600, g=8, p=0.3, kind=0, flat=False),
    dict(B=600, g=8, p=0.3, kind=0, flat=True),
    dict(B=700, g=6, p=0.2, kind=1, flat=True),
    dict(B=520, g=11, p=0.6, kind=1, flat=False),
    dict(B=600, g=8, p=0.3, kind=0, flat=True, forced=1234),
    dict(B=600, g=8, p=0.999, kind=0, flat=True, eps=2.0 ** -14),
    dict(B=64, g=8, p=0.3, kind=0, flat=True),
    dict(B=600, g=8, p=0.3, kind=2, flat=True),
    dict(B=600, g=8, p=0.3, kind=2, flat=False, forced=777),
    dict(B=520, g=11, p=0.6, kind=2, flat=False),
])
def test_plan_dense_path_crowded_bins(dev, orc, case):
    """Dense tables (more than 31 entries: the single-CTA dense path) and
    interpolated tables (the single-CTA interp path) over crowded bins and
    flat tables, against the oracle's fp64 evaluation of every budget."""
    P = _crowded_problem(**case)
    from confidence_scheduled_speculative_gb300 import api
    assert api.planner_path(P["B"] * P["gamma"], P["kind"], P["M"].size) == (
        "interp" if P["kind"] == 2 else "dense")
    g = _gpu_plan(dev, P)
    ref = orc.plan(P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], P["forced"], P["kind"],
                   P["M"], P["val"], P["bias"], P["alpha"])
    exp = compare_plan(f"crowded/{case}", g, ref, P["B"], P["gamma"], P["min_len"],
                       _restage(orc, P))
    assert int(g["status"][0]) == exp.status


@pytest.mark.parametrize("kind,bad", [(0, 0.0), (0, -3.0), (0, float("nan")), (1, -1.8),
                                      (1, float("inf"))])
def test_plan_dense_path_flags_bad_values_far_from_the_maximum(dev, orc, kind, bad):
    """An invalid cost at a small budget, where theta is far below the
    maximum: the dense path must still flag it (DSPARK_STATUS_BAD_COST), as
    the oracle does, and plan as the oracle does."""
    rng = np.random.default_rng(5151)
    B, g = 256, 16
    z = rng.normal(1.5, 1.2, (B, g)).astype(np.float32)
    M = np.arange(B, B + B * g + 1, dtype=np.int32)
    val = 1.0 / (3e-3 + 3e-6 * M) if kind == 0 else 0.002 * M
    val = val.astype(np.float64)
    val[3] = bad
    P = dict(B=B, gamma=g, z=z, T=np.ones(g, np.float32), eps=1e-4, min_len=1, max_len=g + 1,
             kind=kind, M=M, val=val, forced=-1, bias=1.0, alpha=0.5)
    gres = _gpu_plan(dev, P)
    ref = orc.plan(z, P["T"], 1e-4, 1, g + 1, -1, kind, M, val, 1.0, 0.5)
    exp = compare_plan(f"bad/{kind}/{bad}", gres, ref, B, g, 1, _restage(orc, P))
    assert int(gres["status"][0]) == exp.status
    assert exp.status & 32  # BAD_COST


def test_plan_dense_and_rank_paths_meet(dev, orc):
    """The largest table the dense path takes and one entry more (the rank
    path) on the same batch, both against the oracle."""
    from confidence_scheduled_speculative_gb300 import api
    rng = np.random.default_rng(4242)
    B, g = 400, 16
    z = rng.normal(1.0, 1.5, (B, g)).astype(np.float32)
    for n in (api.DENSE_MAX_ENTRIES, api.DENSE_MAX_ENTRIES + 1):
        M = np.arange(1, n + 1, dtype=np.int32)
        P = dict(B=B, gamma=g, z=z, T=np.ones(g, np.float32), eps=1e-4, min_len=1,
                 max_len=g + 1, kind=1, M=M, val=0.0025 * M, forced=-1, bias=1.0, alpha=0.3)
        assert api.planner_path(B * g, 1, n) == ("dense" if n == api.DENSE_MAX_ENTRIES else "rank")
        gres = _gpu_plan(dev, P)
        ref = orc.plan(P["z"], P["T"], P["eps"], 1, g + 1, -1, 1, M, P["val"], 1.0, 0.3)
        exp = compare_plan(f"meet/{n}", gres, ref, B, g, 1, _restage(orc, P))
        assert int(gres["status"][0]) == exp.status


def _rank_case(name):
    """Tables that are not interpolated and have more than 6143 entries:
    the multi-CTA rank path (prefix sums in the last CTA's shared memory,
    every entry bounded in fp32, fp64 where the bounds cannot decide)."""
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    B, g = 512, 16
    z = rng.normal(1.2, 1.4, (B, g)).astype(np.float32)
    every_M = np.arange(B, B + B * g + 1, dtype=np.int32)  # 8193 entries
    base = dict(B=B, gamma=g, z=z, T=np.ones(g, np.float32), eps=1e-4, min_len=1, max_len=g + 1,
                forced=-1, bias=1.0, alpha=0.3)
    sps = 1.0 / (3e-3 + 3e-6 * every_M)
    if name == "sps_every_M":
        return dict(base, kind=0, M=every_M, val=sps)
    if name == "sps_every_M_forced":
        return dict(base, kind=0, M=every_M, val=sps, forced=3000)
    add_M = np.arange(1, 8001, dtype=np.int32)
    if name == "additive_8000":
        return dict(base, kind=1, M=add_M, val=0.0025 * add_M)
    if name == "additive_forced_bad_value":  # T < 0 at one entry: BAD_COST
        val = 0.0025 * add_M
        val[1000] = -50.0
        return dict(base, kind=1, M=add_M, val=val, forced=777)
    if name == "sps_unordered":  # M not increasing at one entry: infeasible
        M = every_M.copy()
        M[4000] = M[3999]
        return dict(base, kind=0, M=M, val=sps)
    raise KeyError(name)


@pytest.mark.parametrize("name", ["sps_every_M", "sps_every_M_forced", "additive_8000",
                                  "additive_forced_bad_value", "sps_unordered"])
def test_plan_rank_path_large_tables(dev, orc, name):
    from confidence_scheduled_speculative_gb300 import api
    P = _rank_case(name)
    assert api.planner_path(P["B"] * P["gamma"], P["kind"], P["M"].size) == "rank"
    g = _gpu_plan(dev, P)
    ref = orc.plan(P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], P["forced"], P["kind"],
                   P["M"], P["val"], P["bias"], P["alpha"])
    exp = compare_plan(f"rank/{name}", g, ref, P["B"], P["gamma"], P["min_len"],
                       _restage(orc, P))
    assert int(g["status"][0]) == exp.status


@pytest.mark.parametrize("name", ["dsv4_like", "stress", "qwen_like"])
def test_plan_interpolated_table_workloads(dev, orc, name):
    """Full-size workloads with their additive tier table read as samples of
    an interpolated cost curve."""
    step = wl.make_step(wl.WORKLOADS[name], seed=3)
    w, c = step.workload, step.cost
    P = dict(B=w.B, gamma=w.gamma, z=step.conf_logits, T=step.sts_temps, eps=w.survival_eps,
             min_len=w.min_verify_len, max_len=w.max_len, forced=-1, kind=2,
             M=np.asarray(c.M, np.int32), val=np.asarray(c.val, np.float64), bias=c.bias_ms,
             alpha=c.alpha_ms)
    gres = _gpu_plan(dev, P)
    ref = orc.plan(P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], -1, 2, P["M"],
                   P["val"], P["bias"], P["alpha"])
    exp = compare_plan(f"interp/{name}", gres, ref, w.B, w.gamma, w.min_verify_len,
                       _restage(orc, P))
    assert int(gres["status"][0]) == exp.status


def _select_case(name):
    """Problems for the few-entry-table planner whose threshold bins hold few
    candidates (ranked by counting) or thousands of equal survivals (radix
    passes, ties resolved by depth then request)."""
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    dsv4_M = np.array([256, 512, 1024, 2048, 4096], np.int32)
    dsv4_val = np.array([0.512, 1.024, 2.048, 4.096, 8.192])
    base = dict(T=np.ones(16, np.float32), eps=1e-4, min_len=1, max_len=17, kind=1, M=dsv4_M,
                val=dsv4_val, forced=-1, bias=1.5, alpha=2.56)
    if name == "all_ones":          # every survival exactly 1.0: one bin of 4096
        return dict(base, B=256, gamma=16, z=np.full((256, 16), 40.0, np.float32))
    if name == "all_ones_forced":
        return dict(base, B=256, gamma=16, z=np.full((256, 16), 40.0, np.float32), forced=1001)
    if name == "half_saturated":    # depths < 8 at 1.0, the rest spread
        z = rng.normal(1.5, 1.0, (256, 16)).astype(np.float32)
        z[:, :8] = 40.0
        return dict(base, B=256, gamma=16, z=z)
    if name == "identical_requests":  # 1000 equal survivals per depth
        z = np.tile(rng.normal(2.0, 1.0, 16).astype(np.float32), (1000, 1))
        return dict(base, B=1000, gamma=16, z=z, kind=0, M=np.array([1000, 3000, 9000], np.int32),
                    val=np.array([90.0, 60.0, 25.0]))
    if name == "identical_forced":
        z = np.tile(rng.normal(2.0, 1.0, 16).astype(np.float32), (1000, 1))
        return dict(base, B=1000, gamma=16, z=z, kind=0, M=np.array([1000, 3000, 9000], np.int32),
                    val=np.array([90.0, 60.0, 25.0]), forced=4321)
    if name == "large_spread":      # 12000 candidates, 16 per thread
        z = rng.normal(1.0, 1.5, (600, 20)).astype(np.float32)
        z[rng.integers(0, 600, 200)] = z[7]
        return dict(base, B=600, gamma=20, z=z, T=np.full(20, 1.3, np.float32), max_len=21,
                    M=np.array([600, 1024, 2048, 4096, 8192, 12600], np.int32),
                    val=np.array([0.5, 0.9, 1.8, 3.5, 7.0, 11.0]))
    if name == "sixteen_entries":
        z = rng.normal(1.0, 1.2, (512, 16)).astype(np.float32)
        M = np.linspace(512, 512 * 17, 16).astype(np.int32)
        return dict(base, B=512, gamma=16, z=z, kind=0, M=M, val=1.0 / (1e-3 + 2e-6 * M))
    if name == "thirty_one_entries":  # the largest table the select path takes
        z = rng.normal(1.0, 1.2, (512, 16)).astype(np.float32)
        M = np.linspace(512, 512 * 17, 31).astype(np.int32)
        return dict(base, B=512, gamma=16, z=z, kind=0, M=M, val=1.0 / (1e-3 + 2e-6 * M))
    if name == "thirty_one_entries_forced":  # 32 slots, few gathered candidates
        # every table entry's range holds budgets <= the 8048 kept candidates
        # and the forced budget takes the 32nd slot; the marked bins gather
        # 187 candidates, ranked by counting (not the radix passes)
        z = rng.normal(1.0, 1.2, (512, 16)).astype(np.float32)
        M = np.linspace(512, 8400, 31).astype(np.int32)
        return dict(base, B=512, gamma=16, z=z, kind=0, M=M, val=1.0 / (1e-3 + 2e-6 * M),
                    forced=2222)
    if name == "thirty_one_entries_ties":  # 32 slots through the radix passes
        z = np.tile(rng.normal(2.0, 1.0, 16).astype(np.float32), (1000, 1))
        M = np.linspace(1000, 16000, 31).astype(np.int32)
        return dict(base, B=1000, gamma=16, z=z, M=M, val=2e-4 * M, forced=4321)
    # the forced budget's theta from the entry covering M = B + budget
    z = rng.normal(1.5, 1.0, (256, 16)).astype(np.float32)
    if name == "forced_below_first_sample":  # 1-D: every sample above B + 100 (entry 0)
        return dict(base, B=256, gamma=16, z=z, kind=0,
                    M=np.array([3256, 3756, 4256], np.int32), val=np.array([500.0, 400.0, 300.0]),
                    forced=100)
    if name == "forced_invalid_sps":  # 1-D: the covering entry's SPS is 0 (theta 0, BAD_COST)
        return dict(base, B=256, gamma=16, z=z, kind=0,
                    M=np.array([256, 1000, 3000], np.int32), val=np.array([500.0, 0.0, 300.0]),
                    forced=1500)
    if name == "forced_invalid_additive":  # additive: the covering tier's cost is negative
        return dict(base, B=256, gamma=16, z=z,
                    val=np.array([0.512, -10.0, 2.048, 4.096, 8.192]), forced=200)
    raise KeyError(name)


@pytest.mark.parametrize("name", ["all_ones", "all_ones_forced", "half_saturated",
                                  "identical_requests", "identical_forced", "large_spread",
                                  "sixteen_entries", "thirty_one_entries",
                                  "thirty_one_entries_forced", "thirty_one_entries_ties",
                                  "forced_below_first_sample", "forced_invalid_sps",
                                  "forced_invalid_additive"])
def test_plan_select_bins(dev, orc, name):
    P = _select_case(name)
    g = _gpu_plan(dev, P)
    ref = orc.plan(P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], P["forced"], P["kind"],
                   P["M"], P["val"], P["bias"], P["alpha"])
    exp = compare_plan(f"select/{name}", g, ref, P["B"], P["gamma"], P["min_len"],
                       _restage(orc, P))
    assert int(g["status"][0]) == exp.status


def test_plan_workspace_reused_across_shapes(dev, orc):
    """One zero-filled workspace serves calls of different shapes in a row:
    each call leaves the survival bins it used cleared."""
    from confidence_scheduled_speculative_gb300 import api
    names = ["half_saturated", "large_spread", "all_ones", "identical_forced", "half_saturated"]
    big = max(api.dspark_plan_workspace_bytes(_select_case(n)["B"], _select_case(n)["gamma"])
              for n in names)
    ws = api.workspace(big, dev)
    for n in names:
        P = _select_case(n)
        B, gm = P["B"], P["gamma"]
        i32 = dict(dtype=torch.int32, device=dev)
        out = dict(survivals=torch.zeros((B, gm), dtype=torch.float32, device=dev),
                   verify_lens=torch.zeros(B, **i32), budget=torch.zeros(1, **i32),
                   tau_theta=torch.zeros(2, dtype=torch.float64, device=dev),
                   status=torch.zeros(1, **i32))
        api.dspark_plan(torch.from_numpy(P["z"]).to(dev), torch.from_numpy(P["T"]).to(dev), B=B,
                        gamma=gm, survival_eps=P["eps"], min_verify_len=P["min_len"],
                        max_verify_len=P["max_len"], forced_budget=P["forced"],
                        cost_kind=P["kind"], cost_M=torch.from_numpy(P["M"]).to(dev),
                        cost_val=torch.from_numpy(P["val"]).to(dev), bias_ms=P["bias"],
                        alpha_ms=P["alpha"], workspace=ws, **out)
        torch.cuda.synchronize()
        g = {k: v.cpu().numpy() for k, v in out.items()}
        ref = orc.plan(P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], P["forced"],
                       P["kind"], P["M"], P["val"], P["bias"], P["alpha"])
        exp = compare_plan(f"reuse/{n}", g, ref, B, gm, P["min_len"], _restage(orc, P))
        assert int(g["status"][0]) == exp.status


def test_plan_edge_cases(dev, orc):
    cases = []
    # every survival below eps: budget 0, all lens = min
    cases.append(dict(B=3, gamma=4, z=np.full((3, 4), -12.0, np.float32), T=np.ones(4, np.float32),
                      eps=0.01, min_len=1, max_len=5, kind=0, M=np.array([1], np.int32),
                      val=np.array([5.0]), forced=-1, bias=0.0, alpha=0.0))
    # B = 1, gamma = 1
    cases.append(dict(B=1, gamma=1, z=np.array([[2.0]], np.float32), T=np.ones(1, np.float32),
                      eps=1e-4, min_len=1, max_len=2, kind=1, M=np.array([1, 2], np.int32),
                      val=np.array([1.0, 1.1]), forced=-1, bias=0.5, alpha=0.1))
    # gamma = 31, many identical requests (ties everywhere)
    z = np.tile(np.linspace(4, -1, 31, dtype=np.float32), (40, 1))
    cases.append(dict(B=40, gamma=31, z=z, T=np.ones(31, np.float32), eps=1e-4, min_len=1,
                      max_len=32, kind=0, M=np.arange(40, 40 + 40 * 31 + 1, dtype=np.int32),
                      val=1.0 / (1e-3 + 2e-6 * np.arange(40, 40 + 40 * 31 + 1)), forced=-1,
                      bias=0.0, alpha=0.0))
    # additive table whose largest tier is below B: infeasible
    cases.append(dict(B=8, gamma=3, z=np.ones((8, 3), np.float32), T=np.ones(3, np.float32),
                      eps=1e-4, min_len=2, max_len=4, kind=1, M=np.array([4], np.int32),
                      val=np.array([1.0]), forced=-1, bias=1.0, alpha=0.0))
    # cost table not ascending, forced budget
    cases.append(dict(B=4, gamma=4, z=np.ones((4, 4), np.float32), T=np.ones(4, np.float32),
                      eps=1e-4, min_len=1, max_len=5, kind=0, M=np.array([5, 5, 9], np.int32),
                      val=np.array([1.0, 2.0, 3.0]), forced=3, bias=0.0, alpha=0.0))
    # NaN confidence and a zero temperature
    zn = np.ones((4, 4), np.float32)
    zn[1, 2] = np.nan
    Tz = np.ones(4, np.float32)
    Tz[3] = 0.0
    cases.append(dict(B=4, gamma=4, z=zn, T=Tz, eps=1e-4, min_len=1, max_len=5, kind=0,
                      M=np.array([1], np.int32), val=np.array([3.0]), forced=-1, bias=0.0,
                      alpha=0.0))
    # the largest planner (16380 candidates, odd B)
    rng = np.random.default_rng(5)
    cases.append(dict(B=1365, gamma=12, z=rng.normal(1, 1.5, (1365, 12)).astype(np.float32),
                      T=np.ones(12, np.float32), eps=1e-4, min_len=1, max_len=13, kind=1,
                      M=(2 ** np.arange(10, 16)).astype(np.int32),
                      val=0.001 * 2.0 ** np.arange(10, 16), forced=-1, bias=2.0, alpha=6.825))
    # a dense 1-D table with more than 1024 entries, forced budget
    cases.append(dict(B=300, gamma=9, z=rng.normal(2, 1, (300, 9)).astype(np.float32),
                      T=np.ones(9, np.float32), eps=1e-3, min_len=1, max_len=10, kind=0,
                      M=np.arange(300, 300 + 2701, dtype=np.int32),
                      val=1.0 / (2e-3 + 3e-6 * np.arange(300, 300 + 2701)), forced=1500,
                      bias=0.0, alpha=0.0))
    cases.append(dict(B=300, gamma=9, z=rng.normal(2, 1, (300, 9)).astype(np.float32),
                      T=np.ones(9, np.float32), eps=1e-3, min_len=1, max_len=10, kind=0,
                      M=np.arange(300, 300 + 2701, dtype=np.int32),
                      val=1.0 / (2e-3 + 3e-6 * np.arange(300, 300 + 2701)), forced=-1,
                      bias=0.0, alpha=0.0))
    for i, P in enumerate(cases):
        g = _gpu_plan(dev, P)
        ref = orc.plan(P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], P["forced"],
                       P["kind"], P["M"], P["val"], P["bias"], P["alpha"])
        exp = compare_plan(f"edge/{i}", g, ref, P["B"], P["gamma"], P["min_len"],
                           _restage(orc, P))
        assert int(g["status"][0]) == exp.status, (i, int(g["status"][0]), exp.status)


def _gpu_pack(dev, anchor, draft, prefix, lens, tiers, cap, sentinel):
    from confidence_scheduled_speculative_gb300 import api
    B, g = draft.shape
    i32 = dict(dtype=torch.int32, device=dev)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    outs = [torch.full((max(cap, 1),), sentinel, **i32) for _ in range(4)]
    cu = torch.full((B + 1,), sentinel, **i32)
    totals = torch.zeros(2, **i32)
    status = torch.zeros(1, **i32)
    api.dspark_pack_verify(t(anchor), t(draft), t(prefix), t(lens), B=B, gamma=g, tiers=tiers,
                           capacity=cap, packed_ids=outs[0], packed_pos=outs[1],
                           packed_req=outs[2], packed_src=outs[3], cu_seqlens=cu, totals=totals,
                           status=status)
    torch.cuda.synchronize()
    names = ["ids", "pos", "req", "src"]
    res = {n: o.cpu().numpy()[:cap] for n, o in zip(names, outs)}
    res.update(cu_seqlens=cu.cpu().numpy(), totals=totals.cpu().numpy(),
               status=int(status.cpu()[0]))
    return res


@pytest.mark.parametrize("seed", range(60))
def test_pack_random(dev, orc, seed):
    rng = np.random.default_rng(90000 + seed)
    gamma = int(rng.integers(1, 32))
    B = int(rng.integers(1, 300))
    lens = rng.integers(1, gamma + 2, size=B).astype(np.int32)
    if rng.random() < 0.2:
        lens[rng.integers(0, B)] = int(rng.choice([0, -3, gamma + 2]))
    total = int(np.clip(lens, 1, gamma + 1).sum())
    tiers = []
    if rng.random() < 0.6:
        tiers = sorted(set(int(x) for x in rng.integers(1, 2 * total + 2, size=int(rng.integers(1, 8)))))
    cap = int(rng.choice([total + 64, total, max(0, total - 5), 2 * total + 2]))
    anchor = rng.integers(0, 1000, B)
    draft = rng.integers(0, 1000, (B, gamma))
    prefix = rng.integers(0, 5000, B)
    g = _gpu_pack(dev, anchor, draft, prefix, lens, tiers, cap, sentinel=-9)
    r = orc.pack(anchor, draft, prefix, lens, tiers, cap, sentinel=-9)
    np.testing.assert_array_equal(g["cu_seqlens"], r.cu_seqlens)
    assert list(g["totals"]) == [r.total, r.padded]
    for k in ("ids", "pos", "req", "src"):
        np.testing.assert_array_equal(g[k], r[k][:cap], err_msg=k)  # incl. untouched rows
    assert g["status"] == r.status


def test_pack_page_layout_on_gpu(dev, orc):
    lens = np.array([2, 1, 4], np.int32)
    anchor = np.array([100, 200, 300])
    draft = np.array([[101, 102, 103], [201, 202, 203], [301, 302, 303]])
    g = _gpu_pack(dev, anchor, draft, np.array([10, 20, 30]), lens, [40, 64, 80], 64, -9)
    assert list(g["cu_seqlens"]) == [0, 2, 3, 7]
    assert list(g["ids"][:7]) == [100, 101, 200, 300, 301, 302, 303]
    assert list(g["totals"]) == [7, 40]
    assert np.all(g["req"][7:40] == -1) and np.all(g["req"][40:] == -9)


# ------------------------------------------------- fused plan + pack (one entry point)

def _fused(dev, P, anchor, prefix, draft, tiers, cap, sentinel=-9):
    from confidence_scheduled_speculative_gb300 import api
    B, g = P["B"], P["gamma"]
    i32 = dict(dtype=torch.int32, device=dev)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    out = dict(survivals=torch.zeros((B, g), dtype=torch.float32, device=dev),
               verify_lens=torch.zeros(B, **i32), budget=torch.zeros(1, **i32),
               tau_theta=torch.zeros(2, dtype=torch.float64, device=dev),
               status=torch.zeros(1, **i32))
    pk = {k: torch.full((max(cap, 1),), sentinel, **i32) for k in ("ids", "pos", "req", "src")}
    cu = torch.full((B + 1,), sentinel, **i32)
    totals = torch.full((2,), sentinel, **i32)
    ws = api.workspace(api.dspark_plan_workspace_bytes(B, g), dev)
    api.dspark_plan_pack(torch.from_numpy(P["z"]).to(dev), torch.from_numpy(P["T"]).to(dev),
                         t(anchor), t(draft), t(prefix), B=B, gamma=g, survival_eps=P["eps"],
                         min_verify_len=P["min_len"], max_verify_len=P["max_len"],
                         forced_budget=P["forced"], cost_kind=P["kind"],
                         cost_M=torch.from_numpy(P["M"]).to(dev),
                         cost_val=torch.from_numpy(P["val"]).to(dev), bias_ms=P["bias"],
                         alpha_ms=P["alpha"], tiers=tiers, capacity=cap,
                         packed_ids=pk["ids"], packed_pos=pk["pos"], packed_req=pk["req"],
                         packed_src=pk["src"], cu_seqlens=cu, totals=totals, workspace=ws, **out)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res.update({k: v.cpu().numpy()[:cap] for k, v in pk.items()})
    res.update(cu_seqlens=cu.cpu().numpy(), totals=totals.cpu().numpy())
    return res


def _pack_inputs(rng, B, g, total_hint):
    anchor = rng.integers(0, 1 << 20, B).astype(np.int32)
    draft = rng.integers(0, 1 << 20, (B, g)).astype(np.int32)
    prefix = rng.integers(1, 8192, B).astype(np.int32)
    mode = rng.integers(0, 4)
    if mode == 0:
        tiers = []
    elif mode == 1:  # every tier below the total: flagged, padded = total
        tiers = [1, 2]
    else:
        tiers = sorted(set(int(x) for x in rng.integers(1, 2 * total_hint + 3, size=int(rng.integers(1, 8)))))
    cap = int(rng.integers(0, 2 * total_hint + 4)) if rng.random() < 0.3 else 2 * total_hint + 8
    return anchor, prefix, draft, tiers, cap


@pytest.mark.parametrize("seed", range(80))
def test_plan_pack_fused_random(dev, orc, seed):
    """dspark_plan_pack equals the oracle's planner followed by its pack,
    including untouched rows past the window, capacity overflow and tier
    lists with no tier above the total; the single-CTA planner kernels pack
    in the same launch, tables beyond them take the rank kernel and then the
    pack kernel."""
    rng = np.random.default_rng(90000 + seed)
    P = _random_problem(rng)
    if seed % 5 == 4:  # a 1-D table at every M: the dense path
        B, g = P["B"], P["gamma"]
        P["kind"] = 0
        P["M"] = np.arange(B, B + max(B * g + 2, 40), dtype=np.int32)
        P["val"] = 1.0 / (1e-3 + 2e-6 * P["M"])
    B, g = P["B"], P["gamma"]
    anchor, prefix, draft, tiers, cap = _pack_inputs(rng, B, g, B * (g + 1))
    got = _fused(dev, P, anchor, prefix, draft, tiers, cap)
    ref = orc.plan(P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], P["forced"], P["kind"],
                   P["M"], P["val"], P["bias"], P["alpha"])
    exp = compare_plan(f"fused/{seed}", got, ref, B, g, P["min_len"], _restage(orc, P))
    pr = orc.pack(anchor, draft, prefix, exp.verify_lens, tiers, cap, sentinel=-9)
    np.testing.assert_array_equal(got["cu_seqlens"], pr.cu_seqlens)
    assert list(got["totals"]) == [pr.total, pr.padded]
    for k in ("ids", "pos", "req", "src"):
        np.testing.assert_array_equal(got[k], pr[k][:cap], err_msg=k)
    assert int(got["status"][0]) == (exp.status | pr.status)


@pytest.mark.parametrize("B,g,forced", [(9000, 1, 5000), (5000, 3, -1), (5000, 3, 4000)])
def test_plan_pack_fused_unstaged(dev, orc, B, g, forced):
    """Batches whose pack inputs (B*(gamma+2) words) do not fit the select
    kernel's shared-memory stage: its fused pack reads anchor / prefix /
    drafts from global memory."""
    rng = np.random.default_rng(B * 100 + g)
    z = rng.normal(1.5, 1.2, (B, g)).astype(np.float32)
    M = np.array([B // 2, B, 2 * B, 4 * B, 8 * B], np.int32)
    P = dict(B=B, gamma=g, z=z, T=np.ones(g, np.float32), eps=1e-4, min_len=1, max_len=g + 1,
             kind=1, M=M, val=1e-4 * M, forced=forced, bias=1.5, alpha=0.5)
    assert B * (g + 2) > 24576
    anchor, prefix, draft, _, _ = _pack_inputs(rng, B, g, B * (g + 1))
    tiers, cap = [B, 2 * B, 4 * B], B * (g + 1)
    got = _fused(dev, P, anchor, prefix, draft, tiers, cap)
    ref = orc.plan(P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], P["forced"], P["kind"],
                   P["M"], P["val"], P["bias"], P["alpha"])
    exp = compare_plan(f"unstaged/{B}/{g}/{forced}", got, ref, B, g, P["min_len"],
                       _restage(orc, P))
    pr = orc.pack(anchor, draft, prefix, exp.verify_lens, tiers, cap, sentinel=-9)
    np.testing.assert_array_equal(got["cu_seqlens"], pr.cu_seqlens)
    assert list(got["totals"]) == [pr.total, pr.padded]
    for k in ("ids", "pos", "req", "src"):
        np.testing.assert_array_equal(got[k], pr[k][:cap], err_msg=k)
    assert int(got["status"][0]) == (exp.status | pr.status)


@pytest.mark.parametrize("name", ["thirty_one_entries", "thirty_one_entries_forced",
                                  "thirty_one_entries_ties"])
def test_plan_pack_fused_select_31_entries(dev, orc, name):
    """The select path's largest table through the fused call: budget,
    verify_lens and the packed window bit for bit against the oracle's
    planner and pack, with both ways of finding the thresholds (counting the
    gathered candidates, radix passes) holding all 32 slots."""
    P = _select_case(name)
    B, g = P["B"], P["gamma"]
    rng = np.random.default_rng(5)
    anchor = rng.integers(0, 1 << 20, B).astype(np.int32)
    draft = rng.integers(0, 1 << 20, (B, g)).astype(np.int32)
    prefix = rng.integers(1, 8192, B).astype(np.int32)
    tiers = [1 << i for i in range(9, 16)]
    cap = 1 << 15
    got = _fused(dev, P, anchor, prefix, draft, tiers, cap)
    ref = orc.plan(P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], P["forced"], P["kind"],
                   P["M"], P["val"], P["bias"], P["alpha"])
    exp = compare_plan(f"fused31/{name}", got, ref, B, g, P["min_len"], _restage(orc, P))
    pr = orc.pack(anchor, draft, prefix, exp.verify_lens, tiers, cap, sentinel=-9)
    np.testing.assert_array_equal(got["cu_seqlens"], pr.cu_seqlens)
    assert list(got["totals"]) == [pr.total, pr.padded]
    for k in ("ids", "pos", "req", "src"):
        np.testing.assert_array_equal(got[k], pr[k][:cap], err_msg=k)
    assert int(got["status"][0]) == (exp.status | pr.status)


@pytest.mark.parametrize("name,seed,forced", CASES)
def test_plan_pack_fused_matches_separate_calls(dev, name, seed, forced):
    """On every workload the fused call gives the two calls' outputs bit for bit."""
    from confidence_scheduled_speculative_gb300.engine import StepConfig, VerifyStep
    step = wl.make_step(wl.WORKLOADS[name], seed=seed)
    cfg = StepConfig.from_step(step)
    if forced is not None:
        cfg.forced_budget = forced
    res = []
    for fused in (False, True):
        vs = VerifyStep(cfg, dev)
        vs.load_inputs(step)
        for t in (vs.packed_ids, vs.packed_pos, vs.packed_req, vs.packed_src):
            t.fill_(-3)
        vs.status.zero_()
        if fused:
            vs.plan_pack()
        else:
            vs.plan()
            vs.pack()
        torch.cuda.synchronize()
        r = vs.result()
        r["packed_all"] = np.stack([t.cpu().numpy() for t in (vs.packed_ids, vs.packed_pos,
                                                                vs.packed_req, vs.packed_src)])
        res.append(r)
    for k in res[0]:
        np.testing.assert_array_equal(np.asarray(res[1][k]), np.asarray(res[0][k]), err_msg=k)


# ----------------------------------------- planner options ([AVS] §三)

def _options(rng, P):
    B, g = P["B"], P["gamma"]
    opt = {}
    if rng.random() < 0.5:
        cg = rng.integers(0, 4, B).astype(np.int32)
        rg = cg.copy()
        flip = rng.random(B) < 0.3
        rg[flip] += 1
        opt["conf_gen"], opt["req_gen"] = cg, rg
    if rng.random() < 0.5:
        opt["lagged_z"] = rng.normal(rng.uniform(-1, 3), rng.uniform(0.2, 2), (B, g)).astype(np.float32)
    if rng.random() < 0.6:
        hi = B * (g + 1) + 3
        opt["align_tiers"] = sorted(set(int(x) for x in rng.integers(1, hi + 1, size=int(rng.integers(1, 6)))))
    return opt


def _gpu_plan_ex(dev, P, opt):
    from confidence_scheduled_speculative_gb300 import api
    B, g = P["B"], P["gamma"]
    i32 = dict(dtype=torch.int32, device=dev)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    out = dict(survivals=torch.zeros((B, g), dtype=torch.float32, device=dev),
               verify_lens=torch.zeros(B, **i32), budget=torch.zeros(1, **i32),
               tau_theta=torch.zeros(2, dtype=torch.float64, device=dev),
               status=torch.zeros(1, **i32))
    ws = api.workspace(api.dspark_plan_workspace_bytes(B, g), dev)
    api.dspark_plan_ex(t(P["z"]), t(P["T"]), B=B, gamma=g, survival_eps=P["eps"],
                       min_verify_len=P["min_len"], max_verify_len=P["max_len"],
                       forced_budget=P["forced"], cost_kind=P["kind"], cost_M=t(P["M"]),
                       cost_val=t(P["val"]), bias_ms=P["bias"], alpha_ms=P["alpha"],
                       workspace=ws, conf_generation=t(opt.get("conf_gen")),
                       req_generation=t(opt.get("req_gen")),
                       lagged_conf_logits=t(opt.get("lagged_z")),
                       align_tiers=opt.get("align_tiers"), **out)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _ex_options(opt):
    return dict(conf_gen=opt.get("conf_gen"), req_gen=opt.get("req_gen"),
                lagged_z=opt.get("lagged_z"), align_tiers=opt.get("align_tiers"))


def _oracle_plan_ex(orc, P, opt):
    return orc.plan_ex(P["z"], P["T"], P["eps"], P["min_len"], P["max_len"], P["forced"], P["kind"],
                       P["M"], P["val"], P["bias"], P["alpha"], **_ex_options(opt))


@pytest.mark.parametrize("seed", range(80))
def test_plan_options_random(dev, orc, seed):
    """dspark_plan_ex with a random mix of the generation mask, a lagged
    budget and tier alignment, on every single-CTA planner path, against the
    oracle's composition of the plain planner."""
    rng = np.random.default_rng(61000 + seed)
    P = _random_problem(rng)
    if seed % 4 == 3:  # a 1-D table at every M: the dense select path
        B, g = P["B"], P["gamma"]
        P["kind"] = 0
        P["M"] = np.arange(B, B + max(B * g + 2, 40), dtype=np.int32)
        P["val"] = 1.0 / (1e-3 + 2e-6 * P["M"])
    elif seed % 4 == 2:  # an interpolated table: the interp select path
        B, g = P["B"], P["gamma"]
        P["kind"] = 2
        P["M"] = np.unique(np.linspace(max(1, B - 3), B + B * g + 4, int(rng.integers(2, 9))).astype(np.int32))
        P["val"] = np.sort(rng.uniform(0.05, 3.0, P["M"].size))
    opt = _options(rng, P)
    g = _gpu_plan_ex(dev, P, opt)
    ref = _oracle_plan_ex(orc, P, opt)
    exp = compare_plan(f"options/{seed}/{sorted(opt)}", g, ref, P["B"], P["gamma"],
                       P["min_len"], _restage(orc, P, **_ex_options(opt)))
    assert int(g["status"][0]) == exp.status


@pytest.mark.parametrize("name,interp", [("dsv4_like", False), ("stress", False),
                                         ("mixed", False), ("dsv4_like", True)])
def test_plan_pack_options_workloads(dev, orc, name, interp):
    """The fused call with every option on a workload: lagged confidences
    from another seed, a third of the slots stale, alignment to the pack's
    tiers (the workload's, or powers of two where it has none); the
    dsv4_like tier table also read as interpolation samples."""
    import dataclasses
    from confidence_scheduled_speculative_gb300 import api
    from confidence_scheduled_speculative_gb300.engine import StepConfig, VerifyStep
    step = wl.make_step(wl.WORKLOADS[name], seed=2)
    if interp:
        step = dataclasses.replace(step, cost=dataclasses.replace(step.cost, kind=2))
    lag = wl.make_step(wl.WORKLOADS[name], seed=3)
    B, g = step.B, step.gamma
    rng = np.random.default_rng(9)
    cg = np.arange(B, dtype=np.int32)
    rg = cg + (rng.random(B) < 0.33).astype(np.int32)
    cfg = StepConfig.from_step(step)
    tiers = list(cfg.tiers) or [1 << i for i in range(4, 16)]
    cfg.tiers = tiers
    cfg.capacity = max(cfg.capacity, tiers[-1])
    vs = VerifyStep(cfg, dev)
    vs.load_inputs(step)
    vs.status.zero_()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    api.dspark_plan_pack(vs.conf_logits, vs.sts_temps, vs.anchor, vs.draft, vs.prefix_lens,
                         B=B, gamma=g, survival_eps=cfg.survival_eps,
                         min_verify_len=cfg.min_verify_len, max_verify_len=cfg.max_verify_len,
                         forced_budget=cfg.forced_budget, cost_kind=cfg.cost_kind,
                         cost_M=vs.cost_M, cost_val=vs.cost_val, bias_ms=cfg.bias_ms,
                         alpha_ms=cfg.alpha_ms, tiers=tiers, capacity=cfg.capacity,
                         survivals=vs.survivals, verify_lens=vs.verify_lens, budget=vs.budget,
                         tau_theta=vs.tau_theta, packed_ids=vs.packed_ids,
                         packed_pos=vs.packed_pos, packed_req=vs.packed_req,
                         packed_src=vs.packed_src, cu_seqlens=vs.cu_seqlens, totals=vs.totals,
                         status=vs.status, workspace=vs.plan_ws, conf_generation=t(cg),
                         req_generation=t(rg), lagged_conf_logits=t(lag.conf_logits),
                         align_to_tiers=True)
    got = vs.result()
    w, c = step.workload, step.cost
    ref = orc.plan_ex(step.conf_logits, step.sts_temps, w.survival_eps, w.min_verify_len, w.max_len,
                      w.forced_budget, c.kind, c.M, c.val, c.bias_ms, c.alpha_ms, conf_gen=cg,
                      req_gen=rg, lagged_z=lag.conf_logits, align_tiers=tiers)
    exp = compare_plan(f"options/{name}", got, ref, B, g, w.min_verify_len,
                       restage(orc, step.conf_logits, step.sts_temps, w.survival_eps,
                               w.min_verify_len, w.max_len, w.forced_budget, c.kind, c.M, c.val,
                               c.bias_ms, c.alpha_ms, conf_gen=cg, req_gen=rg,
                               lagged_z=lag.conf_logits, align_tiers=tiers))
    p = orc.pack(step.anchor, step.draft, step.prefix_lens, exp.verify_lens, tiers, cfg.capacity)
    np.testing.assert_array_equal(got["cu_seqlens"], p.cu_seqlens)
    assert list(got["totals"]) == [p.total, p.padded]
