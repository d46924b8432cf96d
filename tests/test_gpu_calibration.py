"""GPU parity of the STS recorder, the calibration statistics and the
sequential temperature fit against the oracle, through the C-ABI.

The recorder is integer and byte work: bit-exact.  The statistics' bin
counts, label counts, confidence sums and ECE are exact integers on both
sides: bit-exact, except when a confidence lands on the other side of an fp32
rounding boundary because CUDA's fp64 exp and the host's differ in the last
bit (probability ~2^-29 per sigmoid); such a case is logged as a near tie and
checked with a tolerance.  Brier and log loss are fp64 sums in different
orders, the GPU's terms are float pairs: 1e-12 relative plus 1e-12 absolute.  The fit's ECE curve is exact and its
choices equal, with the same near-tie fallback.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import log_near_tie, require_gpu
from confidence_scheduled_speculative_gb300 import api
from confidence_scheduled_speculative_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _t(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


# ------------------------------------------------------------------ recorder

def _record_case(orc, dev, B, gamma, cap, cursor0, seed, with_select, with_lens, bad=False):
    rng = np.random.default_rng(seed)
    z = rng.normal(0, 2, size=(B, gamma)).astype(np.float32)
    vl = rng.integers(1, gamma + 2, size=B).astype(np.int32)
    correct = np.array([rng.integers(0, (v - 1 if with_lens else gamma) + 1) for v in vl],
                       np.int32)
    if bad:
        vl[:: 7] = 0
        vl[3:: 11] = gamma + 5
        correct[1:: 5] = gamma + 3
        correct[2:: 13] = -2
    sel = (rng.random(B) < 0.6).astype(np.uint8) if with_select else None
    # oracle on host copies of the ring
    rz = rng.normal(size=(cap, gamma)).astype(np.float32)
    rc = rng.integers(-5, 5, size=cap).astype(np.int32)
    rt = rng.integers(-5, 5, size=cap).astype(np.int32)
    g_rz, g_rc, g_rt = _t(rz, dev), _t(rc, dev), _t(rt, dev)
    cur_ref, mask_ref, st_ref = orc.sts_record(z, correct, vl if with_lens else None, sel, rz, rc,
                                               rt, cursor0)
    cursor = torch.tensor([cursor0], dtype=torch.int64, device=dev)
    mask = torch.full((B, gamma), 7, dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dspark_sts_record(_t(z, dev), num_correct=_t(correct, dev), B=B, gamma=gamma,
                          rec_logits=g_rz, rec_correct=g_rc, rec_tested=g_rt, cursor=cursor,
                          status=st, verify_lens=_t(vl, dev) if with_lens else None,
                          select=_t(sel, dev) if with_select else None, prefix_mask=mask)
    torch.cuda.synchronize()
    assert int(cursor.item()) == cur_ref
    np.testing.assert_array_equal(g_rz.cpu().numpy().view(np.uint32), rz.view(np.uint32))
    np.testing.assert_array_equal(g_rc.cpu().numpy(), rc)
    np.testing.assert_array_equal(g_rt.cpu().numpy(), rt)
    np.testing.assert_array_equal(mask.cpu().numpy(), mask_ref)
    assert int(st.item()) == st_ref


@pytest.mark.parametrize("B,gamma,cap,cursor0", [
    (1, 1, 1, 0), (7, 4, 100, 0), (1000, 8, 5000, 4990), (1025, 16, 4096, 123456789),
    (3000, 31, 700, 17), (4096, 16, 4096, 2 ** 40 + 5), (50, 3, 20, 0),
])
@pytest.mark.parametrize("with_select,with_lens", [(False, False), (True, True), (True, False)])
def test_record_parity(orc, dev, B, gamma, cap, cursor0, with_select, with_lens):
    _record_case(orc, dev, B, gamma, cap, cursor0, B * 31 + gamma, with_select, with_lens)


@pytest.mark.parametrize("B,gamma,cap", [(64, 8, 1000), (2048, 16, 300)])
def test_record_parity_bad_lengths(orc, dev, B, gamma, cap):
    _record_case(orc, dev, B, gamma, cap, 5, 99, True, True, bad=True)


def test_record_ring_over_many_steps(orc, dev):
    """Forty steps into one ring that wraps several times."""
    B, gamma, cap = 96, 8, 500
    rng = np.random.default_rng(1)
    rz = np.zeros((cap, gamma), np.float32)
    rc = np.zeros(cap, np.int32)
    rt = np.zeros(cap, np.int32)
    g_rz, g_rc, g_rt = _t(rz, dev), _t(rc, dev), _t(rt, dev)
    cursor = torch.zeros(1, dtype=torch.int64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    cur = 0
    for step in range(40):
        z = rng.normal(size=(B, gamma)).astype(np.float32)
        vl = rng.integers(1, gamma + 2, size=B).astype(np.int32)
        correct = np.array([rng.integers(0, v) for v in vl], np.int32)
        sel = (rng.random(B) < 0.3).astype(np.uint8)
        cur, _, _ = orc.sts_record(z, correct, vl, sel, rz, rc, rt, cur, want_mask=False)
        api.dspark_sts_record(_t(z, dev), num_correct=_t(correct, dev), B=B, gamma=gamma,
                              rec_logits=g_rz, rec_correct=g_rc, rec_tested=g_rt, cursor=cursor,
                              status=st, verify_lens=_t(vl, dev), select=_t(sel, dev))
    torch.cuda.synchronize()
    assert int(cursor.item()) == cur and int(st.item()) == 0
    np.testing.assert_array_equal(g_rz.cpu().numpy(), rz)
    np.testing.assert_array_equal(g_rc.cpu().numpy(), rc)
    np.testing.assert_array_equal(g_rt.cpu().numpy(), rt)


# -------------------------------------------------------------------- stats

def _samples(N, gamma, seed, nan=False, bad_len=False):
    cs = wl.calibration_samples(N, gamma, 1.0 + 0.1 * np.arange(gamma), seed=seed)
    z, correct, tested = cs.conf_logits.copy(), cs.correct.copy(), cs.tested.copy()
    if nan and N > 3:
        z[1, gamma // 2] = np.nan
        z[N - 1, 0] = np.nan
    if bad_len and N > 10:
        tested[::9] = gamma + 2
        correct[::7] = -1
        correct[5] = gamma + 9
    return z, correct, tested


def run_stats(dev, z, correct, tested, T, M, ws=None):
    N, gamma = z.shape
    metrics = torch.zeros((2, gamma, 4), dtype=torch.float64, device=dev)
    hist = torch.zeros((2, gamma, M, 3), dtype=torch.int64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    if ws is None:
        ws = api.workspace(api.dspark_calibration_workspace_bytes(gamma, M), dev)
    api.dspark_calibration_stats(_t(z, dev), rec_correct=_t(correct, dev),
                                 rec_tested=_t(tested, dev), N=N, gamma=gamma,
                                 sts_temps=_t(np.asarray(T, np.float32), dev), n_bins=M,
                                 metrics=metrics, workspace=ws, status=st, hist=hist)
    torch.cuda.synchronize()
    return hist.cpu().numpy().astype(np.uint64), metrics.cpu().numpy(), int(st.item())


def compare_stats(tag, gpu, ref):
    hist, met, st = gpu
    assert st == ref.status, (tag, st, ref.status)
    if np.array_equal(hist, ref.hist):
        np.testing.assert_array_equal(met[..., :2], ref.metrics[..., :2], err_msg=tag)
    else:
        # a confidence rounded to the other side of an fp32 boundary: the
        # counts agree, a few samples move between adjacent bins
        d = np.abs(hist.astype(np.int64) - ref.hist.astype(np.int64))
        log_near_tie({"tag": tag, "max_count_diff": int(d[..., 0].max())})
        np.testing.assert_array_equal(hist[..., 0].sum(-1), ref.hist[..., 0].sum(-1))
        assert d[..., 0].sum() <= 4, tag
        np.testing.assert_allclose(met[..., 1], ref.metrics[..., 1], rtol=0, atol=1e-5)
    # Brier / log loss: float-pair terms (log term within 2^-43 absolute)
    np.testing.assert_allclose(met[..., 2:], ref.metrics[..., 2:], rtol=1e-12, atol=1e-12,
                               err_msg=tag)


@pytest.mark.parametrize("N,gamma,M", [
    (0, 4, 10), (1, 1, 1), (255, 3, 2), (257, 8, 10), (5000, 16, 15), (70001, 8, 32),
    (3000, 31, 10), (40000, 16, 10), (2000, 31, 32),
])
def test_stats_parity(orc, dev, N, gamma, M):
    z, correct, tested = _samples(N, gamma, seed=N + gamma)
    T = (0.6 + 0.1 * np.arange(gamma)).astype(np.float32)
    ref = orc.calib_stats(z, correct, tested, T, M)
    compare_stats(f"stats N={N} g={gamma} M={M}", run_stats(dev, z, correct, tested, T, M), ref)


def test_stats_parity_edge_inputs(orc, dev):
    """NaN logits, lengths out of range and a non-positive temperature."""
    z, correct, tested = _samples(3000, 8, seed=11, nan=True, bad_len=True)
    T = np.ones(8, np.float32)
    T[5] = 0.0
    ref = orc.calib_stats(z, correct, tested, T, 10)
    assert ref.status & orc.ST_BAD_INPUT and ref.status & orc.ST_BAD_LEN
    compare_stats("stats edge", run_stats(dev, z, correct, tested, T, 10), ref)


def test_stats_hand_table(orc, dev):
    """The hand-derived table of the golden fixtures, through the GPU."""
    from conftest import golden
    g = golden("calibration_examples.json")["stats_by_hand"]
    z = np.array([[float(v) for v in r] for r in g["z"]], np.float32)
    hist, met, st = run_stats(dev, z, np.array(g["correct"], np.int32),
                              np.array(g["tested"], np.int32), np.ones(3, np.float32), 2)
    assert st == 0
    assert met[0, :, 0].tolist() == g["cumulative"]["n"]
    assert met[0, :, 1].tolist() == g["cumulative"]["ece"]
    assert met[1, :, 1].tolist() == g["per_position"]["ece"]


def test_stats_workspace_reuse(orc, dev):
    """The workspace comes back zeroed: a second call on other data matches."""
    ws = api.workspace(api.dspark_calibration_workspace_bytes(8, 10), dev)
    for seed in (1, 2, 3):
        z, correct, tested = _samples(9000, 8, seed=seed)
        T = np.full(8, 1.1, np.float32)
        ref = orc.calib_stats(z, correct, tested, T, 10)
        compare_stats(f"reuse {seed}", run_stats(dev, z, correct, tested, T, 10, ws), ref)


# ---------------------------------------------------------------------- fit

def run_fit(dev, z, correct, tested, grid, M, ws=None):
    N, gamma = z.shape
    J = len(grid)
    T = torch.zeros(gamma, dtype=torch.float32, device=dev)
    choice = torch.full((gamma,), -7, dtype=torch.int32, device=dev)
    curve = torch.zeros((gamma, J), dtype=torch.float64, device=dev)
    n_obs = torch.zeros(gamma, dtype=torch.int64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    if ws is None:
        ws = api.workspace(api.dspark_sts_fit_workspace_bytes(N, J, M), dev)
    api.dspark_sts_fit(_t(z, dev), rec_correct=_t(correct, dev), rec_tested=_t(tested, dev), N=N,
                       gamma=gamma, temp_grid=list(grid), n_bins=M, sts_temps_out=T,
                       choice=choice, workspace=ws, status=st, ece_curve=curve, n_obs=n_obs)
    torch.cuda.synchronize()
    return dict(T=T.cpu().numpy(), choice=choice.cpu().numpy(), ece_curve=curve.cpu().numpy(),
                n_obs=n_obs.cpu().numpy(), status=int(st.item()))


def compare_fit(tag, gpu, ref):
    assert gpu["status"] == ref.status, (tag, gpu["status"], ref.status)
    np.testing.assert_array_equal(gpu["n_obs"], ref.n_obs, err_msg=tag)
    if np.array_equal(gpu["ece_curve"], ref.ece_curve):
        np.testing.assert_array_equal(gpu["choice"], ref.choice, err_msg=tag)
        np.testing.assert_array_equal(gpu["T"], ref.T, err_msg=tag)
        return
    # a near tie in a sigmoid: the curves agree closely; the choices agree
    # up to the first depth whose choice the difference could change
    log_near_tie({"tag": tag,
                  "max_ece_diff": float(np.abs(gpu["ece_curve"] - ref.ece_curve).max())})
    np.testing.assert_allclose(gpu["ece_curve"], ref.ece_curve, rtol=0, atol=1e-5)
    for k in range(len(ref.choice)):
        if gpu["choice"][k] != ref.choice[k]:
            c = ref.ece_curve[k]
            assert abs(c[gpu["choice"][k]] - c[ref.choice[k]]) <= 1e-5, tag
            break


@pytest.mark.parametrize("N,gamma,J,M", [
    (0, 3, 4, 10), (1, 1, 1, 1), (300, 4, 7, 10), (4097, 8, 32, 15), (20000, 8, 64, 10),
    (4097, 5, 256, 10), (2000, 31, 16, 32), (513, 6, 100, 3), (1500, 31, 256, 32),
])
def test_fit_parity(orc, dev, N, gamma, J, M):
    z, correct, tested = _samples(N, gamma, seed=3 * N + J)
    grid = wl.temperature_grid(J, 0.3, 3.0)
    ref = orc.sts_fit(z, correct, tested, grid, M)
    compare_fit(f"fit N={N} g={gamma} J={J} M={M}", run_fit(dev, z, correct, tested, grid, M), ref)


def test_fit_parity_edge_inputs(orc, dev):
    z, correct, tested = _samples(5000, 8, seed=12, nan=True, bad_len=True)
    grid = wl.temperature_grid(24)
    ref = orc.sts_fit(z, correct, tested, grid, 10)
    assert ref.status & orc.ST_BAD_INPUT and ref.status & orc.ST_BAD_LEN
    compare_fit("fit edge", run_fit(dev, z, correct, tested, grid, 10), ref)


def test_fit_degenerate(orc, dev):
    z, correct, tested = _samples(1000, 4, seed=5)
    # nothing observed: T = 1, choice -1 everywhere
    r = run_fit(dev, z, correct * 0, tested * 0, wl.temperature_grid(8), 10)
    assert r["choice"].tolist() == [-1] * 4 and r["T"].tolist() == [1.0] * 4
    # duplicate candidates: the lower index
    grid = np.array([2.0, 2.0, 0.5, 0.5], np.float32)
    ref = orc.sts_fit(z, correct, tested, grid, 10)
    compare_fit("fit dup", run_fit(dev, z, correct, tested, grid, 10), ref)


def test_fit_workspace_reuse_and_recovery(orc, dev):
    """Two fits through one workspace; the second recovers known temperatures."""
    true_T = [1.0, 1.5, 0.7, 2.0, 1.0, 1.2, 0.8, 1.0]
    grid = wl.temperature_grid(32)
    ws = api.workspace(api.dspark_sts_fit_workspace_bytes(100000, 32, 10), dev)
    cs = wl.calibration_samples(20000, 8, true_T, seed=7)
    ref = orc.sts_fit(cs.conf_logits, cs.correct, cs.tested, grid, 10)
    compare_fit("reuse 1", run_fit(dev, cs.conf_logits, cs.correct, cs.tested, grid, 10, ws), ref)
    cs = wl.calibration_samples(100000, 8, true_T, seed=1)
    ref = orc.sts_fit(cs.conf_logits, cs.correct, cs.tested, grid, 10)
    r = run_fit(dev, cs.conf_logits, cs.correct, cs.tested, grid, 10, ws)
    compare_fit("reuse 2", r, ref)
    step = np.log(grid[1] / grid[0])
    assert (np.abs(np.log(r["T"] / np.array(true_T))) / step <= 3.0).all()


def test_fit_full_size_sampled(orc, dev):
    """The benchmark's fit configuration (262144 samples, gamma 16, 64
    temperatures, 15 bins): the oracle runs the whole fit once and every
    output is compared."""
    N, gamma, J, M = 262144, 16, 64, 15
    cs = wl.calibration_samples(N, gamma, 1.0 + 0.05 * np.arange(gamma), seed=2026)
    grid = wl.temperature_grid(J)
    ref = orc.sts_fit(cs.conf_logits, cs.correct, cs.tested, grid, M)
    compare_fit("fit full", run_fit(dev, cs.conf_logits, cs.correct, cs.tested, grid, M), ref)


# ------------------------------------------------------------- STS sigmoid

def _sts_gpu(dev, z, T):
    out = torch.empty(z.shape, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dspark_sts_confidence(_t(z, dev), sts_temps=_t(T, dev), conf_out=out, status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(st.item())


def _check_near_ties(t, got, ref):
    """Elements where the GPU and the host differ must sit on an fp32
    rounding midpoint to within a few fp64 ulps (CUDA's and the host's fp64
    exp may differ in the last bit there); none is expected."""
    bad = np.flatnonzero(got.view(np.uint32) != ref.view(np.uint32))
    for i in bad[:16]:
        v = 1.0 / (1.0 + np.exp(-np.float64(t[i])))
        a, b = sorted((np.float64(got[i]), np.float64(ref[i])))
        assert np.nextafter(np.float32(a), np.float32(2)) == np.float32(b), (t[i], got[i], ref[i])
        mid = (a + b) / 2
        assert abs(v - mid) <= 8 * np.spacing(v), (t[i], v, mid)
        log_near_tie({"tag": "sts sweep", "t": float(t[i])})
    return bad.size


def test_sts_confidence_sweep(orc, dev):
    """Every 64th fp32 value with |t| <= 70, both signs, T = 1: the fp32
    evaluation (|t| <= 60) and the fp64 formula beyond it against the host."""
    top = int(np.float32(70.0).view(np.uint32))
    pos = np.arange(0, top + 1, 64, dtype=np.uint32).view(np.float32)
    t = np.concatenate([pos, -pos]).reshape(-1, 1)
    got, st = _sts_gpu(dev, t, np.ones(1, np.float32))
    ref, st_ref = orc.sts_rows(t, np.ones(1, np.float32))
    assert st == st_ref == 0
    assert _check_near_ties(t.ravel(), got.ravel(), ref.ravel()) <= 2


def test_sts_confidence_random_and_edges(orc, dev):
    rng = np.random.default_rng(8)
    z = np.concatenate([rng.normal(0, 3, 200000), rng.normal(0, 40, 50000),
                        rng.uniform(-1e-30, 1e-30, 1000)]).astype(np.float32)
    z[:8] = [np.inf, -np.inf, 0.0, -0.0, 3e38, -3e38, 1e-45, -1e-45]
    gamma = 5
    z = z[: (z.size // gamma) * gamma].reshape(-1, gamma)
    T = np.array([1.0, 0.37, 2.5, 1e-3, 7.0], np.float32)
    got, st = _sts_gpu(dev, z, T)
    ref, st_ref = orc.sts_rows(z, T)
    assert st == st_ref == 0
    assert _check_near_ties((z / T).ravel(), got.ravel(), ref.ravel()) <= 1
    # NaN logits and a zero temperature flag BAD_INPUT and propagate like the host
    z[3, 1] = np.nan
    T[4] = 0.0
    got, st = _sts_gpu(dev, z, T)
    ref, st_ref = orc.sts_rows(z, T)
    assert st == st_ref == orc.ST_BAD_INPUT
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
