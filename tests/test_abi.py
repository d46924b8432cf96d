"""The C-ABI library builds, loads and exports every symbol include/*.h
declares; host-side argument checks return their error codes.  No call here
reaches the GPU: each rejected call returns before anything is enqueued."""

import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT

FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: rejected before any CUDA call


@pytest.fixture(scope="module")
def lib():
    from confidence_scheduled_speculative_gb300 import build
    try:
        path = build.build()
    except RuntimeError as e:  # pragma: no cover - toolkit missing
        pytest.skip(str(e))
    return ctypes.CDLL(path)


def declared_symbols():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        with open(h) as f:
            text = f.read()
        names += re.findall(r"DSPARK_API[^;(]*?\b(dspark_\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_four_calls():
    names = declared_symbols()
    for n in ("dspark_plan", "dspark_pack_verify", "dspark_greedy_accept", "dspark_cap_accept"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_and_version(lib):
    lib.dspark_strerror.restype = ctypes.c_char_p
    assert lib.dspark_strerror(0) == b"ok"
    assert b"invalid" in lib.dspark_strerror(-1)
    assert b"workspace" in lib.dspark_strerror(-2)
    assert lib.dspark_version() >= 100


class Params(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("gamma", ctypes.c_int32), ("eps", ctypes.c_float),
                ("min_len", ctypes.c_int32), ("max_len", ctypes.c_int32),
                ("forced", ctypes.c_int32)]


class Cost(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("n", ctypes.c_int32), ("M", ctypes.c_void_p),
                ("val", ctypes.c_void_p), ("bias", ctypes.c_double), ("alpha", ctypes.c_double)]


def _plan(lib, p, c, null_out=False):
    f = lib.dspark_plan
    f.restype = ctypes.c_int
    out = None if null_out else FAKE
    return f(FAKE, FAKE, ctypes.byref(p), ctypes.byref(c), FAKE, out, FAKE, FAKE, None,
             ctypes.c_size_t(0), FAKE, None)


def test_plan_argument_checks(lib):
    good = dict(B=4, gamma=4, eps=1e-4, min_len=1, max_len=5, forced=-1)
    cost = Cost(0, 3, FAKE.value, FAKE.value, 0.0, 0.0)
    assert _plan(lib, Params(**good), cost, null_out=True) == -1
    assert _plan(lib, Params(**{**good, "B": 0}), cost) == -1
    assert _plan(lib, Params(**{**good, "gamma": 32}), cost) == -4
    assert _plan(lib, Params(**{**good, "eps": 1e-6}), cost) == -4
    assert _plan(lib, Params(**{**good, "eps": 2.0}), cost) == -4
    assert _plan(lib, Params(**{**good, "eps": float("nan")}), cost) == -1
    assert _plan(lib, Params(**{**good, "min_len": 3, "max_len": 2}), cost) == -1
    assert _plan(lib, Params(**{**good, "max_len": 6}), cost) == -1
    assert _plan(lib, Params(**{**good, "B": 2048, "gamma": 16}), cost) == -4  # 2048*17 > 2^16
    assert _plan(lib, Params(**{**good, "B": 1025, "gamma": 16}), cost) == -4  # > 16384 candidates
    assert _plan(lib, Params(**good), Cost(3, 3, FAKE.value, FAKE.value, 0, 0)) == -1
    # kind 2 (interpolated additive) passes the kind check and stops at the workspace
    assert _plan(lib, Params(**good), Cost(2, 3, FAKE.value, FAKE.value, 0, 0)) == -2
    assert _plan(lib, Params(**good), Cost(0, 0, FAKE.value, FAKE.value, 0, 0)) == -1
    assert _plan(lib, Params(**good), Cost(1, 3, None, FAKE.value, 0, 0)) == -1
    lib.dspark_plan_workspace_bytes.restype = ctypes.c_size_t
    need = lib.dspark_plan_workspace_bytes(256, 16)
    assert need >= 12 * 256 * 16 and need % 256 == 0
    # a missing or short planner workspace is rejected before any launch
    f = lib.dspark_plan
    assert f(FAKE, FAKE, ctypes.byref(Params(**good)), ctypes.byref(cost), FAKE, FAKE, FAKE,
             FAKE, None, ctypes.c_size_t(0), FAKE, None) == -2
    assert f(FAKE, FAKE, ctypes.byref(Params(**{**good, "B": 256, "gamma": 16, "max_len": 17})),
             ctypes.byref(cost), FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.c_size_t(need - 256), FAKE,
             None) == -2


def test_pack_argument_checks(lib):
    f = lib.dspark_pack_verify
    f.restype = ctypes.c_int
    tiers = (ctypes.c_int32 * 65)(*range(1, 66))

    def call(B=4, gamma=4, n_tiers=0, cap=16, t=tiers, first=FAKE):
        return f(first, FAKE, FAKE, FAKE, B, gamma, t, n_tiers, cap, FAKE, FAKE, FAKE, FAKE,
                 FAKE, FAKE, FAKE, None)

    assert call(first=None) == -1
    assert call(B=0) == -1
    assert call(gamma=32) == -1
    assert call(cap=-1) == -1
    assert call(n_tiers=65) == -1
    bad = (ctypes.c_int32 * 3)(8, 4, 16)
    assert call(n_tiers=3, t=bad) == -1


def test_accept_argument_checks(lib):
    g = lib.dspark_greedy_accept
    g.restype = ctypes.c_int
    lib.dspark_accept_workspace_bytes.restype = ctypes.c_size_t
    need = lib.dspark_accept_workspace_bytes(100, 1000)
    assert need >= 100 * 8 and need % 256 == 0

    def call(dtype=0, ld=1024, V=1000, max_rows=100, ws_bytes=None, new_seq=None, prefix=FAKE,
             ws=FAKE):
        wb = need if ws_bytes is None else ws_bytes
        return g(FAKE, dtype, ctypes.c_int64(ld), V, max_rows, FAKE, FAKE, prefix, 4, 4, None,
                 FAKE, FAKE, FAKE, new_seq, FAKE, ws, ctypes.c_size_t(wb), FAKE, None)

    assert call(dtype=2) == -1
    assert call(ld=999) == -1
    assert call(V=0) == -1
    assert call(max_rows=-1) == -1
    assert call(new_seq=FAKE, prefix=None) == -1
    assert call(ws_bytes=need - 8) == -2
    assert call(ws=None) == -2
    assert call(ws=ctypes.c_void_p(0x10010)) == -2  # not 256-byte aligned
    c = lib.dspark_cap_accept
    c.restype = ctypes.c_int
    assert c(FAKE, 0, ctypes.c_int64(1024), 1000, FAKE, FAKE, FAKE, 4, 4, None, FAKE, FAKE,
             FAKE, None, FAKE, None, FAKE, FAKE, ctypes.c_size_t(need), FAKE, None) == -1


def test_static_accept_rejects_rows_beyond_its_maximum(lib):
    f = lib.dspark_greedy_accept_static
    f.restype = ctypes.c_int
    assert f(FAKE, 0, ctypes.c_int64(1024), 1000, 32769, FAKE, FAKE, FAKE, 4, 4, None, FAKE, FAKE,
             FAKE, None, FAKE, FAKE, None) == -4
    assert f(FAKE, 0, ctypes.c_int64(1024), 1000, -1, FAKE, FAKE, FAKE, 4, 4, None, FAKE, FAKE,
             FAKE, None, FAKE, FAKE, None) == -1


def test_plan_pack_argument_checks(lib):
    f = lib.dspark_plan_pack
    f.restype = ctypes.c_int
    good = dict(B=4, gamma=4, eps=1e-4, min_len=1, max_len=5, forced=-1)
    cost = Cost(1, 3, FAKE.value, FAKE.value, 0.0, 0.0)
    lib.dspark_plan_workspace_bytes.restype = ctypes.c_size_t
    need = lib.dspark_plan_workspace_bytes(4, 4)
    tiers = (ctypes.c_int32 * 3)(8, 16, 32)
    bad_tiers = (ctypes.c_int32 * 3)(8, 4, 32)

    def call(p=good, anchor=FAKE, t=tiers, n_t=3, cap=16, ws=FAKE, wsb=need, cu=FAKE):
        return f(FAKE, FAKE, ctypes.byref(Params(**p)), ctypes.byref(cost), FAKE, FAKE, FAKE, FAKE,
                 anchor, FAKE, FAKE, t, n_t, cap, FAKE, FAKE, FAKE, FAKE, cu, FAKE, ws,
                 ctypes.c_size_t(wsb), FAKE, None)

    assert call(p={**good, "gamma": 32}) == -4       # planner checks first
    assert call(ws=None) == -2
    assert call(wsb=need - 256) == -2
    assert call(anchor=None) == -1                   # then the pack's
    assert call(cu=None) == -1
    assert call(cap=-1) == -1
    assert call(t=bad_tiers) == -1
    assert call(n_t=65) == -1


def test_scatter_argument_checks(lib):
    f = lib.dspark_scatter_compact_to_strided
    f.restype = ctypes.c_int

    def call(src=FAKE, ld_src=8, width=8, eb=2, rows=4, ld_dst=8, dst_rows=10, dst=FAKE):
        return f(src, ctypes.c_int64(ld_src), width, eb, FAKE, FAKE, rows, dst,
                 ctypes.c_int64(ld_dst), dst_rows, FAKE, None)

    assert call(src=None) == -1
    assert call(dst=None) == -1
    assert call(eb=3) == -1
    assert call(width=0) == -1
    assert call(ld_src=7) == -1
    assert call(ld_dst=4) == -1
    assert call(rows=-1) == -1
    g = lib.dspark_scatter_compact_to_strided_ex
    g.restype = ctypes.c_int
    assert g(None, ctypes.c_int64(8), 8, 2, FAKE, FAKE, 4, FAKE, ctypes.c_int64(8), 10,
             ctypes.c_int64(0), FAKE, None) == -1
    assert g(FAKE, ctypes.c_int64(8), 8, 3, FAKE, FAKE, 4, FAKE, ctypes.c_int64(8), 10,
             ctypes.c_int64(-1), FAKE, None) == -1


def test_pad_to_tier_argument_checks(lib):
    f = lib.dspark_pad_to_tier
    f.restype = ctypes.c_int
    assert f(None, 8, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == -1
    assert f(FAKE, -1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == -1
    assert f(FAKE, 8, FAKE, FAKE, FAKE, None, FAKE, FAKE, None) == -1
    assert f(FAKE, 8, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == -1


def test_sampling_argument_checks(lib):
    f = lib.dspark_sampling_accept
    f.restype = ctypes.c_int
    lib.dspark_sampling_workspace_bytes.restype = ctypes.c_size_t
    need = lib.dspark_sampling_workspace_bytes(100, 4, 4)
    assert need % 256 == 0 and need >= 16 * 104

    def call(dtype=0, ld=1024, V=1000, B=4, g=4, ws=FAKE, wsb=need, u=FAKE, prefix=FAKE, new_seq=None):
        return f(FAKE, dtype, ctypes.c_int64(ld), V, 100, FAKE, FAKE, ctypes.c_int64(ld), FAKE,
                 prefix, B, g, u, FAKE, FAKE, FAKE, FAKE, new_seq, FAKE, ws, ctypes.c_size_t(wsb),
                 FAKE, None)

    assert call(dtype=3) == -1
    assert call(ld=999) == -1
    assert call(u=None) == -1
    assert call(g=32) == -1
    assert call(new_seq=FAKE, prefix=None) == -1
    assert call(B=5000) == -4
    assert call(ws=None) == -2
    assert call(wsb=need - 256) == -2
    fx = lib.dspark_sampling_accept_ex
    fx.restype = ctypes.c_int

    def call_ex(dtype=0, lse=FAKE):
        return fx(FAKE, dtype, ctypes.c_int64(1024), 1000, 100, FAKE, FAKE, ctypes.c_int64(1024),
                  lse, FAKE, FAKE, 4, 4, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None,
                  ctypes.c_size_t(need), FAKE, None)

    assert call_ex(dtype=3) == -1
    assert call_ex(lse=None, dtype=3) == -1
    assert call_ex() == -2  # null workspace


def test_calibration_argument_checks(lib):
    conf = lib.dspark_sts_confidence
    conf.restype = ctypes.c_int
    assert conf(FAKE, None, ctypes.c_int64(4), 4, FAKE, FAKE, None) == -1
    assert conf(FAKE, FAKE, ctypes.c_int64(-1), 4, FAKE, FAKE, None) == -1
    assert conf(FAKE, FAKE, ctypes.c_int64(4), 0, FAKE, FAKE, None) == -1
    assert conf(None, FAKE, ctypes.c_int64(4), 4, FAKE, FAKE, None) == -1
    assert conf(None, FAKE, ctypes.c_int64(0), 4, None, FAKE, None) == 0  # nothing to do

    rec = lib.dspark_sts_record
    rec.restype = ctypes.c_int

    def record(z=FAKE, corr=FAKE, B=4, g=4, cap=10, cursor=FAKE):
        return rec(z, corr, None, None, B, g, FAKE, FAKE, FAKE, ctypes.c_int64(cap), cursor, None,
                   FAKE, None)

    assert record(z=None) == -1
    assert record(corr=None) == -1
    assert record(cursor=None) == -1
    assert record(B=0) == -1
    assert record(g=32) == -1
    assert record(cap=0) == -1

    lib.dspark_calibration_workspace_bytes.restype = ctypes.c_size_t
    need = lib.dspark_calibration_workspace_bytes(8, 10)
    assert need % 256 == 0 and need >= 2 * 8 * 10 * 3 * 8
    assert lib.dspark_calibration_workspace_bytes(8, 33) == 0
    assert lib.dspark_calibration_workspace_bytes(0, 10) == 0
    stats = lib.dspark_calibration_stats
    stats.restype = ctypes.c_int

    def call_stats(N=100, g=8, M=10, T=FAKE, ws=FAKE, wsb=need, met=FAKE):
        return stats(FAKE, FAKE, FAKE, ctypes.c_int64(N), g, T, M, None, met, ws,
                     ctypes.c_size_t(wsb), FAKE, None)

    assert call_stats(N=-1) == -1
    assert call_stats(T=None) == -1
    assert call_stats(met=None) == -1
    assert call_stats(M=0) == -1
    assert call_stats(M=33) == -1
    assert call_stats(ws=None) == -2
    assert call_stats(wsb=need - 1) == -2
    assert call_stats(ws=ctypes.c_void_p(0x10010)) == -2

    lib.dspark_sts_fit_workspace_bytes.restype = ctypes.c_size_t
    need = lib.dspark_sts_fit_workspace_bytes(ctypes.c_int64(1000), 2, 10)
    assert need % 256 == 0 and need >= 1000 * 4 + 2 * 10 * 24
    assert lib.dspark_sts_fit_workspace_bytes(ctypes.c_int64(10), 257, 10) == 0
    fit = lib.dspark_sts_fit
    fit.restype = ctypes.c_int

    def call_fit(grid=(1.0, 2.0), N=1000, g=8, M=10, ws=FAKE, wsb=need, out=FAKE):
        arr = (ctypes.c_float * max(1, len(grid)))(*grid)
        return fit(FAKE, FAKE, FAKE, ctypes.c_int64(N), g, arr, len(grid), M, out, FAKE, None,
                   None, ws, ctypes.c_size_t(wsb), FAKE, None)

    assert call_fit(grid=()) == -1
    assert call_fit(grid=[1.0] * 257) == -1
    assert call_fit(grid=(1.0, 0.0)) == -1
    assert call_fit(grid=(1.0, -2.0)) == -1
    assert call_fit(grid=(1.0, float("inf"))) == -1
    assert call_fit(grid=(float("nan"),)) == -1
    assert call_fit(out=None) == -1
    assert call_fit(g=0) == -1
    assert call_fit(M=40) == -1
    assert call_fit(ws=None) == -2
    assert call_fit(wsb=need - 256) == -2


def test_checked_variant_builds_and_reports_itself():
    """The bounds-checked library exports the same calls and says which it
    is; the normal one says it is not checked."""
    from confidence_scheduled_speculative_gb300 import build
    try:
        normal, checked = build.build(), build.build(checked=True)
    except RuntimeError as e:  # pragma: no cover - toolkit missing
        pytest.skip(str(e))
    assert checked != normal
    libs = ctypes.CDLL(normal), ctypes.CDLL(checked)
    for n in declared_symbols():
        assert all(hasattr(lib, n) for lib in libs), n
    assert [lib.dspark_checked_build() for lib in libs] == [0, 1]
