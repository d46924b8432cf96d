"""ctypes binding of the plain-C CPU oracle (``dspark_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU-baseline leg, never by the product library.  The oracle shares
no code with the CUDA path; the only module both sides read is the seeded
input generator.

``build()`` compiles the C source with gcc (``-O2 -ffp-contract=off``, no
fused multiply-add, single thread).  All wrappers take and return numpy
arrays.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libdspark_oracle.so")

# status bits (same values as the library's device status word)
ST_CAPACITY = 1
ST_TOKEN_RANGE = 2
ST_NAN_LOGIT = 4
ST_BAD_INPUT = 8
ST_BAD_LEN = 16
ST_BAD_COST = 32
ST_INFEASIBLE = 64
ST_BAD_INDEX = 128
ST_BAD_TIER = 512

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libdspark_oracle.so``."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _P(t):
    return ctypes.POINTER(t)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            f32p, f64p, i32p, u8p, u16p = (_P(ctypes.c_float), _P(ctypes.c_double),
                                           _P(ctypes.c_int32), _P(ctypes.c_uint8),
                                           _P(ctypes.c_uint16))
            ci, cf, cd, cl = ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_int64
            L.orc_sts.argtypes = [cf, cf]
            L.orc_sts.restype = cf
            L.orc_sts_rows.argtypes = [f32p, f32p, ctypes.c_int64, ci, f32p, i32p]
            L.orc_sts_rows.restype = None
            L.orc_survival.argtypes = [f32p, f32p, ci, ci, cf, f32p, f32p, i32p]
            L.orc_survival.restype = None
            L.orc_plan_from_survivals.argtypes = [f32p, ci, ci, cf, ci, ci, ci, ci, ci, i32p, f64p,
                                                  cd, cd, i32p, i32p, f64p, f64p, f64p, u8p, i32p]
            L.orc_plan_from_survivals.restype = ci
            L.orc_plan.argtypes = [f32p, f32p, ci, ci, cf, ci, ci, ci, ci, ci, i32p, f64p, cd, cd,
                                   f32p, i32p, i32p, f64p, i32p]
            L.orc_plan.restype = ci
            L.orc_pack.argtypes = [i32p, i32p, i32p, i32p, ci, ci, i32p, ci, ci, i32p, i32p, i32p,
                                   i32p, i32p, i32p, i32p]
            L.orc_pack.restype = None
            L.orc_pad_to_tier.argtypes = [ci, ci, i32p, i32p, i32p, i32p, i32p, i32p]
            L.orc_pad_to_tier.restype = None
            L.orc_sampling_accept.argtypes = [f32p, cl, ci, ci, i32p, f32p, cl, i32p, i32p, ci, ci,
                                              f32p, f32p, i32p, i32p, i32p, i32p, i32p, i32p]
            L.orc_sampling_accept.restype = None
            u8p = ctypes.POINTER(ctypes.c_uint8)
            L.orc_scatter_rows.argtypes = [u8p, cl, cl, i32p, ci, ci, u8p, cl, ci, i32p]
            L.orc_scatter_rows.restype = None
            L.orc_argmax_rows_f32.argtypes = [f32p, cl, ci, ci, i32p, i32p]
            L.orc_argmax_rows_f32.restype = None
            L.orc_argmax_rows_bf16.argtypes = [u16p, cl, ci, ci, i32p, i32p]
            L.orc_argmax_rows_bf16.restype = None
            L.orc_greedy_finalize.argtypes = [i32p, ci, i32p, i32p, i32p, ci, ci, ci, i32p, i32p,
                                              i32p, i32p, i32p, i32p]
            L.orc_greedy_finalize.restype = None
            L.orc_cap_finalize.argtypes = [i32p, i32p, i32p, i32p, ci, ci, ci, i32p, i32p, i32p,
                                           i32p, i32p, i32p, i32p, i32p]
            L.orc_cap_finalize.restype = None
            u64p, i64p = _P(ctypes.c_uint64), _P(ctypes.c_int64)
            L.orc_sts_record.argtypes = [f32p, i32p, i32p, u8p, ci, ci, f32p, i32p, i32p, cl,
                                         u64p, u8p, i32p]
            L.orc_sts_record.restype = None
            L.orc_reliability.argtypes = [f32p, u8p, cl, ci, u64p, f64p]
            L.orc_reliability.restype = ctypes.c_uint64
            L.orc_calib_stats.argtypes = [f32p, i32p, i32p, cl, ci, f32p, ci, u64p, f64p, i32p]
            L.orc_calib_stats.restype = None
            L.orc_sts_fit.argtypes = [f32p, i32p, i32p, cl, ci, f32p, ci, ci, f32p, i32p, f64p,
                                      i64p, i32p]
            L.orc_sts_fit.restype = None
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return ctypes.cast(None, ctypes.POINTER(ctype))
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ planner

def sts(z: float, T: float) -> float:
    return float(lib().orc_sts(ctypes.c_float(z), ctypes.c_float(T)))


def sts_rows(z, T):
    """(c [n, gamma] fp32, status): c = sigmoid(z / T_k) elementwise."""
    z = _c(z, np.float32)
    T = _c(T, np.float32)
    n, g = z.shape
    c = np.empty((n, g), np.float32)
    st = np.zeros(1, np.int32)
    lib().orc_sts_rows(_ptr(z, ctypes.c_float), _ptr(T, ctypes.c_float), n, g,
                       _ptr(c, ctypes.c_float), _ptr(st, ctypes.c_int32))
    return c, int(st[0])


def survival(z, T, eps):
    """Returns (s_raw, s_out, status) for confidence logits z [B, gamma]."""
    z = _c(z, np.float32)
    T = _c(T, np.float32)
    B, g = z.shape
    s_raw = np.empty((B, g), np.float32)
    s_out = np.empty((B, g), np.float32)
    st = np.zeros(1, np.int32)
    lib().orc_survival(_ptr(z, ctypes.c_float), _ptr(T, ctypes.c_float), B, g, float(eps),
                       _ptr(s_raw, ctypes.c_float), _ptr(s_out, ctypes.c_float),
                       _ptr(st, ctypes.c_int32))
    return s_raw, s_out, int(st[0])


class PlanResult(dict):
    __getattr__ = dict.__getitem__


def plan_from_survivals(s_raw, eps, min_len, max_len, forced, kind, M, val, bias=0.0, alpha=0.0):
    s_raw = _c(s_raw, np.float32)
    B, g = s_raw.shape
    M = _c(M, np.int32)
    val = _c(val, np.float64)
    lens = np.empty(B, np.int32)
    budget = np.zeros(1, np.int32)
    tt = np.zeros(2, np.float64)
    tau = np.zeros(B * g + 1, np.float64)
    theta = np.zeros(B * g + 1, np.float64)
    feas = np.zeros(B * g + 1, np.uint8)
    st = np.zeros(1, np.int32)
    n_kept = lib().orc_plan_from_survivals(
        _ptr(s_raw, ctypes.c_float), B, g, float(eps), int(min_len), int(max_len), int(forced),
        int(kind), int(M.size), _ptr(M, ctypes.c_int32), _ptr(val, ctypes.c_double), float(bias),
        float(alpha), _ptr(lens, ctypes.c_int32), _ptr(budget, ctypes.c_int32),
        _ptr(tt, ctypes.c_double), _ptr(tau, ctypes.c_double), _ptr(theta, ctypes.c_double),
        _ptr(feas, ctypes.c_uint8), _ptr(st, ctypes.c_int32))
    return PlanResult(verify_lens=lens, budget=int(budget[0]), tau=float(tt[0]),
                      theta=float(tt[1]), tau_curve=tau[:n_kept + 1],
                      theta_curve=theta[:n_kept + 1], feasible=feas[:n_kept + 1].astype(bool),
                      n_kept=int(n_kept), status=int(st[0]))


def plan(z, T, eps, min_len, max_len, forced, kind, M, val, bias=0.0, alpha=0.0):
    z = _c(z, np.float32)
    T = _c(T, np.float32)
    B, g = z.shape
    M = _c(M, np.int32)
    val = _c(val, np.float64)
    s = np.empty((B, g), np.float32)
    lens = np.empty(B, np.int32)
    budget = np.zeros(1, np.int32)
    tt = np.zeros(2, np.float64)
    st = np.zeros(1, np.int32)
    n_kept = lib().orc_plan(
        _ptr(z, ctypes.c_float), _ptr(T, ctypes.c_float), B, g, float(eps), int(min_len),
        int(max_len), int(forced), int(kind), int(M.size), _ptr(M, ctypes.c_int32),
        _ptr(val, ctypes.c_double), float(bias), float(alpha), _ptr(s, ctypes.c_float),
        _ptr(lens, ctypes.c_int32), _ptr(budget, ctypes.c_int32), _ptr(tt, ctypes.c_double),
        _ptr(st, ctypes.c_int32))
    return PlanResult(survivals=s, verify_lens=lens, budget=int(budget[0]), tau=float(tt[0]),
                      theta=float(tt[1]), n_kept=int(n_kept), status=int(st[0]))


def plan_ex(z, T, eps, min_len, max_len, forced, kind, M, val, bias=0.0, alpha=0.0,
            conf_gen=None, req_gen=None, lagged_z=None, align_tiers=None, survivals=None):
    """The planner with the options of [AVS] §三, composed from the plain
    planner's definitions:
      * generation mask: a request whose confidences belong to another
        generation of its slot has survival 1 at every depth;
      * lagged_z: the budget is the plain plan's budget on the lagged
        confidences; the allocation (lens, tau, theta) is the plan on the
        current confidences with that budget forced;
      * align_tiers: with T rows at the chosen budget b and the smallest tier
        t >= T, the executed budget is b + (t - T) (then clipped to the
        in-range candidates like any forced budget); no tier >= T: b.
    ``survivals`` (optional, [B, gamma] fp32) replaces the current
    confidences' survivals computed from z: the later steps then run on
    those values (staged parity: another implementation's survivals)."""
    z = _c(z, np.float32)
    B, g = z.shape
    live = np.ones(B, bool) if conf_gen is None else (np.asarray(conf_gen) == np.asarray(req_gen))

    def surv(zz):
        s_raw = np.ones((B, g), np.float32)
        st = 0
        if live.any():
            r, _, st = survival(_c(zz, np.float32)[live], T, eps)
            s_raw[live] = r
        s_out = np.where(s_raw >= np.float32(eps), s_raw, np.float32(0)).astype(np.float32)
        return s_raw, s_out, st

    status = 0
    if lagged_z is not None:
        lag_raw, _, st = surv(lagged_z)
        status |= st
        first = plan_from_survivals(lag_raw, eps, min_len, max_len, forced, kind, M, val, bias, alpha)
        status |= first.status
        forced = first.budget
    s_raw, s_out, st = surv(z)
    status |= st
    if survivals is not None:
        s_raw = _c(survivals, np.float32)
        s_out = np.where(s_raw >= np.float32(eps), s_raw, np.float32(0)).astype(np.float32)
    res = plan_from_survivals(s_raw, eps, min_len, max_len, forced, kind, M, val, bias, alpha)
    if align_tiers is not None and len(align_tiers) > 0:
        status |= res.status
        total = int(res.verify_lens.sum())
        tiers = [int(t) for t in align_tiers]
        tier = next((t for t in tiers if t >= total), None)
        b_exec = res.budget if tier is None else res.budget + (tier - total)
        res = plan_from_survivals(s_raw, eps, min_len, max_len, b_exec, kind, M, val, bias, alpha)
    res["status"] = res.status | status
    res["survivals"] = s_out
    return res


def plan_step(step):
    """Run the planner on a ``workloads.StepInputs``."""
    w, c = step.workload, step.cost
    return plan(step.conf_logits, step.sts_temps, w.survival_eps, w.min_verify_len, w.max_len,
                w.forced_budget, c.kind, c.M, c.val, c.bias_ms, c.alpha_ms)


# --------------------------------------------------------------------- pack

def pack(anchor, draft, prefix, lens, tiers, capacity, sentinel=-7):
    anchor, prefix, lens = _c(anchor, np.int32), _c(prefix, np.int32), _c(lens, np.int32)
    draft = _c(draft, np.int32)
    tiers = _c(tiers, np.int32)
    B, g = draft.shape
    outs = [np.full(capacity, sentinel, np.int32) for _ in range(4)]
    cu = np.empty(B + 1, np.int32)
    totals = np.zeros(2, np.int32)
    st = np.zeros(1, np.int32)
    lib().orc_pack(_ptr(anchor, ctypes.c_int32), _ptr(draft, ctypes.c_int32),
                   _ptr(prefix, ctypes.c_int32), _ptr(lens, ctypes.c_int32), B, g,
                   _ptr(tiers if tiers.size else np.zeros(1, np.int32), ctypes.c_int32),
                   int(tiers.size), int(capacity), *[_ptr(o, ctypes.c_int32) for o in outs],
                   _ptr(cu, ctypes.c_int32), _ptr(totals, ctypes.c_int32),
                   _ptr(st, ctypes.c_int32))
    return PlanResult(ids=outs[0], pos=outs[1], req=outs[2], src=outs[3], cu_seqlens=cu,
                      total=int(totals[0]), padded=int(totals[1]), status=int(st[0]))


def pad_to_tier(packed, pad_to, capacity):
    """The data-parallel shared tier applied to one rank's pack result (a
    ``pack`` PlanResult): a copy with rows [total, pad_to) turned into pad
    rows and padded = pad_to (reading R30)."""
    outs = [np.array(packed[k], np.int32, copy=True) for k in ("ids", "pos", "req", "src")]
    totals = np.array([packed.total, packed.padded], np.int32)
    st = np.zeros(1, np.int32)
    lib().orc_pad_to_tier(int(pad_to), int(capacity), *[_ptr(o, ctypes.c_int32) for o in outs],
                          _ptr(totals, ctypes.c_int32), _ptr(st, ctypes.c_int32))
    return PlanResult(ids=outs[0], pos=outs[1], req=outs[2], src=outs[3],
                      cu_seqlens=packed.cu_seqlens, total=int(totals[0]), padded=int(totals[1]),
                      status=int(st[0]))


def scatter_rows(src, src_of, total, dst, max_rows=None):
    """ScatterCompactToStrided: returns (a copy of dst with packed row i <
    total written at row src_of[i], status).  src and dst are 2-D arrays of
    the same dtype; their row widths may differ, the copied width is src's."""
    src = np.ascontiguousarray(src)
    out = np.array(dst, copy=True, order="C")
    src_of = _c(src_of, np.int32)
    max_rows = src.shape[0] if max_rows is None else max_rows
    st = np.zeros(1, np.int32)
    u8 = ctypes.POINTER(ctypes.c_uint8)
    lib().orc_scatter_rows(src.ctypes.data_as(u8), src.strides[0], src.shape[1] * src.itemsize,
                           _ptr(src_of, ctypes.c_int32), int(total), int(max_rows),
                           out.ctypes.data_as(u8), out.strides[0], out.shape[0],
                           _ptr(st, ctypes.c_int32))
    return out, int(st[0])


# ------------------------------------------------------------------- accept

def argmax_rows(logits, V=None, rows=None, dtype=None):
    """Row argmax; ``logits`` is float32 [rows, ld] or uint16 bf16 bits."""
    logits = np.ascontiguousarray(logits)
    n, ld = logits.shape
    V = ld if V is None else V
    rows = n if rows is None else rows
    am = np.zeros(max(rows, 1), np.int32)
    st = np.zeros(1, np.int32)
    if logits.dtype == np.float32:
        lib().orc_argmax_rows_f32(_ptr(logits, ctypes.c_float), ld, V, rows,
                                  _ptr(am, ctypes.c_int32), _ptr(st, ctypes.c_int32))
    elif logits.dtype == np.uint16:
        lib().orc_argmax_rows_bf16(_ptr(logits, ctypes.c_uint16), ld, V, rows,
                                   _ptr(am, ctypes.c_int32), _ptr(st, ctypes.c_int32))
    else:
        raise TypeError(logits.dtype)
    return am[:rows], int(st[0])


def greedy_finalize(am, rows, cu, draft, prefix, V):
    draft = _c(draft, np.int32)
    B, g = draft.shape
    am = _c(am if len(am) else np.zeros(1, np.int32), np.int32)
    cu = _c(cu, np.int32)
    prefix = _c(prefix, np.int32)
    o = [np.empty(B, np.int32) for _ in range(4)]
    out = np.empty((B, g + 1), np.int32)
    st = np.zeros(1, np.int32)
    lib().orc_greedy_finalize(_ptr(am, ctypes.c_int32), int(rows), _ptr(cu, ctypes.c_int32),
                              _ptr(draft, ctypes.c_int32), _ptr(prefix, ctypes.c_int32), B, g,
                              int(V), *[_ptr(x, ctypes.c_int32) for x in o],
                              _ptr(out, ctypes.c_int32), _ptr(st, ctypes.c_int32))
    return PlanResult(num_accepted=o[0], bonus=o[1], commit_lens=o[2], new_seq_lens=o[3],
                      out_tokens=out, status=int(st[0]))


def greedy_accept(logits, V, cu, draft, prefix, max_rows=None):
    """Compact-mode accept: argmax of rows [0, min(cu[B], max_rows)), then
    the per-request first mismatch, finalize and out tokens."""
    cu = _c(cu, np.int32)
    B = cu.size - 1
    max_rows = logits.shape[0] if max_rows is None else max_rows
    want = int(cu[B])
    status = 0
    rows = max(0, min(want, max_rows))
    if want > max_rows:
        status |= ST_CAPACITY
    am, st = argmax_rows(logits, V=V, rows=rows)
    fin = greedy_finalize(am, rows, cu, draft, prefix, V)
    fin["argmax"] = am
    fin["status"] = fin.status | st | status
    return fin


def cap_accept(logits, V, lens, draft, prefix):
    draft = _c(draft, np.int32)
    B, g = draft.shape
    am, st = argmax_rows(logits, V=V, rows=B * (g + 1))
    lens = _c(lens, np.int32)
    prefix = _c(prefix, np.int32)
    o = [np.empty(B, np.int32) for _ in range(5)]
    out = np.empty((B, g + 1), np.int32)
    totals = np.zeros(2, np.int32)
    st2 = np.zeros(1, np.int32)
    lib().orc_cap_finalize(_ptr(am, ctypes.c_int32), _ptr(lens, ctypes.c_int32),
                           _ptr(draft, ctypes.c_int32), _ptr(prefix, ctypes.c_int32), B, g,
                           int(V), *[_ptr(x, ctypes.c_int32) for x in o[:4]],
                           _ptr(out, ctypes.c_int32), _ptr(o[4], ctypes.c_int32),
                           _ptr(totals, ctypes.c_int32), _ptr(st2, ctypes.c_int32))
    return PlanResult(argmax=am, num_accepted=o[0], bonus=o[1], commit_lens=o[2],
                      new_seq_lens=o[3], out_tokens=out, ceiling=o[4],
                      sum_commit=int(totals[0]), sum_ceiling=int(totals[1]),
                      status=st | int(st2[0]))


def _as_f32_rows(x):
    """fp32 rows from fp32 or bf16-bit (uint16) logits."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32)
    return x.astype(np.float32, copy=False)


def sampling_accept(target, V, cu, draft_logits, draft, prefix, u_accept, u_bonus, max_rows=None):
    """Speculative sampling accept over compact target rows (cu_seqlens) and
    the draft's proposal rows [B*gamma, ld] (row r*gamma + j = q_j of request
    r), with the given uniforms u_accept [B, gamma] and u_bonus [B]."""
    tgt = _as_f32_rows(target)
    dft = _as_f32_rows(draft_logits)
    cu = _c(cu, np.int32)
    draft = _c(draft, np.int32)
    B, g = draft.shape
    prefix = _c(prefix, np.int32)
    ua = _c(u_accept, np.float32)
    ub = _c(u_bonus, np.float32)
    max_rows = tgt.shape[0] if max_rows is None else max_rows
    want = int(cu[B])
    status = ST_CAPACITY if want > max_rows else 0
    rows = max(0, min(want, max_rows))
    o = [np.empty(B, np.int32) for _ in range(4)]
    out = np.empty((B, g + 1), np.int32)
    st = np.zeros(1, np.int32)
    lib().orc_sampling_accept(_ptr(tgt, ctypes.c_float), tgt.shape[1], int(V), rows,
                              _ptr(cu, ctypes.c_int32), _ptr(dft, ctypes.c_float), dft.shape[1],
                              _ptr(draft, ctypes.c_int32), _ptr(prefix, ctypes.c_int32), B, g,
                              _ptr(ua, ctypes.c_float), _ptr(ub, ctypes.c_float),
                              *[_ptr(x, ctypes.c_int32) for x in o], _ptr(out, ctypes.c_int32),
                              _ptr(st, ctypes.c_int32))
    return PlanResult(num_accepted=o[0], bonus=o[1], commit_lens=o[2], new_seq_lens=o[3],
                      out_tokens=out, status=int(st[0]) | status)


# -------------------------------------------------------------- calibration

def sts_record(z, correct, verify_lens, B_select, rec_z, rec_correct, rec_tested, cursor,
               want_mask=True):
    """Append the selected requests' (z, correct, tested) rows to the ring
    buffers rec_* (modified in place) starting at ``cursor``.  B_select is a
    uint8 [B] mask or None (every request); verify_lens None = full block.
    Returns (new_cursor, prefix_mask or None, status)."""
    z = _c(z, np.float32)
    B, g = z.shape
    correct = _c(correct, np.int32)
    vl = None if verify_lens is None else _c(verify_lens, np.int32)
    sel = None if B_select is None else _c(B_select, np.uint8)
    cap = rec_correct.shape[0]
    cur = np.array([cursor], np.uint64)
    mask = np.empty((B, g), np.uint8) if want_mask else None
    st = np.zeros(1, np.int32)
    lib().orc_sts_record(_ptr(z, ctypes.c_float), _ptr(correct, ctypes.c_int32),
                         _ptr(vl, ctypes.c_int32), _ptr(sel, ctypes.c_uint8), B, g,
                         _ptr(rec_z, ctypes.c_float), _ptr(rec_correct, ctypes.c_int32),
                         _ptr(rec_tested, ctypes.c_int32), cap, _ptr(cur, ctypes.c_uint64),
                         _ptr(mask, ctypes.c_uint8), _ptr(st, ctypes.c_int32))
    return int(cur[0]), mask, int(st[0])


def reliability(p, y, n_bins):
    """(hist [n_bins, 3] uint64, metrics [4] = n, ECE, Brier, log loss,
    E = ECE*n*2^32 as an exact integer) of (prediction, label) pairs."""
    p = _c(p, np.float32).reshape(-1)
    y = _c(y, np.uint8).reshape(-1)
    hist = np.zeros((n_bins, 3), np.uint64)
    met = np.zeros(4, np.float64)
    E = lib().orc_reliability(_ptr(p, ctypes.c_float), _ptr(y, ctypes.c_uint8), p.shape[0],
                              int(n_bins), _ptr(hist, ctypes.c_uint64),
                              _ptr(met, ctypes.c_double))
    return hist, met, int(E)


def calib_stats(z, correct, tested, T, n_bins):
    """Per-depth calibration of recorded samples: hist [2, gamma, n_bins, 3]
    and metrics [2, gamma, 4] (flavour 0 cumulative S_k, 1 per-position c_k)."""
    z = _c(z, np.float32)
    N, g = z.shape
    correct = _c(correct, np.int32)
    tested = _c(tested, np.int32)
    T = _c(T, np.float32)
    hist = np.zeros((2, g, n_bins, 3), np.uint64)
    met = np.zeros((2, g, 4), np.float64)
    st = np.zeros(1, np.int32)
    lib().orc_calib_stats(_ptr(z, ctypes.c_float), _ptr(correct, ctypes.c_int32),
                          _ptr(tested, ctypes.c_int32), N, g, _ptr(T, ctypes.c_float),
                          int(n_bins), _ptr(hist, ctypes.c_uint64), _ptr(met, ctypes.c_double),
                          _ptr(st, ctypes.c_int32))
    return PlanResult(hist=hist, metrics=met, status=int(st[0]))


def sts_fit(z, correct, tested, grid, n_bins):
    """Sequential per-depth temperature fit over a grid of temperatures."""
    z = _c(z, np.float32)
    N, g = z.shape
    correct = _c(correct, np.int32)
    tested = _c(tested, np.int32)
    grid = _c(grid, np.float32)
    J = grid.shape[0]
    T = np.zeros(g, np.float32)
    choice = np.zeros(g, np.int32)
    curve = np.zeros((g, J), np.float64)
    n_obs = np.zeros(g, np.int64)
    st = np.zeros(1, np.int32)
    lib().orc_sts_fit(_ptr(z, ctypes.c_float), _ptr(correct, ctypes.c_int32),
                      _ptr(tested, ctypes.c_int32), N, g, _ptr(grid, ctypes.c_float), J,
                      int(n_bins), _ptr(T, ctypes.c_float), _ptr(choice, ctypes.c_int32),
                      _ptr(curve, ctypes.c_double), _ptr(n_obs, ctypes.c_int64),
                      _ptr(st, ctypes.c_int32))
    return PlanResult(T=T, choice=choice, ece_curve=curve, n_obs=n_obs, status=int(st[0]))
