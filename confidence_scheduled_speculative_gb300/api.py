"""Thin Python binding of libdspark.so (include/dspark.h).

Argument marshalling only: every function here forwards device pointers,
sizes and the current CUDA stream to the C entry point of the same name, and
raises :class:`DsparkError` on a non-zero return code.  PyTorch provides the
device buffers and the stream; every step of the computation runs in the
library's CUDA kernels.  There is no fallback: if the library is missing the
import of a function raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

DSPARK_OK = 0
DSPARK_ERR_INVALID_ARG = -1
DSPARK_ERR_WORKSPACE = -2
DSPARK_ERR_CUDA = -3
DSPARK_ERR_UNSUPPORTED = -4

STATUS_CAPACITY = 1
STATUS_TOKEN_RANGE = 2
STATUS_NAN_LOGIT = 4
STATUS_BAD_INPUT = 8
STATUS_BAD_LEN = 16
STATUS_BAD_COST = 32
STATUS_INFEASIBLE = 64
STATUS_BAD_INDEX = 128
STATUS_TIMEOUT = 256
STATUS_BAD_TIER = 512
STATUS_OUT_OF_BOUNDS = 1024  # only the bounds-checked library sets it

# cost tables of at most SELECT_MAX_ENTRIES entries take the planner's
# single-CTA select path, larger ones up to DENSE_MAX_ENTRIES its single-CTA
# dense path, interpolated tables of at most INTERP_MAX_SAMPLES samples its
# single-CTA interp path (all three with the pack fused in); the rest the
# multi-CTA rank path
SELECT_MAX_ENTRIES = 31
DENSE_MAX_ENTRIES = 6143
INTERP_MAX_SAMPLES = 2048
COST_SPS_1D = 0
COST_ADDITIVE = 1
COST_ADDITIVE_INTERP = 2
DTYPE_BF16 = 0
DTYPE_F32 = 1
MAX_TIERS = 64


def planner_path(n_candidates: int, cost_kind: int, n_entries: int) -> str:
    """Which planner kernel a call takes: "select", "dense", "interp" or "rank"."""
    if cost_kind == COST_ADDITIVE_INTERP:
        return "interp" if n_entries <= INTERP_MAX_SAMPLES else "rank"
    if n_entries <= SELECT_MAX_ENTRIES:
        return "select"
    return "dense" if n_entries <= DENSE_MAX_ENTRIES else "rank"


class DsparkError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {dspark_strerror(code)} ({code})")
        self.code = code


class dspark_plan_params(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("gamma", ctypes.c_int32),
                ("survival_eps", ctypes.c_float), ("min_verify_len", ctypes.c_int32),
                ("max_verify_len", ctypes.c_int32), ("forced_budget", ctypes.c_int32)]


class dspark_cost_table(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("n", ctypes.c_int32), ("M", ctypes.c_void_p),
                ("val", ctypes.c_void_p), ("bias_ms", ctypes.c_double),
                ("alpha_ms", ctypes.c_double)]


class dspark_plan_options(ctypes.Structure):
    _fields_ = [("conf_generation", ctypes.c_void_p), ("req_generation", ctypes.c_void_p),
                ("lagged_conf_logits", ctypes.c_void_p), ("align_to_tiers", ctypes.c_int32),
                ("host_tiers", ctypes.POINTER(ctypes.c_int32)), ("n_tiers", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None

_VP, _I32, _I64, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t

_SIGS = {
    "dspark_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "dspark_version": (ctypes.c_int, []),
    "dspark_checked_build": (ctypes.c_int, []),
    "dspark_plan_workspace_bytes": (_SZ, [_I32, _I32]),
    "dspark_plan": (ctypes.c_int, [_VP, _VP, ctypes.POINTER(dspark_plan_params),
                                   ctypes.POINTER(dspark_cost_table), _VP, _VP, _VP, _VP, _VP,
                                   _SZ, _VP, _VP]),
    "dspark_pack_verify": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I32, _I32,
                                          ctypes.POINTER(ctypes.c_int32), _I32, _I32, _VP, _VP,
                                          _VP, _VP, _VP, _VP, _VP, _VP]),
    "dspark_plan_ex": (ctypes.c_int, [_VP, _VP, ctypes.POINTER(dspark_plan_params),
                                      ctypes.POINTER(dspark_cost_table),
                                      ctypes.POINTER(dspark_plan_options), _VP, _VP, _VP, _VP, _VP,
                                      _SZ, _VP, _VP]),
    "dspark_plan_pack_ex": (ctypes.c_int, [_VP, _VP, ctypes.POINTER(dspark_plan_params),
                                           ctypes.POINTER(dspark_cost_table),
                                           ctypes.POINTER(dspark_plan_options), _VP, _VP, _VP, _VP,
                                           _VP, _VP, _VP, ctypes.POINTER(ctypes.c_int32), _I32,
                                           _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
    "dspark_plan_pack": (ctypes.c_int, [_VP, _VP, ctypes.POINTER(dspark_plan_params),
                                        ctypes.POINTER(dspark_cost_table), _VP, _VP, _VP, _VP,
                                        _VP, _VP, _VP, ctypes.POINTER(ctypes.c_int32), _I32, _I32,
                                        _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
    "dspark_scatter_compact_to_strided": (ctypes.c_int, [_VP, _I64, _I32, _I32, _VP, _VP, _I32,
                                                         _VP, _I64, _I32, _VP, _VP]),
    "dspark_pad_to_tier": (ctypes.c_int, [_VP, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "dspark_scatter_compact_to_strided_ex": (ctypes.c_int, [_VP, _I64, _I32, _I32, _VP, _VP,
                                                            _I32, _VP, _I64, _I32, _I64, _VP,
                                                            _VP]),
    "dspark_sampling_workspace_bytes": (_SZ, [_I32, _I32, _I32]),
    "dspark_sampling_accept": (ctypes.c_int, [_VP, _I32, _I64, _I32, _I32, _VP, _VP, _I64, _VP,
                                              _VP, _I32, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                              _VP, _SZ, _VP, _VP]),
    "dspark_sampling_accept_ex": (ctypes.c_int, [_VP, _I32, _I64, _I32, _I32, _VP, _VP, _I64,
                                                 _VP, _VP, _VP, _I32, _I32, _VP, _VP, _VP, _VP,
                                                 _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
    "dspark_accept_workspace_bytes": (_SZ, [_I32, _I32]),
    "dspark_greedy_accept": (ctypes.c_int, [_VP, _I32, _I64, _I32, _I32, _VP, _VP, _VP, _I32,
                                            _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP,
                                            _VP]),
    "dspark_cap_accept": (ctypes.c_int, [_VP, _I32, _I64, _I32, _VP, _VP, _VP, _I32, _I32, _VP,
                                         _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
    "dspark_greedy_accept_static": (ctypes.c_int, [_VP, _I32, _I64, _I32, _I32, _VP, _VP, _VP,
                                                   _I32, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                                   _VP]),
    "dspark_sts_confidence": (ctypes.c_int, [_VP, _VP, _I64, _I32, _VP, _VP, _VP]),
    "dspark_sts_record": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I32, _I32, _VP, _VP, _VP, _I64,
                                         _VP, _VP, _VP, _VP]),
    "dspark_calibration_workspace_bytes": (_SZ, [_I32, _I32]),
    "dspark_calibration_stats": (ctypes.c_int, [_VP, _VP, _VP, _I64, _I32, _VP, _I32, _VP, _VP,
                                                _VP, _SZ, _VP, _VP]),
    "dspark_sts_fit_workspace_bytes": (_SZ, [_I64, _I32, _I32]),
    "dspark_sts_fit": (ctypes.c_int, [_VP, _VP, _VP, _I64, _I32, ctypes.POINTER(ctypes.c_float),
                                      _I32, _I32, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]),
}


def library_path() -> str:
    """The normal library, or the bounds-checked one when DSPARK_CHECKED=1."""
    if os.environ.get("DSPARK_CHECKED", "0") == "1":
        return _build.CHECKED_LIB_PATH
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load libdspark.so; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{os.path.basename(path)} not found at {path}: build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _p(t: torch.Tensor | None, dtype: torch.dtype | None = None, name: str = "") -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn: str, rc: int) -> None:
    if rc != DSPARK_OK:
        raise DsparkError(fn, rc)


# ------------------------------------------------------------------- calls

def dspark_strerror(code: int) -> str:
    return load().dspark_strerror(int(code)).decode()


def dspark_version() -> int:
    return int(load().dspark_version())


def dspark_checked_build() -> bool:
    return bool(load().dspark_checked_build())


def dspark_plan_workspace_bytes(B: int, gamma: int) -> int:
    return int(load().dspark_plan_workspace_bytes(B, gamma))


def dspark_accept_workspace_bytes(max_rows: int, V: int) -> int:
    return int(load().dspark_accept_workspace_bytes(max_rows, V))


def dspark_plan(conf_logits, sts_temps, *, B, gamma, survival_eps, min_verify_len,
                max_verify_len, forced_budget, cost_kind, cost_M, cost_val, bias_ms=0.0,
                alpha_ms=0.0, survivals, verify_lens, budget, tau_theta, status,
                workspace, stream=None) -> None:
    """Planner: STS survivals -> budget -> verify_lens (all outputs on device).
    ``workspace``: a device byte buffer of dspark_plan_workspace_bytes(B, gamma)."""
    params = dspark_plan_params(B, gamma, survival_eps, min_verify_len, max_verify_len,
                                forced_budget)
    cost = dspark_cost_table(cost_kind, int(cost_M.numel()), _p(cost_M, torch.int32, "cost_M"),
                             _p(cost_val, torch.float64, "cost_val"), bias_ms, alpha_ms)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().dspark_plan(
        _p(conf_logits, torch.float32, "conf_logits"), _p(sts_temps, torch.float32, "sts_temps"),
        ctypes.byref(params), ctypes.byref(cost), _p(survivals, torch.float32, "survivals"),
        _p(verify_lens, torch.int32, "verify_lens"), _p(budget, torch.int32, "budget"),
        _p(tau_theta, torch.float64, "tau_theta"), _p(workspace), ws_bytes,
        _p(status, torch.int32, "status"), _stream(stream))
    _check("dspark_plan", rc)


def dspark_pack_verify(anchor, draft, prefix_lens, verify_lens, *, B, gamma, tiers, capacity,
                       packed_ids, packed_pos, packed_req, packed_src, cu_seqlens, totals,
                       status, stream=None) -> None:
    """Front-pack the verify rows; ``tiers`` is a host sequence of ints."""
    tiers = [int(t) for t in tiers]
    arr = (ctypes.c_int32 * max(1, len(tiers)))(*tiers)
    rc = load().dspark_pack_verify(
        _p(anchor, torch.int32, "anchor"), _p(draft, torch.int32, "draft"),
        _p(prefix_lens, torch.int32, "prefix_lens"), _p(verify_lens, torch.int32, "verify_lens"),
        B, gamma, arr, len(tiers), capacity, _p(packed_ids, torch.int32, "packed_ids"),
        _p(packed_pos, torch.int32, "packed_pos"), _p(packed_req, torch.int32, "packed_req"),
        _p(packed_src, torch.int32, "packed_src"), _p(cu_seqlens, torch.int32, "cu_seqlens"),
        _p(totals, torch.int32, "totals"), _p(status, torch.int32, "status"), _stream(stream))
    _check("dspark_pack_verify", rc)


def plan_options(conf_generation=None, req_generation=None, lagged_conf_logits=None,
                 align_tiers=None):
    """A dspark_plan_options (kept alive by the returned tuple's second item)
    from device tensors and a host tier list; None when no option is set."""
    if conf_generation is None and req_generation is None and lagged_conf_logits is None \
            and not align_tiers:
        return None, None
    tiers = [int(t) for t in (align_tiers or [])]
    arr = (ctypes.c_int32 * max(1, len(tiers)))(*tiers)
    opt = dspark_plan_options(_p(conf_generation, torch.int32, "conf_generation"),
                              _p(req_generation, torch.int32, "req_generation"),
                              _p(lagged_conf_logits, torch.float32, "lagged_conf_logits"),
                              1 if tiers else 0, arr, len(tiers))
    return opt, arr


def dspark_plan_ex(conf_logits, sts_temps, *, B, gamma, survival_eps, min_verify_len,
                   max_verify_len, forced_budget, cost_kind, cost_M, cost_val, bias_ms=0.0,
                   alpha_ms=0.0, survivals, verify_lens, budget, tau_theta, status, workspace,
                   conf_generation=None, req_generation=None, lagged_conf_logits=None,
                   align_tiers=None, stream=None) -> None:
    """dspark_plan with the planner options (generation mask, lagged-
    confidence budget, graph-tier alignment to ``align_tiers``)."""
    params = dspark_plan_params(B, gamma, survival_eps, min_verify_len, max_verify_len,
                                forced_budget)
    cost = dspark_cost_table(cost_kind, int(cost_M.numel()), _p(cost_M, torch.int32, "cost_M"),
                             _p(cost_val, torch.float64, "cost_val"), bias_ms, alpha_ms)
    opt, _keep = plan_options(conf_generation, req_generation, lagged_conf_logits, align_tiers)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().dspark_plan_ex(
        _p(conf_logits, torch.float32, "conf_logits"), _p(sts_temps, torch.float32, "sts_temps"),
        ctypes.byref(params), ctypes.byref(cost), None if opt is None else ctypes.byref(opt),
        _p(survivals, torch.float32, "survivals"), _p(verify_lens, torch.int32, "verify_lens"),
        _p(budget, torch.int32, "budget"), _p(tau_theta, torch.float64, "tau_theta"),
        _p(workspace), ws_bytes, _p(status, torch.int32, "status"), _stream(stream))
    _check("dspark_plan_ex", rc)


def dspark_plan_pack(conf_logits, sts_temps, anchor, draft, prefix_lens, *, B, gamma,
                     survival_eps, min_verify_len, max_verify_len, forced_budget, cost_kind,
                     cost_M, cost_val, bias_ms=0.0, alpha_ms=0.0, tiers, capacity, survivals,
                     verify_lens, budget, tau_theta, packed_ids, packed_pos, packed_req,
                     packed_src, cu_seqlens, totals, status, workspace, conf_generation=None,
                     req_generation=None, lagged_conf_logits=None, align_to_tiers=False,
                     stream=None) -> None:
    """dspark_plan then dspark_pack_verify on its verify_lens, in fewer launches
    (the pack runs inside the planner's last kernel for tables of <= 31
    entries).  The planner options as in dspark_plan_ex; alignment uses the
    pack's ``tiers``."""
    params = dspark_plan_params(B, gamma, survival_eps, min_verify_len, max_verify_len,
                                forced_budget)
    cost = dspark_cost_table(cost_kind, int(cost_M.numel()), _p(cost_M, torch.int32, "cost_M"),
                             _p(cost_val, torch.float64, "cost_val"), bias_ms, alpha_ms)
    tiers = [int(t) for t in tiers]
    arr = (ctypes.c_int32 * max(1, len(tiers)))(*tiers)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    opt, _keep = plan_options(conf_generation, req_generation, lagged_conf_logits,
                              tiers if align_to_tiers else None)
    rc = load().dspark_plan_pack_ex(
        _p(conf_logits, torch.float32, "conf_logits"), _p(sts_temps, torch.float32, "sts_temps"),
        ctypes.byref(params), ctypes.byref(cost), None if opt is None else ctypes.byref(opt),
        _p(survivals, torch.float32, "survivals"),
        _p(verify_lens, torch.int32, "verify_lens"), _p(budget, torch.int32, "budget"),
        _p(tau_theta, torch.float64, "tau_theta"), _p(anchor, torch.int32, "anchor"),
        _p(draft, torch.int32, "draft"), _p(prefix_lens, torch.int32, "prefix_lens"), arr,
        len(tiers), capacity, _p(packed_ids, torch.int32, "packed_ids"),
        _p(packed_pos, torch.int32, "packed_pos"), _p(packed_req, torch.int32, "packed_req"),
        _p(packed_src, torch.int32, "packed_src"), _p(cu_seqlens, torch.int32, "cu_seqlens"),
        _p(totals, torch.int32, "totals"), _p(workspace), ws_bytes,
        _p(status, torch.int32, "status"), _stream(stream))
    _check("dspark_plan_pack", rc)


def dspark_scatter_compact_to_strided(src, packed_src, totals, dst, *, status,
                                      wait_limit_ns=None, stream=None) -> None:
    """Copy packed row i < totals[0] of ``src`` [max_rows, width] to row
    packed_src[i] of ``dst`` [B*(gamma+1), >= width] (2-D, same dtype:
    bfloat16, float16 or float32, unit inner stride).  ``wait_limit_ns``
    (dspark_scatter_compact_to_strided_ex) bounds one pipeline wait of the
    TMA path; None keeps the 200 ms default."""
    for name, t in (("src", src), ("dst", dst)):
        if not t.is_cuda or t.dim() != 2 or t.stride(1) != 1:
            raise ValueError(f"{name}: expected a 2-D CUDA tensor with unit inner stride")
    if src.dtype != dst.dtype or src.element_size() not in (2, 4):
        raise ValueError("src and dst: same dtype of 2 or 4 bytes")
    args = (src.data_ptr(), src.stride(0), src.size(1), src.element_size(),
            _p(packed_src, torch.int32, "packed_src"), _p(totals, torch.int32, "totals"),
            src.size(0), dst.data_ptr(), dst.stride(0), dst.size(0))
    if wait_limit_ns is None:
        name = "dspark_scatter_compact_to_strided"
        rc = load().dspark_scatter_compact_to_strided(*args, _p(status, torch.int32, "status"),
                                                      _stream(stream))
    else:
        name = "dspark_scatter_compact_to_strided_ex"
        rc = load().dspark_scatter_compact_to_strided_ex(*args, int(wait_limit_ns),
                                                         _p(status, torch.int32, "status"),
                                                         _stream(stream))
    _check(name, rc)


def dspark_pad_to_tier(pad_to, *, packed_ids, packed_pos, packed_req, packed_src, totals,
                       status, capacity=None, stream=None) -> None:
    """Pad one rank's packed window to the verify tier the data-parallel
    ranks share (``pad_to``: device int32 [1], may be ``totals[1:2]``)."""
    capacity = packed_ids.numel() if capacity is None else capacity
    rc = load().dspark_pad_to_tier(
        _p(pad_to, torch.int32, "pad_to"), int(capacity), _p(packed_ids, torch.int32, "packed_ids"),
        _p(packed_pos, torch.int32, "packed_pos"), _p(packed_req, torch.int32, "packed_req"),
        _p(packed_src, torch.int32, "packed_src"), _p(totals, torch.int32, "totals"),
        _p(status, torch.int32, "status"), _stream(stream))
    _check("dspark_pad_to_tier", rc)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise ValueError(f"logits: expected bfloat16 or float32, got {t.dtype}")


def _logits_ptr(logits: torch.Tensor, V: int) -> tuple[int, int]:
    """Device or pinned host logits: pinned host memory is device-accessible
    at the same address (unified addressing), and the kernels then read it
    over the host link."""
    if not (logits.is_cuda or logits.is_pinned()) or logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits: expected a 2-D CUDA or pinned tensor with unit column stride")
    if logits.size(1) < V:
        raise ValueError("logits: fewer columns than V")
    return logits.data_ptr(), logits.stride(0)


def dspark_greedy_accept(logits, *, V, cu_seqlens, draft, prefix_lens, B, gamma, num_accepted,
                         bonus, commit_lens, out_tokens, workspace, status, argmax=None,
                         new_seq_lens=None, max_rows=None, stream=None) -> None:
    """Compact-mode greedy accept over the packed rows of ``logits``."""
    ptr, ld = _logits_ptr(logits, V)
    max_rows = logits.size(0) if max_rows is None else max_rows
    rc = load().dspark_greedy_accept(
        ptr, _dtype_code(logits), ld, V, max_rows, _p(cu_seqlens, torch.int32, "cu_seqlens"),
        _p(draft, torch.int32, "draft"), _p(prefix_lens, torch.int32, "prefix_lens"), B, gamma,
        _p(argmax, torch.int32, "argmax"), _p(num_accepted, torch.int32, "num_accepted"),
        _p(bonus, torch.int32, "bonus"), _p(commit_lens, torch.int32, "commit_lens"),
        _p(new_seq_lens, torch.int32, "new_seq_lens"), _p(out_tokens, torch.int32, "out_tokens"),
        _p(workspace), workspace.numel() * workspace.element_size(),
        _p(status, torch.int32, "status"), _stream(stream))
    _check("dspark_greedy_accept", rc)


def dspark_sampling_workspace_bytes(max_rows: int, B: int, gamma: int) -> int:
    return int(load().dspark_sampling_workspace_bytes(max_rows, B, gamma))


def dspark_sampling_accept(logits, draft_logits, *, V, cu_seqlens, draft, prefix_lens, B, gamma,
                           u_accept, u_bonus, num_accepted, bonus, commit_lens, out_tokens,
                           workspace, status, new_seq_lens=None, max_rows=None,
                           draft_lse=None, stream=None) -> None:
    """Speculative sampling accept: packed target rows ``logits`` and the
    draft's proposal rows ``draft_logits`` [B*gamma, >= V] (same dtype);
    ``u_accept`` [B, gamma] and ``u_bonus`` [B] are fp32 uniforms.  With
    ``draft_lse`` ([B*gamma] fp32, each draft row's log-sum-exp) the call is
    dspark_sampling_accept_ex and the draft rows are not normalised here."""
    ptr, ld = _logits_ptr(logits, V)
    dptr, dld = _logits_ptr(draft_logits, V)
    if draft_logits.dtype != logits.dtype:
        raise ValueError("draft_logits: expected the dtype of logits")
    max_rows = logits.size(0) if max_rows is None else max_rows
    if draft_lse is not None:
        rc = load().dspark_sampling_accept_ex(
            ptr, _dtype_code(logits), ld, V, max_rows, _p(cu_seqlens, torch.int32, "cu_seqlens"),
            dptr, dld, _p(draft_lse, torch.float32, "draft_lse"), _p(draft, torch.int32, "draft"),
            _p(prefix_lens, torch.int32, "prefix_lens"), B, gamma,
            _p(u_accept, torch.float32, "u_accept"), _p(u_bonus, torch.float32, "u_bonus"),
            _p(num_accepted, torch.int32, "num_accepted"), _p(bonus, torch.int32, "bonus"),
            _p(commit_lens, torch.int32, "commit_lens"),
            _p(new_seq_lens, torch.int32, "new_seq_lens"), _p(out_tokens, torch.int32, "out_tokens"),
            _p(workspace), workspace.numel() * workspace.element_size(),
            _p(status, torch.int32, "status"), _stream(stream))
        _check("dspark_sampling_accept_ex", rc)
        return
    rc = load().dspark_sampling_accept(
        ptr, _dtype_code(logits), ld, V, max_rows, _p(cu_seqlens, torch.int32, "cu_seqlens"),
        dptr, dld, _p(draft, torch.int32, "draft"), _p(prefix_lens, torch.int32, "prefix_lens"),
        B, gamma, _p(u_accept, torch.float32, "u_accept"), _p(u_bonus, torch.float32, "u_bonus"),
        _p(num_accepted, torch.int32, "num_accepted"), _p(bonus, torch.int32, "bonus"),
        _p(commit_lens, torch.int32, "commit_lens"), _p(new_seq_lens, torch.int32, "new_seq_lens"),
        _p(out_tokens, torch.int32, "out_tokens"), _p(workspace),
        workspace.numel() * workspace.element_size(), _p(status, torch.int32, "status"),
        _stream(stream))
    _check("dspark_sampling_accept", rc)


def dspark_cap_accept(logits, *, V, verify_lens, draft, prefix_lens, B, gamma, num_accepted,
                      bonus, commit_lens, out_tokens, ceiling, totals, workspace, status,
                      argmax=None, new_seq_lens=None, stream=None) -> None:
    """cap-accept over the strided [B*(gamma+1), V] verify rows."""
    ptr, ld = _logits_ptr(logits, V)
    rc = load().dspark_cap_accept(
        ptr, _dtype_code(logits), ld, V, _p(verify_lens, torch.int32, "verify_lens"),
        _p(draft, torch.int32, "draft"), _p(prefix_lens, torch.int32, "prefix_lens"), B, gamma,
        _p(argmax, torch.int32, "argmax"), _p(num_accepted, torch.int32, "num_accepted"),
        _p(bonus, torch.int32, "bonus"), _p(commit_lens, torch.int32, "commit_lens"),
        _p(new_seq_lens, torch.int32, "new_seq_lens"), _p(out_tokens, torch.int32, "out_tokens"),
        _p(ceiling, torch.int32, "ceiling"), _p(totals, torch.int32, "totals"), _p(workspace),
        workspace.numel() * workspace.element_size(), _p(status, torch.int32, "status"),
        _stream(stream))
    _check("dspark_cap_accept", rc)


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled device byte buffer usable as a workspace (256-byte
    aligned by the caching allocator).  The planner's workspace must start
    out zero; the accept workspaces need not, but zeroing is done once, at
    allocation, off the step."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


STATIC_MAX_ROWS = 32768


def dspark_greedy_accept_static(logits, *, V, cu_seqlens, draft, prefix_lens, B, gamma,
                                num_accepted, bonus, commit_lens, out_tokens, status,
                                argmax=None, new_seq_lens=None, max_rows=None,
                                stream=None) -> None:
    """dspark_greedy_accept for callers that cannot allocate device memory:
    the scratch is a library-owned device array (at most STATIC_MAX_ROWS
    rows).  Calls that overlap on the GPU race on that array."""
    ptr, ld = _logits_ptr(logits, V)
    max_rows = logits.size(0) if max_rows is None else max_rows
    rc = load().dspark_greedy_accept_static(
        ptr, _dtype_code(logits), ld, V, max_rows, _p(cu_seqlens, torch.int32, "cu_seqlens"),
        _p(draft, torch.int32, "draft"), _p(prefix_lens, torch.int32, "prefix_lens"), B, gamma,
        _p(argmax, torch.int32, "argmax"), _p(num_accepted, torch.int32, "num_accepted"),
        _p(bonus, torch.int32, "bonus"), _p(commit_lens, torch.int32, "commit_lens"),
        _p(new_seq_lens, torch.int32, "new_seq_lens"), _p(out_tokens, torch.int32, "out_tokens"),
        _p(status, torch.int32, "status"), _stream(stream))
    _check("dspark_greedy_accept_static", rc)


# -------------------------------------------------------------- calibration

def dspark_sts_confidence(conf_logits, *, sts_temps, conf_out, status, stream=None) -> None:
    """c = sigmoid(z / T) elementwise over conf_logits [n_rows, gamma]."""
    n_rows, gamma = conf_logits.shape
    rc = load().dspark_sts_confidence(
        _p(conf_logits, torch.float32, "conf_logits"), _p(sts_temps, torch.float32, "sts_temps"),
        n_rows, gamma, _p(conf_out, torch.float32, "conf_out"), _p(status, torch.int32, "status"),
        _stream(stream))
    _check("dspark_sts_confidence", rc)


def dspark_sts_record(conf_logits, *, num_correct, B, gamma, rec_logits, rec_correct, rec_tested,
                      cursor, status, verify_lens=None, select=None, prefix_mask=None,
                      stream=None) -> None:
    """Append the selected requests of one step to the recorded-sample ring
    (rec_logits [capacity, gamma] fp32, rec_correct / rec_tested [capacity]
    int32) at the device cursor (an int64 [1] tensor, bit-identical to the
    C ABI's uint64)."""
    rc = load().dspark_sts_record(
        _p(conf_logits, torch.float32, "conf_logits"), _p(num_correct, torch.int32, "num_correct"),
        _p(verify_lens, torch.int32, "verify_lens"), _p(select, torch.uint8, "select"), B, gamma,
        _p(rec_logits, torch.float32, "rec_logits"), _p(rec_correct, torch.int32, "rec_correct"),
        _p(rec_tested, torch.int32, "rec_tested"), rec_correct.numel(),
        _p(cursor, torch.int64, "cursor"), _p(prefix_mask, torch.uint8, "prefix_mask"),
        _p(status, torch.int32, "status"), _stream(stream))
    _check("dspark_sts_record", rc)


def dspark_calibration_workspace_bytes(gamma: int, n_bins: int) -> int:
    return int(load().dspark_calibration_workspace_bytes(gamma, n_bins))


def dspark_calibration_stats(rec_logits, *, rec_correct, rec_tested, N, gamma, sts_temps, n_bins,
                             metrics, workspace, status, hist=None, stream=None) -> None:
    """Per-depth calibration (metrics [2, gamma, 4] fp64; hist [2, gamma,
    n_bins, 3] int64 holding the C ABI's uint64 counts)."""
    rc = load().dspark_calibration_stats(
        _p(rec_logits, torch.float32, "rec_logits"), _p(rec_correct, torch.int32, "rec_correct"),
        _p(rec_tested, torch.int32, "rec_tested"), N, gamma,
        _p(sts_temps, torch.float32, "sts_temps"), n_bins, _p(hist, torch.int64, "hist"),
        _p(metrics, torch.float64, "metrics"), _p(workspace),
        workspace.numel() * workspace.element_size(), _p(status, torch.int32, "status"),
        _stream(stream))
    _check("dspark_calibration_stats", rc)


def dspark_sts_fit_workspace_bytes(N: int, n_temps: int, n_bins: int) -> int:
    return int(load().dspark_sts_fit_workspace_bytes(N, n_temps, n_bins))


def dspark_sts_fit(rec_logits, *, rec_correct, rec_tested, N, gamma, temp_grid, n_bins,
                   sts_temps_out, choice, workspace, status, ece_curve=None, n_obs=None,
                   stream=None) -> None:
    """Sequential per-depth temperature fit over ``temp_grid`` (a host
    sequence of positive temperatures)."""
    grid = (ctypes.c_float * len(temp_grid))(*[float(t) for t in temp_grid])
    rc = load().dspark_sts_fit(
        _p(rec_logits, torch.float32, "rec_logits"), _p(rec_correct, torch.int32, "rec_correct"),
        _p(rec_tested, torch.int32, "rec_tested"), N, gamma, grid, len(temp_grid), n_bins,
        _p(sts_temps_out, torch.float32, "sts_temps_out"), _p(choice, torch.int32, "choice"),
        _p(ece_curve, torch.float64, "ece_curve"), _p(n_obs, torch.int64, "n_obs"),
        _p(workspace), workspace.numel() * workspace.element_size(),
        _p(status, torch.int32, "status"), _stream(stream))
    _check("dspark_sts_fit", rc)
