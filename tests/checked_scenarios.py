"""Calls that the bounds-checked library is run through (test_gpu_checked.py).

`scenarios(dev)` drives every entry point of the C ABI over the workloads
and the edge cases where a kernel's computed indices come closest to the
ends of their buffers, and returns every output (status words included) as
numpy arrays keyed "scenario/output".  test_gpu_checked.py runs it once in
its own process on the normal library and once in a child process started
with DSPARK_CHECKED=1, which loads libdspark_checked.so; run as a script
(`python tests/checked_scenarios.py OUT.npz`) it is that child and writes
the arrays to OUT.npz.

The inputs are seeded and synthetic (the workloads module); no expected
value comes from here: the normal library's parity with the oracle is
checked by the other GPU tests, and here the two builds are checked against
each other.
"""

from __future__ import annotations

import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from confidence_scheduled_speculative_gb300 import api  # noqa: E402
from confidence_scheduled_speculative_gb300 import workloads as wl  # noqa: E402
from confidence_scheduled_speculative_gb300.engine import StepConfig, VerifyStep  # noqa: E402

I32, F32, F64 = torch.int32, torch.float32, torch.float64


def _np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().copy()


def _i32(dev, a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def _dev_logits(a: np.ndarray, dev) -> torch.Tensor:
    """numpy logits (bf16 bits as uint16, or fp32) on the device."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def _steps(dev, out: dict) -> None:
    """Each workload through the engine: the fused plan + pack and the
    separate planner and pack, greedy accept on the compact rows, cap-accept
    on the strided rows.  The stress workload (B=1024, gamma=16: the largest
    candidate count) runs the planner and pack only."""
    for name in ("tiny", "qwen_like", "dsv4_like", "mixed", "stress"):
        for seed in (0, 1):
            step = wl.make_step(wl.WORKLOADS[name], seed=seed)
            vs = VerifyStep(StepConfig.from_step(step), dev)
            vs.load_inputs(step)
            vs.plan_pack()
            torch.cuda.synchronize()
            fused = vs.result()
            vs.load_inputs(step)
            vs.plan()
            vs.pack()
            torch.cuda.synchronize()
            sep = vs.result()
            for k in ("survivals", "verify_lens", "budget", "tau_theta", "cu_seqlens", "totals",
                      "status"):
                out[f"step/{name}/{seed}/fused/{k}"] = np.asarray(fused[k])
                out[f"step/{name}/{seed}/separate/{k}"] = np.asarray(sep[k])
            n = int(sep["totals"][1])
            for k in ("packed_ids", "packed_pos", "packed_req", "packed_src"):
                out[f"step/{name}/{seed}/fused/{k}"] = np.asarray(fused[k])[:n]
            if name == "stress":
                continue
            strided = _dev_logits(wl.strided_logits(step), dev)
            total = int(sep["totals"][0])
            compact = strided.index_select(0, vs.packed_src[:total].long()).contiguous()
            vs.greedy_accept(compact)
            torch.cuda.synchronize()
            res = vs.result()
            for k in ("argmax", "num_accepted", "bonus", "commit_lens", "new_seq_lens",
                      "out_tokens", "status"):
                v = np.asarray(res[k])
                out[f"step/{name}/{seed}/greedy/{k}"] = v[:total] if k == "argmax" else v
            vs.cap_accept(strided)
            torch.cuda.synchronize()
            res = vs.result()
            for k in ("argmax", "num_accepted", "bonus", "commit_lens", "out_tokens", "status"):
                out[f"step/{name}/{seed}/cap/{k}"] = np.asarray(res[k])
            del strided, compact


def _plan(dev, out, tag, z, T, *, eps, min_len, max_len, forced, kind, M, val, bias=0.0,
          alpha=0.0, **options) -> None:
    B, g = z.shape
    o = dict(survivals=torch.zeros((B, g), dtype=F32, device=dev),
             verify_lens=torch.zeros(B, dtype=I32, device=dev),
             budget=torch.zeros(1, dtype=I32, device=dev),
             tau_theta=torch.zeros(2, dtype=F64, device=dev),
             status=torch.zeros(1, dtype=I32, device=dev))
    ws = api.workspace(api.dspark_plan_workspace_bytes(B, g), dev)
    api.dspark_plan_ex(torch.from_numpy(z).to(dev), torch.from_numpy(T).to(dev), B=B, gamma=g,
                       survival_eps=eps, min_verify_len=min_len, max_verify_len=max_len,
                       forced_budget=forced, cost_kind=kind,
                       cost_M=_i32(dev, M), cost_val=torch.from_numpy(np.asarray(val, np.float64)).to(dev),
                       bias_ms=bias, alpha_ms=alpha, workspace=ws, **o, **options)
    torch.cuda.synchronize()
    for k, v in o.items():
        out[f"plan/{tag}/{k}"] = _np(v)


def _planner_cases(dev, out) -> None:
    """Cost tables on both planner paths and their edges: a 1-D table at
    every M (staged in shared memory), a table past the stage (global
    memory), additive tables of 5, 31, 32 and 61 entries, interpolated tables
    of 8 and 100 samples; budgets 0 and everything; every candidate below
    eps; B=1 and gamma=1; the dense path over crowded bins; the planner
    options."""
    rng = np.random.default_rng(1234)
    B, g = 256, 16
    z = rng.normal(1.5, 1.2, (B, g)).astype(np.float32)
    T = rng.uniform(0.8, 1.3, g).astype(np.float32)
    base = dict(eps=1e-4, min_len=1, max_len=g + 1, forced=-1)
    M1 = np.arange(B, B + B * g + 1, dtype=np.int32)
    _plan(dev, out, "sps_every_M", z, T, kind=api.COST_SPS_1D, M=M1,
          val=1.0 / (1e-3 + 2e-6 * M1), **base)
    Bl, gl = 600, 24  # 14400 candidates: a table of 15004 entries, past the stage
    zl = rng.normal(1.0, 1.5, (Bl, gl)).astype(np.float32)
    Ml = np.arange(1, Bl + Bl * gl + 5, dtype=np.int32)
    _plan(dev, out, "additive_unstaged", zl, np.ones(gl, np.float32), kind=api.COST_ADDITIVE,
          M=Ml, val=0.003 * Ml, eps=1e-4, min_len=1, max_len=gl + 1, forced=-1)
    for n in (5, 31, 32, 61):
        Mt = np.linspace(B + 16, B * (g + 1), n).astype(np.int32)
        Mt = np.unique(Mt)
        _plan(dev, out, f"additive_{n}", z, T, kind=api.COST_ADDITIVE, M=Mt,
              val=0.002 * Mt + 0.5, bias=1.0, alpha=0.2, **base)
    for n in (8, 100, 2100):  # 2100 samples: the rank path
        Mi = np.unique(np.linspace(B, B * (g + 1) + 8, n).astype(np.int32))
        _plan(dev, out, f"interp_{n}", z, T, kind=api.COST_ADDITIVE_INTERP, M=Mi,
              val=0.0025 * Mi + 0.3 * np.sin(Mi / 97.0) ** 2, bias=0.8, alpha=0.1, **base)
    Mt = np.array([B + 64, B + 512, B + 2048, B * (g + 1)], np.int32)
    for forced in (0, B * g):
        _plan(dev, out, f"forced_{forced}", z, T, kind=api.COST_ADDITIVE, M=Mt,
              val=0.002 * Mt, **{**base, "forced": forced})
        _plan(dev, out, f"forced_{forced}_rank", z, T, kind=api.COST_SPS_1D, M=M1,
              val=1.0 / (1e-3 + 2e-6 * M1), **{**base, "forced": forced})
    zlow = np.full((B, g), -30.0, np.float32)
    _plan(dev, out, "all_dropped", zlow, T, kind=api.COST_ADDITIVE, M=Mt, val=0.002 * Mt, **base)
    _plan(dev, out, "all_dropped_rank", zlow, T, kind=api.COST_SPS_1D, M=M1,
          val=1.0 / (1e-3 + 2e-6 * M1), **base)
    _plan(dev, out, "min_len_3", z, T, kind=api.COST_ADDITIVE, M=Mt, val=0.002 * Mt,
          **{**base, "min_len": 3, "max_len": 9})
    z11 = np.array([[2.0]], np.float32)
    _plan(dev, out, "B1_g1", z11, np.ones(1, np.float32), kind=api.COST_ADDITIVE,
          M=np.array([1, 2], np.int32), val=np.array([1.0, 1.5]), eps=1e-4, min_len=1,
          max_len=2, forced=-1)
    # the dense path's crowded bins (every request with the same
    # confidences: 600 equal keys a bin) and a flat table: the entries left
    # go through the threshold slots 32 at a time
    Bc, gc = 600, 8
    zc = np.full((Bc, gc), np.log(0.3 / 0.7), np.float32)
    Mc = np.arange(Bc, Bc + Bc * gc + 1, dtype=np.int32)
    for forced in (-1, 1234):
        _plan(dev, out, f"dense_crowded_{forced}", zc, np.ones(gc, np.float32),
              kind=api.COST_SPS_1D, M=Mc, val=np.full(Mc.size, 500.0), eps=1e-4, min_len=1,
              max_len=gc + 1, forced=forced)
    gen = _i32(dev, np.arange(B))
    stale = _i32(dev, np.where(np.arange(B) % 5 == 0, -1, np.arange(B)))
    lag = torch.from_numpy((z + rng.normal(0, 0.3, z.shape)).astype(np.float32)).to(dev)
    for tag, kind, M, val in (("select", api.COST_ADDITIVE, Mt, 0.002 * Mt),
                              ("rank", api.COST_SPS_1D, M1, 1.0 / (1e-3 + 2e-6 * M1))):
        _plan(dev, out, f"options_{tag}", z, T, kind=kind, M=M, val=val,
              conf_generation=gen, req_generation=stale, lagged_conf_logits=lag,
              align_tiers=[64, 256, 1024, 4352], **base)


def _accept_cases(dev, out) -> None:
    """The allocation-free greedy accept, the shared-tier pad, both scatter
    paths and the sampling accept with and without the draft normalizers."""
    rng = np.random.default_rng(77)
    step = wl.make_step(wl.QWEN, seed=5)
    vs = VerifyStep(StepConfig.from_step(step), dev)
    vs.load_inputs(step)
    vs.plan_pack()
    torch.cuda.synchronize()
    total = int(vs.totals[0].item())
    strided = _dev_logits(wl.strided_logits(step), dev)
    compact = strided.index_select(0, vs.packed_src[:total].long()).contiguous()
    B, g = step.B, step.gamma
    o = {k: torch.zeros(B, dtype=I32, device=dev) for k in ("num", "bonus", "commit", "seq")}
    o["out"] = torch.zeros((B, g + 1), dtype=I32, device=dev)
    o["argmax"] = torch.full((compact.size(0),), -1, dtype=I32, device=dev)
    o["status"] = torch.zeros(1, dtype=I32, device=dev)
    api.dspark_greedy_accept_static(compact, V=step.workload.V, cu_seqlens=vs.cu_seqlens,
                                    draft=vs.draft, prefix_lens=vs.prefix_lens, B=B, gamma=g,
                                    num_accepted=o["num"], bonus=o["bonus"],
                                    commit_lens=o["commit"], new_seq_lens=o["seq"],
                                    out_tokens=o["out"], argmax=o["argmax"], status=o["status"])
    torch.cuda.synchronize()
    for k, v in o.items():
        out[f"static/{k}"] = _np(v)
    pad_to = torch.tensor([int(vs.totals[1].item()) + 40], dtype=I32, device=dev)
    vs.pad_to_tier(pad_to)
    torch.cuda.synchronize()
    res = vs.result()
    for k in ("packed_ids", "packed_pos", "packed_req", "packed_src", "totals", "status"):
        out[f"pad_to_tier/{k}"] = np.asarray(res[k])

    Bs, gs = 24, 7
    lens = rng.integers(1, gs + 2, size=Bs).astype(np.int32)
    src_rows = np.concatenate([r * (gs + 1) + np.arange(L) for r, L in enumerate(lens)])
    n = src_rows.size
    for width in (8192, 1003):  # bulk copies (16 KB rows), 2-byte copies
        src = torch.from_numpy(rng.integers(0, 2 ** 15, size=(n, width)).astype(np.int16)).to(dev)
        dst = torch.full((Bs * (gs + 1), width), 7, dtype=torch.int16, device=dev)
        st = torch.zeros(1, dtype=I32, device=dev)
        api.dspark_scatter_compact_to_strided(src.view(torch.bfloat16), _i32(dev, src_rows),
                                              _i32(dev, [n]), dst.view(torch.bfloat16), status=st)
        torch.cuda.synchronize()
        out[f"scatter/{width}/dst"] = _np(dst)
        out[f"scatter/{width}/status"] = _np(st)

    V, Bq, gq = 32000, 12, 6
    cu = np.concatenate([[0], np.cumsum(rng.integers(1, gq + 2, size=Bq))]).astype(np.int32)
    tgt = torch.from_numpy(rng.normal(0, 2, (int(cu[-1]), V)).astype(np.float32)).to(dev)
    dft = torch.from_numpy(rng.normal(0, 2, (Bq * gq, V)).astype(np.float32)).to(dev)
    drafts = _i32(dev, rng.integers(0, V, (Bq, gq)))
    ua = torch.from_numpy(rng.random((Bq, gq)).astype(np.float32)).to(dev)
    ub = torch.from_numpy(rng.random(Bq).astype(np.float32)).to(dev)
    lse = torch.logsumexp(dft.double(), dim=1).float()
    for dtype in (torch.float32, torch.bfloat16):
        for with_lse in (False, True):
            s = {k: torch.zeros(Bq, dtype=I32, device=dev) for k in ("num", "bonus", "commit", "seq")}
            s["out"] = torch.zeros((Bq, gq + 1), dtype=I32, device=dev)
            s["status"] = torch.zeros(1, dtype=I32, device=dev)
            ws = api.workspace(api.dspark_sampling_workspace_bytes(int(cu[-1]), Bq, gq), dev)
            api.dspark_sampling_accept(tgt.to(dtype), dft.to(dtype), V=V, cu_seqlens=_i32(dev, cu),
                                       draft=drafts, prefix_lens=_i32(dev, np.arange(Bq)), B=Bq,
                                       gamma=gq, u_accept=ua, u_bonus=ub, num_accepted=s["num"],
                                       bonus=s["bonus"], commit_lens=s["commit"],
                                       new_seq_lens=s["seq"], out_tokens=s["out"], workspace=ws,
                                       status=s["status"], draft_lse=lse if with_lse else None)
            torch.cuda.synchronize()
            tag = f"sampling/{str(dtype).split('.')[-1]}/{'lse' if with_lse else 'norm'}"
            for k, v in s.items():
                out[f"{tag}/{k}"] = _np(v)


def _calibration_cases(dev, out) -> None:
    """The recorder into a ring shorter than a step's selection (it wraps),
    with a selection mask and verify lengths; the elementwise confidences;
    the calibration statistics; the temperature fit."""
    rng = np.random.default_rng(9)
    B, g, capr = 300, 8, 170
    z = torch.from_numpy(rng.normal(1, 1, (B, g)).astype(np.float32)).to(dev)
    lens = rng.integers(1, g + 2, B).astype(np.int32)
    corr = _i32(dev, [int(rng.integers(0, L)) for L in lens])
    sel = torch.from_numpy((rng.random(B) < 0.8).astype(np.uint8)).to(dev)
    r = dict(rz=torch.zeros((capr, g), dtype=F32, device=dev),
             rc=torch.full((capr,), -1, dtype=I32, device=dev),
             rt=torch.full((capr,), -1, dtype=I32, device=dev),
             cur=torch.tensor([123], dtype=torch.int64, device=dev),
             mask=torch.zeros((B, g), dtype=torch.uint8, device=dev),
             status=torch.zeros(1, dtype=I32, device=dev))
    for _ in range(2):  # the second call starts from the advanced cursor
        api.dspark_sts_record(z, num_correct=corr, B=B, gamma=g, rec_logits=r["rz"],
                              rec_correct=r["rc"], rec_tested=r["rt"], cursor=r["cur"],
                              status=r["status"], prefix_mask=r["mask"],
                              verify_lens=_i32(dev, lens), select=sel)
    torch.cuda.synchronize()
    for k, v in r.items():
        out[f"record/{k}"] = _np(v)
    c = torch.zeros((B, g), dtype=F32, device=dev)
    st = torch.zeros(1, dtype=I32, device=dev)
    api.dspark_sts_confidence(z, sts_temps=torch.full((g,), 1.3, dtype=F32, device=dev),
                              conf_out=c, status=st)
    torch.cuda.synchronize()
    out["confidence/c"], out["confidence/status"] = _np(c), _np(st)

    N, G, J, M = 20000, 12, 24, 15
    cs = wl.calibration_samples(N, G, 0.9 + 0.05 * np.arange(G), seed=4)
    zc = torch.from_numpy(cs.conf_logits).to(dev)
    cc, tc = torch.from_numpy(cs.correct).to(dev), torch.from_numpy(cs.tested).to(dev)
    s = dict(metrics=torch.zeros((2, G, 4), dtype=F64, device=dev),
             hist=torch.zeros((2, G, M, 3), dtype=torch.int64, device=dev),
             status=torch.zeros(1, dtype=I32, device=dev))
    api.dspark_calibration_stats(zc, rec_correct=cc, rec_tested=tc, N=N, gamma=G,
                                 sts_temps=torch.ones(G, dtype=F32, device=dev), n_bins=M,
                                 workspace=api.workspace(api.dspark_calibration_workspace_bytes(G, M), dev),
                                 **s)
    torch.cuda.synchronize()
    for k, v in s.items():
        out[f"stats/{k}"] = _np(v)
    f = dict(sts_temps_out=torch.zeros(G, dtype=F32, device=dev),
             choice=torch.zeros(G, dtype=I32, device=dev),
             ece_curve=torch.zeros((G, J), dtype=F64, device=dev),
             n_obs=torch.zeros(G, dtype=torch.int64, device=dev),
             status=torch.zeros(1, dtype=I32, device=dev))
    api.dspark_sts_fit(zc, rec_correct=cc, rec_tested=tc, N=N, gamma=G,
                       temp_grid=wl.temperature_grid(J), n_bins=M,
                       workspace=api.workspace(api.dspark_sts_fit_workspace_bytes(N, J, M), dev), **f)
    torch.cuda.synchronize()
    for k, v in f.items():
        out[f"fit/{k}"] = _np(v)


def scenarios(dev) -> dict[str, np.ndarray]:
    out: dict[str, np.ndarray] = {}
    _steps(dev, out)
    _planner_cases(dev, out)
    _accept_cases(dev, out)
    _calibration_cases(dev, out)
    return out


def main(path: str) -> None:
    if not api.dspark_checked_build():
        raise SystemExit("DSPARK_CHECKED=1 did not load the bounds-checked library")
    out = scenarios(torch.device("cuda:0"))
    np.savez(path, **out)


if __name__ == "__main__":
    main(sys.argv[1])
