"""Canary guard bands around every output buffer and workspace.

Each entry point gets its outputs and its workspace cut from the middle of a
larger device buffer whose borders hold a sentinel byte pattern.  After the
call the borders must be unchanged (no write outside the buffers the caller
described) and the outputs must equal those of the same call on plain
buffers.  Sizes follow the workloads (a full dsv4_like step, the mixed
workload's rank path) and edge cases where a write could run past an end
(a capacity below the padded total, a shared tier past the capacity, a
recorder ring shorter than one step's selection)."""

import numpy as np
import pytest
import torch

from confidence_scheduled_speculative_gb300 import workloads as wl
from gpu_helpers import require_gpu, to_dev_logits

pytestmark = pytest.mark.gpu

SENTINEL = 0xA5
GUARD_BYTES = 1024  # a multiple of 256: every payload keeps 256-byte alignment


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


class Guarded:
    """`view` ([shape], dtype) sits between two GUARD_BYTES bands of SENTINEL."""

    def __init__(self, shape, dtype, device, init=0):
        shape = tuple(shape) if isinstance(shape, (tuple, list)) else (shape,)
        n = int(np.prod(shape)) if shape else 1
        esz = torch.empty(0, dtype=dtype).element_size()
        self.nbytes = n * esz
        self.raw = torch.full((GUARD_BYTES * 2 + self.nbytes,), SENTINEL, dtype=torch.uint8,
                              device=device)
        self.view = self.raw[GUARD_BYTES:GUARD_BYTES + self.nbytes].view(dtype).view(shape)
        if init is not None:
            self.view.fill_(init)

    def intact(self) -> bool:
        head = self.raw[:GUARD_BYTES]
        tail = self.raw[GUARD_BYTES + self.nbytes:]
        return bool((head == SENTINEL).all()) and bool((tail == SENTINEL).all())


def _all_intact(bufs):
    bad = [k for k, g in bufs.items() if not g.intact()]
    assert not bad, f"guard bands overwritten: {bad}"


def _i32(dev, a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def _interpolated(step):
    """The step with its additive tier table read as interpolation samples."""
    import dataclasses
    return dataclasses.replace(step, cost=dataclasses.replace(step.cost, kind=2))


def _step_guarded(dev, name, fused, interp=False):
    """One plan + pack + greedy accept + cap-accept of a workload through the
    binding, every output and workspace guarded."""
    from confidence_scheduled_speculative_gb300 import api
    step = wl.make_step(wl.WORKLOADS[name], seed=2)
    if interp:
        step = _interpolated(step)
    w, c = step.workload, step.cost
    B, g, cap = step.B, step.gamma, step.capacity
    i32, f32, f64 = torch.int32, torch.float32, torch.float64
    gb = {
        "survivals": Guarded((B, g), f32, dev), "verify_lens": Guarded(B, i32, dev),
        "budget": Guarded(1, i32, dev), "tau_theta": Guarded(2, f64, dev),
        "status": Guarded(1, i32, dev),
        "plan_ws": Guarded(api.dspark_plan_workspace_bytes(B, g), torch.uint8, dev),
        "ids": Guarded(cap, i32, dev, -3), "pos": Guarded(cap, i32, dev, -3),
        "req": Guarded(cap, i32, dev, -3), "src": Guarded(cap, i32, dev, -3),
        "cu": Guarded(B + 1, i32, dev), "totals": Guarded(2, i32, dev),
    }
    z = torch.from_numpy(step.conf_logits).to(dev)
    T = torch.from_numpy(step.sts_temps).to(dev)
    anchor, draft, prefix = _i32(dev, step.anchor), _i32(dev, step.draft), _i32(dev, step.prefix_lens)
    cM = torch.from_numpy(np.asarray(c.M, np.int32)).to(dev)
    cV = torch.from_numpy(np.asarray(c.val, np.float64)).to(dev)
    common = dict(B=B, gamma=g, survival_eps=w.survival_eps, min_verify_len=w.min_verify_len,
                  max_verify_len=w.max_len, forced_budget=w.forced_budget, cost_kind=c.kind,
                  cost_M=cM, cost_val=cV, bias_ms=c.bias_ms, alpha_ms=c.alpha_ms,
                  survivals=gb["survivals"].view, verify_lens=gb["verify_lens"].view,
                  budget=gb["budget"].view, tau_theta=gb["tau_theta"].view,
                  status=gb["status"].view, workspace=gb["plan_ws"].view)
    packed = dict(packed_ids=gb["ids"].view, packed_pos=gb["pos"].view,
                  packed_req=gb["req"].view, packed_src=gb["src"].view,
                  cu_seqlens=gb["cu"].view, totals=gb["totals"].view)
    if fused:
        api.dspark_plan_pack(z, T, anchor, draft, prefix, tiers=step.tiers, capacity=cap,
                             **common, **packed)
    else:
        api.dspark_plan(z, T, **common)
        api.dspark_pack_verify(anchor, draft, prefix, gb["verify_lens"].view, B=B, gamma=g,
                               tiers=step.tiers, capacity=cap, status=gb["status"].view,
                               **packed)
    torch.cuda.synchronize()
    total = int(gb["totals"].view[0])
    strided = to_dev_logits(wl.strided_logits(step), dev)
    compact = strided.index_select(0, gb["src"].view[:total].long()).contiguous()
    rows_max = max(cap, B * (g + 1))
    acc = {
        "argmax": Guarded(rows_max, i32, dev, -5), "num_acc": Guarded(B, i32, dev),
        "bonus": Guarded(B, i32, dev), "commit": Guarded(B, i32, dev),
        "new_seq": Guarded(B, i32, dev), "out": Guarded((B, g + 1), i32, dev),
        "acc_ws": Guarded(api.dspark_accept_workspace_bytes(rows_max, w.V), torch.uint8, dev),
        "ceiling": Guarded(B, i32, dev), "cap_totals": Guarded(2, i32, dev),
        "acc_status": Guarded(1, i32, dev),
    }
    outs = dict(num_accepted=acc["num_acc"].view, bonus=acc["bonus"].view,
                commit_lens=acc["commit"].view, new_seq_lens=acc["new_seq"].view,
                out_tokens=acc["out"].view, argmax=acc["argmax"].view[:compact.size(0)],
                workspace=acc["acc_ws"].view, status=acc["acc_status"].view)
    api.dspark_greedy_accept(compact, V=w.V, cu_seqlens=gb["cu"].view, draft=draft,
                             prefix_lens=prefix, B=B, gamma=g, **outs)
    torch.cuda.synchronize()
    greedy = {k: v.cpu().numpy().copy() for k, v in outs.items() if k != "workspace"}
    outs["argmax"] = acc["argmax"].view[:strided.size(0)]
    api.dspark_cap_accept(strided, V=w.V, verify_lens=gb["verify_lens"].view, draft=draft,
                          prefix_lens=prefix, B=B, gamma=g, ceiling=acc["ceiling"].view,
                          totals=acc["cap_totals"].view, **outs)
    torch.cuda.synchronize()
    gb.update(acc)
    res = {k: v.view.cpu().numpy() for k, v in gb.items() if not k.endswith("ws")}
    res["greedy"] = greedy
    return step, gb, res


@pytest.mark.parametrize("name,fused,interp", [("dsv4_like", True, False), ("mixed", False, False),
                                               ("dsv4_like", True, True), ("qwen_like", True, False),
                                               ("tiny", False, False)])
def test_step_outputs_stay_inside_their_buffers(dev, name, fused, interp):
    """Planner (select, dense select or interp select path), pack (fused or
    its own kernel), greedy accept and cap-accept write nothing outside the
    buffers they are given, and give the outputs of the same step on plain
    buffers."""
    from confidence_scheduled_speculative_gb300.engine import StepConfig, VerifyStep
    step, gb, res = _step_guarded(dev, name, fused, interp)
    _all_intact(gb)
    vs = VerifyStep(StepConfig.from_step(step), dev)
    vs.load_inputs(step)
    vs.plan_pack() if fused else (vs.plan(), vs.pack())
    total = int(vs.totals[0].item())
    strided = to_dev_logits(wl.strided_logits(step), dev)
    vs.greedy_accept(strided.index_select(0, vs.packed_src[:total].long()).contiguous())
    ref = vs.result()
    for k, rk in (("survivals", "survivals"), ("verify_lens", "verify_lens"), ("budget", "budget"),
                  ("tau_theta", "tau_theta"), ("cu", "cu_seqlens"), ("totals", "totals")):
        np.testing.assert_array_equal(res[k], ref[rk], err_msg=k)
    n = int(ref["totals"][1])
    for k in ("ids", "pos", "req", "src"):
        np.testing.assert_array_equal(res[k][:n], ref["packed_" + k][:n], err_msg=k)
        assert np.all(res[k][max(n, total):] == -3), k  # past the padded window: untouched
    g = res["greedy"]
    for k, rk in (("num_accepted", "num_accepted"), ("bonus", "bonus"),
                  ("commit_lens", "commit_lens"), ("out_tokens", "out_tokens")):
        np.testing.assert_array_equal(g[k], ref[rk], err_msg=k)
    np.testing.assert_array_equal(g["argmax"][:total], ref["argmax"][:total])


def test_capacity_edges_stay_inside(dev, orc):
    """A capacity below the padded total, and a shared tier past the
    capacity: rows stop at the capacity (CAPACITY flagged), the bands hold."""
    from confidence_scheduled_speculative_gb300 import api
    step = wl.make_step(wl.QWEN, seed=3)
    B, g = step.B, step.gamma
    r = orc.plan_step(step)
    lens = _i32(dev, r.verify_lens)
    total = int(r.verify_lens.sum())
    cap = total - 7
    gb = {k: Guarded(cap, torch.int32, dev, -3) for k in ("ids", "pos", "req", "src")}
    gb.update(cu=Guarded(B + 1, torch.int32, dev), totals=Guarded(2, torch.int32, dev),
              status=Guarded(1, torch.int32, dev))
    anchor, draft, prefix = _i32(dev, step.anchor), _i32(dev, step.draft), _i32(dev, step.prefix_lens)
    api.dspark_pack_verify(anchor, draft, prefix, lens, B=B, gamma=g, tiers=step.tiers,
                           capacity=cap, packed_ids=gb["ids"].view, packed_pos=gb["pos"].view,
                           packed_req=gb["req"].view, packed_src=gb["src"].view,
                           cu_seqlens=gb["cu"].view, totals=gb["totals"].view,
                           status=gb["status"].view)
    torch.cuda.synchronize()
    _all_intact(gb)
    assert int(gb["status"].view.item()) & api.STATUS_CAPACITY
    pad_to = torch.tensor([cap + 1000], dtype=torch.int32, device=dev)
    api.dspark_pad_to_tier(pad_to, packed_ids=gb["ids"].view, packed_pos=gb["pos"].view,
                           packed_req=gb["req"].view, packed_src=gb["src"].view,
                           totals=gb["totals"].view, status=gb["status"].view, capacity=cap)
    torch.cuda.synchronize()
    _all_intact(gb)


def test_scatter_and_sampling_stay_inside(dev, orc):
    """ScatterCompactToStrided into a guarded strided buffer (TMA path and
    2-byte path) and the sampling accept with guarded outputs and workspace."""
    from confidence_scheduled_speculative_gb300 import api
    rng = np.random.default_rng(8)
    B, g = 24, 7
    lens = rng.integers(1, g + 2, size=B).astype(np.int32)
    p = orc.pack(np.zeros(B), np.zeros((B, g)), np.zeros(B), lens, [], B * (g + 1))
    for width in (8192, 1003):  # 16 KB rows (bulk copies), unaligned rows (2-byte copies)
        src = torch.from_numpy(rng.integers(0, 2 ** 15, size=(p.total, width)).astype(np.int16)).to(dev)
        dst = Guarded((B * (g + 1), width), torch.int16, dev, 7)
        st = Guarded(1, torch.int32, dev)
        api.dspark_scatter_compact_to_strided(src.view(torch.bfloat16), _i32(dev, p.src[:p.total]),
                                              _i32(dev, [p.total]), dst.view.view(torch.bfloat16),
                                              status=st.view)
        torch.cuda.synchronize()
        _all_intact({"dst": dst, "status": st})
        assert int(st.view.item()) == 0
    V, Bs, gs = 5000, 6, 4
    cu = np.concatenate([[0], np.cumsum(rng.integers(1, gs + 2, size=Bs))]).astype(np.int32)
    tgt = to_dev_logits(rng.normal(0, 2, (int(cu[-1]), V)).astype(np.float32), dev)
    dft = to_dev_logits(rng.normal(0, 2, (Bs * gs, V)).astype(np.float32), dev)
    drafts = _i32(dev, rng.integers(0, V, (Bs, gs)))
    ua = torch.from_numpy(rng.random((Bs, gs)).astype(np.float32)).to(dev)
    ub = torch.from_numpy(rng.random(Bs).astype(np.float32)).to(dev)
    gbs = {"num": Guarded(Bs, torch.int32, dev), "bonus": Guarded(Bs, torch.int32, dev),
           "commit": Guarded(Bs, torch.int32, dev), "seq": Guarded(Bs, torch.int32, dev),
           "out": Guarded((Bs, gs + 1), torch.int32, dev), "status": Guarded(1, torch.int32, dev),
           "ws": Guarded(api.dspark_sampling_workspace_bytes(int(cu[-1]), Bs, gs), torch.uint8, dev)}
    api.dspark_sampling_accept(tgt, dft, V=V, cu_seqlens=_i32(dev, cu), draft=drafts,
                               prefix_lens=_i32(dev, np.arange(Bs)), B=Bs, gamma=gs, u_accept=ua,
                               u_bonus=ub, num_accepted=gbs["num"].view, bonus=gbs["bonus"].view,
                               commit_lens=gbs["commit"].view, new_seq_lens=gbs["seq"].view,
                               out_tokens=gbs["out"].view, workspace=gbs["ws"].view,
                               status=gbs["status"].view)
    torch.cuda.synchronize()
    _all_intact(gbs)


def test_calibration_stays_inside(dev):
    """The STS recorder into a ring shorter than one step's selection, the
    calibration statistics and the temperature fit, all guarded."""
    from confidence_scheduled_speculative_gb300 import api
    rng = np.random.default_rng(9)
    B, g, capr = 40, 8, 25
    z = torch.from_numpy(rng.normal(1, 1, (B, g)).astype(np.float32)).to(dev)
    corr = _i32(dev, rng.integers(0, g + 1, B))
    gbr = {"rz": Guarded((capr, g), torch.float32, dev), "rc": Guarded(capr, torch.int32, dev),
           "rt": Guarded(capr, torch.int32, dev), "cur": Guarded(1, torch.int64, dev),
           "mask": Guarded((B, g), torch.uint8, dev), "status": Guarded(1, torch.int32, dev)}
    api.dspark_sts_record(z, num_correct=corr, B=B, gamma=g, rec_logits=gbr["rz"].view,
                          rec_correct=gbr["rc"].view, rec_tested=gbr["rt"].view,
                          cursor=gbr["cur"].view, status=gbr["status"].view,
                          prefix_mask=gbr["mask"].view)
    torch.cuda.synchronize()
    _all_intact(gbr)
    assert int(gbr["status"].view.item()) & api.STATUS_CAPACITY
    N, G, J, M = 3000, 8, 16, 10
    cs = wl.calibration_samples(N, G, 1.0 + 0.05 * np.arange(G), seed=4)
    zc = torch.from_numpy(cs.conf_logits).to(dev)
    cc, tc = torch.from_numpy(cs.correct).to(dev), torch.from_numpy(cs.tested).to(dev)
    gbs = {"metrics": Guarded((2, G, 4), torch.float64, dev),
           "hist": Guarded((2, G, M, 3), torch.int64, dev), "status": Guarded(1, torch.int32, dev),
           "ws": Guarded(api.dspark_calibration_workspace_bytes(G, M), torch.uint8, dev)}
    api.dspark_calibration_stats(zc, rec_correct=cc, rec_tested=tc, N=N, gamma=G,
                                 sts_temps=torch.ones(G, dtype=torch.float32, device=dev),
                                 n_bins=M, metrics=gbs["metrics"].view, hist=gbs["hist"].view,
                                 workspace=gbs["ws"].view, status=gbs["status"].view)
    torch.cuda.synchronize()
    _all_intact(gbs)
    grid = wl.temperature_grid(J)
    gbf = {"T": Guarded(G, torch.float32, dev), "choice": Guarded(G, torch.int32, dev),
           "ece": Guarded((G, J), torch.float64, dev), "nobs": Guarded(G, torch.int64, dev),
           "status": Guarded(1, torch.int32, dev),
           "ws": Guarded(api.dspark_sts_fit_workspace_bytes(N, J, M), torch.uint8, dev)}
    api.dspark_sts_fit(zc, rec_correct=cc, rec_tested=tc, N=N, gamma=G, temp_grid=grid, n_bins=M,
                       sts_temps_out=gbf["T"].view, choice=gbf["choice"].view,
                       ece_curve=gbf["ece"].view, n_obs=gbf["nobs"].view,
                       workspace=gbf["ws"].view, status=gbf["status"].view)
    torch.cuda.synchronize()
    _all_intact(gbf)
