"""GPU parity of the greedy accept (compact mode) and of cap-accept against
the CPU oracle, through the C-ABI: per-row argmax, num_accepted, bonus,
commit_lens, new_seq_lens, out_tokens, ceiling and totals, all bit-exact.

Covers small cases that span several CTAs and a ragged tail, the edge cases
of the argmax (ties across CTA split boundaries, NaN, -0/+0, rows of -inf,
V not a multiple of the 16-byte chunk, padded and unaligned row strides,
capacity overflow, bad ranges, out-of-range tokens), every workload at its
full size in the launch configuration the benchmark times, and the stress
workload at 17408 packed rows (4.5 GB) on sampled requests."""

import numpy as np
import pytest
import torch

from confidence_scheduled_speculative_gb300 import workloads as wl
from gpu_helpers import (compare_plan, oracle_plan, oracle_restage, require_gpu, run_plan_pack,
                         to_dev_logits)

pytestmark = pytest.mark.gpu

OUT_KEYS = ("num_accepted", "bonus", "commit_lens", "new_seq_lens", "out_tokens")


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _gpu_greedy(dev, logits_dev, V, cu, draft, prefix, max_rows=None, with_argmax=True, ws=None):
    """Compact greedy accept through the C ABI, with or without the per-row
    argmax output."""
    from confidence_scheduled_speculative_gb300 import api
    B, g = draft.shape
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    i32 = dict(dtype=torch.int32, device=dev)
    rows_cap = logits_dev.size(0) if max_rows is None else max_rows
    o = dict(num_accepted=torch.full((B,), -5, **i32), bonus=torch.full((B,), -5, **i32),
             commit_lens=torch.full((B,), -5, **i32), new_seq_lens=torch.full((B,), -5, **i32),
             out_tokens=torch.full((B, g + 1), -5, **i32))
    am = torch.full((max(rows_cap, 1),), -5, **i32)
    st = torch.zeros(1, **i32)
    if ws is None:
        ws = api.workspace(api.dspark_accept_workspace_bytes(rows_cap, V), dev)
    api.dspark_greedy_accept(logits_dev, V=V, cu_seqlens=t(cu), draft=t(draft),
                             prefix_lens=t(prefix), B=B, gamma=g, workspace=ws, status=st,
                             argmax=am if with_argmax else None, max_rows=rows_cap, **o)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in o.items()}
    res["argmax"] = am.cpu().numpy() if with_argmax else None
    res["status"] = int(st.cpu()[0])
    return res


def _gpu_cap(dev, logits_dev, V, lens, draft, prefix):
    from confidence_scheduled_speculative_gb300 import api
    B, g = draft.shape
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    i32 = dict(dtype=torch.int32, device=dev)
    rows = B * (g + 1)
    o = dict(num_accepted=torch.full((B,), -5, **i32), bonus=torch.full((B,), -5, **i32),
             commit_lens=torch.full((B,), -5, **i32), new_seq_lens=torch.full((B,), -5, **i32),
             out_tokens=torch.full((B, g + 1), -5, **i32), ceiling=torch.full((B,), -5, **i32),
             totals=torch.full((2,), -5, **i32))
    am = torch.full((rows,), -5, **i32)
    st = torch.zeros(1, **i32)
    ws = api.workspace(api.dspark_accept_workspace_bytes(rows, V), dev)
    api.dspark_cap_accept(logits_dev, V=V, verify_lens=t(lens), draft=t(draft),
                          prefix_lens=t(prefix), B=B, gamma=g, workspace=ws, status=st, argmax=am,
                          **o)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in o.items()}
    res["argmax"] = am.cpu().numpy()
    res["status"] = int(st.cpu()[0])
    return res


def _cmp_greedy(tag, g, r, rows):
    if g["argmax"] is not None:
        np.testing.assert_array_equal(g["argmax"][:rows], r.argmax[:rows], err_msg=f"{tag} argmax")
    for k in OUT_KEYS:
        np.testing.assert_array_equal(g[k], r[k], err_msg=f"{tag} {k}")
    assert g["status"] == r.status, (tag, g["status"], r.status)


# ------------------------------------------------------------ small cases

def _logits(rng, rows, V, ld, dtype):
    x = rng.normal(0, 1, size=(rows, ld)).astype(np.float32)
    return x if dtype == "fp32" else wl.to_bf16_bits(x)


def _plant(rng, x, rows_peaks, V):
    """Put a clear maximum at the given column of each listed row."""
    for row, col in rows_peaks:
        if x.dtype == np.uint16:
            x[row, col] = wl.to_bf16_bits(np.array([9.0], np.float32))[0]
        else:
            x[row, col] = 9.0


@pytest.mark.parametrize("with_argmax", [True, False], ids=["argmax-out", "no-argmax-out"])
@pytest.mark.parametrize("seed", range(40))
def test_greedy_random_small(dev, orc, seed, with_argmax):
    rng = np.random.default_rng(123000 + seed)
    dtype = "fp32" if seed % 2 else "bf16"
    V = int(rng.choice([1024, 1001, 517, 4096, 33, 8, 1]))
    ld = V + int(rng.choice([0, 0, 8, 3, 16]))
    gamma = int(rng.integers(1, 32))
    B = int(rng.integers(1, 24))
    lens = rng.integers(1, gamma + 2, size=B)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    rows = int(cu[-1])
    x = _logits(rng, rows + int(rng.integers(0, 3)), V, ld, dtype)
    draft = rng.integers(0, V, size=(B, gamma)).astype(np.int32)
    # make most target rows agree with the draft so the first mismatch varies
    peaks = []
    for r in range(B):
        for j in range(int(lens[r])):
            if j < gamma and rng.random() < 0.8:
                peaks.append((int(cu[r]) + j, int(draft[r, j])))
    _plant(rng, x, peaks, V)
    prefix = rng.integers(0, 9000, size=B).astype(np.int32)
    g = _gpu_greedy(dev, to_dev_logits(x, dev), V, cu, draft, prefix, with_argmax=with_argmax)
    r = orc.greedy_accept(np.ascontiguousarray(x), V, cu, draft, prefix)
    _cmp_greedy(f"small/{seed}", g, r, rows)


@pytest.mark.parametrize("with_argmax", [True, False], ids=["argmax-out", "no-argmax-out"])
def test_argmax_edge_rows(dev, orc, with_argmax):
    rng = np.random.default_rng(77)
    V, gamma = 129280, 3
    rows = 12
    x = np.zeros((rows, V), np.float32)
    x[0] = 0.0                                        # all equal -> 0
    x[1] = -np.inf                                    # nothing above -inf -> 0
    x[2, :] = -1.0
    x[2, [5000, 70000, 129279]] = 3.0                 # tie far apart -> 5000
    x[3, :] = -1.0
    x[3, 129279] = 2.0                                # max in the last element
    x[4] = rng.normal(size=V)
    x[4, 1234] = np.nan                               # NaN skipped, flagged
    x[4, 99] = 50.0
    x[5, :] = -3.0
    x[5, 17] = -0.0
    x[5, 16] = 0.0                                    # -0 == +0 -> 16
    x[6] = rng.normal(size=V)
    x[6, ::4096] = 40.0                               # ties at many chunk / CTA boundaries
    x[7, :] = np.nan
    x[8] = rng.normal(size=V)
    x[9] = rng.normal(size=V)
    x[9, 64639:64642] = 7.5                           # ties around the middle of the row
    x[10, :] = -1.0
    x[10, 0] = -1.0
    x[11] = rng.normal(size=V)
    cu = np.array([0, 4, 8, 12], np.int32)
    draft = np.zeros((3, gamma), np.int32)
    prefix = np.zeros(3, np.int32)
    for dtype in ("fp32", "bf16"):
        xx = x if dtype == "fp32" else wl.to_bf16_bits(x)
        g = _gpu_greedy(dev, to_dev_logits(xx, dev), V, cu, draft, prefix,
                        with_argmax=with_argmax)
        r = orc.greedy_accept(np.ascontiguousarray(xx), V, cu, draft, prefix)
        _cmp_greedy(f"edge/{dtype}", g, r, rows)
        if with_argmax:
            assert g["argmax"][2] == 5000 and g["argmax"][5] == 16 and g["argmax"][4] == 99
        assert g["status"] & 4


@pytest.mark.parametrize("with_argmax", [True, False], ids=["argmax-out", "no-argmax-out"])
def test_unaligned_and_capacity(dev, orc, with_argmax):
    rng = np.random.default_rng(78)
    V, gamma, B = 3001, 5, 6
    lens = np.array([6, 1, 3, 6, 2, 4])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    draft = rng.integers(0, V, size=(B, gamma)).astype(np.int32)
    draft[2, 1] = V + 5  # out of range -> TOKEN_RANGE
    prefix = rng.integers(0, 100, size=B).astype(np.int32)
    big = wl.to_bf16_bits(rng.normal(size=(cu[-1] + 1, V + 1)).astype(np.float32))
    # a view starting one element in: base not 16-byte aligned -> scalar path
    dev_big = to_dev_logits(big, dev)
    view = dev_big.view(-1)[1:1 + cu[-1] * (V + 1)].view(cu[-1], V + 1)
    host_view = big.reshape(-1)[1:1 + cu[-1] * (V + 1)].reshape(cu[-1], V + 1)
    kw = dict(with_argmax=with_argmax)
    g = _gpu_greedy(dev, view, V, cu, draft, prefix, **kw)
    r = orc.greedy_accept(np.ascontiguousarray(host_view), V, cu, draft, prefix)
    _cmp_greedy("unaligned", g, r, int(cu[-1]))
    # fewer rows available than cu[B]: CAPACITY, requests past them are bad ranges
    g2 = _gpu_greedy(dev, view, V, cu, draft, prefix, max_rows=10, **kw)
    r2 = orc.greedy_accept(np.ascontiguousarray(host_view), V, cu, draft, prefix, max_rows=10)
    _cmp_greedy("capacity", g2, r2, 10)
    assert g2["status"] & 1 and g2["status"] & 16
    # a decreasing cu_seqlens entry is a bad range
    cu_bad = cu.copy()
    cu_bad[3] = cu_bad[2] - 1
    g3 = _gpu_greedy(dev, view, V, cu_bad, draft, prefix, **kw)
    r3 = orc.greedy_accept(np.ascontiguousarray(host_view), V, cu_bad, draft, prefix)
    _cmp_greedy("bad-cu", g3, r3, int(cu_bad[-1]))
    # negative start, empty request, and a request longer than gamma + 1
    for i, cu_b in enumerate(([-1, 6, 7, 10, 16, 18, 22], [0, 6, 6, 9, 15, 17, 21],
                              [0, 6, 7, 10, 20, 21, 22])):
        cu_b = np.array(cu_b, np.int32)
        g4 = _gpu_greedy(dev, view, V, cu_b, draft, prefix, **kw)
        r4 = orc.greedy_accept(np.ascontiguousarray(host_view), V, cu_b, draft, prefix)
        _cmp_greedy(f"bad-cu/{i}", g4, r4, max(int(cu_b[-1]), 0))


@pytest.mark.parametrize("seed", range(16))
def test_cap_random_small(dev, orc, seed):
    rng = np.random.default_rng(321000 + seed)
    dtype = "bf16" if seed % 2 else "fp32"
    V = int(rng.choice([1024, 999, 2048]))
    gamma = int(rng.integers(1, 32))
    B = int(rng.integers(1, 20))
    rows = B * (gamma + 1)
    x = _logits(rng, rows, V, V, dtype)
    draft = rng.integers(0, V, size=(B, gamma)).astype(np.int32)
    peaks = [(r * (gamma + 1) + j, int(draft[r, j])) for r in range(B) for j in range(gamma)
             if rng.random() < 0.85]
    _plant(rng, x, peaks, V)
    lens = rng.integers(1, gamma + 2, size=B).astype(np.int32)
    if seed % 5 == 0:
        lens[0] = gamma + 7  # clamped, BAD_LEN
    prefix = rng.integers(0, 9000, size=B).astype(np.int32)
    g = _gpu_cap(dev, to_dev_logits(x, dev), V, lens, draft, prefix)
    r = orc.cap_accept(np.ascontiguousarray(x), V, lens, draft, prefix)
    np.testing.assert_array_equal(g["argmax"], r.argmax)
    for k in OUT_KEYS + ("ceiling",):
        np.testing.assert_array_equal(g[k], r[k], err_msg=k)
    assert list(g["totals"]) == [r.sum_commit, r.sum_ceiling]
    assert g["status"] == r.status


# ---------------------------------------------------- workloads, full size

def _compact_from_gpu(vs, strided_dev):
    total = int(vs.totals[0].item())
    src = vs.packed_src[:total].long()
    return strided_dev.index_select(0, src).contiguous(), total


@pytest.mark.parametrize("name", ["tiny", "qwen_like", "dsv4_like", "mixed"])
def test_step_workloads_full_size(dev, orc, name):
    """plan -> pack -> compact accept, and cap-accept, at the workload's full
    size with the launch configuration the benchmark uses (VerifyStep)."""
    step = wl.make_step(wl.WORKLOADS[name], seed=0)
    strided = wl.strided_logits(step)
    strided_dev = to_dev_logits(strided, dev)
    vs, g = run_plan_pack(dev, step)
    ref = compare_plan(name, g, oracle_plan(orc, step), step.B, step.gamma,
                       step.workload.min_verify_len, oracle_restage(orc, step))
    p = orc.pack(step.anchor, step.draft, step.prefix_lens, ref.verify_lens, step.tiers,
                 step.capacity)
    compact_dev, total = _compact_from_gpu(vs, strided_dev)
    assert total == p.total
    vs.greedy_accept(compact_dev)
    gg = vs.result()
    compact = strided[p.src[:p.total]]
    rg = orc.greedy_accept(compact, step.V, p.cu_seqlens, step.draft, step.prefix_lens)
    np.testing.assert_array_equal(gg["argmax"][:total], rg.argmax)
    for k in OUT_KEYS:
        np.testing.assert_array_equal(gg[k], rg[k], err_msg=k)
    assert int(gg["status"][0]) == rg.status == 0
    # the benchmark's call: no per-row argmax output
    for t in (vs.num_accepted, vs.bonus, vs.commit_lens, vs.new_seq_lens, vs.out_tokens):
        t.fill_(-9)
    vs.greedy_accept(compact_dev, write_argmax=False)
    gf = vs.result()
    for k in OUT_KEYS:
        np.testing.assert_array_equal(gf[k], rg[k], err_msg="no argmax out: " + k)
    assert int(gf["status"][0]) == 0
    # cap-accept over the strided rows commits the same, and reports the ceiling
    vs.status.zero_()
    vs.cap_accept(strided_dev)
    gc = vs.result()
    rc = orc.cap_accept(strided, step.V, ref.verify_lens, step.draft, step.prefix_lens)
    np.testing.assert_array_equal(gc["argmax"][:step.workload.strided_rows], rc.argmax)
    for k in OUT_KEYS + ("ceiling",):
        np.testing.assert_array_equal(gc[k], rc[k], err_msg=k)
    assert list(gc["cap_totals"]) == [rc.sum_commit, rc.sum_ceiling]
    for k in ("num_accepted", "bonus", "commit_lens", "out_tokens"):
        np.testing.assert_array_equal(gc[k], gg[k], err_msg="compact vs cap " + k)
    assert np.all(gc["ceiling"] >= gc["num_accepted"])


def test_step_is_deterministic(dev):
    """The same step twice gives the same bits; the second time the plan,
    pack and accept run again through VerifyStep.compact_step."""
    step = wl.make_step(wl.DSV4, seed=1)
    strided_dev = to_dev_logits(wl.strided_logits(step), dev)
    outs = []
    for it in range(2):
        vs, _ = run_plan_pack(dev, step)
        compact, _ = _compact_from_gpu(vs, strided_dev)
        if it == 0:
            vs.greedy_accept(compact)
        else:
            for t in (vs.survivals, vs.verify_lens, vs.packed_ids, vs.num_accepted, vs.bonus,
                      vs.commit_lens, vs.new_seq_lens, vs.out_tokens):
                t.fill_(-9)
            vs.compact_step(compact)
        outs.append(vs.result())
    for k in ("survivals", "verify_lens", "tau_theta") + OUT_KEYS:
        np.testing.assert_array_equal(outs[0][k], outs[1][k], err_msg=k)
    padded = int(outs[0]["totals"][1])
    assert int(outs[1]["totals"][1]) == padded
    np.testing.assert_array_equal(outs[0]["packed_ids"][:padded], outs[1]["packed_ids"][:padded])
    assert np.all(outs[1]["packed_ids"][padded:] == -9)  # rows past the padded total untouched
    assert int(outs[1]["status"][0]) == 0


def test_stress_full_size_sampled(dev, orc):
    """B=1024, gamma=16 with the largest forced budget: every planner and pack
    output is compared; the accept runs over all packed rows (4.5 GB of bf16
    at the forced budget) and is compared on sampled requests whose rows come
    from the shared generator (the other rows are filler)."""
    step = wl.make_step(wl.STRESS, seed=0, forced_budget=16384)
    vs, g = run_plan_pack(dev, step)
    ref = compare_plan("stress/16384", g, oracle_plan(orc, step), step.B, step.gamma,
                       step.workload.min_verify_len, oracle_restage(orc, step))
    p = orc.pack(step.anchor, step.draft, step.prefix_lens, ref.verify_lens, step.tiers,
                 step.capacity)
    np.testing.assert_array_equal(g["cu_seqlens"], p.cu_seqlens)
    total = p.total
    V = step.V
    gen = torch.Generator(device=dev).manual_seed(0)
    logits = torch.randn((total, V), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    sample = sorted(set(np.random.default_rng(0).integers(0, step.B, size=24).tolist()) | {0, step.B - 1})
    cu = p.cu_seqlens
    host_rows = {}
    for r in sample:
        rows = wl.target_rows(step, [(r, j) for j in range(int(cu[r + 1] - cu[r]))])
        host_rows[r] = rows
        logits[int(cu[r]):int(cu[r + 1])] = to_dev_logits(rows, dev)
    vs.greedy_accept(logits)
    gg = vs.result()
    for r in sample:
        L = int(cu[r + 1] - cu[r])
        sub = orc.greedy_accept(host_rows[r], V, np.array([0, L], np.int32),
                                step.draft[r:r + 1], step.prefix_lens[r:r + 1])
        np.testing.assert_array_equal(gg["argmax"][cu[r]:cu[r + 1]], sub.argmax)
        for k in OUT_KEYS:
            np.testing.assert_array_equal(gg[k][r], sub[k][0], err_msg=f"r={r} {k}")
    assert int(gg["status"][0]) == 0
    assert int(gg["commit_lens"].min()) >= 1


def test_greedy_accept_reads_pinned_host_logits(dev, orc):
    """The accept over packed logits in pinned host memory (read by the
    kernels through unified addressing) equals the device-memory call."""
    from confidence_scheduled_speculative_gb300 import api
    rng = np.random.default_rng(21)
    B, g, V = 24, 6, 5000
    lens = rng.integers(1, g + 2, size=B)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    rows = int(cu[-1])
    logits = rng.normal(size=(rows, V)).astype(np.float32)
    draft = rng.integers(0, V, size=(B, g)).astype(np.int32)
    for r in range(B):  # plant matches so some chains run long
        for j in range(lens[r] - 1):
            if rng.random() < 0.7:
                logits[cu[r] + j, draft[r, j]] = 9.0
    bf = torch.from_numpy(logits).to(torch.bfloat16)
    outs = []
    for src in (bf.to(dev), bf.pin_memory()):
        i32 = dict(dtype=torch.int32, device=dev)
        o = dict(num_accepted=torch.zeros(B, **i32), bonus=torch.zeros(B, **i32),
                 commit_lens=torch.zeros(B, **i32), out_tokens=torch.zeros((B, g + 1), **i32))
        st = torch.zeros(1, **i32)
        ws = api.workspace(api.dspark_accept_workspace_bytes(rows, V), dev)
        api.dspark_greedy_accept(src, V=V, cu_seqlens=torch.from_numpy(cu).to(dev),
                                 draft=torch.from_numpy(draft).to(dev), prefix_lens=None, B=B,
                                 gamma=g, workspace=ws, status=st, **o)
        torch.cuda.synchronize()
        outs.append({k: v.cpu().numpy() for k, v in o.items()} | {"status": int(st.item())})
    for k in outs[0]:
        np.testing.assert_array_equal(outs[0][k], outs[1][k], err_msg=k)


@pytest.mark.parametrize("name", ["qwen_like", "tiny"])
def test_run_host_end_to_end(dev, orc, name):
    """engine.run_host from pinned host buffers (inputs in one copy, the
    status and outputs back in one copy), with the accept reading the packed
    logits over the host link and with them copied in first: every output
    equals the oracle's plan + pack + greedy accept."""
    from confidence_scheduled_speculative_gb300.engine import (HostStepIO, StepConfig, VerifyStep,
                                                               run_host)
    step = wl.make_step(wl.WORKLOADS[name], seed=3)
    w = step.workload
    ref = oracle_plan(orc, step)
    p = orc.pack(step.anchor, step.draft, step.prefix_lens, ref.verify_lens, step.tiers,
                 step.capacity)
    cu = np.asarray(p.cu_seqlens)
    rows_rj = [(r, j) for r in range(w.B) for j in range(int(cu[r + 1] - cu[r]))]
    host_rows = wl.target_rows(step, rows_rj)
    acc = orc.greedy_accept(host_rows, w.V, cu, step.draft, step.prefix_lens)
    if w.logits_dtype == "fp32":
        host = torch.from_numpy(host_rows)
    else:
        host = torch.from_numpy(host_rows.view(np.int16)).view(torch.bfloat16)
    host = host.pin_memory()
    vs = VerifyStep(StepConfig.from_step(step), dev)
    io = HostStepIO(vs)
    io.fill(step)
    for dev_logits in (None, torch.empty(host.shape, dtype=host.dtype, device=dev)):
        io.out_host.fill_(-7)
        nbytes = run_host(vs, io, host, dev_logits)
        assert nbytes == p.total * host.stride(0) * host.element_size()
        assert int(io.status.item()) == 0
        assert list(io.totals.numpy()) == [p.total, p.padded]
        np.testing.assert_array_equal(io.verify_lens.numpy(), ref.verify_lens)
        np.testing.assert_array_equal(io.out_tokens.numpy(), acc.out_tokens)
        np.testing.assert_array_equal(io.commit_lens.numpy(), acc.commit_lens)
        np.testing.assert_array_equal(io.new_seq_lens.numpy(), acc.new_seq_lens)
