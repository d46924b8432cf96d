"""GPU parity of the speculative sampling accept (dspark_sampling_accept)
against the oracle, through the C ABI.

Decisions are compared exactly.  The GPU sums exps in fp32 per thread and
fp64 beyond (the oracle in fp64, index order) and the two sides call
different exp implementations, so p and q differ at about 1e-6 relative: a
decision may differ only where it sits that close to its threshold.  Every
request whose outputs differ is checked to be such a case (the margin of the
first differing decision, evaluated independently in fp64 here, is below
1e-5 relative) and logged; everything else must match."""

import numpy as np
import pytest
import torch

from confidence_scheduled_speculative_gb300 import workloads as wl
from gpu_helpers import log_near_tie, require_gpu, to_dev_logits

pytestmark = pytest.mark.gpu

KEYS = ("num_accepted", "bonus", "commit_lens", "new_seq_lens", "out_tokens")
REL = 1e-5


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _gpu_sampling(dev, tgt, dft, V, cu, draft, prefix, ua, ub, max_rows=None, draft_lse=None):
    from confidence_scheduled_speculative_gb300 import api
    B, g = draft.shape
    t = lambda a, d=np.int32: torch.from_numpy(np.ascontiguousarray(a, dtype=d)).to(dev)
    i32 = dict(dtype=torch.int32, device=dev)
    rows_cap = tgt.shape[0] if max_rows is None else max_rows
    o = dict(num_accepted=torch.full((B,), -5, **i32), bonus=torch.full((B,), -5, **i32),
             commit_lens=torch.full((B,), -5, **i32), new_seq_lens=torch.full((B,), -5, **i32),
             out_tokens=torch.full((B, g + 1), -5, **i32))
    st = torch.zeros(1, **i32)
    ws = api.workspace(api.dspark_sampling_workspace_bytes(rows_cap, B, g), dev)
    api.dspark_sampling_accept(to_dev_logits(tgt, dev), to_dev_logits(dft, dev), V=V,
                               cu_seqlens=t(cu), draft=t(draft), prefix_lens=t(prefix), B=B,
                               gamma=g, u_accept=t(ua, np.float32), u_bonus=t(ub, np.float32),
                               workspace=ws, status=st, max_rows=rows_cap,
                               draft_lse=None if draft_lse is None else t(draft_lse, np.float32), **o)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in o.items()}
    res["status"] = int(st.item())
    return res


def _f32(x):
    x = np.ascontiguousarray(x)
    return (x.astype(np.uint32) << 16).view(np.float32) if x.dtype == np.uint16 else x.astype(np.float32)


def _probs(row, V):
    z = _f32(row[:V]).astype(np.float64)
    ok = ~np.isnan(z)
    m = z[ok].max() if ok.any() else -np.inf
    e = np.where(ok, np.exp(z - m), 0.0)
    return e / e.sum() if e.sum() > 0 else e


def _near_boundary(r, got, ref, tgt, dft, V, cu, draft, ua, ub):
    """True when request r's first differing decision is within REL of its
    threshold (fp64 evaluation, independent of both implementations)."""
    g = draft.shape[1]
    lo, hi = int(cu[r]), int(cu[r + 1])
    L = hi - lo
    for j in range(L - 1):
        x = int(draft[r, j])
        inside = 0 <= x < V
        p = _probs(tgt[lo + j], V)[x] if inside else 0.0
        q = _probs(dft[r * g + j], V)[x] if inside else 0.0
        lhs = float(ua[r, j]) * q
        accept = lhs < p
        gpu_acc = got["num_accepted"][r] > j
        ref_acc = ref.num_accepted[r] > j
        if gpu_acc != ref_acc:
            return abs(lhs - p) <= REL * max(p, lhs, 1e-300)
        if not accept:
            break
    c = int(ref.num_accepted[r])
    if int(got["num_accepted"][r]) != c:
        return False
    p = _probs(tgt[lo + c], V)
    w = np.maximum(p - _probs(dft[r * g + c], V), 0.0) if c < L - 1 else p
    if w.sum() <= 0:
        w = p
    C = np.cumsum(w)
    target = float(ub[r]) * C[-1]
    a, b = sorted((int(got["bonus"][r]), int(ref.bonus[r])))
    edges = [C[a], C[b - 1] if b > 0 else 0.0]
    return min(abs(e - target) for e in edges) <= REL * C[-1]


def _compare(tag, got, ref, tgt, dft, V, cu, draft, ua, ub):
    B = draft.shape[0]
    bad = [r for r in range(B) if any(
        not np.array_equal(np.asarray(got[k])[r], np.asarray(ref[k])[r]) for k in KEYS)]
    for r in bad:
        assert _near_boundary(r, got, ref, tgt, dft, V, cu, draft, ua, ub), (tag, r)
        log_near_tie({"tag": f"sampling/{tag}", "request": r})
    assert len(bad) <= max(1, B // 50), (tag, bad)
    assert got["status"] == ref.status, (tag, got["status"], ref.status)


def _problem(rng, B, g, V, dtype, accept_bias=1.0, ld_pad=0):
    """Target rows ~ N(0, 2) with a peak; draft rows = target + noise (the
    closer, the more drafts pass); drafts drawn from q; uniforms."""
    lens = rng.integers(1, g + 2, size=B)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    rows = int(cu[-1])
    tgt = np.zeros((max(rows, 1), V + ld_pad), np.float32)
    dft = np.zeros((B * g, V + ld_pad), np.float32)
    draft = np.zeros((B, g), np.int32)
    for r in range(B):
        for j in range(g):
            base = rng.normal(0, 2, V).astype(np.float32)
            base[rng.integers(0, V)] += 6
            d = base + rng.normal(0, accept_bias, V).astype(np.float32)
            dft[r * g + j, :V] = d
            if j < lens[r]:
                tgt[cu[r] + j, :V] = base
            q = np.exp(d.astype(np.float64) - d.max())
            draft[r, j] = rng.choice(V, p=q / q.sum())
        if lens[r] == g + 1:
            tgt[cu[r] + g, :V] = rng.normal(0, 2, V)
    if dtype == "bf16":
        tgt, dft = wl.to_bf16_bits(tgt), wl.to_bf16_bits(dft)
    prefix = rng.integers(0, 9000, B).astype(np.int32)
    ua = rng.random((B, g)).astype(np.float32)
    ub = rng.random(B).astype(np.float32)
    return tgt, dft, cu, draft, prefix, ua, ub


@pytest.mark.parametrize("seed", range(24))
def test_sampling_random(dev, orc, seed):
    rng = np.random.default_rng(8100 + seed)
    dtype = "bf16" if seed % 2 == 0 else "fp32"
    V = int(rng.choice([33, 1000, 4099, 8, 20000]))
    g = int(rng.integers(1, 9))
    B = int(rng.integers(1, 20))
    pad = int(rng.choice([0, 0, 3, 8]))
    tgt, dft, cu, draft, prefix, ua, ub = _problem(rng, B, g, V, dtype, float(rng.choice([0.05, 0.5, 2.0])), pad)
    got = _gpu_sampling(dev, tgt, dft, V, cu, draft, prefix, ua, ub)
    ref = orc.sampling_accept(tgt, V, cu, dft, draft, prefix, ua, ub)
    _compare(f"random/{seed}", got, ref, tgt, dft, V, cu, draft, ua, ub)


@pytest.mark.parametrize("B", [80, 100, 120, 160, 220])
def test_sampling_cluster_splits(dev, orc, B):
    """Batch sizes whose bonus draws are split over 7, 6, 5, 3 and 2 CTAs
    per request on a 152-SM GPU (the split is floor(4 * SMs / B), 1..8):
    the integer round sums make the draw independent of the split."""
    rng = np.random.default_rng(9300 + B)
    V, g = 4099, 4
    tgt, dft, cu, draft, prefix, ua, ub = _problem(rng, B, g, V, "bf16", 0.5)
    got = _gpu_sampling(dev, tgt, dft, V, cu, draft, prefix, ua, ub)
    ref = orc.sampling_accept(tgt, V, cu, dft, draft, prefix, ua, ub)
    _compare(f"split/{B}", got, ref, tgt, dft, V, cu, draft, ua, ub)


def _lse_rows(dft, V):
    """log(sum exp(z)) of every draft row in fp64 (NaN weighs 0), as fp32:
    what the drafting step's sampler hands over."""
    z = _f32(dft[:, :V]).astype(np.float64)
    z = np.where(np.isnan(z), -np.inf, z)
    m = z.max(axis=1)
    ok = np.isfinite(m)
    s = np.exp(z - np.where(ok, m, 0.0)[:, None]).sum(axis=1)
    return np.where(ok, m + np.log(np.where(ok, s, 1.0)), -np.inf).astype(np.float32)


@pytest.mark.parametrize("seed", range(8))
def test_sampling_with_draft_normalizers(dev, orc, seed):
    """dspark_sampling_accept_ex: with each draft row's log-sum-exp supplied
    the draft rows are not normalised by the library; the decisions equal
    the oracle's (which normalises them itself) up to its near-tie
    tolerance."""
    rng = np.random.default_rng(8700 + seed)
    dtype = "bf16" if seed % 2 == 0 else "fp32"
    V = int(rng.choice([33, 1000, 4099, 20000]))
    g = int(rng.integers(1, 9))
    B = int(rng.choice([3, 17, 90]))
    tgt, dft, cu, draft, prefix, ua, ub = _problem(rng, B, g, V, dtype, float(rng.choice([0.05, 0.5])))
    got = _gpu_sampling(dev, tgt, dft, V, cu, draft, prefix, ua, ub, draft_lse=_lse_rows(dft, V))
    ref = orc.sampling_accept(tgt, V, cu, dft, draft, prefix, ua, ub)
    _compare(f"lse/{seed}", got, ref, tgt, dft, V, cu, draft, ua, ub)


def test_sampling_edge_cases(dev, orc):
    rng = np.random.default_rng(77)
    V, g, B = 1000, 4, 6
    tgt, dft, cu, draft, prefix, ua, ub = _problem(rng, B, g, V, "fp32", 0.3)
    # equal distributions for request 0: every draft passes
    lo = int(cu[0])
    for j in range(int(cu[1] - cu[0]) - 1):
        dft[0 * g + j] = tgt[lo + j]
    # a NaN in a target row and an out-of-range draft token
    tgt[int(cu[2]), 17] = np.nan
    draft[3, 0] = V + 4
    got = _gpu_sampling(dev, tgt, dft, V, cu, draft, prefix, ua, ub)
    ref = orc.sampling_accept(tgt, V, cu, dft, draft, prefix, ua, ub)
    _compare("edge", got, ref, tgt, dft, V, cu, draft, ua, ub)
    assert got["num_accepted"][0] == cu[1] - cu[0] - 1
    assert got["status"] & 4 and got["status"] & 2
    # p == q with the draft token at -inf in both: rejected (0 < 0 fails),
    # the residual is empty, the bonus is drawn from p
    r1 = next(r for r in range(B) if r != 3 and cu[r + 1] - cu[r] >= 2)
    t2, d2 = tgt.copy(), dft.copy()
    lo1 = int(cu[r1])
    d2[r1 * g] = t2[lo1]
    x = int(draft[r1, 0])
    t2[lo1, x] = -np.inf
    d2[r1 * g, x] = -np.inf
    got2 = _gpu_sampling(dev, t2, d2, V, cu, draft, prefix, ua, ub)
    ref2 = orc.sampling_accept(t2, V, cu, d2, draft, prefix, ua, ub)
    _compare("empty-residual", got2, ref2, t2, d2, V, cu, draft, ua, ub)
    assert got2["num_accepted"][r1] == 0 and got2["bonus"][r1] >= 0
    # bad ranges and fewer rows than cu[B]
    cu_bad = cu.copy()
    cu_bad[2] = cu_bad[1]
    got3 = _gpu_sampling(dev, tgt, dft, V, cu_bad, draft, prefix, ua, ub)
    ref3 = orc.sampling_accept(tgt, V, cu_bad, dft, draft, prefix, ua, ub)
    _compare("bad-cu", got3, ref3, tgt, dft, V, cu_bad, draft, ua, ub)
    assert got3["bonus"][1] == -1 and got3["status"] & 16
    got4 = _gpu_sampling(dev, tgt, dft, V, cu, draft, prefix, ua, ub, max_rows=int(cu[3]))
    ref4 = orc.sampling_accept(tgt, V, cu, dft, draft, prefix, ua, ub, max_rows=int(cu[3]))
    _compare("capacity", got4, ref4, tgt, dft, V, cu, draft, ua, ub)
    assert got4["status"] & 1


def test_sampling_first_token_is_distributed_as_p(dev):
    """With drafts drawn from q, the first committed token follows p
    (chi-square over 4 x 4096 requests), as for the oracle."""
    rng = np.random.default_rng(34)
    V, B = 5, 4096
    p = np.array([0.35, 0.05, 0.3, 0.2, 0.1])
    q = np.array([0.1, 0.4, 0.1, 0.25, 0.15])
    lp, lq = np.log(p).astype(np.float32), np.log(q).astype(np.float32)
    tgt = np.tile(lp, (2 * B, 1))
    dft = np.tile(lq, (B, 1))
    cu = np.arange(0, 2 * B + 1, 2, dtype=np.int32)
    counts = np.zeros(V)
    for _ in range(4):
        draft = rng.choice(V, size=(B, 1), p=q).astype(np.int32)
        got = _gpu_sampling(dev, tgt, dft, V, cu, draft, np.zeros(B), rng.random((B, 1)), rng.random(B))
        counts += np.bincount(got["out_tokens"][:, 0], minlength=V)
    n = counts.sum()
    chi2 = float(((counts - n * p) ** 2 / (n * p)).sum())
    assert chi2 < 20.5, (chi2, counts / n)


def test_sampling_dsv4_like_full_size(dev, orc):
    """B=256, gamma=16, V=129280 bf16 with the planner's lengths: every
    request runs on the GPU; 12 sampled requests are rebuilt as a small
    problem for the oracle (a request's outputs depend only on its rows)."""
    from gpu_helpers import run_plan_pack
    step = wl.make_step(wl.DSV4, seed=0)
    vs, g_plan = run_plan_pack(dev, step)
    cu = g_plan["cu_seqlens"]
    B, g, V = step.B, step.gamma, step.V
    rows = int(cu[-1])
    gen = torch.Generator(device=dev).manual_seed(5)
    tgt_dev = (torch.randn((rows, V), generator=gen, device=dev) * 2).to(torch.bfloat16)
    dft_dev = (tgt_dev[:1].float().repeat(B * g, 1) * 0).to(torch.bfloat16)
    # draft rows: the target row of the same depth plus noise, so that drafts pass often
    for r in range(B):
        lo, hi = int(cu[r]), int(cu[r + 1])
        n = hi - lo - 1
        if n > 0:
            noise = torch.randn((n, V), generator=gen, device=dev) * 0.3
            dft_dev[r * g:r * g + n] = (tgt_dev[lo:lo + n].float() + noise).to(torch.bfloat16)
    rng = np.random.default_rng(6)
    # drafts drawn from q on the device (a seeded generator)
    draft = np.zeros((B, g), np.int32)
    gen2 = torch.Generator(device=dev).manual_seed(7)
    for r in range(B):
        n = int(cu[r + 1] - cu[r]) - 1
        if n > 0:
            q = torch.softmax(dft_dev[r * g:r * g + n].float(), dim=1)
            draft[r, :n] = torch.multinomial(q, 1, generator=gen2).squeeze(1).cpu().numpy()
    ua = rng.random((B, g)).astype(np.float32)
    ub = rng.random(B).astype(np.float32)
    from confidence_scheduled_speculative_gb300 import api
    t = lambda a, d=np.int32: torch.from_numpy(np.ascontiguousarray(a, dtype=d)).to(dev)
    i32 = dict(dtype=torch.int32, device=dev)
    o = dict(num_accepted=torch.zeros(B, **i32), bonus=torch.zeros(B, **i32),
             commit_lens=torch.zeros(B, **i32), new_seq_lens=torch.zeros(B, **i32),
             out_tokens=torch.zeros((B, g + 1), **i32))
    st = torch.zeros(1, **i32)
    ws = api.workspace(api.dspark_sampling_workspace_bytes(rows, B, g), dev)
    api.dspark_sampling_accept(tgt_dev, dft_dev, V=V, cu_seqlens=t(cu), draft=t(draft),
                               prefix_lens=vs.prefix_lens, B=B, gamma=g, u_accept=t(ua, np.float32),
                               u_bonus=t(ub, np.float32), workspace=ws, status=st, **o)
    torch.cuda.synchronize()
    got = {k: v.cpu().numpy() for k, v in o.items()}
    assert int(st.item()) == 0
    assert np.all(got["num_accepted"] <= np.diff(cu) - 1) and np.all(got["bonus"] >= 0)
    sample = sorted(set(rng.integers(0, B, 10).tolist()) | {0, B - 1})
    tgt_bits = tgt_dev.view(torch.int16).cpu().numpy().view(np.uint16)
    dft_bits = dft_dev.view(torch.int16).cpu().numpy().view(np.uint16)
    prefix = step.prefix_lens
    sub_cu, sub_t, sub_d = [0], [], []
    for r in sample:
        lo, hi = int(cu[r]), int(cu[r + 1])
        sub_t.append(tgt_bits[lo:hi])
        sub_d.append(dft_bits[r * g:(r + 1) * g])
        sub_cu.append(sub_cu[-1] + hi - lo)
    sub_t, sub_d = np.concatenate(sub_t), np.concatenate(sub_d)
    sub_cu = np.array(sub_cu, np.int32)
    ref = orc.sampling_accept(sub_t, V, sub_cu, sub_d, draft[sample], prefix[sample], ua[sample], ub[sample])
    sub_got = {k: got[k][sample] for k in KEYS}
    sub_got["status"] = ref.status
    _compare("dsv4", sub_got, ref, sub_t, sub_d, V, sub_cu, draft[sample], ua[sample], ub[sample])


def test_sampling_residual_mass_threshold(dev, orc):
    """The empty-residual cut-off on the GPU, on the oracle pin's hand case
    (V = 2, residual masses 2^-19 and 2^-21 on the two sides of 2^-20): the
    larger residual is drawn from (bonus 0), the smaller one is read as
    empty and the bonus is drawn from p (u_bonus 0.75 -> token 1)."""
    b = np.array([-(2.0 ** -17), -(2.0 ** -19)], np.float32)
    tgt = np.zeros((4, 2), np.float32)
    dft = np.stack([[b[0], 0.0], [b[1], 0.0]]).astype(np.float32)
    cu = np.array([0, 2, 4], np.int32)
    draft = np.array([[1], [1]], np.int32)
    ua = np.full((2, 1), np.float32(1.0 - 2.0 ** -24), np.float32)
    for ub, want in ((0.75, [0, 1]), (0.25, [0, 0])):
        ubv = np.full(2, ub, np.float32)
        got = _gpu_sampling(dev, tgt, dft, 2, cu, draft, np.zeros(2), ua, ubv)
        ref = orc.sampling_accept(tgt, 2, cu, dft, draft, np.zeros(2), ua, ubv)
        assert got["num_accepted"].tolist() == [0, 0] and ref.num_accepted.tolist() == [0, 0]
        assert got["bonus"].tolist() == want == ref.bonus.tolist()
        assert got["status"] == 0
