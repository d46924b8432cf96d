"""GPU parity of the data-parallel shared verify tier (dspark_pad_to_tier)
against the oracle, through the C ABI ([AVS] §六: each rank's local verify
tier is gathered and every rank replays the largest; [SGL] "Ragged
verify").  The ranks' MAX all-reduce is host logic, covered with gloo ranks
in test_multirank.py; here one GPU applies given shared tiers to real packs,
and every row of the packed buffers is compared, untouched ones included."""

import numpy as np
import pytest
import torch

from confidence_scheduled_speculative_gb300 import workloads as wl
from gpu_helpers import compare_plan, oracle_plan, oracle_restage, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _packed(vs):
    return {k: getattr(vs, "packed_" + k).cpu().numpy() for k in ("ids", "pos", "req", "src")}


def _case(dev, orc, name, forced, shared, in_place):
    """GPU: plan + pack, then the pad to `shared`.  Oracle: its planner (held
    to the GPU's lens by the staged comparison), its pack over the same
    sentinel-filled buffers, then its pad.  Returns (oracle pack, oracle
    padded result)."""
    from confidence_scheduled_speculative_gb300.engine import StepConfig, VerifyStep
    step = wl.make_step(wl.WORKLOADS[name], seed=4, forced_budget=forced)
    vs = VerifyStep(StepConfig.from_step(step), dev)
    vs.load_inputs(step)
    for t in (vs.packed_ids, vs.packed_pos, vs.packed_req, vs.packed_src):
        t.fill_(-3)
    vs.status.zero_()
    vs.plan_pack()
    g = vs.result()
    exp = compare_plan(f"dp/{name}/{forced}", g, oracle_plan(orc, step), step.B, step.gamma,
                       step.workload.min_verify_len, oracle_restage(orc, step))
    base = orc.pack(step.anchor, step.draft, step.prefix_lens, exp.verify_lens, step.tiers,
                    step.capacity, sentinel=-3)
    assert list(g["totals"]) == [base.total, base.padded]
    vs.status.zero_()
    if in_place:
        vs.totals[1:2].fill_(shared)  # as an in-place all-reduce leaves it
        vs.pad_to_tier()
    else:
        vs.pad_to_tier(torch.tensor([shared], dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    got = _packed(vs)
    ref = orc.pad_to_tier(base, shared, step.capacity)
    for k in ("ids", "pos", "req", "src"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=f"{name} {shared} {k}")
    assert vs.totals.cpu().tolist() == [ref.total, ref.padded]
    assert int(vs.status.item()) == ref.status
    return base, ref


@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("name,forced", [("qwen_like", 40), ("qwen_like", None),
                                          ("dsv4_like", 300), ("dsv4_like", None),
                                          ("stress", 2048)])
def test_pad_to_shared_tier(dev, orc, name, forced, in_place):
    """Shared tiers at and above the rank's own: every tier of the workload
    from its local one up, and the capacity itself."""
    w = wl.WORKLOADS[name]
    step = wl.make_step(w, seed=4, forced_budget=forced)
    tiers = [int(t) for t in step.tiers] or [step.capacity]
    r = orc.plan_step(step)
    local = orc.pack(step.anchor, step.draft, step.prefix_lens, r.verify_lens, step.tiers,
                     step.capacity).padded
    for shared in [t for t in tiers if t >= local] + [step.capacity]:
        base, ref = _case(dev, orc, name, forced, shared, in_place)
        assert ref.padded == shared and ref.status == 0
        assert base.padded == local


def test_pad_to_shared_tier_edges(dev, orc):
    """A shared tier below the rank's real rows (BAD_TIER, nothing written)
    and one above the capacity (pad rows up to the capacity, CAPACITY)."""
    from confidence_scheduled_speculative_gb300 import api
    step = wl.make_step(wl.QWEN, seed=4, forced_budget=40)
    total = int(orc.plan_step(step).verify_lens.sum())
    base, low = _case(dev, orc, "qwen_like", 40, total - 1, False)
    assert low.status == api.STATUS_BAD_TIER and low.padded == base.padded
    _, over = _case(dev, orc, "qwen_like", 40, step.capacity + 100, True)
    assert over.status == api.STATUS_CAPACITY and over.padded == step.capacity + 100
