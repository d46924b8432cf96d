"""GPU parity of ScatterCompactToStrided (dspark_scatter_compact_to_strided)
against the oracle's row copy, through the C ABI: the whole strided buffer is
compared byte for byte, so rows the scatter must not touch (pad rows, rows
no request selected) are checked too."""

import numpy as np
import pytest
import torch

from confidence_scheduled_speculative_gb300 import workloads as wl
from gpu_helpers import require_gpu, run_plan_pack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def _scatter(dev, src_np, src_of, total, dst_np, torch_dtype, max_rows=None, dst_ld=None):
    from confidence_scheduled_speculative_gb300 import api
    t32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    ints = np.int16 if src_np.itemsize == 2 else np.int32
    src = torch.from_numpy(np.ascontiguousarray(src_np).view(ints)).to(dev).view(torch_dtype)
    dst_full = torch.from_numpy(np.ascontiguousarray(dst_np).view(ints)).to(dev).view(torch_dtype)
    dst = dst_full if dst_ld is None else dst_full[:, :dst_ld]
    if max_rows is not None:
        src = src[:max_rows]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    src_of_full = np.full(max(src.size(0), len(src_of)), -1, np.int32)
    src_of_full[:len(src_of)] = src_of
    api.dspark_scatter_compact_to_strided(src, t32(src_of_full), t32([total]), dst, status=st)
    torch.cuda.synchronize()
    return dst_full.cpu().view(torch.int16 if src_np.itemsize == 2 else torch.int32).numpy(), int(st.item())


@pytest.mark.parametrize("seed", range(24))
def test_scatter_random(dev, orc, seed):
    rng = np.random.default_rng(5150 + seed)
    B, g = int(rng.integers(1, 40)), int(rng.integers(1, 32))
    lens = rng.integers(1, g + 2, size=B).astype(np.int32)
    p = orc.pack(np.zeros(B), np.zeros((B, g)), np.zeros(B), lens, [], B * (g + 1))
    dtype = [np.uint16, np.uint32][seed % 2]
    torch_dtype = [torch.bfloat16, torch.float32][seed % 2]
    width = int(rng.choice([1, 7, 8, 64, 1000, 4096 + 3]))
    src = rng.integers(0, 2 ** 15, size=(p.total, width)).astype(dtype)
    dst = rng.integers(0, 2 ** 15, size=(B * (g + 1), width + int(rng.choice([0, 8, 5])))).astype(dtype)
    got, st = _scatter(dev, src, p.src[:p.total], p.total, dst, torch_dtype)
    ref, rst = orc.scatter_rows(src, p.src[:p.total], p.total, dst)
    np.testing.assert_array_equal(got, ref.view(got.dtype))
    assert st == rst == 0


def test_scatter_bad_index_and_clamped_total(dev, orc):
    rng = np.random.default_rng(7)
    src = rng.integers(0, 1000, size=(6, 16)).astype(np.uint16)
    dst = np.zeros((5, 16), np.uint16)
    src_of = np.array([4, 9, -2, 0, 1, 3], np.int32)
    got, st = _scatter(dev, src, src_of, 6, dst, torch.bfloat16)
    ref, rst = orc.scatter_rows(src, src_of, 6, dst)
    np.testing.assert_array_equal(got, ref.view(got.dtype))
    assert st == rst == orc.ST_BAD_INDEX
    # totals above the rows available: only max_rows rows are copied
    got2, st2 = _scatter(dev, src, src_of[[0, 3, 4, 5, 1, 2]], 50, dst, torch.bfloat16, max_rows=3)
    ref2, rst2 = orc.scatter_rows(src[:3], src_of[[0, 3, 4, 5, 1, 2]], 50, dst, max_rows=3)
    np.testing.assert_array_equal(got2, ref2.view(got2.dtype))
    assert st2 == rst2 == 0


def test_scatter_workload_full_size(dev, orc):
    """dsv4_like: the packed rows' logits (2048 x 129280 bf16) back into the
    4352-row strided buffer; compared on every selected row and on a sample of
    untouched rows."""
    step = wl.make_step(wl.DSV4, seed=0)
    vs, g = run_plan_pack(dev, step)
    total = int(g["totals"][0])
    V = step.V
    gen = torch.Generator(device=dev).manual_seed(3)
    compact = torch.randn((vs.packed_src.numel(), V), generator=gen, device=dev).to(torch.bfloat16)
    strided = torch.full((step.B * (step.gamma + 1), V), -7.0, device=dev, dtype=torch.bfloat16)
    from confidence_scheduled_speculative_gb300 import api
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dspark_scatter_compact_to_strided(compact, vs.packed_src, vs.totals, strided, status=st)
    torch.cuda.synchronize()
    src = vs.packed_src[:total].long()
    assert torch.equal(strided.index_select(0, src), compact[:total])
    mask = torch.ones(strided.size(0), dtype=torch.bool, device=dev)
    mask[src] = False
    assert bool((strided[mask] == -7.0).all()) and int(st.item()) == 0


def test_scatter_gives_up_and_returns(dev, orc):
    """Failure detection without a fault: with the pipeline wait limited to 0
    (one test per wait) the TMA path's first wait finds its copy still in
    flight, gives up, flags DSPARK_STATUS_TIMEOUT, lets its in-flight copies
    land and returns.  The context stays usable: the same call with the
    default limit, and with a long explicit one, then matches the oracle."""
    from confidence_scheduled_speculative_gb300 import api
    rng = np.random.default_rng(17)
    B, g, width = 24, 7, 24576  # 48 KB bf16 rows: three 16 KB segments each
    lens = rng.integers(1, g + 2, size=B).astype(np.int32)
    p = orc.pack(np.zeros(B), np.zeros((B, g)), np.zeros(B), lens, [], B * (g + 1))
    src_np = rng.integers(0, 2 ** 15, size=(p.total, width)).astype(np.uint16)
    dst_np = rng.integers(0, 2 ** 15, size=(B * (g + 1), width)).astype(np.uint16)
    t32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    src = torch.from_numpy(src_np.view(np.int16)).to(dev).view(torch.bfloat16)
    src_of, totals = t32(p.src[:p.total]), t32([p.total])
    ref, _ = orc.scatter_rows(src_np, p.src[:p.total], p.total, dst_np)
    for limit, want in ((0, api.STATUS_TIMEOUT), (None, 0), (10 ** 10, 0)):
        dst = torch.from_numpy(dst_np.view(np.int16)).to(dev).view(torch.bfloat16)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        api.dspark_scatter_compact_to_strided(src, src_of, totals, dst, status=st,
                                              wait_limit_ns=limit)
        torch.cuda.synchronize()
        assert int(st.item()) == want, (limit, int(st.item()))
        if want == 0:
            np.testing.assert_array_equal(dst.cpu().view(torch.int16).numpy(), ref.view(np.int16))
