"""The allocation-free greedy accept (dspark_greedy_accept_static) against the
workspace version (dspark_greedy_accept), through the C ABI.

Some callers cannot allocate device memory -- embeddings that only pass in
buffers they own, runtimes whose device memory is fixed at start-up and that
forbid cudaMalloc afterwards -- so the library offers this variant whose
scratch is a library-owned device array.  Two calls in a row, on inputs of
different sizes, must each match the workspace version exactly (the outputs
are token ids and counts), also when the second call runs over the scratch
the first one left behind.  This file is collected last."""

import numpy as np
import pytest
import torch

from confidence_scheduled_speculative_gb300 import workloads as wl
from gpu_helpers import require_gpu, to_dev_logits

pytestmark = pytest.mark.gpu

KEYS = ("argmax", "num_accepted", "bonus", "commit_lens", "new_seq_lens", "out_tokens", "status")


def _problem(seed, B, gamma, V, dtype):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, gamma + 2, size=B)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    rows = int(cu[-1])
    x = rng.normal(0, 1, size=(rows, V)).astype(np.float32)
    draft = rng.integers(0, V, size=(B, gamma)).astype(np.int32)
    for r in range(B):
        for j in range(min(int(lens[r]), gamma)):
            if rng.random() < 0.8:
                x[cu[r] + j, draft[r, j]] = 9.0
    if dtype == "bf16":
        x = wl.to_bf16_bits(x)
    prefix = rng.integers(1, 8192, size=B).astype(np.int32)
    return x, cu, draft, prefix


def _run(dev, fn, x, cu, draft, prefix, V, with_ws, max_rows=None):
    from confidence_scheduled_speculative_gb300 import api
    B, g = draft.shape
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    i32 = dict(dtype=torch.int32, device=dev)
    logits = to_dev_logits(x, dev)
    rows = logits.size(0)
    out = dict(num_accepted=torch.full((B,), -5, **i32), bonus=torch.full((B,), -5, **i32),
               commit_lens=torch.full((B,), -5, **i32), new_seq_lens=torch.full((B,), -5, **i32),
               out_tokens=torch.full((B, g + 1), -5, **i32), argmax=torch.full((rows,), -5, **i32))
    status = torch.zeros(1, **i32)
    kw = dict(V=V, cu_seqlens=t(cu), draft=t(draft), prefix_lens=t(prefix), B=B, gamma=g,
              status=status, **out)
    if max_rows is not None:
        kw["max_rows"] = max_rows
    if with_ws:
        kw["workspace"] = api.workspace(api.dspark_accept_workspace_bytes(rows, V), dev)
    fn(logits, **kw)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["status"] = int(status.item())
    return res


def test_static_scratch_matches_workspace_version_twice():
    dev = require_gpu()
    from confidence_scheduled_speculative_gb300 import api
    cases = [(11, 96, 16, 129280, "bf16"), (12, 13, 7, 4099, "fp32")]
    problems = [(_problem(seed, B, gamma, V, dtype), V) for seed, B, gamma, V, dtype in cases]
    refs = [_run(dev, api.dspark_greedy_accept, *p, V, with_ws=True) for p, V in problems]
    # two calls in a row on the shared scratch, the second over what the first left
    gots = [_run(dev, api.dspark_greedy_accept_static, *p, V, with_ws=False) for p, V in problems]
    for i, (got, ref) in enumerate(zip(gots, refs)):
        for k in KEYS:
            np.testing.assert_array_equal(got[k], ref[k], err_msg=f"call {i}: {k}")


def test_static_scratch_rejects_rows_beyond_its_maximum():
    dev = require_gpu()
    from confidence_scheduled_speculative_gb300 import api
    x, cu, draft, prefix = _problem(3, 2, 3, 64, "fp32")
    logits = to_dev_logits(x, dev)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    z = lambda *s: torch.zeros(*s, dtype=torch.int32, device=dev)
    with pytest.raises(api.DsparkError) as e:
        api.dspark_greedy_accept_static(
            logits, V=64, cu_seqlens=t(cu), draft=t(draft), prefix_lens=t(prefix), B=2, gamma=3,
            num_accepted=z(2), bonus=z(2), commit_lens=z(2), out_tokens=z(2, 4), status=z(1),
            max_rows=api.STATIC_MAX_ROWS + 1)
    assert e.value.code == api.DSPARK_ERR_UNSUPPORTED


def test_static_scratch_clamps_device_rows_above_max_rows():
    """cu_seqlens[B] above max_rows: both versions clamp the rows to max_rows,
    flag DSPARK_STATUS_CAPACITY, leave the argmax of later rows untouched and
    give the requests past the clamp no acceptance (BAD_LEN), identically."""
    dev = require_gpu()
    from confidence_scheduled_speculative_gb300 import api
    x, cu, draft, prefix = _problem(21, 40, 8, 20000, "bf16")
    max_rows = int(cu[-1]) - 13
    ref = _run(dev, api.dspark_greedy_accept, x, cu, draft, prefix, 20000, True, max_rows)
    got = _run(dev, api.dspark_greedy_accept_static, x, cu, draft, prefix, 20000, False,
               max_rows)
    for k in KEYS:
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    assert got["status"] & api.STATUS_CAPACITY and got["status"] & api.STATUS_BAD_LEN
    assert np.all(got["argmax"][max_rows:] == -5) and np.all(got["argmax"][:max_rows] >= 0)
    cut = int(np.searchsorted(cu, max_rows, side="right")) - 1  # first request past the clamp
    assert np.all(got["num_accepted"][cut:] == 0) and np.all(got["bonus"][cut:] == -1)
