"""Layout of the step arena that the end-to-end path moves with one copy each
way (inputs and a zero status word in, the status and outputs out): every
piece 16-byte aligned, no two pieces overlapping, the status word the last
word copied in and the first copied out.  Host-only (CPU tensors)."""

import pytest
import torch

from confidence_scheduled_speculative_gb300 import engine


@pytest.mark.parametrize("B,g", [(1, 1), (4, 3), (32, 8), (256, 16), (1024, 31)])
def test_step_arena_layout(B, g):
    arena, views, n_in, out_lo = engine._arena(B, g, "cpu")
    base = arena.data_ptr()
    spans = []
    for name, v in views.items():
        off = v.data_ptr() - base
        assert off % 16 == 0, name
        assert v.is_contiguous(), name
        spans.append((off, off + v.numel() * v.element_size(), name))
    spans.sort()
    for (a0, a1, na), (b0, b1, nb) in zip(spans, spans[1:]):
        assert a1 <= b0, (na, nb)
    assert spans[-1][1] <= arena.numel() * 4
    status = views["status"].data_ptr() - base
    assert out_lo * 4 == status and n_in == out_lo + 1
    for name in ("conf_logits", "sts_temps", "anchor", "draft", "prefix_lens"):
        assert views[name].data_ptr() - base < status, name
    for name in ("totals", "out_tokens", "commit_lens", "new_seq_lens", "verify_lens"):
        assert views[name].data_ptr() - base > status, name
    assert views["conf_logits"].dtype == torch.float32 and views["draft"].dtype == torch.int32
    assert tuple(views["out_tokens"].shape) == (B, g + 1)


def test_select_path_limit_matches_kernel():
    """The step's launch count follows the planner's dispatch: the binding's
    select-path table limit is the kernel source's."""
    import os
    import re

    from confidence_scheduled_speculative_gb300 import api
    src = os.path.join(os.path.dirname(api.__file__), "csrc", "plan.cu")
    with open(src) as f:
        m = re.search(r"constexpr int kMaxSelect = (\d+);", f.read())
    assert m is not None
    assert api.SELECT_MAX_ENTRIES == int(m.group(1))
    with open(src) as f:
        text = f.read()
    stage = re.search(r"constexpr int kStage = (\d+);", text)
    assert "constexpr int kDenseMaxEntries = (kStage * 4 - 16) / 16;" in text
    assert api.DENSE_MAX_ENTRIES == (int(stage.group(1)) * 4 - 16) // 16
    interp = re.search(r"constexpr int kInterpMaxSamples = (\d+);", text)
    assert api.INTERP_MAX_SAMPLES == int(interp.group(1))


def test_binding_planner_paths():
    """api.planner_path restates plan.cu's routing (the select path's table
    limit is checked against the kernel source above)."""
    from confidence_scheduled_speculative_gb300 import api
    assert api.planner_path(4096, api.COST_ADDITIVE, 5) == "select"
    assert api.planner_path(4096, api.COST_SPS_1D, 31) == "select"
    assert api.planner_path(4096, api.COST_SPS_1D, 32) == "dense"
    assert api.planner_path(4096, api.COST_SPS_1D, 4097) == "dense"
    assert api.planner_path(4096, api.COST_ADDITIVE, api.DENSE_MAX_ENTRIES) == "dense"
    assert api.planner_path(16384, api.COST_SPS_1D, api.DENSE_MAX_ENTRIES + 1) == "rank"
    assert api.planner_path(64, api.COST_ADDITIVE_INTERP, 5) == "interp"
    assert api.planner_path(4096, api.COST_ADDITIVE_INTERP, api.INTERP_MAX_SAMPLES) == "interp"
    assert api.planner_path(4096, api.COST_ADDITIVE_INTERP, api.INTERP_MAX_SAMPLES + 1) == "rank"
