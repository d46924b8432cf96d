"""The bounds-checked build on the GPU.

libdspark_checked.so is the library compiled with -DDSPARK_CHECKED: every
index a kernel computes from data (packed rows, ranks, prefix-sum and table
positions, histogram bins, partial slots, recorder slots) is tested against
the extent of the buffer it addresses before the access, and one outside it
sets DSPARK_STATUS_OUT_OF_BOUNDS instead of being used.  A child process
started with DSPARK_CHECKED=1 runs checked_scenarios.py on it; this process
runs the same calls on the normal library.  Every output must be equal bit
for bit, and no status word of either may carry the out-of-bounds bit."""

import os
import subprocess
import sys

import numpy as np
import pytest

from conftest import ROOT
from gpu_helpers import require_gpu

pytestmark = pytest.mark.gpu


def test_checked_build_matches_and_flags_nothing(tmp_path):
    dev = require_gpu()
    from confidence_scheduled_speculative_gb300 import api
    from confidence_scheduled_speculative_gb300 import build as _b
    import checked_scenarios

    if api.dspark_checked_build():
        pytest.skip("this process already runs the checked library (DSPARK_CHECKED=1): "
                    "there is no normal build to compare with")
    _b.build(checked=True)
    path = str(tmp_path / "checked.npz")
    env = dict(os.environ, DSPARK_CHECKED="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_scenarios.py"), path],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert p.returncode == 0, p.stdout[-2000:] + p.stderr[-4000:]
    normal = checked_scenarios.scenarios(dev)
    with np.load(path) as f:
        checked = {k: f[k] for k in f.files}
    assert sorted(checked) == sorted(normal)
    assert len(normal) > 300
    statuses = [k for k in normal if k.endswith("/status")]
    assert len(statuses) > 40
    for k in statuses:
        for build, res in (("normal", normal), ("checked", checked)):
            assert not int(res[k].ravel()[0]) & api.STATUS_OUT_OF_BOUNDS, (build, k)
    diff = [k for k in normal
            if normal[k].shape != checked[k].shape or normal[k].tobytes() != checked[k].tobytes()]
    assert not diff, diff[:20]
