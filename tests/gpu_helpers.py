"""Shared helpers of the GPU parity tests: run the CUDA path through the
C-ABI binding and the oracle on the same seeded inputs, compare."""

import json
import os
import warnings

import numpy as np
import torch

from confidence_scheduled_speculative_gb300 import workloads as wl

NEAR_TIE_LOG = os.environ.get("DSPARK_NEAR_TIE_LOG")


def require_gpu():
    assert torch.cuda.is_available(), "the gpu-marked tests need a CUDA device"
    from confidence_scheduled_speculative_gb300 import api, build
    build.build()
    api.load()
    return torch.device("cuda:0")


def to_dev_logits(arr: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bits or float32 -> device tensor of the same bits."""
    if arr.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(device)


def log_near_tie(record: dict) -> None:
    warnings.warn(f"near tie: {record}")
    if NEAR_TIE_LOG:
        with open(NEAR_TIE_LOG, "a") as f:
            f.write(json.dumps(record) + "\n")


def compare_plan(tag, gpu: dict, ref, B: int, gamma: int, min_len: int) -> bool:
    """Bit-exact planner parity.  Returns False (after logging) when the
    survivals differ in the last bit (an fp64 exp rounding to the other side
    of an fp32 boundary), in which case the discrete outputs are checked for
    validity instead of equality."""
    sg, so = gpu["survivals"], ref.survivals
    if np.array_equal(sg.view(np.uint32), so.view(np.uint32)):
        np.testing.assert_array_equal(gpu["verify_lens"], ref.verify_lens, err_msg=f"{tag} lens")
        assert int(gpu["budget"][0]) == ref.budget, (tag, int(gpu["budget"][0]), ref.budget)
        assert gpu["tau_theta"][0] == ref.tau, (tag, gpu["tau_theta"][0], ref.tau)
        assert gpu["tau_theta"][1] == ref.theta, (tag, gpu["tau_theta"][1], ref.theta)
        return True
    diff = float(np.max(np.abs(sg.astype(np.float64) - so.astype(np.float64))))
    assert diff <= 1e-6, (tag, "survivals differ by", diff)
    idx = np.argwhere(sg.view(np.uint32) != so.view(np.uint32))
    log_near_tie({"tag": tag, "elements": idx[:8].tolist(), "max_abs_diff": diff})
    assert abs(float(gpu["tau_theta"][0]) - ref.tau) <= 1e-6 * max(1.0, ref.tau) + 1e-6 * B * gamma
    lens = gpu["verify_lens"]
    assert lens.min() >= min_len
    return False


def run_plan_pack(device, step, forced=None):
    """GPU planner + pack on a workloads.StepInputs; returns (VerifyStep, host results)."""
    from confidence_scheduled_speculative_gb300.engine import StepConfig, VerifyStep
    cfg = StepConfig.from_step(step)
    if forced is not None:
        cfg.forced_budget = forced
    vs = VerifyStep(cfg, device)
    vs.load_inputs(step)
    vs.status.zero_()
    vs.plan()
    vs.pack()
    return vs, vs.result()


def oracle_plan(orc, step, forced=None):
    w, c = step.workload, step.cost
    fb = w.forced_budget if forced is None else forced
    return orc.plan(step.conf_logits, step.sts_temps, w.survival_eps, w.min_verify_len,
                    w.max_len, fb, c.kind, c.M, c.val, c.bias_ms, c.alpha_ms)
