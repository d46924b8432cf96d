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


def restage(orc, z, T, eps, min_len, max_len, forced, kind, M, val, bias=0.0, alpha=0.0,
            **options):
    """The oracle's planner steps after the survivals (order, tau, theta,
    budget, lens; with ``options``, the composition of ``orc.plan_ex``) as a
    function of given survivals: ``restage(...)(s)`` plans on ``s`` in place
    of the survivals the oracle would compute from z."""
    def run(s):
        return orc.plan_ex(z, T, eps, min_len, max_len, forced, kind, M, val, bias, alpha,
                           survivals=s, **options)
    return run


def compare_plan(tag, gpu: dict, ref, B: int, gamma: int, min_len: int, restaged):
    """Staged, bit-exact planner parity.

    When the GPU's survivals equal the oracle's bit for bit, verify_lens,
    budget, tau and theta must equal ``ref``.  When some survival differs in
    its last bit (the fp64 sigmoid landing on the other side of an fp32
    rounding boundary; logged as a near tie, at most 1e-6 apart), the
    oracle's later steps are rerun on the GPU's own survivals
    (``restaged(survivals)``, see ``restage``) and the GPU's outputs must
    equal that result bit for bit: the order, tau, theta, budget and lens are
    defined exactly from whatever survivals they are given ([AVS] §一).

    Returns the oracle result the outputs were held to; the stages after the
    planner (the pack, the status word) are checked against it."""
    sg, so = gpu["survivals"], ref.survivals
    exp = ref
    if not np.array_equal(sg.view(np.uint32), so.view(np.uint32)):
        diff = float(np.max(np.abs(sg.astype(np.float64) - so.astype(np.float64))))
        assert diff <= 1e-6, (tag, "survivals differ by", diff)
        idx = np.argwhere(sg.view(np.uint32) != so.view(np.uint32))
        log_near_tie({"tag": tag, "elements": idx[:8].tolist(), "max_abs_diff": diff})
        exp = restaged(sg)
    np.testing.assert_array_equal(gpu["verify_lens"], exp.verify_lens, err_msg=f"{tag} lens")
    assert int(gpu["budget"][0]) == exp.budget, (tag, int(gpu["budget"][0]), exp.budget)
    assert gpu["tau_theta"][0] == exp.tau, (tag, gpu["tau_theta"][0], exp.tau)
    assert gpu["tau_theta"][1] == exp.theta, (tag, gpu["tau_theta"][1], exp.theta)
    return exp


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


def oracle_restage(orc, step, forced=None):
    w, c = step.workload, step.cost
    fb = w.forced_budget if forced is None else forced
    return restage(orc, step.conf_logits, step.sts_temps, w.survival_eps, w.min_verify_len,
                   w.max_len, fb, c.kind, c.M, c.val, c.bias_ms, c.alpha_ms)
