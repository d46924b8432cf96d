"""Benchmark of the DSpark verify hot path on GB300: plan + pack + greedy
accept steps/s at B=256, gamma=16, V=129280 (bf16 target logits), compact
mode, and the accept kernel's HBM bandwidth against the measured peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  Under torchrun every rank runs its own batch
of B requests (weak scaling); the one exchange per step is the MAX
all-reduce of the ranks' verify tiers, after which each rank pads its window
to the shared tier (dspark_pad_to_tier).  The elapsed time is the maximum
over ranks.

A step = dspark_plan + dspark_pack_verify + dspark_greedy_accept over one
batch, with every input resident in HBM when the timed region starts.  The
target logits of the packed rows (~2048 rows x 129280 x 2 B = 529 MB) are
larger than the 129 MB L2, so each step streams them from HBM.  ``e2e``
times the same step through ``engine.run_host``: inputs from pinned host
memory and the packed rows' logits read by the accept straight from a pinned
host buffer over the link, results read back; ``e2e.copy_then_accept`` is
the variant that reads the packed total back first and copies that many
rows in before the accept.

--impl reference times the CPU oracle (the reference arm: the pages print
no runnable implementation) on the host cores with the same metric and
workload.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "plan+pack+accept steps/s at B=256 gamma=16 V=129280; accept HBM GB/s % of peak"
UNIT = "steps/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dsv4_like")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-cap", action="store_true")
    ap.add_argument("--separate-plan-pack", action="store_true",
                    help="issue dspark_plan and dspark_pack_verify instead of dspark_plan_pack")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the stress row sweep, the qwen_like cold-L2 step and the mixed report")
    ap.add_argument("--no-calib", action="store_true",
                    help="skip the calibration (recorder, statistics, fit) measurements")
    ap.add_argument("--event-every", type=int, default=16,
                    help="bracket the accept call with events on every n-th timed step")
    ap.add_argument("--out", default=None, help="also append the JSON line to this file")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def ncu_traffic(workload: str):
    """Per-launch DRAM bytes (read + write) of the accept kernel from the
    committed ncu summary, or None when no capture exists for this workload
    or the kernel sources changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not d:
        return None
    h = hashlib.sha256()
    for rel in ("csrc/accept.cu", "csrc/logits.cuh", "csrc/dspark_common.cuh",
                "csrc/sigmoid.cuh"):
        with open(os.path.join(ROOT, "confidence_scheduled_speculative_gb300", rel), "rb") as f:
            h.update(f.read())
    return d["bytes_per_launch"] if h.hexdigest() == d.get("sources_sha256") else None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.strip().split(",") for ln in self.file if ln.strip()]
        os.unlink(self.file.name)
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                power.append(float(r[3]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def oracle_step_timing(step, compact, budget_s, max_steps=None, row_fraction=1.0):
    """Time the CPU oracle on the workload: the full planner and pack, and
    the accept over a sample of the packed rows.  Returns the full-step rate
    estimated as 1 / (t_plan_pack + rows * t_per_row)."""
    import oracle
    oracle.build()
    w = step.workload
    rows = compact.shape[0]
    n_rows = max(1, int(round(rows * row_fraction)))
    t_pp, t_acc, rows_done, steps = 0.0, 0.0, 0, 0
    start = time.perf_counter()
    cursor = 0
    while True:
        t0 = time.perf_counter()
        r = oracle.plan_step(step)
        p = oracle.pack(step.anchor, step.draft, step.prefix_lens, r.verify_lens, step.tiers,
                        step.capacity)
        t1 = time.perf_counter()
        # n_rows consecutive packed rows from the cursor, wrapping around at
        # the end: every step samples the same number of rows
        lo = cursor % rows
        hi = lo + n_rows
        full_am = np.zeros(rows, np.int32)
        am, _ = oracle.argmax_rows(compact[lo:min(hi, rows)], V=w.V)
        full_am[lo:min(hi, rows)] = am
        if hi > rows:
            am2, _ = oracle.argmax_rows(compact[:hi - rows], V=w.V)
            full_am[:hi - rows] = am2
        oracle.greedy_finalize(full_am, rows, p.cu_seqlens, step.draft, step.prefix_lens, w.V)
        t2 = time.perf_counter()
        cursor = hi % rows
        t_pp += t1 - t0
        t_acc += t2 - t1
        rows_done += n_rows
        steps += 1
        if time.perf_counter() - start >= budget_s or (max_steps and steps >= max_steps):
            break
    per_step = t_pp / steps + rows * (t_acc / rows_done)
    return {"value": 1.0 / per_step, "steps": steps, "t_plan_pack_ms": 1e3 * t_pp / steps,
            "t_accept_row_us": 1e6 * t_acc / rows_done, "rows_sampled": rows_done,
            "elapsed_s": time.perf_counter() - start}


def make_inputs(name: str, seed: int):
    from confidence_scheduled_speculative_gb300 import workloads as wl
    step = wl.make_step(wl.WORKLOADS[name], seed=seed)
    strided = wl.strided_logits(step)  # [B*(gamma+1), V] bf16 bits
    return step, strided


# Arm Ltd. (implementer 0x41) part numbers of the server cores this may run on
ARM_PARTS = {0xd0c: "Neoverse-N1", 0xd40: "Neoverse-V1", 0xd49: "Neoverse-N2",
             0xd4f: "Neoverse-V2", 0xd84: "Neoverse-V3", 0xd8e: "Neoverse-N3"}


def cpu_info():
    """Host CPU: the x86 model name, else lscpu's model name, else the Arm
    part number named from ARM_PARTS."""
    model, part, impl = None, None, None
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key, _, val = ln.partition(":")
                key, val = key.strip().lower(), val.strip()
                if key in ("model name", "processor name") and model is None:
                    model = val
                elif key == "cpu part" and part is None:
                    part = val
                elif key == "cpu implementer" and impl is None:
                    impl = val
    except OSError:
        pass
    if model is None:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for ln in out.splitlines():
                if ln.lower().startswith("model name:"):
                    model = ln.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    if (model is None or model.startswith("-")) and part is not None:
        try:
            name = ARM_PARTS.get(int(part, 16)) if impl in (None, "0x41") else None
        except ValueError:
            name = None
        model = name or f"cpu part {part}"
    return {"nproc": os.cpu_count(), "model": model}


# ---------------------------------------------------------------- reference

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from confidence_scheduled_speculative_gb300 import workloads as wl
    step = wl.make_step(wl.WORKLOADS[args.workload], seed=args.seed)
    import oracle
    r = oracle.plan_step(step)
    p = oracle.pack(step.anchor, step.draft, step.prefix_lens, r.verify_lens, step.tiers,
                    step.capacity)
    rows = [(int(s) // (step.gamma + 1), int(s) % (step.gamma + 1)) for s in p.src[:p.total]]
    compact = wl.target_rows(step, rows)
    # bound the whole run to about two minutes: each timed step processes the
    # planner, the pack and a slice of the packed rows
    k = max(1, args.steps)
    est = oracle_step_timing(step, compact, budget_s=3.0)
    full_step_s = 1.0 / est["value"]
    per_step_budget = min(full_step_s, 120.0 / (k + max(3, args.warmup)))
    frac = max(1.0 / compact.shape[0],
               min(1.0, (per_step_budget - est["t_plan_pack_ms"] / 1e3) / max(full_step_s, 1e-9)))
    oracle_step_timing(step, compact, budget_s=0.0, max_steps=max(3, args.warmup),
                       row_fraction=frac)
    res = oracle_step_timing(step, compact, budget_s=1e9, max_steps=k, row_fraction=frac)
    sample = (f"{res['steps']} oracle steps: full planner + pack each step, accept over "
              f"{res['rows_sampled']} of {compact.shape[0]}*{res['steps']} packed rows "
              f"(fraction {frac:.4f} per step); full-step rate = 1/(t_plan_pack + rows*t_row)")
    line = {
        "impl": "reference", "metric": METRIC, "value": res["value"], "unit": UNIT,
        "n_gpus": args.gpus, "steps": res["steps"], "warmup": max(3, args.warmup),
        "ms_per_step": 1e3 / res["value"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload} B={step.B} gamma={step.gamma} V={step.V} compact",
                   "seed": args.seed},
        "cpu_baseline": {"value": res["value"], "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, "host": cpu_info()},
        "e2e": {"value": res["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    emit(line, args)


def max_over_ranks(x: float, dev, world: int) -> float:
    """The largest x over the ranks: the job's time is its slowest rank's."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput: every rank processes its own units (weak
    scaling, no data exchanged), all within the slowest rank's time."""
    return world * units_per_rank / seconds


def rank_seed(seed: int, rank: int) -> int:
    """Each rank draws its own requests (an independent data-parallel shard)."""
    return seed + rank


def emit(line, args):
    s = json.dumps(line)
    print(s, flush=True)
    if args.out:
        with open(args.out, "a") as f:
            f.write(s + "\n")


# --------------------------------------------------------------------- ours

CAL_N, CAL_GAMMA, CAL_TEMPS, CAL_BINS = 262144, 16, 64, 15


def plan_kind_timing(dev, stream, vs, kind, reps=32, table=None):
    """GPU time of one dspark_plan call (survival + planner pass) with the
    step's cost table (or `table` = (M, val) tensors) read as `kind`: 32
    calls captured in a CUDA graph."""
    import torch
    from confidence_scheduled_speculative_gb300 import api as _api
    c = vs.cfg
    cM, cval = (vs.cost_M, vs.cost_val) if table is None else table
    out = {}

    def call():
        _api.dspark_plan(vs.conf_logits, vs.sts_temps, B=c.B, gamma=c.gamma,
                         survival_eps=c.survival_eps, min_verify_len=c.min_verify_len,
                         max_verify_len=c.max_verify_len, forced_budget=c.forced_budget,
                         cost_kind=kind, cost_M=cM, cost_val=cval,
                         bias_ms=c.bias_ms, alpha_ms=c.alpha_ms, survivals=vs.survivals,
                         verify_lens=vs.verify_lens, budget=vs.budget, tau_theta=vs.tau_theta,
                         status=vs.status, workspace=vs.plan_ws)

    try:
        for _ in range(3):
            call()
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=gs):
            for _ in range(reps):
                call()
        torch.cuda.synchronize()
        cg.replay()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record(stream)
        for _ in range(5):
            cg.replay()
        ev[1].record(stream)
        torch.cuda.synchronize()
        out["us"] = ev[0].elapsed_time(ev[1]) * 1e3 / (5 * reps)
        out["budget"] = int(vs.budget.item())
        out["status"] = int(vs.status.item())
    except Exception as e:  # report, do not fail the run
        out["error"] = f"{type(e).__name__}: {e}"[:200]
    return out


def accept_rows_sweep(dev, stream, seed, reps=20):
    """Accept bandwidth against the packed row count on the stress workload
    (B=1024, gamma=16, V=129280): forced budgets 0..16384 step 1024 give
    1024..17408 packed rows (0.26..4.5 GB of bf16, every point larger than
    L2).  Per point: the real planner + pack with that forced budget, then
    the accept calls back to back over filler logits (N(0,1) bf16; the
    argmax results are not checked here, the parity tests do that)."""
    import torch
    from confidence_scheduled_speculative_gb300 import workloads as wl
    from confidence_scheduled_speculative_gb300.engine import StepConfig, VerifyStep
    w = wl.STRESS
    peak = load_peaks()[0]
    out = {"workload": f"stress B={w.B} gamma={w.gamma} V={w.V} compact, forced budgets",
           "points": []}
    try:
        buf = torch.empty((w.B * (w.gamma + 1), w.V), dtype=torch.bfloat16, device=dev)
        buf.normal_(generator=torch.Generator(device=dev).manual_seed(seed))
        for f in range(0, w.B * w.gamma + 1, 1024):
            step = wl.make_step(w, seed=seed, forced_budget=f)
            vs = VerifyStep(StepConfig.from_step(step), dev)
            vs.load_inputs(step)
            vs.plan_pack()
            torch.cuda.synchronize()
            total = int(vs.totals[0].item())
            _, _, _, acc_fn = vs.bind_compact(buf[:total])
            for _ in range(3):
                acc_fn()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            ev[0].record(stream)
            for _ in range(reps):
                acc_fn()
            ev[1].record(stream)
            torch.cuda.synchronize()
            us = ev[0].elapsed_time(ev[1]) * 1e3 / reps
            nbytes = total * w.V * w.elem_bytes
            gbs = nbytes / (us * 1e-6) / 1e9
            out["points"].append({"forced_budget": f, "rows": total, "accept_us": us,
                                  "gbs": gbs, "frac": gbs / peak,
                                  "status": int(vs.status.item())})
            del vs
        del buf
    except Exception as e:  # report, do not fail the run
        out["error"] = f"{type(e).__name__}: {e}"[:200]
    return out


def mixed_cap_report(dev, n_steps=200):
    """The mixed-traffic report of cap-accept (B=128, gamma=12, three
    acceptance classes, 1-D SPS table): over independent steps (seeds
    0..n_steps-1, no state carried) the planner's tau at its budget (the
    expected commit under calibrated confidences), the delivered commit
    sum(min(raw, len - 1) + 1) and the ceiling sum(raw + 1) of verifying
    every depth, overall and per class (request r has class r mod 3, match
    probability 0.9 / 0.6 / 0.3 per depth): a class's tau is the number of
    its requests plus its selected survivals.  The target rows follow the
    workload recipe -- N(0,1) with a +8 peak at the draft token with the
    row's match probability, else at another uniform token -- drawn on the
    device (a statistical report: the rows are not the shared generator's
    bits)."""
    import torch
    from confidence_scheduled_speculative_gb300 import workloads as wl
    from confidence_scheduled_speculative_gb300.engine import StepConfig, VerifyStep
    w = wl.MIXED
    out = {"workload": f"mixed B={w.B} gamma={w.gamma} V={w.V} cap-accept, 1-D SPS table",
           "steps": n_steps, "seeds": f"0..{n_steps - 1}"}
    try:
        rows = w.B * (w.gamma + 1)
        logits = torch.empty((rows, w.V), dtype=torch.bfloat16, device=dev)
        gen = torch.Generator(device=dev)
        cls = np.arange(w.B) % 3
        names = ("p0.9", "p0.6", "p0.3")
        acc = {k: np.zeros(3) for k in ("tau", "delivered", "ceiling", "rows")}
        budget = 0
        for seed in range(n_steps):
            step = wl.make_step(w, seed=seed)
            rng = np.random.default_rng(np.random.SeedSequence([7919, seed]))
            peak = rng.integers(0, w.V - 1, size=(w.B, w.gamma + 1))
            d = step.draft.astype(np.int64)
            other = peak[:, :w.gamma] + (peak[:, :w.gamma] >= d)
            hit = rng.random((w.B, w.gamma)) < step.match_prob
            peak[:, :w.gamma] = np.where(hit, d, other)
            gen.manual_seed(seed)
            logits.normal_(generator=gen)
            flat = torch.from_numpy(peak.reshape(-1)).to(dev)
            logits[torch.arange(rows, device=dev), flat] += wl.PEAK
            vs = VerifyStep(StepConfig.from_step(step), dev)
            vs.load_inputs(step)
            vs.plan()
            vs.cap_accept(logits, write_argmax=False)
            lens = vs.verify_lens.cpu().numpy().astype(np.int64)
            s = vs.survivals.cpu().numpy().astype(np.float64)
            commit = vs.commit_lens.cpu().numpy().astype(np.int64)
            raw = vs.ceiling.cpu().numpy().astype(np.int64)
            sel = np.arange(w.gamma)[None, :] < (lens - 1)[:, None]  # selected candidates
            tau_r = 1.0 + (s * sel).sum(axis=1)
            for c in range(3):
                m = cls == c
                acc["tau"][c] += tau_r[m].sum()
                acc["delivered"][c] += commit[m].sum()
                acc["ceiling"][c] += (raw[m] + 1).sum()
                acc["rows"][c] += lens[m].sum()
            budget += int(vs.budget.item())
            out["status"] = out.get("status", 0) | int(vs.status.item())
        n_cls = np.bincount(cls, minlength=3)
        per = {}
        for c in range(3):
            per[names[c]] = {
                "requests": int(n_cls[c]),
                "mean_verify_len": acc["rows"][c] / (n_steps * n_cls[c]),
                "mean_tau": acc["tau"][c] / n_steps,
                "mean_delivered": acc["delivered"][c] / n_steps,
                "mean_ceiling": acc["ceiling"][c] / n_steps,
                "delivered_over_ceiling": acc["delivered"][c] / acc["ceiling"][c],
                "delivered_over_tau": acc["delivered"][c] / acc["tau"][c]}
        tau, deliv, ceil = (acc[k].sum() for k in ("tau", "delivered", "ceiling"))
        out.update({"mean_budget": budget / n_steps, "mean_tau": tau / n_steps,
                    "mean_delivered": deliv / n_steps, "mean_ceiling": ceil / n_steps,
                    "delivered_over_ceiling": deliv / ceil, "delivered_over_tau": deliv / tau,
                    "per_class": per})
        del logits
    except Exception as e:  # report, do not fail the run
        out["error"] = f"{type(e).__name__}: {e}"[:200]
    return out


def configs_report(dev, stream, seed, reps=20, e2e_reps=10):
    """Every workload's step through the same calls: packed rows, the device
    step (plan + pack + greedy accept, back to back), the planner alone, and
    end-to-end steps/s through engine.run_host (inputs from pinned host
    buffers, the accept reading the packed logits over the host link).  The
    target logits are N(0,1) filler of the packed rows' shape (timing only;
    the parity tests check values); stress runs at its largest forced
    budget."""
    import torch
    from confidence_scheduled_speculative_gb300 import workloads as wl
    from confidence_scheduled_speculative_gb300.engine import (HostStepIO, StepConfig,
                                                               VerifyStep, run_host)
    out = {}
    for name in ("tiny", "qwen_like", "dsv4_like", "mixed", "stress"):
        try:
            w = wl.WORKLOADS[name]
            step = wl.make_step(w, seed=seed, forced_budget=w.B * w.gamma if name == "stress" else None)
            vs = VerifyStep(StepConfig.from_step(step), dev)
            vs.load_inputs(step)
            vs.plan_pack()
            torch.cuda.synchronize()
            total = int(vs.totals[0].item())
            dt = torch.float32 if w.logits_dtype == "fp32" else torch.bfloat16
            logits = torch.empty((max(total, 1), w.V), dtype=dt, device=dev)
            logits.normal_(generator=torch.Generator(device=dev).manual_seed(seed))
            plan_pack_fn, plan_fn, _, acc_fn = vs.bind_compact(logits)

            def timed(fn, n):
                for _ in range(3):
                    fn()
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                ev[0].record(stream)
                for _ in range(n):
                    fn()
                ev[1].record(stream)
                torch.cuda.synchronize()
                return ev[0].elapsed_time(ev[1]) * 1e3 / n

            step_us = timed(lambda: (plan_pack_fn(), acc_fn()), reps)
            plan_us = timed(plan_fn, reps)
            io = HostStepIO(vs)
            io.fill(step)
            host = torch.empty(logits.shape, dtype=dt).pin_memory()
            host.copy_(logits)
            for _ in range(2):
                run_host(vs, io, host, None)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(e2e_reps):
                run_host(vs, io, host, None)
            e2e = e2e_reps / (time.perf_counter() - t0)
            out[name] = {"B": w.B, "gamma": w.gamma, "V": w.V, "rows": total,
                         "step_us": step_us, "plan_us": plan_us, "e2e_steps_per_s": e2e,
                         "accept_gbs_in_step": total * w.V * w.elem_bytes / (step_us * 1e-6) / 1e9,
                         "status": int(vs.status.item()) | int(io.status.item())}
            del logits, host, vs, io
        except Exception as e:  # report, do not fail the run
            out[name] = {"error": f"{type(e).__name__}: {e}"[:200]}
    return out


def small_step_timing(dev, stream, name, seed, reps=48, copies=4):
    """plan + pack + accept step time of a workload whose logits fit in L2
    (qwen_like: 256 packed rows x 151936 bf16 = 77.8 MB).  Each timed step
    reads its own copy of the packed logits, rotating over `copies` copies
    (311 MB together, more than twice L2), so each step's accept streams its
    rows from HBM; only the step is bracketed by events.  For comparison, the
    same step after rewriting a 256 MB buffer before every step (that flush
    leaves L2 full of dirty lines, which the accept's reads then write back)."""
    import torch
    from confidence_scheduled_speculative_gb300.engine import StepConfig, VerifyStep
    out = {}
    try:
        step, strided = make_inputs(name, seed)
        w = step.workload
        vs = VerifyStep(StepConfig.from_step(step), dev)
        vs.load_inputs(step)
        vs.plan_pack()
        torch.cuda.synchronize()
        total = int(vs.totals[0].item())
        strided_dev = torch.from_numpy(strided.view(np.int16)).to(dev).view(torch.bfloat16)
        compact = strided_dev.index_select(0, vs.packed_src[:total].long()).contiguous()
        bufs = [compact] + [compact.clone() for _ in range(copies - 1)]
        fns = [vs.bind_compact(b) for b in bufs]
        nbytes = total * w.V * w.elem_bytes

        def timed(flush):
            for i in range(3):
                fns[i % copies][0]()
                fns[i % copies][3]()
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
            for i, e in enumerate(evs):
                plan_pack_fn, _, _, acc_fn = fns[0] if flush is not None else fns[i % copies]
                if flush is not None:
                    flush.fill_(1)
                e[0].record(stream)
                plan_pack_fn()
                e[1].record(stream)
                acc_fn()
                e[2].record(stream)
            torch.cuda.synchronize()
            step_us = np.array([e[0].elapsed_time(e[2]) for e in evs]) * 1e3
            acc_us = np.array([e[1].elapsed_time(e[2]) for e in evs]) * 1e3
            return float(np.median(step_us)), float(np.median(acc_us))

        step_p50, acc_p50 = timed(None)
        # accept calls back to back over the rotating copies (each call's rows
        # are still cold: the three other copies were read since): the
        # per-call cost once launches overlap, as inside a pipelined step
        n_b2b = 64
        for i in range(copies):
            fns[i][3]()
        eb = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        eb[0].record(stream)
        for i in range(n_b2b):
            fns[i % copies][3]()
        eb[1].record(stream)
        torch.cuda.synchronize()
        b2b_us = eb[0].elapsed_time(eb[1]) * 1e3 / n_b2b
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        f_step, f_acc = timed(flush)
        del flush
        out = {"workload": f"{w.name} B={w.B} gamma={w.gamma} V={w.V} compact",
               "rows": total,
               "l2": f"{copies} copies of the packed logits ({copies * nbytes / 1e6:.0f} MB) in rotation",
               "step_us_p50": step_p50, "accept_us_p50": acc_p50,
               "accept_gbs": nbytes / (acc_p50 * 1e-6) / 1e9,
               "accept_frac": nbytes / (acc_p50 * 1e-6) / 1e9 / load_peaks()[0],
               "accept_back_to_back_cold": {"us": b2b_us, "calls": n_b2b,
                                            "gbs": nbytes / (b2b_us * 1e-6) / 1e9,
                                            "frac": nbytes / (b2b_us * 1e-6) / 1e9 / load_peaks()[0]},
               "with_l2_write_flush": {"step_us_p50": f_step, "accept_us_p50": f_acc,
                                       "accept_gbs": nbytes / (f_acc * 1e-6) / 1e9},
               "status": int(vs.status.item())}
    except Exception as e:  # report, do not fail the run
        out["error"] = f"{type(e).__name__}: {e}"[:200]
    return out


def calibration_timing(dev, stream, vs, w, K):
    """Recorder, statistics and fit timings (CUDA events on the stream)."""
    import torch
    from confidence_scheduled_speculative_gb300 import api as _api
    from confidence_scheduled_speculative_gb300 import workloads as wl
    out = {}
    i32 = dict(dtype=torch.int32, device=dev)
    cap_rows = 1 << 16
    rz = torch.zeros((cap_rows, w.gamma), dtype=torch.float32, device=dev)
    rc = torch.zeros(cap_rows, **i32)
    rt = torch.zeros(cap_rows, **i32)
    cur = torch.zeros(1, dtype=torch.int64, device=dev)
    st = torch.zeros(1, **i32)
    mask = torch.zeros((w.B, w.gamma), dtype=torch.uint8, device=dev)

    def rec():
        _api.dspark_sts_record(vs.conf_logits, num_correct=vs.num_accepted, B=w.B,
                               gamma=w.gamma, rec_logits=rz, rec_correct=rc, rec_tested=rt,
                               cursor=cur, status=st, verify_lens=vs.verify_lens,
                               prefix_mask=mask)

    def timed(fn, n):
        for _ in range(3):
            fn()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        torch.cuda.synchronize()
        ev[0].record(stream)
        for _ in range(n):
            fn()
        ev[1].record(stream)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) * 1e3 / n

    out["record_us_stream"] = timed(rec, min(K, 200))
    # GPU time per call: 64 calls captured in one CUDA graph (the device
    # cursor makes the recorder capturable), replayed
    try:
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=gs):
            for _ in range(64):
                rec()
        torch.cuda.synchronize()
        out["record_us"] = timed(cg.replay, 10) / 64
    except Exception as e:  # report, do not fail the run
        out["record_us"] = None
        out["record_graph_error"] = f"{type(e).__name__}: {e}"[:200]
    out["record_rows_per_call"] = w.B
    cs = wl.calibration_samples(CAL_N, CAL_GAMMA, 1.0 + 0.05 * np.arange(CAL_GAMMA), seed=2026)
    z = torch.from_numpy(cs.conf_logits).to(dev)
    cor = torch.from_numpy(cs.correct).to(dev)
    tst = torch.from_numpy(cs.tested).to(dev)
    T = torch.ones(CAL_GAMMA, dtype=torch.float32, device=dev)
    met = torch.zeros((2, CAL_GAMMA, 4), dtype=torch.float64, device=dev)
    ws_s = _api.workspace(_api.dspark_calibration_workspace_bytes(CAL_GAMMA, CAL_BINS), dev)

    def stats():
        _api.dspark_calibration_stats(z, rec_correct=cor, rec_tested=tst, N=CAL_N,
                                      gamma=CAL_GAMMA, sts_temps=T, n_bins=CAL_BINS, metrics=met,
                                      workspace=ws_s, status=st)

    grid = wl.temperature_grid(CAL_TEMPS)
    T_fit = torch.zeros(CAL_GAMMA, dtype=torch.float32, device=dev)
    choice = torch.zeros(CAL_GAMMA, **i32)
    ws_f = _api.workspace(_api.dspark_sts_fit_workspace_bytes(CAL_N, CAL_TEMPS, CAL_BINS), dev)

    def fit():
        _api.dspark_sts_fit(z, rec_correct=cor, rec_tested=tst, N=CAL_N, gamma=CAL_GAMMA,
                            temp_grid=grid, n_bins=CAL_BINS, sts_temps_out=T_fit, choice=choice,
                            workspace=ws_f, status=st)

    s_us = timed(stats, 20)
    f_us = timed(fit, 5)
    # sigmoids the fit evaluates: every (sample, candidate) at each depth the
    # sample's window reached, plus one per sample and depth for S
    reached = int(np.minimum(cs.tested, CAL_GAMMA).sum())
    evals = reached * (CAL_TEMPS + 1)
    out.update({
        "samples": CAL_N, "gamma": CAL_GAMMA, "temps": CAL_TEMPS, "bins": CAL_BINS,
        "stats_us": s_us, "stats_samples_per_s": CAL_N / (s_us * 1e-6),
        "fit_us": f_us, "fit_sigmoids": evals, "fit_sigmoids_per_s": evals / (f_us * 1e-6),
        "fit_T": [float(x) for x in T_fit.cpu().tolist()],
        "status": int(st.item()),
    })
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    from confidence_scheduled_speculative_gb300 import api
    from confidence_scheduled_speculative_gb300 import build as _b
    from confidence_scheduled_speculative_gb300.engine import (HostStepIO, StepConfig, VerifyStep,
                                                               run_host)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    _b.build()
    api.load()

    step, strided = make_inputs(args.workload, rank_seed(args.seed, rank))
    w = step.workload
    vs = VerifyStep(StepConfig.from_step(step), dev)
    vs.load_inputs(step)
    vs.plan()
    vs.pack()
    torch.cuda.synchronize()
    total, padded = (int(x) for x in vs.totals.cpu())
    strided_dev = torch.from_numpy(strided.view(np.int16)).to(dev).view(torch.bfloat16)
    compact = strided_dev.index_select(0, vs.packed_src[:total].long()).contiguous()
    accept_bytes = total * w.V * w.elem_bytes

    plan_pack_fn, plan_fn, pack_fn, acc_fn = vs.bind_compact(compact)
    stream = torch.cuda.current_stream()

    if args.separate_plan_pack:
        def plan_pack_fn():
            plan_fn()
            pack_fn()

    if world > 1:
        # data-parallel ranks replay one verify tier: after each rank's plan
        # + pack, the MAX all-reduce of the local tiers (one int32, NCCL, on
        # the stream) and the pad to the shared tier
        local_plan_pack = plan_pack_fn

        def plan_pack_fn():
            local_plan_pack()
            vs.share_tier()

    def one_step():
        plan_pack_fn()
        acc_fn()

    warm = max(3, args.warmup)
    vs.status.zero_()

    # ---- timed region: K steps, bracketed by two events and nothing else
    # inside (an event between two steps would keep the next step's first
    # kernel from launching while the previous step finishes)
    K = max(1, args.steps)
    every = max(1, args.event_every)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    sampler.start()  # (waits 0.3 s for nvidia-smi to start: before the warm-up, so the GPU stays busy)
    for _ in range(warm):
        one_step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for _ in range(K):
        plan_pack_fn()
        acc_fn()
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    elapsed_ms = max_over_ranks(elapsed_ms, dev, world)
    status = int(vs.status.item())

    # ---- step percentiles (after the timed region): n_pct steps with an
    # event at every step boundary; every `every`-th step also brackets its
    # accept call (those steps are left out of the percentiles)
    n_pct = max(256, min(K, 1024))
    sampled = list(range(0, n_pct, every))
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(n_pct + 1)]
    ev_a = {i: torch.cuda.Event(enable_timing=True) for i in sampled}
    ev_b = {i: torch.cuda.Event(enable_timing=True) for i in sampled}
    for i in range(n_pct):
        ev_s[i].record(stream)
        plan_pack_fn()
        if i % every == 0:
            ev_a[i].record(stream)
            acc_fn()
            ev_b[i].record(stream)
        else:
            acc_fn()
    ev_s[n_pct].record(stream)
    torch.cuda.synchronize()
    accept_ms = [ev_a[i].elapsed_time(ev_b[i]) for i in sampled]
    step_all = np.array([ev_s[i].elapsed_time(ev_s[i + 1]) for i in range(n_pct)]) * 1e3
    clean = [i for i in range(n_pct) if i % every != 0]
    step_us = step_all[clean]

    # ---- the accept call's duration for the roofline: n_roof steps after the
    # timed region, each one's accept bracketed by events after its plan +
    # pack (the bracket keeps the accept from launching early, so a sample
    # includes that launch gap); the mean over the samples gives
    # roofline.achieved, reported with its spread
    n_roof = max(256, min(K, 1024))
    ra = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_roof)]
    for e in ra:
        plan_pack_fn()
        e[0].record(stream)
        acc_fn()
        e[1].record(stream)
    torch.cuda.synchronize()
    roof_us = np.array([a.elapsed_time(b) for a, b in ra]) * 1e3

    # ---- breakdown (outside the timed region): per call on the same stream,
    # the fused plan+pack and, for reference, the two separate calls
    n_b = min(K, 200)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_b)]
    for e in evs:
        e[0].record(stream)
        plan_pack_fn()
        e[1].record(stream)
        acc_fn()
        e[2].record(stream)
        plan_fn()
        e[3].record(stream)
        pack_fn()
        e[4].record(stream)
        acc_fn()
        e[5].record(stream)
    torch.cuda.synchronize()
    br = np.array([[e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]), e[2].elapsed_time(e[3]),
                    e[3].elapsed_time(e[4])] for e in evs]) * 1e3
    # accept calls back to back (each launched while the previous one runs):
    # the accept's own duration without the launch gap a bracketing event adds
    n_acc = min(K, 200)
    b2b = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    b2b[0].record(stream)
    for _ in range(n_acc):
        acc_fn()
    b2b[1].record(stream)
    torch.cuda.synchronize()
    acc_b2b_us = b2b[0].elapsed_time(b2b[1]) * 1e3 / n_acc

    # ---- the same step replayed from a CUDA graph (secondary): 16 steps per
    # graph, captured on a side stream with the calls bound to it
    graph = None
    if not args.no_graph and world == 1:
        try:
            gs = torch.cuda.Stream()
            bound = vs.bind_compact(compact, stream=gs)
            calls = bound[1:] if args.separate_plan_pack else (bound[0], bound[3])
            per_graph = 16
            cg = torch.cuda.CUDAGraph()
            gs.wait_stream(stream)
            with torch.cuda.graph(cg, stream=gs):
                for _ in range(per_graph):
                    for fn in calls:
                        fn()
            torch.cuda.synchronize()
            for _ in range(3):
                cg.replay()
            torch.cuda.synchronize()
            reps = max(1, K // per_graph)
            ge = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            ge[0].record(torch.cuda.current_stream())
            for _ in range(reps):
                cg.replay()
            ge[1].record(torch.cuda.current_stream())
            torch.cuda.synchronize()
            g_ms = ge[0].elapsed_time(ge[1])
            graph = {"value": world * reps * per_graph / (g_ms / 1e3), "unit": UNIT,
                     "steps": reps * per_graph, "steps_per_graph": per_graph,
                     "us_per_step": g_ms * 1e3 / (reps * per_graph)}
        except Exception as e:  # report, do not fail the run
            graph = {"error": f"{type(e).__name__}: {e}"[:200]}

    # ---- ScatterCompactToStrided of the packed logits (secondary): read and
    # write total x V x 2 bytes; calls back to back
    scat = None
    if not args.no_cap:
        from confidence_scheduled_speculative_gb300 import api as _api
        scat_dst = torch.empty_like(strided_dev)
        st_s = torch.zeros(1, dtype=torch.int32, device=dev)
        for _ in range(3):
            _api.dspark_scatter_compact_to_strided(compact, vs.packed_src, vs.totals, scat_dst,
                                                   status=st_s)
        n_s = min(K, 200)
        se = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        se[0].record(stream)
        for _ in range(n_s):
            _api.dspark_scatter_compact_to_strided(compact, vs.packed_src, vs.totals, scat_dst,
                                                   status=st_s)
        se[1].record(stream)
        torch.cuda.synchronize()
        s_us = se[0].elapsed_time(se[1]) * 1e3 / n_s
        s_bytes = 2 * total * w.V * w.elem_bytes
        scat = {"us": s_us, "rows": total, "bytes": s_bytes,
                "gbs": s_bytes / (s_us * 1e-6) / 1e9,
                "frac": s_bytes / (s_us * 1e-6) / 1e9 / load_peaks()[0],
                "status": int(st_s.item())}
        del scat_dst

    # ---- speculative sampling accept over the same packed rows (secondary):
    # draft proposal rows = the strided target rows of the same depth, so
    # drafts pass often; calls back to back
    samp = None
    if not args.no_cap:
        from confidence_scheduled_speculative_gb300 import api as _api
        g_ = w.gamma
        sel = torch.arange(w.B * g_, device=dev)
        sel = (sel // g_) * (g_ + 1) + sel % g_
        dft_dev = strided_dev.index_select(0, sel)
        gen = torch.Generator(device=dev).manual_seed(11)
        ua = torch.rand((w.B, g_), generator=gen, device=dev)
        ub = torch.rand((w.B,), generator=gen, device=dev)
        i32 = dict(dtype=torch.int32, device=dev)
        so = dict(num_accepted=torch.zeros(w.B, **i32), bonus=torch.zeros(w.B, **i32),
                  commit_lens=torch.zeros(w.B, **i32), new_seq_lens=torch.zeros(w.B, **i32),
                  out_tokens=torch.zeros((w.B, g_ + 1), **i32))
        st_p = torch.zeros(1, **i32)
        sws = _api.workspace(_api.dspark_sampling_workspace_bytes(compact.size(0), w.B, g_), dev)

        def samp_call():
            _api.dspark_sampling_accept(compact, dft_dev, V=w.V, cu_seqlens=vs.cu_seqlens,
                                        draft=vs.draft, prefix_lens=vs.prefix_lens, B=w.B,
                                        gamma=g_, u_accept=ua, u_bonus=ub, workspace=sws,
                                        status=st_p, **so)

        for _ in range(3):
            samp_call()
        n_p = min(K, 200)
        pe = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        pe[0].record(stream)
        for _ in range(n_p):
            samp_call()
        pe[1].record(stream)
        torch.cuda.synchronize()
        p_us = pe[0].elapsed_time(pe[1]) * 1e3 / n_p
        tested = int((torch.diff(vs.cu_seqlens) - 1).clamp(min=0).sum().item())
        p_bytes = (total + tested) * w.V * w.elem_bytes  # the normalizer's rows, read once
        samp = {"us": p_us, "target_rows": total, "draft_rows": tested,
                "normalizer_bytes": p_bytes,
                "gbs_normalizer_bytes": p_bytes / (p_us * 1e-6) / 1e9,
                "frac_of_peak": p_bytes / (p_us * 1e-6) / 1e9 / load_peaks()[0],
                "mean_accepted": float(so["num_accepted"].float().mean().item()),
                "status": int(st_p.item())}
        # the same call with the draft rows' log-sum-exp supplied (as the
        # drafting step's sampler has it): only the target rows are normalised
        lse = torch.logsumexp(dft_dev.float(), dim=1).contiguous()

        def samp_call_lse():
            _api.dspark_sampling_accept(compact, dft_dev, V=w.V, cu_seqlens=vs.cu_seqlens,
                                        draft=vs.draft, prefix_lens=vs.prefix_lens, B=w.B,
                                        gamma=g_, u_accept=ua, u_bonus=ub, workspace=sws,
                                        status=st_p, draft_lse=lse, **so)

        ref_out = so["out_tokens"].clone()
        for _ in range(3):
            samp_call_lse()
        pe2 = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        pe2[0].record(stream)
        for _ in range(n_p):
            samp_call_lse()
        pe2[1].record(stream)
        torch.cuda.synchronize()
        l_us = pe2[0].elapsed_time(pe2[1]) * 1e3 / n_p
        l_bytes = total * w.V * w.elem_bytes
        samp["with_draft_lse"] = {"us": l_us, "normalizer_bytes": l_bytes,
                                  "gbs_normalizer_bytes": l_bytes / (l_us * 1e-6) / 1e9,
                                  "same_out_tokens": bool(torch.equal(ref_out, so["out_tokens"])),
                                  "status": int(st_p.item())}
        del dft_dev, sws

    # ---- calibration (secondary): the STS recorder on this step's accept
    # outputs, then statistics and the sequential fit over a log of recorded
    # samples
    calib = None
    if not args.no_cap and not args.no_calib:
        calib = calibration_timing(dev, stream, vs, w, K)

    # ---- the planner alone from a CUDA graph, with the step's additive table
    # and with the same samples interpolated (secondary)
    plan_kinds = None
    if not args.no_cap and w.name == "dsv4_like":
        from confidence_scheduled_speculative_gb300 import api as _api
        vs.status.zero_()
        # the same tier costs at every 128 rows: 31 entries, the select
        # path's largest table; at every 64 rows: 61 entries, the dense path
        dM = torch.arange(256, 4097, 128, dtype=torch.int32, device=dev)
        dense = (dM, 0.002 * dM.to(torch.float64))
        dM2 = torch.arange(256, 4097, 64, dtype=torch.int32, device=dev)
        dense2 = (dM2, 0.002 * dM2.to(torch.float64))
        # the pages' 1-D table: SPS sampled at every integer M in [B, B + B*gamma]
        sM = torch.arange(w.B, w.B + w.B * w.gamma + 1, dtype=torch.int32, device=dev)
        sps = (sM, 1.0 / (3e-3 + 3e-6 * sM.to(torch.float64)))
        plan_kinds = {"additive_tier": plan_kind_timing(dev, stream, vs, _api.COST_ADDITIVE),
                      "sps_1d_every_M":
                          plan_kind_timing(dev, stream, vs, _api.COST_SPS_1D, table=sps),
                      "additive_tier_31_entries":
                          plan_kind_timing(dev, stream, vs, _api.COST_ADDITIVE, table=dense),
                      "additive_tier_61_entries":
                          plan_kind_timing(dev, stream, vs, _api.COST_ADDITIVE, table=dense2),
                      "additive_interpolated":
                          plan_kind_timing(dev, stream, vs, _api.COST_ADDITIVE_INTERP)}
        for k, (kind, n) in {"additive_tier": (_api.COST_ADDITIVE, int(vs.cost_M.numel())),
                             "sps_1d_every_M": (_api.COST_SPS_1D, int(sM.numel())),
                             "additive_tier_31_entries": (_api.COST_ADDITIVE, int(dM.numel())),
                             "additive_tier_61_entries": (_api.COST_ADDITIVE, int(dM2.numel())),
                             "additive_interpolated": (_api.COST_ADDITIVE_INTERP,
                                                       int(vs.cost_M.numel()))}.items():
            plan_kinds[k]["path"] = _api.planner_path(w.B * w.gamma, kind, n)
        vs.status.zero_()

    # ---- accept bandwidth against packed rows (stress workload) and the
    # small workload whose logits fit in L2 (secondary)
    sweep = small = mixed = by_config = None
    if not args.no_cap and not args.no_sweep and w.name == "dsv4_like":
        sweep = accept_rows_sweep(dev, stream, args.seed)
        small = small_step_timing(dev, stream, "qwen_like", args.seed)
        mixed = mixed_cap_report(dev)
        by_config = configs_report(dev, stream, args.seed)

    # ---- cap-accept over the full strided block (secondary)
    cap = None
    if not args.no_cap:
        n_c = min(K, 200)
        ce = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_c)]
        for _ in range(3):
            vs.cap_accept(strided_dev, write_argmax=False)
        for e in ce:
            e[0].record(stream)
            vs.cap_accept(strided_dev, write_argmax=False)
            e[1].record(stream)
        torch.cuda.synchronize()
        cap_us = float(np.median([a.elapsed_time(b) for a, b in ce])) * 1e3
        cap_bytes = w.strided_rows * w.V * w.elem_bytes
        tot = vs.cap_totals.cpu().tolist()
        cap = {"accept_us": cap_us, "rows": w.strided_rows,
               "hbm_gbs": cap_bytes / (cap_us * 1e-6) / 1e9,
               "sum_commit": tot[0], "sum_ceiling_plus1": tot[1]}

    # ---- end to end from pinned host buffers
    io = HostStepIO(vs)
    io.fill(step)
    host_logits = torch.empty((total, w.V), dtype=torch.bfloat16, pin_memory=True)
    host_logits.copy_(compact)
    e2e_dev = torch.empty_like(compact)
    n_e = max(1, min(args.e2e_steps, K))

    def e2e_run(dev_logits):
        """n_e end-to-end steps; (seconds over ranks, logits bytes, outputs ok)."""
        for _ in range(3):
            run_host(vs, io, host_logits, dev_logits)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        nbytes = 0
        for _ in range(n_e):
            nbytes = run_host(vs, io, host_logits, dev_logits)
        torch.cuda.synchronize()
        secs = max_over_ranks(time.perf_counter() - t0, dev, world)
        ok = (np.array_equal(io.out_tokens.numpy(), vs.out_tokens.cpu().numpy())
              and int(io.status.item()) == 0)
        return secs, nbytes, ok

    # the accept reads the packed rows from the pinned buffer over the host
    # link (no host synchronisation inside a step); for comparison, the host
    # reads the packed total and copies that many rows in first
    e2e_s, logit_bytes, e2e_ok = e2e_run(None)
    e2e_copy_s, copy_bytes, copy_ok = e2e_run(e2e_dev)

    # ---- CPU oracle baseline (rank 0, N=1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        host_compact = strided[vs.packed_src[:total].cpu().numpy()]
        res = oracle_step_timing(step, host_compact, budget_s=args.cpu_seconds)
        cpu = {"value": res["value"], "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": (f"{res['steps']} oracle steps in {res['elapsed_s']:.1f} s: full "
                          f"planner + pack each, accept over {res['rows_sampled']} packed rows "
                          f"in total; full-step rate = 1/(t_plan_pack + {total}*t_row)"),
               "t_plan_pack_ms": res["t_plan_pack_ms"], "t_accept_row_us": res["t_accept_row_us"],
               "host": cpu_info()}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peak, peak_kind = load_peaks()
    acc_us = float(np.mean(accept_ms)) * 1e3  # the step-percentile loop's sampled accepts
    roof_mean = float(np.mean(roof_us))
    achieved = accept_bytes / (roof_mean * 1e-6) / 1e9
    in_step = accept_bytes / (acc_us * 1e-6) / 1e9
    ms_per_step = elapsed_ms / K
    value = job_rate(K, world, elapsed_ms / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": warm, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{w.name} B={w.B} gamma={w.gamma} V={w.V} compact",
                   "B": w.B, "gamma": w.gamma, "V": w.V, "mode": "compact",
                   "packed_rows": total, "padded_rows": padded, "seed": args.seed,
                   "plan_pack": "separate calls" if args.separate_plan_pack else "dspark_plan_pack",
                   "l2": f"inputs larger than L2: {accept_bytes / 1e6:.1f} MB of logits per step",
                   "parallelism": (f"dp{world}: own requests per rank, MAX all-reduce of the "
                                   "verify tier each step" if world > 1 else "replicas x1")},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "kernel": "dspark_greedy_accept (argmax + finalize)",
                     "bytes_per_launch": accept_bytes,
                     "traffic": ncu_traffic(w.name),
                     "samples": int(roof_us.size),
                     "accept_us": {"mean": roof_mean,
                                   "p10": float(np.percentile(roof_us, 10)),
                                   "p50": float(np.percentile(roof_us, 50)),
                                   "p90": float(np.percentile(roof_us, 90))},
                     "method": (f"{roof_us.size} steps after the timed region, each accept "
                                "call bracketed by CUDA events after its plan + pack; "
                                "achieved = bytes_per_launch / mean"),
                     "in_step": {"achieved": in_step, "frac": in_step / peak,
                                 "samples": len(accept_ms),
                                 "method": (f"every {every}-th step of the step-percentile "
                                            "loop brackets its accept")}},
        "e2e": {"value": job_rate(n_e, world, e2e_s), "unit": UNIT,
                "h2d_bytes_per_step": io.h2d_input_bytes() + logit_bytes,
                "d2h_bytes_per_step": io.d2h_output_bytes(), "steps": n_e,
                "matches_device_path": bool(e2e_ok),
                "mode": "accept reads the pinned host logits over the link",
                "copy_then_accept": {"value": job_rate(n_e, world, e2e_copy_s),
                                     "h2d_bytes_per_step": io.h2d_input_bytes() + copy_bytes,
                                     "matches_device_path": bool(copy_ok)}},
        "cpu_baseline": cpu,
        "gpu_launches": (vs.kernels_per_step(args.separate_plan_pack) + (world > 1)) * K,
        "clocks": clocks,
        "step_us": {"p10": float(np.percentile(step_us, 10)),
                    "p50": float(np.percentile(step_us, 50)),
                    "p90": float(np.percentile(step_us, 90)),
                    "steps": int(step_us.size),
                    "method": ("after the timed region: an event at every step boundary "
                               "(which keeps the next step from launching early, so these "
                               "are slightly above ms_per_step)")},
        "breakdown_us": {"plan_pack": float(np.median(br[:, 0])),
                         "accept": float(np.median(br[:, 1])),
                         "plan_alone": float(np.median(br[:, 2])),
                         "pack_alone": float(np.median(br[:, 3])),
                         "accept_timed_mean": acc_us, "step_timed_mean": 1e3 * ms_per_step,
                         "accept_back_to_back": acc_b2b_us,
                         "accept_back_to_back_gbs": accept_bytes / (acc_b2b_us * 1e-6) / 1e9,
                         "accept_rows_per_s": total / (acc_b2b_us * 1e-6),
                         "planner_calls_per_s": 1e6 / float(np.median(br[:, 2]))},
        "cuda_graph": graph,
        "scatter_compact_to_strided": scat,
        "sampling_accept": samp,
        "calibration": calib,
        "plan_by_cost_kind": plan_kinds,
        "cap_accept": cap,
        "accept_by_rows": sweep,
        "qwen_like_cold_l2": small,
        "mixed_cap_report": mixed,
        "by_config": by_config,
        "status": status,
    }
    emit(line, args)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
