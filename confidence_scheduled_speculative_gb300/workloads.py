"""Seeded synthetic inputs for the DSpark verify planner and greedy accept.

This module only *draws data*: confidence logits, STS temperatures, draft and
anchor tokens, prefix lengths, cost tables, graph tiers and target-logit rows.
It contains none of the planner's or the accept's arithmetic (no sigmoid, no
survival product, no sort, no argmax), so the CPU oracle and the CUDA path can
both consume what it produces without sharing any of the method.

The pages the workloads imitate measure DeepSeek-V4-Flash and Qwen3 serving on
gsm8k / arena-hard / poetry traffic.  Neither those models nor those datasets
exist here; the generators below stand in for their *shapes*: vocabulary size
V, batch B, block length gamma, per-depth acceptance decay and the traffic mix.

Target logits are drawn per verify row, keyed by (seed, request r, depth j), so
any subset of rows (for example the packed rows of a compact window) can be
produced without materialising the full strided [B, gamma+1, V] tensor:

* every row is N(0, 1) noise;
* row j < gamma of request r gets +8 at ``draft[r, j]`` with probability
  ``match_prob[r, j]``, otherwise at a uniformly drawn token != draft[r, j];
* row gamma (the bonus row after a fully accepted block) gets +8 at a
  uniformly drawn token.

bf16 rows are rounded to nearest-even from the fp32 draw and returned as raw
uint16 bit patterns.

Recorded calibration samples (``calibration_samples``) stand in for a log of
served steps: each sample has a true per-depth acceptance probability drawn
in probability space, a confidence-head logit that is that probability's
logit scaled by a known "true" temperature (a head miscalibrated by exactly
that temperature), the greedy prefix outcome drawn depth by depth, and a
verify window that is the full block for a fraction of the samples and a
random compact window otherwise.
"""

from __future__ import annotations

import dataclasses
from typing import Iterable, Sequence

import numpy as np

# cost-table kinds, matching the C-ABI's dspark_cost_table.kind
COST_SPS_1D = 0
COST_ADDITIVE = 1
COST_ADDITIVE_INTERP = 2

_ROW_TAG = 0x5EED_0001
_STEP_TAG = 0x5EED_0002
PEAK = 8.0


@dataclasses.dataclass(frozen=True)
class Workload:
    """Static description of one synthetic workload."""

    name: str
    B: int
    gamma: int
    V: int
    logits_dtype: str  # "bf16" | "fp32"
    survival_eps: float = 1e-4
    min_verify_len: int = 1
    max_verify_len: int = 0  # 0 -> gamma + 1
    forced_budget: int = -1
    description: str = ""

    @property
    def max_len(self) -> int:
        return self.max_verify_len if self.max_verify_len > 0 else self.gamma + 1

    @property
    def strided_rows(self) -> int:
        return self.B * (self.gamma + 1)

    @property
    def elem_bytes(self) -> int:
        return 2 if self.logits_dtype == "bf16" else 4


@dataclasses.dataclass
class CostTable:
    kind: int
    M: np.ndarray  # int32, strictly ascending
    val: np.ndarray  # float64 (SPS in steps/s, or token-side cost in ms)
    bias_ms: float = 0.0
    alpha_ms: float = 0.0


@dataclasses.dataclass
class StepInputs:
    """One planner+pack+accept step's inputs (host numpy arrays)."""

    workload: Workload
    seed: int
    conf_logits: np.ndarray  # float32 [B, gamma]
    sts_temps: np.ndarray  # float32 [gamma]
    draft: np.ndarray  # int32 [B, gamma]
    anchor: np.ndarray  # int32 [B]
    prefix_lens: np.ndarray  # int32 [B]
    match_prob: np.ndarray  # float64 [B, gamma], data-generation only
    cost: CostTable
    tiers: np.ndarray  # int32 graph tiers for the pack round-up (may be empty)
    capacity: int

    @property
    def B(self) -> int:
        return self.workload.B

    @property
    def gamma(self) -> int:
        return self.workload.gamma

    @property
    def V(self) -> int:
        return self.workload.V


# ---------------------------------------------------------------- workloads

TINY = Workload("tiny", B=4, gamma=4, V=1024, logits_dtype="fp32", max_verify_len=5,
                description="B=4 gamma=4 V=1024 fp32, 1-D SPS table")
QWEN = Workload("qwen_like", B=32, gamma=8, V=151936, logits_dtype="bf16",
                description="Qwen3-like dense: B=32 gamma=8 V=151936 bf16, additive table")
DSV4 = Workload("dsv4_like", B=256, gamma=16, V=129280, logits_dtype="bf16", max_verify_len=17,
                description="DeepSeek-V4-like: B=256 gamma=16 V=129280 bf16, additive table")
MIXED = Workload("mixed", B=128, gamma=12, V=129280, logits_dtype="bf16",
                 description="Mixed traffic: B=128 gamma=12 V=129280 bf16, 3 classes, 1-D SPS")
STRESS = Workload("stress", B=1024, gamma=16, V=129280, logits_dtype="bf16",
                  description="Stress: B=1024 gamma=16 V=129280 bf16, additive, forced budgets")

WORKLOADS = {w.name: w for w in (TINY, QWEN, DSV4, MIXED, STRESS)}


def _logit(p: np.ndarray) -> np.ndarray:
    p = np.asarray(p, dtype=np.float64)
    return np.log(p) - np.log1p(-p)


def _step_rng(w: Workload, seed: int) -> np.random.Generator:
    name_key = sum(ord(ch) * (i + 1) for i, ch in enumerate(w.name))
    return np.random.default_rng(np.random.SeedSequence([_STEP_TAG, name_key, seed]))


def make_step(w: Workload, seed: int = 0, forced_budget: int | None = None) -> StepInputs:
    """Draw one step's planner/pack/accept inputs for workload ``w``."""
    rng = _step_rng(w, seed)
    B, g, V = w.B, w.gamma, w.V
    k = np.arange(g, dtype=np.float64)

    if w.name == "tiny":
        z = rng.normal(1.5, 1.0, size=(B, g))
        temps = np.ones(g)
        match = np.full((B, g), 0.8)
    elif w.name == "qwen_like":
        c = 0.9 - 0.05 * k
        z = _logit(c)[None, :] + rng.normal(0.0, 0.5, size=(B, g))
        temps = 1.0 + 0.1 * k
        match = np.broadcast_to(c, (B, g)).copy()
    elif w.name == "dsv4_like":
        c = 0.92 - 0.03 * k
        z = _logit(c)[None, :] + rng.normal(0.0, 0.7, size=(B, g))
        temps = 1.0 + 0.05 * k
        match = np.broadcast_to(c, (B, g)).copy()
    elif w.name == "mixed":
        p_class = np.array([0.9, 0.6, 0.3])
        p = p_class[np.arange(B) % 3]
        z = _logit(p)[:, None] + rng.normal(0.0, 0.5, size=(B, g))
        temps = np.ones(g)
        match = np.broadcast_to(p[:, None], (B, g)).copy()
    elif w.name == "stress":
        z = rng.normal(1.0, 1.5, size=(B, g))
        temps = 1.0 + 0.05 * k
        match = np.full((B, g), 0.7)
    else:  # pragma: no cover - guarded by WORKLOADS
        raise ValueError(w.name)

    draft = rng.integers(0, V, size=(B, g), dtype=np.int64).astype(np.int32)
    anchor = rng.integers(0, V, size=B, dtype=np.int64).astype(np.int32)
    prefix = rng.integers(1, 8193, size=B, dtype=np.int64).astype(np.int32)

    cost, tiers = cost_table_for(w)
    cap = max(w.strided_rows, int(tiers.max()) if tiers.size else 0)
    fb = w.forced_budget if forced_budget is None else forced_budget
    if fb != w.forced_budget:
        w = dataclasses.replace(w, forced_budget=fb)
    return StepInputs(
        workload=w, seed=seed,
        conf_logits=np.ascontiguousarray(z, dtype=np.float32),
        sts_temps=np.ascontiguousarray(temps, dtype=np.float32),
        draft=np.ascontiguousarray(draft), anchor=anchor, prefix_lens=prefix,
        match_prob=match, cost=cost, tiers=tiers, capacity=cap)


def cost_table_for(w: Workload) -> tuple[CostTable, np.ndarray]:
    """The cost table (planner input) and the pack's graph tiers for ``w``."""
    B, g = w.B, w.gamma
    if w.name in ("tiny", "mixed"):
        a, bcoef = (2.0e-3, 4e-6) if w.name == "tiny" else (3.0e-3, 3e-6)
        M = np.arange(B, B + B * g + 1, dtype=np.int32)
        val = 1.0 / (a + bcoef * M.astype(np.float64))
        return CostTable(COST_SPS_1D, M, val), np.zeros(0, dtype=np.int32)
    if w.name in ("qwen_like", "dsv4_like"):
        tiers = (np.array([32, 64, 128, 256, 512], dtype=np.int32) if w.name == "qwen_like"
                 else np.array([256, 512, 1024, 2048, 4096], dtype=np.int32))
        return CostTable(COST_ADDITIVE, tiers, 0.002 * tiers.astype(np.float64),
                         bias_ms=1.5, alpha_ms=0.01 * B), tiers
    if w.name == "stress":
        tiers = (2 ** np.arange(10, 16)).astype(np.int32)
        return CostTable(COST_ADDITIVE, tiers, 0.001 * tiers.astype(np.float64),
                         bias_ms=2.0, alpha_ms=0.005 * B), tiers
    raise ValueError(w.name)


# ----------------------------------------------------------- target logits

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest-even); return the raw uint16 patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _row_f32(step: StepInputs, r: int, j: int) -> np.ndarray:
    w = step.workload
    rng = np.random.default_rng(np.random.SeedSequence([_ROW_TAG, step.seed, w.B, w.gamma, r, j]))
    row = rng.standard_normal(w.V, dtype=np.float32)
    u = rng.random()
    if j < w.gamma:
        d = int(step.draft[r, j])
        if u < step.match_prob[r, j]:
            peak = d
        else:
            peak = int(rng.integers(0, w.V - 1))
            if peak >= d:
                peak += 1
    else:
        peak = int(rng.integers(0, w.V))
    row[peak] += np.float32(PEAK)
    return row


def target_rows(step: StepInputs, rows_rj: Iterable[tuple[int, int]]) -> np.ndarray:
    """Target logits for the listed (request, depth) rows, one row each.

    Returns float32 [n, V] for fp32 workloads, uint16 bf16 bits otherwise.
    """
    rows_rj = list(rows_rj)
    w = step.workload
    out = np.empty((len(rows_rj), w.V), dtype=np.float32 if w.logits_dtype == "fp32" else np.uint16)
    for i, (r, j) in enumerate(rows_rj):
        row = _row_f32(step, int(r), int(j))
        out[i] = row if w.logits_dtype == "fp32" else to_bf16_bits(row)
    return out


def strided_logits(step: StepInputs) -> np.ndarray:
    """All B*(gamma+1) verify rows in request-major order [B*(gamma+1), V]."""
    w = step.workload
    return target_rows(step, ((r, j) for r in range(w.B) for j in range(w.gamma + 1)))


def strided_row_index(r: int, j: int, gamma: int) -> int:
    return r * (gamma + 1) + j


# ------------------------------------------------------ the pages' example

def pages_example_confidences() -> np.ndarray:
    """The two-request teaching example of the adaptive-verify page (section 一):
    conditional confidences [0.9, 0.8] and [0.6, 0.5]."""
    return np.array([[0.9, 0.8], [0.6, 0.5]], dtype=np.float64)


def confidence_logits_for(probs: np.ndarray) -> np.ndarray:
    """Confidence logits whose STS output at T=1 is the given probabilities
    (the inverse of the logistic link, used to build test inputs)."""
    return np.ascontiguousarray(_logit(probs), dtype=np.float32)


@dataclasses.dataclass(frozen=True)
class CalibrationSamples:
    """Recorded (z, correct, tested) rows and the truth they were drawn from."""

    conf_logits: np.ndarray  # [N, gamma] fp32
    correct: np.ndarray      # [N] int32, accepted drafts inside the window
    tested: np.ndarray       # [N] int32, drafts the target checked
    true_temps: np.ndarray   # [gamma] fp32
    true_probs: np.ndarray   # [N, gamma] fp64


_CAL_TAG = 0x5EED_0003


def calibration_samples(N: int, gamma: int, true_temps, seed: int = 0, full_frac: float = 0.25,
                        concentration: float = 6.0) -> CalibrationSamples:
    """N recorded steps of one request each.  Depth k's true acceptance
    probability is Beta-distributed with mean 0.92 - 0.03 k (the DSV4-like
    decay) and the given concentration; the head logit is
    logit(probability) * true_temps[k]; the prefix survives depth k with that
    probability; the window is the whole block for ``full_frac`` of the
    samples (cap-accept style) and 0..gamma drafts uniformly otherwise; the
    recorded count is the accepted prefix cut to the window."""
    rng = np.random.default_rng(np.random.SeedSequence([_CAL_TAG, N, gamma, seed]))
    Tt = np.broadcast_to(np.asarray(true_temps, np.float64), (gamma,)).copy()
    k = np.arange(gamma, dtype=np.float64)
    mean = np.clip(0.92 - 0.03 * k, 0.05, 0.95)
    a = mean * concentration
    b = (1.0 - mean) * concentration
    prob = np.clip(rng.beta(a[None, :], b[None, :], size=(N, gamma)), 1e-4, 1.0 - 1e-4)
    z = _logit(prob) * Tt[None, :]
    u = rng.random((N, gamma))
    fail = u >= prob
    raw = np.where(fail.any(axis=1), fail.argmax(axis=1), gamma)
    full = rng.random(N) < full_frac
    win = rng.integers(0, gamma + 1, size=N)
    tested = np.where(full, gamma, win)
    correct = np.minimum(raw, tested)
    return CalibrationSamples(conf_logits=np.ascontiguousarray(z, dtype=np.float32),
                              correct=correct.astype(np.int32), tested=tested.astype(np.int32),
                              true_temps=Tt.astype(np.float32), true_probs=prob)


def temperature_grid(n: int = 64, lo: float = 0.25, hi: float = 4.0) -> np.ndarray:
    """n log-spaced candidate temperatures from lo to hi (fp32)."""
    return np.geomspace(lo, hi, n).astype(np.float32)


def seeds(n: int, start: int = 0) -> Sequence[int]:
    return range(start, start + n)


def approx_bytes(w: Workload, rows: int) -> int:
    return int(rows) * w.V * w.elem_bytes


def describe(w: Workload) -> str:
    return f"{w.name}: B={w.B} gamma={w.gamma} V={w.V} {w.logits_dtype} ({w.description})"


__all__ = [
    "Workload", "CostTable", "StepInputs", "WORKLOADS", "TINY", "QWEN", "DSV4", "MIXED", "STRESS",
    "COST_SPS_1D", "COST_ADDITIVE", "COST_ADDITIVE_INTERP", "make_step", "cost_table_for", "target_rows", "strided_logits",
    "to_bf16_bits", "bf16_bits_to_f32", "strided_row_index", "pages_example_confidences",
    "confidence_logits_for", "seeds", "approx_bytes", "describe", "PEAK",
    "CalibrationSamples", "calibration_samples", "temperature_grid",
]
