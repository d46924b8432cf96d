"""Device buffers for one planner + pack + accept step, and the calls that
run it.

``VerifyStep`` owns every device buffer a DSpark decode step needs on the
verify side (planner outputs, packed window, accept outputs, workspaces and
the cost table), allocated once through PyTorch, and enqueues the C-ABI
calls on one stream.  It adds no computation of its own: the numbers all
come from the library's kernels.

``run_host`` is the end-to-end entry a caller with host buffers uses: it
copies the step's inputs from pinned host memory, runs the planner and the
pack, reads back the packed totals (the host needs them to pick the verify
graph tier), copies the target logits of the packed rows, runs the accept
and reads the results back.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import api


@dataclasses.dataclass
class StepConfig:
    B: int
    gamma: int
    V: int
    logits_dtype: torch.dtype
    survival_eps: float
    min_verify_len: int
    max_verify_len: int
    forced_budget: int
    cost_kind: int
    cost_M: np.ndarray
    cost_val: np.ndarray
    bias_ms: float
    alpha_ms: float
    tiers: tuple
    capacity: int

    @classmethod
    def from_step(cls, step) -> "StepConfig":
        """Build from a ``workloads.StepInputs``."""
        w, c = step.workload, step.cost
        return cls(B=w.B, gamma=w.gamma, V=w.V,
                   logits_dtype=torch.bfloat16 if w.logits_dtype == "bf16" else torch.float32,
                   survival_eps=w.survival_eps, min_verify_len=w.min_verify_len,
                   max_verify_len=w.max_len, forced_budget=w.forced_budget, cost_kind=c.kind,
                   cost_M=np.asarray(c.M, np.int32), cost_val=np.asarray(c.val, np.float64),
                   bias_ms=c.bias_ms, alpha_ms=c.alpha_ms,
                   tiers=tuple(int(t) for t in step.tiers), capacity=int(step.capacity))


_IN_PIECES = (("conf_logits", torch.float32, "Bg"), ("sts_temps", torch.float32, "g"),
              ("anchor", torch.int32, "B"), ("draft", torch.int32, "Bg"),
              ("prefix_lens", torch.int32, "B"))
_OUT_PIECES = (("status", torch.int32, "1"), ("totals", torch.int32, "2"),
               ("out_tokens", torch.int32, "Bg1"), ("commit_lens", torch.int32, "B"),
               ("new_seq_lens", torch.int32, "B"), ("verify_lens", torch.int32, "B"))


def _shape(kind: str, B: int, g: int) -> tuple[int, ...]:
    return {"Bg": (B, g), "g": (g,), "B": (B,), "1": (1,), "2": (2,), "Bg1": (B, g + 1)}[kind]


def _arena(B: int, g: int, device, pin: bool = False):
    """One zeroed int32 arena laid out as [inputs | status | outputs], each
    piece starting on a 16-byte boundary; returns (arena, named views, words
    of the inputs and the status, first word of the status)."""
    offsets, at = {}, 0
    for name, _, kind in _IN_PIECES + _OUT_PIECES:
        at = (at + 3) & ~3
        offsets[name] = at
        n = 1
        for d in _shape(kind, B, g):
            n *= d
        at += n
    if pin:
        arena = torch.zeros(at, dtype=torch.int32).pin_memory()
    else:
        arena = torch.zeros(at, dtype=torch.int32, device=device)
    views = {}
    for name, dt, kind in _IN_PIECES + _OUT_PIECES:
        shp = _shape(kind, B, g)
        n = 1
        for d in shp:
            n *= d
        v = arena[offsets[name]:offsets[name] + n]
        views[name] = (v.view(dt) if dt != torch.int32 else v).view(shp)
    n_in = offsets["status"] + 1  # the inputs and the status word
    return arena, views, n_in, offsets["status"]


class VerifyStep:
    """All device state of one verify-side step for a fixed configuration."""

    def __init__(self, cfg: StepConfig, device: str | torch.device = "cuda"):
        self.cfg = cfg
        self.device = torch.device(device)
        B, g, cap = cfg.B, cfg.gamma, cfg.capacity
        i32 = dict(dtype=torch.int32, device=self.device)
        f32 = dict(dtype=torch.float32, device=self.device)
        # the step's inputs, the status word and the outputs a host reads
        # back share one arena of 4-byte words ([inputs | status | outputs],
        # each piece 16-byte aligned): the end-to-end path moves the inputs
        # (with a zero status) in one copy and the status and outputs out in
        # another
        self.arena, views, self.n_in, self.out_lo = _arena(B, g, self.device)
        self.conf_logits = views["conf_logits"]
        self.sts_temps = views["sts_temps"]
        self.sts_temps.fill_(1.0)
        self.anchor = views["anchor"]
        self.draft = views["draft"]
        self.prefix_lens = views["prefix_lens"]
        self.cost_M = torch.as_tensor(cfg.cost_M, dtype=torch.int32, device=self.device)
        self.cost_val = torch.as_tensor(cfg.cost_val, dtype=torch.float64, device=self.device)
        # planner outputs
        self.survivals = torch.zeros((B, g), **f32)
        self.verify_lens = views["verify_lens"]
        self.budget = torch.zeros(1, **i32)
        self.tau_theta = torch.zeros(2, dtype=torch.float64, device=self.device)
        self.status = views["status"]
        # pack outputs
        self.packed_ids = torch.zeros(cap, **i32)
        self.packed_pos = torch.zeros(cap, **i32)
        self.packed_req = torch.zeros(cap, **i32)
        self.packed_src = torch.zeros(cap, **i32)
        self.cu_seqlens = torch.zeros(B + 1, **i32)
        self.totals = views["totals"]
        # accept outputs
        rows_max = max(cap, B * (g + 1))
        self.argmax = torch.zeros(rows_max, **i32)
        self.num_accepted = torch.zeros(B, **i32)
        self.bonus = torch.zeros(B, **i32)
        self.commit_lens = views["commit_lens"]
        self.new_seq_lens = views["new_seq_lens"]
        self.out_tokens = views["out_tokens"]
        self.ceiling = torch.zeros(B, **i32)
        self.cap_totals = torch.zeros(2, **i32)
        self.accept_ws = api.workspace(api.dspark_accept_workspace_bytes(rows_max, cfg.V),
                                       self.device)
        self.plan_ws = None
        nb = api.dspark_plan_workspace_bytes(B, g)
        if nb:
            self.plan_ws = api.workspace(nb, self.device)

    # ------------------------------------------------------------- inputs
    def load_inputs(self, step) -> None:
        """Copy a ``workloads.StepInputs``'s planner/pack inputs to the device."""
        self.conf_logits.copy_(torch.from_numpy(step.conf_logits))
        self.sts_temps.copy_(torch.from_numpy(step.sts_temps))
        self.anchor.copy_(torch.from_numpy(step.anchor))
        self.draft.copy_(torch.from_numpy(step.draft))
        self.prefix_lens.copy_(torch.from_numpy(step.prefix_lens))

    # -------------------------------------------------------------- calls
    def plan(self, stream=None) -> None:
        c = self.cfg
        api.dspark_plan(self.conf_logits, self.sts_temps, B=c.B, gamma=c.gamma,
                        survival_eps=c.survival_eps, min_verify_len=c.min_verify_len,
                        max_verify_len=c.max_verify_len, forced_budget=c.forced_budget,
                        cost_kind=c.cost_kind, cost_M=self.cost_M, cost_val=self.cost_val,
                        bias_ms=c.bias_ms, alpha_ms=c.alpha_ms, survivals=self.survivals,
                        verify_lens=self.verify_lens, budget=self.budget,
                        tau_theta=self.tau_theta, status=self.status, workspace=self.plan_ws,
                        stream=stream)

    def pack(self, stream=None) -> None:
        c = self.cfg
        api.dspark_pack_verify(self.anchor, self.draft, self.prefix_lens, self.verify_lens,
                               B=c.B, gamma=c.gamma, tiers=c.tiers, capacity=c.capacity,
                               packed_ids=self.packed_ids, packed_pos=self.packed_pos,
                               packed_req=self.packed_req, packed_src=self.packed_src,
                               cu_seqlens=self.cu_seqlens, totals=self.totals,
                               status=self.status, stream=stream)

    def plan_pack(self, stream=None) -> None:
        """plan then pack in fewer launches (dspark_plan_pack)."""
        c = self.cfg
        api.dspark_plan_pack(self.conf_logits, self.sts_temps, self.anchor, self.draft,
                             self.prefix_lens, B=c.B, gamma=c.gamma,
                             survival_eps=c.survival_eps, min_verify_len=c.min_verify_len,
                             max_verify_len=c.max_verify_len, forced_budget=c.forced_budget,
                             cost_kind=c.cost_kind, cost_M=self.cost_M, cost_val=self.cost_val,
                             bias_ms=c.bias_ms, alpha_ms=c.alpha_ms, tiers=c.tiers,
                             capacity=c.capacity, survivals=self.survivals,
                             verify_lens=self.verify_lens, budget=self.budget,
                             tau_theta=self.tau_theta, packed_ids=self.packed_ids,
                             packed_pos=self.packed_pos, packed_req=self.packed_req,
                             packed_src=self.packed_src, cu_seqlens=self.cu_seqlens,
                             totals=self.totals, status=self.status, workspace=self.plan_ws,
                             stream=stream)

    def pad_to_tier(self, pad_to: torch.Tensor | None = None, stream=None) -> None:
        """Pad the packed window to a verify tier shared with other ranks
        (dspark_pad_to_tier); ``pad_to`` defaults to totals[1] itself, as
        left by ``share_tier``'s in-place all-reduce."""
        api.dspark_pad_to_tier(self.totals[1:2] if pad_to is None else pad_to,
                               packed_ids=self.packed_ids, packed_pos=self.packed_pos,
                               packed_req=self.packed_req, packed_src=self.packed_src,
                               totals=self.totals, status=self.status,
                               capacity=self.cfg.capacity, stream=stream)

    def share_tier(self, group=None, stream=None) -> None:
        """The data-parallel step's one exchange: the max of the ranks' local
        verify tiers (in place on totals[1]), then the pad to it."""
        share_tier(self.totals, group)
        self.pad_to_tier(None, stream)

    def kernels_per_step(self, separate_plan_pack: bool = False) -> int:
        """Kernels one compact step launches: survival + one single-CTA
        planner kernel (select, dense or interp; the pack inside), else
        survival + rank + pack (separate plan and pack calls add the pack
        kernel); then argmax + finalize."""
        c = self.cfg
        select = api.planner_path(c.B * c.gamma, c.cost_kind, len(c.cost_M)) != "rank"
        return (3 if (separate_plan_pack or not select) else 2) + 2

    def greedy_accept(self, logits: torch.Tensor, write_argmax: bool = True, stream=None) -> None:
        c = self.cfg
        api.dspark_greedy_accept(logits, V=c.V, cu_seqlens=self.cu_seqlens, draft=self.draft,
                                 prefix_lens=self.prefix_lens, B=c.B, gamma=c.gamma,
                                 num_accepted=self.num_accepted, bonus=self.bonus,
                                 commit_lens=self.commit_lens, out_tokens=self.out_tokens,
                                 workspace=self.accept_ws, status=self.status,
                                 argmax=self.argmax if write_argmax else None,
                                 new_seq_lens=self.new_seq_lens, stream=stream)

    def cap_accept(self, logits: torch.Tensor, write_argmax: bool = True, stream=None) -> None:
        c = self.cfg
        api.dspark_cap_accept(logits, V=c.V, verify_lens=self.verify_lens, draft=self.draft,
                              prefix_lens=self.prefix_lens, B=c.B, gamma=c.gamma,
                              num_accepted=self.num_accepted, bonus=self.bonus,
                              commit_lens=self.commit_lens, out_tokens=self.out_tokens,
                              ceiling=self.ceiling, totals=self.cap_totals,
                              workspace=self.accept_ws, status=self.status,
                              argmax=self.argmax if write_argmax else None,
                              new_seq_lens=self.new_seq_lens, stream=stream)

    def compact_step(self, logits: torch.Tensor, stream=None) -> None:
        """plan + pack -> greedy accept, enqueued back to back."""
        self.plan_pack(stream)
        self.greedy_accept(logits, write_argmax=False, stream=stream)

    def bind_compact(self, logits: torch.Tensor, stream=None):
        """Marshal the calls of a compact step once; returns zero-argument
        callables (plan_pack, plan, pack, accept) that re-issue the same C
        calls with the same device pointers (for tight timing loops);
        plan_pack is plan then pack in fewer launches."""
        lib = api.load()
        c = self.cfg
        s = api._stream(stream)
        p = lambda t: None if t is None else t.data_ptr()
        self._params = api.dspark_plan_params(c.B, c.gamma, c.survival_eps, c.min_verify_len,
                                              c.max_verify_len, c.forced_budget)
        self._cost = api.dspark_cost_table(c.cost_kind, int(self.cost_M.numel()),
                                           p(self.cost_M), p(self.cost_val), c.bias_ms,
                                           c.alpha_ms)
        self._tiers = (api.ctypes.c_int32 * max(1, len(c.tiers)))(*c.tiers)
        plan_args = (p(self.conf_logits), p(self.sts_temps), api.ctypes.byref(self._params),
                     api.ctypes.byref(self._cost), p(self.survivals), p(self.verify_lens),
                     p(self.budget), p(self.tau_theta), p(self.plan_ws),
                     0 if self.plan_ws is None else self.plan_ws.numel(), p(self.status), s)
        pack_args = (p(self.anchor), p(self.draft), p(self.prefix_lens), p(self.verify_lens),
                     c.B, c.gamma, self._tiers, len(c.tiers), c.capacity, p(self.packed_ids),
                     p(self.packed_pos), p(self.packed_req), p(self.packed_src),
                     p(self.cu_seqlens), p(self.totals), p(self.status), s)
        plan_pack_args = (plan_args[:8] + (p(self.anchor), p(self.draft), p(self.prefix_lens),
                                           self._tiers, len(c.tiers), c.capacity,
                                           p(self.packed_ids), p(self.packed_pos),
                                           p(self.packed_req), p(self.packed_src),
                                           p(self.cu_seqlens), p(self.totals)) + plan_args[8:])
        ptr, ld = api._logits_ptr(logits, c.V)
        acc_args = (ptr, api._dtype_code(logits), ld, c.V, logits.size(0), p(self.cu_seqlens),
                    p(self.draft), p(self.prefix_lens), c.B, c.gamma, None,
                    p(self.num_accepted), p(self.bonus), p(self.commit_lens),
                    p(self.new_seq_lens), p(self.out_tokens), p(self.accept_ws),
                    self.accept_ws.numel(), p(self.status), s)

        def call(fn, args, name):
            def run():
                rc = fn(*args)
                if rc != api.DSPARK_OK:
                    raise api.DsparkError(name, rc)
            return run

        return (call(lib.dspark_plan_pack, plan_pack_args, "dspark_plan_pack"),
                call(lib.dspark_plan, plan_args, "dspark_plan"),
                call(lib.dspark_pack_verify, pack_args, "dspark_pack_verify"),
                call(lib.dspark_greedy_accept, acc_args, "dspark_greedy_accept"))

    # ------------------------------------------------------- host round trip
    def result(self) -> dict:
        """Copy every output to host numpy arrays (synchronises)."""
        torch.cuda.synchronize(self.device)
        names = ["survivals", "verify_lens", "budget", "tau_theta", "status", "packed_ids",
                 "packed_pos", "packed_req", "packed_src", "cu_seqlens", "totals", "argmax",
                 "num_accepted", "bonus", "commit_lens", "new_seq_lens", "out_tokens", "ceiling",
                 "cap_totals"]
        return {n: getattr(self, n).cpu().numpy() for n in names}


def share_tier(totals: torch.Tensor, group=None) -> torch.Tensor:
    """The exchange data-parallel ranks make each step ([AVS] §六: local
    verify tier -> DP gather -> DP-global max token tier; [SGL] "Ragged
    verify": the ranks share the largest tier any rank needs).  ``totals`` is
    a rank's pack output (real rows, padded rows = its local tier); totals[1]
    becomes the largest local tier over the ranks of ``group`` by one int32
    MAX all-reduce in place (NCCL on the current stream, no host
    synchronisation, or gloo on CPU tensors).  Nothing else crosses ranks:
    each rank plans, packs and accepts its own requests.  With one rank (or
    no process group) nothing happens.  Returns the view totals[1:2], the
    shared tier, for dspark_pad_to_tier."""
    import torch.distributed as dist
    tier = totals[1:2]
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(tier, op=dist.ReduceOp.MAX, group=group)
    return tier


class HostStepIO:
    """Pinned host buffers for the end-to-end path (``run_host``)."""

    def __init__(self, vs: VerifyStep):
        c = vs.cfg
        # the device arena's layout in pinned memory: the inputs (and a
        # status word that stays zero) go in with one copy, the status and
        # the outputs come back with one copy
        self.arena, views, self.n_in, self.out_lo = _arena(c.B, c.gamma, None, pin=True)
        self.in_arena = self.arena[:self.n_in]
        self.out_host = torch.zeros(self.arena.numel() - self.out_lo, dtype=torch.int32).pin_memory()
        self.conf_logits = views["conf_logits"]
        self.sts_temps = views["sts_temps"]
        self.anchor = views["anchor"]
        self.draft = views["draft"]
        self.prefix_lens = views["prefix_lens"]
        # outputs: views of out_host at the device arena's offsets
        _, oviews, _, _ = _arena(c.B, c.gamma, None, pin=False)
        base = self.out_lo
        def out_view(name):
            v = oviews[name]
            off = v.storage_offset() - base
            return self.out_host[off:off + v.numel()].view(v.shape)
        self.status = out_view("status")
        self.totals = out_view("totals")
        self.out_tokens = out_view("out_tokens")
        self.commit_lens = out_view("commit_lens")
        self.new_seq_lens = out_view("new_seq_lens")
        self.verify_lens = out_view("verify_lens")

    def fill(self, step) -> None:
        self.conf_logits.copy_(torch.from_numpy(step.conf_logits))
        self.sts_temps.copy_(torch.from_numpy(step.sts_temps))
        self.anchor.copy_(torch.from_numpy(step.anchor))
        self.draft.copy_(torch.from_numpy(step.draft))
        self.prefix_lens.copy_(torch.from_numpy(step.prefix_lens))

    def h2d_input_bytes(self) -> int:
        return self.in_arena.numel() * 4

    def d2h_output_bytes(self) -> int:
        return self.out_host.numel() * 4


def run_host(vs: VerifyStep, io: HostStepIO, host_logits: torch.Tensor,
             dev_logits: torch.Tensor | None, stream=None) -> int:
    """One end-to-end compact step from pinned host buffers.

    ``host_logits`` (pinned, [rows, V]) holds the target logits of the packed
    rows in packed order, standing in for the verify forward's output.  With
    ``dev_logits`` (a device buffer) the host reads the packed total after the
    plan and copies that many rows in; with ``dev_logits=None`` the accept
    reads the packed rows straight from the pinned buffer over the host link
    (no host synchronisation inside the step).  Returns the number of logits
    bytes moved host -> device.
    """
    s = torch.cuda.current_stream() if stream is None else stream
    with torch.cuda.stream(s):
        # the inputs and a zero status word: one copy
        vs.arena[:vs.n_in].copy_(io.in_arena, non_blocking=True)
        vs.plan_pack(s)
        if dev_logits is None:
            vs.greedy_accept(host_logits, write_argmax=False, stream=s)
            rows = -1
        else:
            io.totals.copy_(vs.totals, non_blocking=True)
            s.synchronize()  # the host needs the packed total to run the verify window
            rows = int(io.totals[0])
            dev_logits[:rows].copy_(host_logits[:rows], non_blocking=True)
            vs.greedy_accept(dev_logits, write_argmax=False, stream=s)
        # the status and every output: one copy
        io.out_host.copy_(vs.arena[vs.out_lo:], non_blocking=True)
        s.synchronize()
    if rows < 0:
        rows = int(io.totals[0])
    return rows * host_logits.stride(0) * host_logits.element_size()
