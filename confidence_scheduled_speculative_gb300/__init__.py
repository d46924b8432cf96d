"""GB300-native DSpark confidence-scheduled speculative decoding hot path.

The per-step verify planner (STS survivals, budget argmax, verify_lens), the
ragged verify pack (cu_seqlens, graph-tier round-up) and the greedy / cap
accept run as hand-written sm_103a CUDA kernels inside ``libdspark.so``,
whose C ABI is declared in ``include/dspark.h``.  ``api`` is the thin Python
binding (argument marshalling only); ``workloads`` draws seeded synthetic
inputs.
"""

__all__ = ["api", "workloads"]
