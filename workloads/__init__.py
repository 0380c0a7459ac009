"""Seeded synthetic inputs for the multi-LoRA delta (shared by the GPU path's
tests/bench and by the CPU oracle's harness; holds none of the method's arithmetic)."""
from .spec import (ALPHA, CONFIGS, Batch, Pool, Workload, config0, config1, config2, config3,
                   config4, decode_workload, mixed_workload, prefill_workload, zipf_probs)

__all__ = ["ALPHA", "CONFIGS", "Batch", "Pool", "Workload", "config0", "config1", "config2",
           "config3", "config4", "decode_workload", "mixed_workload", "prefill_workload",
           "zipf_probs"]
