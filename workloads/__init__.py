"""Seeded synthetic inputs for the multi-LoRA delta (shared by the GPU path's
tests/bench and by the CPU oracle's harness; holds none of the method's arithmetic)."""
from .spec import (ALPHA, WORKLOADS, Batch, Pool, Workload, decode_workload, llama3_8b_decode,
                   llama3_8b_mixed, llama3_8b_prefill, llama7b_decode, llama7b_prefill, mixed_13b, mixed_workload,
                   pool_stress, prefill_workload, tiny_decode, zipf_probs)

__all__ = ["ALPHA", "WORKLOADS", "Batch", "Pool", "Workload", "decode_workload", "llama3_8b_decode",
           "llama3_8b_mixed", "llama3_8b_prefill", "llama7b_decode", "llama7b_prefill", "mixed_13b", "mixed_workload",
           "pool_stress", "prefill_workload", "tiny_decode", "zipf_probs"]
