"""ORACLE — test infrastructure only.

A plain fp64 CPU implementation of the multi-LoRA delta and of its integer steps,
written from the pages' definitions.  Only tests/, __graft_entry__.smoke() and
bench.py's CPU-baseline / reference legs may use it; it shares no code with the
CUDA path (heterogeneous_adapters_gb300) and neither imports the other.
"""
from .oracle import (ERRORS, OracleError, build, group_tokens, lora_delta,
                     lora_expand, page_list)

__all__ = ["ERRORS", "OracleError", "build", "group_tokens",
           "lora_delta", "lora_expand", "page_list"]
