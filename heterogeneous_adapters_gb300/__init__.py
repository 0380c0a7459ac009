"""GB300-native multi-LoRA delta: BGMV (decode) and SGMV (prefill) over a unified
paged adapter pool, as hand-written sm_103a CUDA kernels behind a C ABI
(include/lora.h, liblora.so).  This package holds the kernels' sources (csrc/),
the in-tree build, the ctypes binding and the byte/flop model used to report
throughput against the HBM roofline."""
from . import costmodel
from ._binding import (DERR, LORA_MAX_PROBLEMS_PER_LAUNCH, LORA_MAX_RANK, LORA_MAX_SEGMENTS,
                       LORA_NOALLOC_MAX_TOKENS, LoraError, Pool, apply_mixed, bgmv, bgmv_noalloc, debug_delta_with_t, debug_page_list,
                       delta_grouped, get_device_error, lib, segment, sgmv, stage_pages, workspace_init,
                       workspace_size, workspace_view)

__all__ = ["costmodel", "DERR", "LORA_MAX_PROBLEMS_PER_LAUNCH", "LORA_MAX_RANK",
           "LORA_MAX_SEGMENTS", "LORA_NOALLOC_MAX_TOKENS", "LoraError", "Pool", "apply_mixed",
           "bgmv", "bgmv_noalloc", "debug_delta_with_t",
           "debug_page_list", "delta_grouped", "get_device_error", "lib", "segment", "sgmv",
           "stage_pages",
           "workspace_init", "workspace_size", "workspace_view"]
