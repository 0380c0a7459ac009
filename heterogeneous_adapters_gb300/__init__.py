"""GB300-native multi-LoRA delta: BGMV (decode) and SGMV (prefill) over a unified
paged adapter pool, as hand-written sm_103a CUDA kernels behind a C ABI
(include/lora.h, liblora.so), and the host runtime around them: the adapter cache over
the pool's pages and the batch scheduler (include/lora_runtime.h).  This package holds
the sources (csrc/), the in-tree build, the ctypes binding and the byte/flop model used
to report throughput against the HBM roofline."""
from . import costmodel
from ._binding import (DERR, LORA_ENOSPACE, LORA_MAX_PROBLEMS_PER_LAUNCH, LORA_MAX_RANK,
                       LORA_MAX_SEGMENTS, LORA_NOALLOC_MAX_TOKENS, LORA_STAGE_MAX_RUNS, LORA_UNIT_ABSENT,
                       LORA_UNIT_LOADING,
                       LORA_UNIT_READY, AdapterCache, LoraError, Pool, Scheduler, apply_mixed, bgmv,
                       bgmv_noalloc, debug_delta_with_t, debug_page_list, debug_wait_limit, delta_grouped,
                       expand, get_device_error, shrink,
                       lib, segment, sgmv, stage_pages, stage_pages_ce, workspace_init, workspace_size,
                       workspace_view)

__all__ = ["costmodel", "DERR", "LORA_ENOSPACE", "LORA_MAX_PROBLEMS_PER_LAUNCH", "LORA_MAX_RANK",
           "LORA_MAX_SEGMENTS", "LORA_NOALLOC_MAX_TOKENS", "LORA_STAGE_MAX_RUNS", "LORA_UNIT_ABSENT",
           "LORA_UNIT_LOADING",
           "LORA_UNIT_READY", "AdapterCache", "LoraError", "Pool", "Scheduler", "apply_mixed",
           "bgmv", "bgmv_noalloc", "debug_delta_with_t", "debug_page_list", "debug_wait_limit",
           "delta_grouped", "expand", "shrink",
           "get_device_error", "lib", "segment", "sgmv", "stage_pages", "stage_pages_ce", "workspace_init",
           "workspace_size", "workspace_view"]
