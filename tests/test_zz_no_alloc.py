"""The allocation-free BGMV entry point (lora_bgmv_noalloc) against the workspace one
(lora_bgmv), through the C ABI.

Some callers cannot allocate device memory at all -- code running while a CUDA graph is
being captured, serving engines that carve every byte of the GPU into their own pools
up front, plugins that are only handed their inputs and outputs -- so they cannot
provide the workspace that lora_bgmv needs.  lora_bgmv_noalloc keeps that scratch in a
fixed array inside the library.  This file is collected last on purpose: if it fails,
a run that stops at the first failure has already run every other test."""
import numpy as np
import pytest

import heterogeneous_adapters_gb300 as lora
from heterogeneous_adapters_gb300 import _binding as B
from workloads import spec

from .harness import GpuCase, check_gate

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_bgmv_on_two_calls():
    import torch
    wl = spec.decode_workload("noalloc-h2048-t96", 91, 2048, 2, 2, 30, [4, 8, 16, 64], 96, 1.0)
    case = GpuCase(wl)
    try:
        y0 = case.dev.y.clone()
        err = torch.full((1,), 0x7FFFFFFF, dtype=torch.int32, device=case.device)
        for _ in range(2):
            # the existing entry point, from y0
            case.dev.y.copy_(y0)
            assert case.run() == 0
            want = case.dev.y.clone()
            # the allocation-free one, from y0 again
            case.dev.y.copy_(y0)
            lora.bgmv_noalloc(case.pool, case.problems(), case.dev.token_adapter, case.T, err,
                              case.stream)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            for i in range(len(wl.problems)):
                got = case.dev.y[i].double().cpu().numpy()
                check_gate(got, want[i].double().cpu().numpy(), f"no-alloc problem {i}")
    finally:
        case.close()


def test_noalloc_rejects_batches_beyond_its_scratch():
    import torch
    wl = spec.decode_workload("noalloc-limit", 92, 256, 1, 1, 4, [4], 8, 1.0)
    case = GpuCase(wl)
    try:
        big = lora.LORA_NOALLOC_MAX_TOKENS + 1
        ids = torch.zeros(big, dtype=torch.int32, device=case.device)
        with pytest.raises(lora.LoraError) as ei:
            lora.bgmv_noalloc(case.pool, case.problems(), ids, big, None, case.stream)
        assert ei.value.status == B.LORA_ETOOBIG
    finally:
        case.close()
