"""The allocation-free BGMV entry point (lora_bgmv_noalloc) against the workspace one
(lora_bgmv) and against the fp64 oracle, through the C ABI.

Some callers have no way to get device memory for a workspace: a serving engine that
reserves all of the GPU's memory for its own pools when it starts, a plugin that its host
framework hands only input and output buffers, a step loop in which a cudaMalloc (which
may synchronise the device) is not allowed.  lora_bgmv_noalloc keeps that scratch in a
fixed array inside the library.  It runs the same kernels as lora_bgmv, chosen by the same
rules, so on the same batch the two must agree bit for bit.

This file is collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test."""
import numpy as np
import pytest

import heterogeneous_adapters_gb300 as lora
from heterogeneous_adapters_gb300 import _binding as B
from workloads import spec

from .harness import GpuCase, full_check

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nprob,path", [(4, "ring"), (1, "cluster")])
def test_noalloc_matches_workspace_bgmv_on_two_calls(nprob, path):
    """Four projections run the ring kernel; one projection of a 96-row batch runs the
    cluster kernel.  Two calls in a row, each from the same y0: bit-identical to lora_bgmv,
    and within the parity gate of the oracle (with y0 = 0, the strict delta-only bound
    too)."""
    import torch
    L, P = (2, 2) if nprob == 4 else (1, 1)
    wl = spec.decode_workload(f"noalloc-h2048-t96-{path}", 91, 2048, L, P, 30, [4, 8, 16, 64], 96, 1.0)
    case = GpuCase(wl, y0_zero=True)
    try:
        assert len(wl.problems) == nprob
        y0 = case.dev.y.clone()
        err = torch.full((1,), 0x7FFFFFFF, dtype=torch.int32, device=case.device)
        for _ in range(2):
            case.dev.y.copy_(y0)
            assert case.run() == 0                     # lora_bgmv with a workspace
            want = case.dev.y.clone()
            case.dev.y.copy_(y0)
            lora.bgmv_noalloc(case.pool, case.problems(), case.dev.token_adapter, case.T, err,
                              case.stream)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            assert torch.equal(case.dev.y.view(torch.int16), want.view(torch.int16)), \
                "lora_bgmv_noalloc differs from lora_bgmv"
            full_check(wl, case, list(range(nprob)))
    finally:
        case.close()


def test_noalloc_reports_device_errors_per_call():
    """A bad adapter id sets the adapter bit in this call's error_bits; the next correct
    call reports 0 (the array's error word is cleared at every call)."""
    import torch
    wl = spec.decode_workload("noalloc-err", 93, 512, 1, 2, 6, [4, 8], 20, 1.0)
    case = GpuCase(wl)
    try:
        err = torch.zeros(1, dtype=torch.int32, device=case.device)
        ids = case.dev.token_adapter.clone()
        bad = ids.clone()
        bad[int(np.nonzero(wl.batch.token_adapter() >= 0)[0][0])] = wl.pool.num_adapters + 1
        lora.bgmv_noalloc(case.pool, case.problems(), bad, case.T, err, case.stream)
        torch.cuda.synchronize()
        assert int(err.item()) & 0x1
        lora.bgmv_noalloc(case.pool, case.problems(), ids, case.T, err, case.stream)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
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
