"""The separate shrink and expand entry points (lora_shrink, lora_expand) and the
tensor-parallel delta built on them, against the fp64 oracle through the C ABI.

The tensor-parallel cases emulate N ranks on one GPU: shard k is a pool made of columns
[k h/N, (k+1) h/N) of every page of the full pool (same page table), with the matching
column shards of x and y; every shard's shrink writes its partial t, the partial t are
summed (what the all-reduce does across GPUs), and every shard expands its own output
columns.  The assembled y must match the oracle's unsharded delta."""
import numpy as np
import pytest

from workloads.materialize import host_inputs

from .harness import T_ACC, GpuCase, full_check, magnitude_sums, oracle_problem
from .test_gpu_parity import _widths_case, small_decode, small_prefill

pytestmark = pytest.mark.gpu


CASES = {
    "decode-h4096": lambda: small_decode(101, 4096, 1, 3, 12, [1, 8, 32, 64], 37, zipf=1.1),
    "decode-h512-ranks-to-256": lambda: small_decode(102, 512, 2, 2, 9, [3, 16, 128, 256], 29),
    "prefill-rows-h2048": lambda: small_prefill(103, 2048, 1, 2, 6, [8, 16, 64], [5, 130, 1, 40]),
    "widths-h1024": lambda: _widths_case("decode", 104, 1024, [(1024, 256), (2560, 1024), (1024, 1032)], 7,
                                         [4, 16, 64], T_dec=25),
    "many-projections": lambda: small_decode(105, 256, 5, 4, 6, [4, 8], 17),   # 20: several launches
}


def _ids(case):
    return case.torch.from_numpy(case.wl.batch.token_adapter()).to(case.device)


@pytest.mark.parametrize("name", list(CASES))
def test_shrink_then_expand(name):
    """t from lora_shrink against the oracle's (scaled) shrink, within the fp32 accumulation
    bound; y after lora_expand against the oracle's delta (y0 = 0: the strict bound too)."""
    import torch
    wl = CASES[name]()
    case = GpuCase(wl, y0_zero=True)
    try:
        ids = _ids(case)
        nprob = len(wl.problems)
        # every row is its own segment here: the workspace for T rows and T segments
        nb = case.lora.workspace_size(case.pool, case.T, case.T)
        ws = torch.empty(nb, dtype=torch.uint8, device=case.device)
        case.lora.workspace_init(ws, nb, case.stream)
        t = torch.zeros((nprob, case.T, wl.pool.r_max), dtype=torch.float32, device=case.device)
        case.lora.shrink(case.pool, case.problems(), ids, case.T, ws, nb, t, case.stream)
        case.lora.expand(case.pool, case.problems(), case.T, ws, nb, t, case.stream)
        assert case.lora.get_device_error(ws, case.stream) == 0
        full_check(wl, case, list(range(nprob)))
        hi = host_inputs(wl)
        tok = wl.batch.token_adapter()
        t_gpu = t.cpu().numpy().astype(np.float64)
        for i, (l, p) in enumerate(case.dev.problems[:4]):
            _, t_ref, _ = oracle_problem(wl, hi, l, p, want_t=True)
            S, _ = magnitude_sums(wl, hi, l, p)
            for row in np.nonzero(tok >= 0)[0]:
                a = tok[row]
                r, s = int(wl.pool.ranks[a]), float(wl.pool.scales[a])
                err = np.abs(t_gpu[i, row, :r] - s * t_ref[row, :r])
                assert np.all(err <= s * T_ACC * S[row, :r]), (i, row, err.max())
    finally:
        case.close()


@pytest.mark.parametrize("n_shards", [2, 4])
@pytest.mark.parametrize("name", ["decode-h4096", "prefill-rows-h2048"])
def test_tensor_parallel_delta_emulated(name, n_shards):
    """N shards of the pool, their partial shrinks summed, each shard's expand into its
    output columns: the whole delta of the oracle (strict bound, y0 = 0)."""
    import torch

    import heterogeneous_adapters_gb300 as lora
    from heterogeneous_adapters_gb300 import tp
    wl = CASES[name]()
    case = GpuCase(wl, y0_zero=True)
    try:
        p = wl.pool
        d = case.dev
        ids = _ids(case)
        nprob = len(wl.problems)
        shards = []
        for k in range(n_shards):
            lo, hi_ = tp.shard_range(p.h, n_shards, k)
            pages = d.pool[:, lo:hi_].contiguous()
            pool_k = lora.Pool(pages, p.num_pages, hi_ - lo, d.pt, p.pt.size, d.pt_off, d.ranks, d.scales,
                               p.num_adapters, p.num_layers, p.num_proj, p.r_max)
            x_k = d.x[:, :, lo:hi_].contiguous()
            y_k = d.y[:, :, lo:hi_].contiguous()
            probs_k = [(x_k[d.x_src[i]], y_k[i], hi_ - lo, hi_ - lo, l, pj) for i, (l, pj) in enumerate(d.problems)]
            nb = lora.workspace_size(pool_k, case.T, case.T)
            ws_k = torch.empty(nb, dtype=torch.uint8, device=case.device)
            lora.workspace_init(ws_k, nb, case.stream)
            t_k = torch.zeros((nprob, case.T, p.r_max), dtype=torch.float32, device=case.device)
            shards.append(dict(lo=lo, hi=hi_, pool=pool_k, pages=pages, x=x_k, y=y_k, probs=probs_k, ws=ws_k,
                               nb=nb, t=t_k))
        for s in shards:
            lora.shrink(s["pool"], s["probs"], ids, case.T, s["ws"], s["nb"], s["t"], case.stream)
        t_sum = torch.stack([s["t"] for s in shards]).sum(0)   # the all-reduce across the GPUs
        for s in shards:
            lora.expand(s["pool"], s["probs"], case.T, s["ws"], s["nb"], t_sum, case.stream)
            d.y[:, :, s["lo"]:s["hi"]] = s["y"]
            assert lora.get_device_error(s["ws"], case.stream) == 0
        full_check(wl, case, list(range(nprob)))
        for s in shards:
            s["pool"].close()
    finally:
        case.close()


def test_shrink_expand_host_checks():
    import torch
    wl = CASES["decode-h4096"]()
    case = GpuCase(wl)
    try:
        ids = _ids(case)
        t = torch.zeros((3, case.T, wl.pool.r_max), dtype=torch.float32, device=case.device)
        with pytest.raises(case.lora.LoraError) as ei:
            case.lora.shrink(case.pool, case.problems(), ids, case.T, case.ws, case.ws_bytes, t.view(-1)[1:],
                             case.stream)   # t not 16-byte aligned
        assert ei.value.status == 2
        with pytest.raises(case.lora.LoraError):
            case.lora.expand(case.pool, case.problems(), case.T, case.ws, case.ws_bytes, None, case.stream)
        assert case.error_bits() == 0
    finally:
        case.close()
