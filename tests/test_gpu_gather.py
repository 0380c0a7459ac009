"""Decode batches in which some adapters serve many tokens (gathered tensor-core tiles) and
prefill batches of short segments (tensor-core tiles packing several K chunks, B^T slices
or y slices per ring stage), against the fp64 oracle through the C ABI.

Every case runs with y0 = 0, so the strict delta-only bound applies as well as the gate;
x rows of the gathered tiles come from anywhere in the batch, and the tiles' padding rows
(beyond the group's tokens) must leave every other row untouched."""
import numpy as np
import pytest

from workloads import spec
from workloads.spec import Batch, Workload, all_problems, make_pool_all_resident

from .harness import GpuCase, full_check
from .test_gpu_parity import _widths_case, small_prefill

pytestmark = pytest.mark.gpu


def hot_decode(seed, h, L, P, hot, cold_tokens, n_cold_adapters, cold_ranks, base_tokens=0):
    """Decode batch: hot adapter k (ids 0, 1, ...) of rank hot[k][1] serves hot[k][0] tokens;
    cold_tokens more tokens draw uniformly among n_cold_adapters others; base_tokens are
    base-only.  Tokens are shuffled through the batch."""
    rng = np.random.default_rng(seed)
    n_hot = len(hot)
    ranks = np.concatenate([np.asarray([r for _, r in hot], np.int32),
                            rng.choice(np.asarray(cold_ranks, np.int32), size=n_cold_adapters)])
    ids = np.concatenate([np.full(n, k, np.int32) for k, (n, _) in enumerate(hot)] +
                         [rng.integers(n_hot, n_hot + n_cold_adapters, size=cold_tokens).astype(np.int32),
                          np.full(base_tokens, -1, np.int32)])
    rng.shuffle(ids)
    pool = make_pool_all_resident(rng, h, L, P, ranks)
    batch = Batch(np.zeros(1, np.int32), np.zeros(0, np.int32), ids)
    return Workload(f"hot-decode-h{h}-t{ids.size}", seed, pool, batch, all_problems(L, P))


HOT = {
    # one adapter with 64 tokens and nothing else (the single-adapter decode batch)
    "h4096-one-adapter-64": lambda: hot_decode(81, 4096, 1, 3, [(64, 16)], 0, 1, [8]),
    # groups of 5 .. 64 tokens, ranks 8 .. 128, beside cold tokens and base-only rows
    "h4096-mixed-groups": lambda: hot_decode(82, 4096, 1, 3, [(5, 8), (9, 64), (33, 128), (64, 32), (16, 1)],
                                             40, 30, [8, 16, 64], base_tokens=7),
    # a group longer than one tile (130 and 257 tokens: two and three tiles, ragged)
    "h2048-multi-tile-groups": lambda: hot_decode(83, 2048, 2, 2, [(130, 16), (257, 64), (8, 24)],
                                                  20, 10, [4, 16]),
    # rank 256 groups stay on the CUDA-core path beside gathered ones
    "h5120-rank256-and-gathered": lambda: hot_decode(84, 5120, 1, 2, [(20, 256), (20, 128), (12, 8)],
                                                     9, 5, [16]),
    # a narrow pool (one 16-byte vector per thread in the ring body)
    "h1024-hot": lambda: hot_decode(85, 1024, 2, 3, [(48, 64), (11, 16)], 30, 12, [4, 8, 32]),
}


@pytest.mark.parametrize("gather", [None, 2, 0])
@pytest.mark.parametrize("name", list(HOT))
def test_hot_adapter_decode(name, gather):
    """Default tuning (groups of 8 or more tokens on gathered tiles), every group of 2 or
    more tokens on them, and none (the CUDA-core ring alone)."""
    wl = HOT[name]()
    tuning = {"split_max_problems": 0}
    if gather is not None:
        tuning["gather_min_rows"] = gather
    case = GpuCase(wl, y0_zero=True, tuning=tuning)
    try:
        assert case.run() == 0
        full_check(wl, case, list(range(len(wl.problems))))
    finally:
        case.close()


def test_hot_adapter_decode_gathered_equals_ring_within_rounding():
    """The same batch through gathered tiles and through the ring: both within the strict
    bound of the oracle (checked above), and the two GPU results differ by at most the
    final bf16 rounding plus fp32 accumulation order."""
    import torch
    wl = HOT["h4096-mixed-groups"]()
    outs = []
    for gather in (2, 0):
        case = GpuCase(wl, y0_zero=True, tuning={"split_max_problems": 0, "gather_min_rows": gather})
        try:
            assert case.run() == 0
            outs.append(case.dev.y.float().cpu())
        finally:
            case.close()
    a, b = outs
    assert torch.all((a - b).abs() <= 2 ** -7 * torch.maximum(a.abs(), b.abs()) + 1e-6)


@pytest.mark.parametrize("kind", ["decode"])
def test_hot_adapter_decode_projection_widths(kind):
    """Gathered tiles over Llama-3-8B widths (k/v outputs of 1,024, MLP of 14,336): the shrink
    K loop and the expand's slices cross page blocks of a vector."""
    dims = [(4096, 4096), (4096, 1024), (4096, 14336), (14336, 4096)]
    wl = _widths_case(kind, 86, 4096, dims, 3, [8, 64], T_dec=40)
    case = GpuCase(wl, y0_zero=True, tuning={"split_max_problems": 0, "gather_min_rows": 2})
    try:
        assert case.run() == 0
        full_check(wl, case, list(range(len(wl.problems))))
    finally:
        case.close()


@pytest.mark.parametrize("rank", [8, 16, 64, 128])
def test_short_segment_tiles_pack_stages(rank):
    """Prefill segments of 2 .. 40 rows, all on the tensor cores: a tile of few rows packs
    several K chunks into a shrink stage, several B^T slices and y slices into theirs."""
    lens = [2, 3, 8, 16, 31, 32, 33, 40, 5, 17, 24]
    wl = small_prefill(87 + rank, 4096, 1, 2, len(lens), [rank], lens, ids=np.arange(len(lens)))
    case = GpuCase(wl, y0_zero=True, tuning={"mma_min_rows": 2})
    try:
        assert case.run() == 0
        full_check(wl, case, list(range(len(wl.problems))))
    finally:
        case.close()
