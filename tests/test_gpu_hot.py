"""Decode batches in which some adapters serve many tokens (groups cut into many chunks of
the CUDA-core kernels) and prefill batches of short segments on the tensor-core tiles,
against the fp64 oracle through the C ABI.

Every case runs with y0 = 0, so the strict delta-only bound applies as well as the gate."""
import numpy as np
import pytest

from workloads import spec
from workloads.spec import Batch, Workload, all_problems, make_pool_all_resident

from .harness import GpuCase, full_check
from .test_gpu_parity import small_prefill

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
    # a rank-256 group (above the tensor-core limit) beside rank-128 and rank-8 groups
    "h5120-rank256-and-gathered": lambda: hot_decode(84, 5120, 1, 2, [(20, 256), (20, 128), (12, 8)],
                                                     9, 5, [16]),
    # a narrow pool (one 16-byte vector per thread in the ring body)
    "h1024-hot": lambda: hot_decode(85, 1024, 2, 3, [(48, 64), (11, 16)], 30, 12, [4, 8, 32]),
}


@pytest.mark.parametrize("path", ["ring", "cluster"])
@pytest.mark.parametrize("name", list(HOT))
def test_hot_adapter_decode(name, path):
    """Adapters with 5 .. 257 tokens of one decode batch, through the ring kernel and through
    the few-projection kernels (every projection of the batch in one launch)."""
    wl = HOT[name]()
    tuning = {"ring": {"split_max_problems": 0}, "cluster": {"split_max_problems": 8}}[path]
    case = GpuCase(wl, y0_zero=True, tuning=tuning)
    try:
        assert case.run() == 0
        full_check(wl, case, list(range(len(wl.problems))))
    finally:
        case.close()


@pytest.mark.parametrize("rank", [8, 16, 64, 128])
def test_short_segment_tiles(rank):
    """Prefill segments of 2 .. 40 rows, all on the tensor-core tiles (ragged 32-row boxes,
    tiles of a few rows), each segment with its own adapter."""
    lens = [2, 3, 8, 16, 31, 32, 33, 40, 5, 17, 24]
    wl = small_prefill(87 + rank, 4096, 1, 2, len(lens), [rank], lens, ids=np.arange(len(lens)))
    case = GpuCase(wl, y0_zero=True, tuning={"mma_min_rows": 2})
    try:
        assert case.run() == 0
        full_check(wl, case, list(range(len(wl.problems))))
    finally:
        case.close()
