"""GPU path vs fp64 oracle, elementwise, through the C ABI (liblora.so).

Small cases cover every element; the five full-size workloads run in the same
launch configuration as the bench (all projections of one step in one call) and
compare sampled projections element by element, plus properties over all of them.
"""
import numpy as np
import pytest

from workloads import spec
from workloads.spec import Batch, Workload, all_problems, make_pool_all_resident

from .harness import GpuCase, check_gate, full_check, oracle_problem

pytestmark = pytest.mark.gpu


def small_decode(seed, h, L, P, N, ranks, T, zipf=1.0, base=False):
    return spec.decode_workload(f"decode-h{h}-t{T}", seed, h, L, P, N, ranks, T,
                                None if base else zipf, base_ids=base)


def small_prefill(seed, h, L, P, N, ranks, lens, ids=None):
    rng = np.random.default_rng(seed)
    ranks_a = rng.choice(np.asarray(ranks, np.int32), size=N)
    pool = make_pool_all_resident(rng, h, L, P, ranks_a, num_pages=None)
    lens = np.asarray(lens)
    if ids is None:
        ids = rng.choice(N, size=lens.size, p=spec.zipf_probs(N, 1.0))
    seg_start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    batch = Batch(seg_start, np.asarray(ids, np.int32), np.zeros(0, np.int32))
    return Workload(f"prefill-h{h}-s{lens.size}", seed, pool, batch, all_problems(L, P))


def _mixed(seed, h, L, P, N, ranks, lens, n_dec, n_base):
    rng = np.random.default_rng(seed)
    ranks_a = rng.choice(np.asarray(ranks, np.int32), size=N)
    n_req = len(lens) + n_dec
    ids = rng.choice(N, size=n_req, p=spec.zipf_probs(N, 0.8))
    ids[rng.choice(n_req, size=n_base, replace=False)] = -1
    pool = make_pool_all_resident(rng, h, L, P, ranks_a, num_pages=None)
    seg_start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    batch = Batch(seg_start, ids[:len(lens)].astype(np.int32), ids[len(lens):].astype(np.int32))
    return Workload(f"mixed-h{h}", seed, pool, batch, all_problems(L, P))


SMALL = {
    "tiny": spec.tiny_decode,
    "decode-h512-ragged-ranks": lambda: small_decode(41, 512, 2, 4, 20, [1, 3, 8, 16, 64], 37),
    "decode-h5120": lambda: small_decode(43, 5120, 1, 2, 10, [8, 128], 20),
    "decode-h4096-r256": lambda: small_decode(44, 4096, 1, 1, 3, [256], 9),
    "decode-h6144": lambda: small_decode(58, 6144, 1, 2, 8, [8, 64], 13),
    "decode-h8192": lambda: small_decode(59, 8192, 1, 1, 6, [16, 128], 11),
    "prefill-h8192": lambda: small_prefill(60, 8192, 1, 1, 5, [8, 64, 128], [150, 40, 3]),
    "mixed-h6144": lambda: _mixed(61, 6144, 1, 1, 9, [16, 128], [140, 7], 12, 2),
    "decode-base-uniform": lambda: small_decode(45, 1024, 1, 2, 6, [4, 16], 25, base=True),
    "prefill-h1024-ragged": lambda: small_prefill(46, 1024, 1, 3, 8, [8, 16, 32],
                                                  [1, 7, 130, 300, 2, 64, 129, 5, 0, 17, 255, 3]),
    "prefill-h4096-r256-and-r8": lambda: small_prefill(49, 4096, 1, 2, 4, [8, 256],
                                                       [200, 40, 33, 128]),
    "prefill-h2048-all-ranks": lambda: small_prefill(50, 2048, 2, 1, 24, [1, 8, 16, 24, 32, 48, 64, 96, 128],
                                                     [129, 257, 31, 32, 500, 128, 7, 64]),
    "mixed-h2048": lambda: _mixed(47, 2048, 2, 2, 30, [8, 16, 32, 64, 128], [5, 260, 131], 40, 5),
    "mixed-h5120": lambda: _mixed(48, 5120, 1, 2, 12, [8, 128], [300, 9], 17, 3),
    # more projections than one launch takes (256 for the CUDA-core kernel, 64 for tiles)
    "decode-320-projections": lambda: small_decode(67, 256, 80, 4, 9, [2, 8, 16], 21),
    "mixed-320-projections": lambda: _mixed(68, 256, 80, 4, 9, [4, 16], [70, 2, 40], 11, 2),
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("y0_zero", [False, True])
def test_small_parity(name, y0_zero):
    wl = SMALL[name]()
    case = GpuCase(wl, y0_zero=y0_zero)
    try:
        assert case.run() == 0
        full_check(wl, case, list(range(len(wl.problems))))
    finally:
        case.close()


@pytest.mark.parametrize("mma_min", [0, 2, 128])
def test_prefill_size_classes(mma_min):
    """The same prefill batch with every segment on the CUDA-core path (0), every segment of
    more than one row on the tensor-core path (2), and only full-tile segments on it (128)."""
    wl = small_prefill(57, 1024, 2, 2, 10, [8, 16, 32, 64, 128], [1, 2, 127, 128, 129, 300, 64, 0, 9])
    case = GpuCase(wl, y0_zero=True, tuning={"mma_min_rows": mma_min})
    try:
        assert case.run() == 0
        full_check(wl, case, list(range(len(wl.problems))))
    finally:
        case.close()


@pytest.mark.parametrize("pages", [4, 8])
def test_decode_ring_stage_shapes(pages):
    """The decode ring with 4 and with 8 rows per stage on the same batch: ranks that are
    not multiples of either and chunks of 1 to 4 rows (a skewed adapter mix)."""
    wl = small_decode(65, 2048, 1, 3, 12, [1, 3, 5, 8, 13, 64, 100], 57, zipf=1.3)
    # the ring kernel, not the cluster kernel
    case = GpuCase(wl, tuning={"ring_rows_per_stage": pages, "split_max_problems": 0})
    try:
        assert case.run() == 0
        full_check(wl, case, list(range(len(wl.problems))))
    finally:
        case.close()


@pytest.mark.parametrize("path", ["ring", "cluster"])
@pytest.mark.parametrize("h", [512, 4096, 5120, 8192])
def test_decode_cluster_and_ring_paths(path, h):
    """The same few-projection decode batch through the cluster kernel (each chunk split over
    8 CTAs) and the ring kernel (6 projections in one launch): ranks not multiples of 8 rows,
    chunks of 1 to 4 rows, base-only rows, ranks up to 128."""
    wl = small_decode(66, h, 2, 3, 10, [1, 5, 8, 16, 64, 128], 47, zipf=1.2)
    wl.batch.dec_adapter[::9] = -1
    tuning = {"ring": {"split_max_problems": 0}, "cluster": {"split_max_problems": 8}}[path]
    case = GpuCase(wl, tuning=tuning)
    try:
        assert case.run() == 0
        full_check(wl, case, list(range(len(wl.problems))))
    finally:
        case.close()


@pytest.mark.parametrize("kind", ["prefill", "mixed", "decode"])
def test_shared_x_inputs(kind):
    """q, k and v of a layer read one x buffer (the other projections' own x buffers hold
    NaN, so reading one of them would show); the tensor-core items of a tile for those
    projections run side by side."""
    import dataclasses

    import torch
    if kind == "prefill":
        wl = small_prefill(67, 1024, 2, 4, 8, [8, 16, 64], [200, 33, 7, 130])
    elif kind == "mixed":
        wl = _mixed(68, 2048, 1, 4, 12, [8, 32, 128], [150, 40], 30, 3)
    else:
        wl = small_decode(69, 2048, 2, 4, 15, [4, 16, 64], 40)
    wl = dataclasses.replace(wl, shared_x=True)
    case = GpuCase(wl)
    try:
        used = set(case.dev.x_src)
        assert len(used) < len(wl.problems)
        for i in range(len(wl.problems)):
            if i not in used:
                case.dev.x[i].fill_(float("nan"))
        torch.cuda.synchronize()
        assert case.run() == 0
        full_check(wl, case, list(range(len(wl.problems))))
    finally:
        case.close()


def test_t_matches_oracle_shrink():
    """fp32 t (the value the expand consumes, scaled) against the oracle's fp64 t."""
    import torch

    from .harness import T_ACC, magnitude_sums
    from workloads.materialize import host_inputs
    wl = small_decode(51, 2048, 1, 2, 12, [2, 8, 32, 64], 33)
    case = GpuCase(wl)
    try:
        lora = case.lora
        b = wl.batch
        lora.segment(case.pool, None, None, 0, case.dev.token_adapter, b.num_decode, case.T,
                     case.ws, case.ws_bytes, case.stream)
        hi = host_inputs(wl)
        ids = b.token_adapter()
        for i, (l, p) in enumerate(case.dev.problems):
            t_out = torch.zeros((case.T, wl.pool.r_max), dtype=torch.float32, device=case.device)
            lora.debug_delta_with_t(case.pool, case.problems()[i], case.ws, case.ws_bytes, t_out,
                                    case.stream)
            assert case.error_bits() == 0
            t_gpu = t_out.cpu().numpy().astype(np.float64)
            _, t_ref, _ = oracle_problem(wl, hi, l, p, want_t=True)
            S, _ = magnitude_sums(wl, hi, l, p)
            for row in np.nonzero(ids >= 0)[0]:
                a = ids[row]
                r = int(wl.pool.ranks[a])
                s = float(wl.pool.scales[a])
                err = np.abs(t_gpu[row, :r] - s * t_ref[row, :r])
                assert np.all(err <= s * T_ACC * S[row, :r]), (row, err.max())
    finally:
        case.close()


def test_repeat_calls_accumulate():
    """Two calls add the delta twice (y is updated in place, the queue resets itself)."""
    wl = small_decode(52, 1024, 1, 2, 9, [4, 8], 21)
    case = GpuCase(wl, y0_zero=True)
    try:
        assert case.run() == 0
        once = [case.y_f64(i) for i in range(len(wl.problems))]
        assert case.run() == 0
        for i in range(len(wl.problems)):
            twice = case.y_f64(i)
            check_gate(twice, 2 * once[i], "second call")
    finally:
        case.close()


def test_zero_B_leaves_y_bit_identical():
    import torch
    wl = small_decode(53, 1024, 2, 2, 10, [8, 16], 30)
    case = GpuCase(wl)
    try:
        pool = wl.pool
        b_pages = np.concatenate([pool.pt[pool.block_entries(a, l, p, 1)]
                                  for a in range(pool.num_adapters) for (l, p) in wl.problems])
        case.dev.pool[torch.from_numpy(b_pages.astype(np.int64)).to(case.device)] = 0
        before = [case.y_bits(i).copy() for i in range(len(wl.problems))]
        assert case.run() == 0
        for i in range(len(wl.problems)):
            after = case.y_bits(i)
            same = (after == before[i]) | ((before[i] == 0x8000) & (after == 0))  # -0 -> +0
            assert same.all()
    finally:
        case.close()


def test_page_placement_and_batch_order_invariance():
    """Moving pages in the pool, or permuting the batch, gives bit-identical rows."""
    import torch
    wl = small_decode(54, 2048, 1, 2, 15, [8, 16, 32], 40)
    base = GpuCase(wl)
    try:
        assert base.run() == 0
        ref = [base.y_bits(i).copy() for i in range(len(wl.problems))]
        # page placement: move every page q to slot perm[q]
        rng = np.random.default_rng(5)
        perm = torch.from_numpy(rng.permutation(wl.pool.num_pages)).to(base.device)
        moved = torch.empty_like(base.dev.pool)
        moved[perm] = base.dev.pool
        base.dev.pool.copy_(moved)
        base.dev.pt.copy_(perm[base.dev.pt.long()].int())
        base.dev.y.copy_(base.y_init)
        assert base.run() == 0
        for i in range(len(wl.problems)):
            assert np.array_equal(base.y_bits(i), ref[i])
        # batch order: permute rows of x, y and the adapter ids
        order = torch.from_numpy(rng.permutation(base.T)).to(base.device)
        base.dev.x.copy_(base.dev.x[:, order])
        base.dev.y.copy_(base.y_init[:, order])
        base.dev.token_adapter.copy_(base.dev.token_adapter[order])
        assert base.run() == 0
        o = order.cpu().numpy()
        for i in range(len(wl.problems)):
            assert np.array_equal(base.y_bits(i), ref[i][o])
    finally:
        base.close()


def test_empty_and_all_base_batches():
    wl = small_decode(55, 512, 1, 1, 4, [4], 8, base=True)
    wl.batch.dec_adapter[:] = -1
    case = GpuCase(wl)
    try:
        before = case.y_bits(0).copy()
        assert case.run() == 0
        assert np.array_equal(case.y_bits(0), before)
    finally:
        case.close()
    # empty batch: T = 0 is a no-op (buffers still valid pointers)
    case = GpuCase(small_decode(56, 512, 1, 1, 4, [4], 3))
    try:
        before = case.y_bits(0).copy()
        case.lora.bgmv(case.pool, case.problems(), case.dev.token_adapter, 0, case.ws,
                       case.ws_bytes, case.stream)
        assert case.error_bits() == 0
        assert np.array_equal(case.y_bits(0), before)
    finally:
        case.close()


# ----------------------------------------------------------------------------- full-size workloads

def _sample(n, k, seed):
    rng = np.random.default_rng(seed)
    return sorted(rng.choice(n, size=min(k, n), replace=False).tolist())


@pytest.mark.parametrize("cfg,k", [("decode", 8), ("prefill", 2), ("mixed", 2), ("stress-distinct", 4),
                                   ("stress-zipf", 4), ("llama3-decode", 7), ("llama3-prefill", 3),
                                   ("llama3-mixed", 3)])
def test_full_workload(cfg, k):
    import torch
    wl = spec.WORKLOADS[cfg]()
    case = GpuCase(wl, nan_dummies=True)
    try:
        assert case.run() == 0
        # properties over every projection: finite, base rows untouched, adapted rows changed
        ids = torch.from_numpy(wl.batch.token_adapter()).to(case.device)
        base_rows = ids == -1
        assert torch.isfinite(case.dev.y).all()
        if case.y_init is not None and base_rows.any():
            assert torch.equal(case.dev.y[:, base_rows], case.y_init[:, base_rows])
        full_check(wl, case, _sample(len(wl.problems), k, seed=sum(map(ord, str(cfg)))),
                   strict=False)
    finally:
        case.close()


@pytest.mark.parametrize("cfg,k", [("decode", 3), ("prefill", 1), ("mixed", 1), ("stress-distinct", 2),
                                   ("stress-zipf", 2), ("llama3-decode", 3), ("llama3-prefill", 2),
                                   ("llama3-mixed", 2)])
def test_full_workload_delta_only(cfg, k):
    """The full workloads with y0 = 0, so that y holds the delta alone (|delta| is ~0.05 of
    |y0| otherwise, where the gate could hide a dropped rank term): every sampled
    projection within the strict delta-only bound, in the launch configuration the bench
    times."""
    wl = spec.WORKLOADS[cfg]()
    case = GpuCase(wl, y0_zero=True, nan_dummies=True)
    try:
        assert case.run() == 0
        full_check(wl, case, _sample(len(wl.problems), k, seed=7 + sum(map(ord, str(cfg)))), strict=True)
    finally:
        case.close()


def _widths_case(kind, seed, h, dims, N, ranks, T_dec=0, lens=()):
    """One layer, one projection per (d_in, d_out) pair in dims, every adapter resident."""
    rng = np.random.default_rng(seed)
    P = len(dims)
    ranks_a = rng.choice(np.asarray(ranks, np.int32), size=N)
    pool = make_pool_all_resident(rng, h, 1, P, ranks_a, num_pages=None, proj_dims=dims)
    lens = np.asarray(lens, np.int64)
    ids = rng.choice(N, size=lens.size + T_dec, p=spec.zipf_probs(N, 1.0)).astype(np.int32)
    ids[::7] = -1
    seg_start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    batch = Batch(seg_start, ids[:lens.size], ids[lens.size:])
    return Workload(f"{kind}-widths-h{h}", seed, pool, batch, all_problems(1, P))


WIDTH_CASES = {
    # narrower k/v outputs, a 2.5-page output and input, an output one page plus 8 columns
    "h1024-mixed-widths": (1024, [(1024, 256), (1024, 2560), (2560, 1024), (1024, 1032),
                                  (1024, 1024)]),
    # Llama-3-8B shapes: q, k, v, o, gate, up, down
    "h4096-llama3-8b": (4096, [(4096, 4096), (4096, 1024), (4096, 1024), (4096, 4096),
                               (4096, 14336), (4096, 14336), (14336, 4096)]),
    # the widest vector a pool allows (16 pages) on both sides
    "h512-max-pages": (512, [(8192, 8), (8, 8192)]),
}


@pytest.mark.parametrize("case_name", list(WIDTH_CASES))
@pytest.mark.parametrize("path", ["decode-cluster", "decode-ring", "prefill", "mixed"])
def test_projection_widths(case_name, path):
    """Projections whose input and output widths differ from h (vectors spanning several
    pool pages, the last one partly used).  x columns past a problem's d_in hold NaN and y
    columns past its d_out must come back unchanged."""
    h, dims = WIDTH_CASES[case_name]
    tuning = {"decode-cluster": {"split_max_problems": 8},
              "decode-ring": {"split_max_problems": 0}}.get(path)
    kind = path.split("-")[0]
    if kind == "decode":
        wl = _widths_case(kind, 70, h, dims, 9, [1, 5, 8, 16, 64], T_dec=29)
    elif kind == "prefill":
        wl = _widths_case(kind, 71, h, dims, 6, [8, 16, 128], lens=[1, 130, 17, 64, 0, 5])
    else:
        wl = _widths_case(kind, 72, h, dims, 7, [4, 16, 32], T_dec=11, lens=[70, 3, 129])
    case = GpuCase(wl, tuning=tuning)
    try:
        for i, (l, p) in enumerate(case.dev.problems):
            d_in, d_out = wl.pool.dims(p)
            case.dev.x[i, :, d_in:] = float("nan")
        y_before = case.dev.y.clone()
        assert case.run() == 0
        full_check(wl, case, list(range(len(wl.problems))))
        for i, (l, p) in enumerate(case.dev.problems):
            d_out = wl.pool.dims(p)[1]
            assert case.torch.equal(case.dev.y[i, :, d_out:].view(case.torch.int16),
                                    y_before[i, :, d_out:].view(case.torch.int16)), (l, p)
    finally:
        case.close()


@pytest.mark.parametrize("mma_min", [2, 32, 0])
@pytest.mark.parametrize("kind", ["prefill", "mixed"])
def test_projection_widths_tensor_core_tiles(mma_min, kind):
    """Prefill tiles of projections whose widths differ from h (d_in a multiple of 64, d_out
    one of 128): the shrink K loop crosses into an A row's next page block and the expand's
    column slices into a B column's next page block, the last block partly used.  Every
    segment of >= 2 rows on the tensor cores (2), the default split (32), none (0)."""
    dims = [(1024, 256), (1024, 2560), (2560, 1024), (1024, 1024), (3072, 640)]
    lens = [1, 2, 127, 128, 129, 300, 33, 0, 9]
    if kind == "prefill":
        wl = _widths_case(kind, 73, 1024, dims, 8, [1, 8, 16, 32, 64, 128], lens=lens)
    else:
        wl = _widths_case(kind, 74, 1024, dims, 8, [3, 16, 64, 100], T_dec=23, lens=lens)
    case = GpuCase(wl, y0_zero=True, tuning={"mma_min_rows": mma_min})
    try:
        for i, (l, p) in enumerate(case.dev.problems):
            case.dev.x[i, :, wl.pool.dims(p)[0]:] = float("nan")
        y_before = case.dev.y.clone()
        assert case.run() == 0
        full_check(wl, case, list(range(len(wl.problems))))
        for i, (l, p) in enumerate(case.dev.problems):
            d_out = wl.pool.dims(p)[1]
            assert case.torch.equal(case.dev.y[i, :, d_out:].view(case.torch.int16),
                                    y_before[i, :, d_out:].view(case.torch.int16)), (l, p)
    finally:
        case.close()
