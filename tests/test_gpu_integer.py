"""Integer steps on the GPU, bit-exact against the oracle: the grouping of the batch by
adapter (scheduler step) and the page-table walk (gathered page list)."""
import numpy as np
import pytest

import oracle
from workloads import spec

from .harness import GpuCase
from .test_gpu_parity import _mixed, small_decode, small_prefill

pytestmark = pytest.mark.gpu


def _grouping_from_ws(case):
    torch = case.torch
    b = case.wl.batch
    v = case.lora.workspace_view(case.pool, case.ws, case.ws_bytes, case.T, case.nseg)
    base = case.ws.data_ptr()

    def arr(ptr, n):
        off = ptr - base
        return case.ws[off:off + 4 * n].view(torch.int32).cpu().numpy()

    counts = arr(v.counts, 4)
    n_ad, G = int(counts[0]), int(counts[1])
    return arr(v.perm, n_ad), arr(v.grp_start, G + 1), arr(v.grp_adapter, G), counts


def _segment(case):
    b, d = case.wl.batch, case.dev
    case.lora.segment(case.pool, d.seg_start if b.num_segments else None,
                      d.seg_adapter if b.num_segments else None, b.num_segments,
                      d.dec_adapter if b.num_decode else None, b.num_decode, case.T, case.ws,
                      case.ws_bytes, case.stream)
    assert case.error_bits() == 0


CASES = {
    "tiny": spec.tiny_decode,
    "decode-zipf": lambda: small_decode(61, 256, 1, 1, 50, [4], 300),
    "decode-base": lambda: small_decode(62, 256, 1, 1, 7, [4], 500, base=True),
    "decode-large": lambda: small_decode(63, 256, 1, 1, 3000, [4], 5000),
    "decode-max-segments": lambda: small_decode(66, 64, 1, 1, 20000, [1, 2], 16384, base=True),
    "prefill": lambda: small_prefill(64, 256, 1, 1, 9, [4], [3, 0, 200, 1, 77, 128, 129, 5]),
    "mixed": lambda: _mixed(65, 256, 1, 1, 40, [4, 8], [5, 260, 131, 1], 300, 30),
}


@pytest.mark.parametrize("name", list(CASES))
def test_grouping_bit_exact(name):
    wl = CASES[name]()
    case = GpuCase(wl)
    try:
        _segment(case)
        perm, gs, ga, counts = _grouping_from_ws(case)
        want_perm, want_gs, want_ga = oracle.group_tokens(wl.batch.token_adapter())
        assert np.array_equal(perm, want_perm)
        assert np.array_equal(gs, want_gs)
        assert np.array_equal(ga, want_ga)
    finally:
        case.close()


def _widths_decode():
    """Two layers of projections 256 -> 64, 256 -> 640 and 640 -> 256 on h = 256."""
    rng = np.random.default_rng(67)
    ranks = rng.choice(np.asarray([1, 3, 8, 16], np.int32), size=12)
    pool = spec.make_pool_all_resident(rng, 256, 2, 3, ranks,
                                       proj_dims=[(256, 64), (256, 640), (640, 256)])
    ids = rng.integers(-1, 12, size=90).astype(np.int32)
    batch = spec.Batch(np.zeros(1, np.int32), np.zeros(0, np.int32), ids)
    return spec.Workload("decode-widths", 67, pool, batch, spec.all_problems(2, 3))


@pytest.mark.parametrize("name", ["tiny", "decode-zipf", "mixed", "decode-widths"])
def test_page_list_bit_exact(name):
    import torch
    wl = _widths_decode() if name == "decode-widths" else CASES[name]()
    case = GpuCase(wl)
    try:
        _segment(case)
        _, _, ga, _ = _grouping_from_ws(case)
        for (l, p) in wl.problems:
            want = oracle.page_list(wl.pool.pt, wl.pool.pt_off, wl.pool.ranks, wl.pool.num_proj,
                                    l, p, ga, h=wl.h, proj_dims=wl.pool.proj_dims)
            cap = want.size + 8
            out = torch.full((cap,), -7, dtype=torch.int32, device=case.device)
            cnt = torch.zeros(1, dtype=torch.int32, device=case.device)
            case.lora.debug_page_list(case.pool, case.ws, case.ws_bytes, l, p, out, cap, cnt,
                                      case.stream)
            assert case.error_bits() == 0
            n = int(cnt.item())
            assert n == want.size
            assert np.array_equal(out[:n].cpu().numpy(), want)
    finally:
        case.close()


@pytest.mark.parametrize("cfg", ["decode", "prefill", "mixed", "stress-distinct"])
def test_grouping_full_workloads(cfg):
    """Grouping of the full-size batches (metadata only; a 1-page dummy pool suffices)."""
    import torch

    import heterogeneous_adapters_gb300 as lora
    wl = spec.WORKLOADS[cfg]()
    dev = "cuda:0"
    b = wl.batch
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)  # noqa: E731
    pages = torch.zeros((1, wl.h), dtype=torch.bfloat16, device=dev)
    pt = t(wl.pool.pt)
    off = torch.from_numpy(wl.pool.pt_off).to(dev)
    ranks = t(wl.pool.ranks)
    scales = torch.from_numpy(wl.pool.scales).to(dev)
    pool = lora.Pool(pages, 1, wl.h, pt, wl.pool.pt.size, off, ranks, scales,
                     wl.pool.num_adapters, wl.pool.num_layers, wl.pool.num_proj, wl.pool.r_max)
    T, nseg = b.num_tokens, b.num_segments + b.num_decode
    nbytes = lora.workspace_size(pool, T, nseg)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    lora.workspace_init(ws, nbytes, stream)
    lora.segment(pool, t(b.seg_start) if b.num_segments else None,
                 t(b.seg_adapter) if b.num_segments else None, b.num_segments,
                 t(b.dec_adapter) if b.num_decode else None, b.num_decode, T, ws, nbytes, stream)
    assert lora.get_device_error(ws, stream) == 0
    v = lora.workspace_view(pool, ws, nbytes, T, nseg)

    def arr(ptr, n):
        o = ptr - ws.data_ptr()
        return ws[o:o + 4 * n].view(torch.int32).cpu().numpy()

    counts = arr(v.counts, 4)
    want_perm, want_gs, want_ga = oracle.group_tokens(b.token_adapter())
    assert counts[0] == want_perm.size and counts[1] == want_ga.size
    assert np.array_equal(arr(v.perm, counts[0]), want_perm)
    assert np.array_equal(arr(v.grp_start, counts[1] + 1), want_gs)
    assert np.array_equal(arr(v.grp_adapter, counts[1]), want_ga)
    pool.close()
