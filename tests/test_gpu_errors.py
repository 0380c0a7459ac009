"""Error behaviour: host-side argument checks return a status and launch nothing;
data errors found on the device set error bits, skip the offending group and leave
the rest of the batch correct.  No test here faults, traps or hangs the GPU: every
bad index is caught by a bounds check before it is dereferenced."""
import numpy as np
import pytest

import heterogeneous_adapters_gb300 as lora
from heterogeneous_adapters_gb300 import _binding as B

from .harness import GpuCase, full_check
from .test_gpu_parity import _widths_case, small_decode, small_prefill

pytestmark = pytest.mark.gpu


def _wl(wide=False):
    if wide:   # projection 0 reads and writes vectors of 3 pages (the last partly used)
        return _widths_case("decode", 72, 512, [(1280, 1040), (512, 512)], 6, [4, 8], T_dec=20)
    return small_decode(71, 512, 1, 2, 6, [4, 8], 20)


# the decode batches here have 2 projections: the cluster kernel when its limit allows
# them, the ring kernel when the cluster kernel is turned off
PATHS = {"cluster": {"split_max_problems": 8}, "ring": {"split_max_problems": 0}}


@pytest.mark.parametrize("path", list(PATHS))
def test_bad_adapter_id_sets_bit_and_skips_only_that_token(path):
    import torch
    wl = _wl()
    case = GpuCase(wl, tuning=PATHS[path])
    try:
        ids = wl.batch.token_adapter().copy()
        victim = int(np.nonzero(ids >= 0)[0][0])
        case.dev.token_adapter[victim] = wl.pool.num_adapters + 5
        before = case.y_bits(0).copy()
        bits = case.run()
        assert bits & 0x1
        assert np.array_equal(case.y_bits(0)[victim], before[victim])
        # every other token is still correct: check against the oracle with the victim as base
        wl.batch.dec_adapter[victim] = -1
        full_check(wl, case, [0, 1])
        case.dev.token_adapter[victim] = -3
        assert case.run() & 0x1
    finally:
        case.close()


@pytest.mark.parametrize("path", list(PATHS))
def test_bad_page_rank_and_block_bits(path):
    import torch
    wl = _wl()
    case = GpuCase(wl, tuning=PATHS[path])
    try:
        ids = wl.batch.token_adapter()
        a = int(ids[ids >= 0][0])
        e = int(wl.pool.block_entries(a, 0, 0, 1)[0])
        case.dev.pt[e] = wl.pool.num_pages          # page id out of range
        assert case.run() & 0x8
        case.dev.pt[e] = int(wl.pool.pt[e])
        case.dev.ranks[a] = wl.pool.r_max + 1       # rank out of range
        assert case.run() & 0x2
        case.dev.ranks[a] = int(wl.pool.ranks[a])
        case.dev.pt_off[a] = wl.pool.pt.size        # block beyond the page table
        assert case.run() & 0x4
        case.dev.pt_off[a] = int(wl.pool.pt_off[a])
        assert case.run() == 0
    finally:
        case.close()


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("ab", [0, 1])
@pytest.mark.parametrize("wide", [False, True])
def test_bad_page_skips_that_adapter_in_that_projection_only(path, ab, wide):
    """An out-of-range A-row (ab=0) or B-column (ab=1) page of adapter a in projection 0
    (for the wide pool, in the last page block of its vectors): the page bit is set, a's
    rows of projection 0 keep their y, everything else is right."""
    wl = _wl(wide)
    case = GpuCase(wl, tuning=PATHS[path])
    try:
        ids = wl.batch.token_adapter()
        a = int(ids[ids >= 0][0])
        l, p = wl.problems[0]
        e = int(wl.pool.block_entries(a, l, p, ab)[-1])
        case.dev.pt[e] = wl.pool.num_pages
        before = case.y_bits(0).copy()
        assert case.run() & 0x8
        rows = ids == a
        assert np.array_equal(case.y_bits(0)[rows], before[rows])
        full_check(wl, case, [1])                          # projection 1 is untouched by the error
        # projection 0's other rows: compare with the oracle taking a's rows as base rows
        wl.batch.dec_adapter[rows] = -1                    # decode only: rows are the decode ids
        full_check(wl, case, [0])
    finally:
        case.close()


def test_bad_segments_bit():
    wl = small_prefill(72, 256, 1, 1, 4, [4], [5, 9, 3])
    case = GpuCase(wl)
    try:
        case.dev.seg_start[1] = 50                  # beyond T (17 rows)
        assert case.run() & 0x10
        case.dev.seg_start[1] = 6
        case.dev.seg_start[2] = 2                   # decreasing
        assert case.run() & 0x10
    finally:
        case.close()


def test_host_side_checks():
    import torch
    wl = _wl()
    case = GpuCase(wl)
    try:
        h = wl.h
        x, y = case.dev.x[0], case.dev.y[0]
        bad = [
            ([(x, y, h + 4, h, 0, 0)], B.LORA_EALIGN),            # ld % 8 != 0
            ([(x.data_ptr() + 2, y, h, h, 0, 0)], B.LORA_EALIGN),  # misaligned x
            ([(x, y, h, h, 1, 0)], B.LORA_EINVAL),                # layer out of range
            ([(x, y, h, h, 0, 2)], B.LORA_EINVAL),                # proj out of range
            ([(x, None, h, h, 0, 0)], B.LORA_EINVAL),             # null y
            ([(x, y, h - 8, h, 0, 0)], B.LORA_EINVAL),            # ld < h
        ]
        for probs, want in bad:
            with pytest.raises(lora.LoraError) as ei:
                lora.bgmv(case.pool, probs, case.dev.token_adapter, case.T, case.ws,
                          case.ws_bytes, case.stream)
            assert ei.value.status == want
        with pytest.raises(lora.LoraError) as ei:
            lora.bgmv(case.pool, case.problems(), case.dev.token_adapter, case.T, case.ws,
                      case.ws_bytes - 256, case.stream)
        assert ei.value.status == B.LORA_EWORKSPACE
        with pytest.raises(lora.LoraError) as ei:
            lora.bgmv(case.pool, case.problems(), case.dev.token_adapter, case.T,
                      case.ws.data_ptr() + 16, case.ws_bytes - 256, case.stream)
        assert ei.value.status == B.LORA_EWORKSPACE
        with pytest.raises(lora.LoraError) as ei:
            lora.segment(case.pool, None, None, 0, case.dev.token_adapter,
                         lora.LORA_MAX_SEGMENTS + 1, 1 << 20, case.ws, case.ws_bytes, case.stream)
        assert ei.value.status == B.LORA_ETOOBIG
        assert case.error_bits() == 0
    finally:
        case.close()


def test_bounded_wait_gives_up_and_reports():
    """The bounded device wait every kernel uses: a barrier nothing completes, a 5 ms limit;
    the timeout bit comes back through the error word, the wait took about the limit, and
    the context stays usable (a correct launch right after)."""
    import torch
    wl = _wl()
    case = GpuCase(wl)
    try:
        el = torch.zeros(1, dtype=torch.int64, device=case.device)
        lora.debug_wait_limit(case.ws, case.ws_bytes, 5_000_000, el, case.stream)
        assert case.error_bits() == 0x20
        waited = int(el.item())
        assert 5_000_000 <= waited < 1_000_000_000, waited
        with pytest.raises(lora.LoraError):
            lora.debug_wait_limit(case.ws, case.ws_bytes, 3_000_000_000, None, case.stream)
        with pytest.raises(lora.LoraError):
            lora.debug_wait_limit(case.ws, case.ws_bytes, 10, None, case.stream)
        assert case.run() == 0
        full_check(wl, case, [0, 1])
    finally:
        case.close()
