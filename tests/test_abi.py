"""The C ABI library loads without a GPU and exports every symbol include/*.h
declares; host-only calls (pool creation checks, sizes, status strings) behave as
documented.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    import glob
    src = "".join(open(f).read() for f in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(lora_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from heterogeneous_adapters_gb300 import build, lib as load
    build.build()
    return load()


def test_header_declares_the_documented_entry_points():
    names = declared_functions()
    for n in ["lora_pool_create", "lora_bgmv", "lora_sgmv", "lora_apply_mixed", "lora_segment"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from heterogeneous_adapters_gb300 import _binding
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), f"liblora.so does not export {n}"
    assert sorted(_binding.EXPORTED) == names


def test_pool_create_host_checks(lib):
    from heterogeneous_adapters_gb300._binding import (LORA_EALIGN, LORA_EINVAL, LORA_ETOOBIG,
                                                       lora_pool_desc)
    h = ctypes.c_void_p()
    fake = 1 << 20   # never dereferenced: creation only records pointers

    def desc(**kw):
        d = dict(pages=fake, num_pages=16, h=256, num_adapters=2, num_layers=1, num_proj=1,
                 r_max=8, reserved=0, page_table=fake, page_table_len=32, adapter_pt_off=fake,
                 ranks=fake, scales=fake, proj_dims=None)
        d.update(kw)
        return lora_pool_desc(**d)

    assert lib.lora_pool_create(ctypes.byref(h), ctypes.byref(desc())) == 0
    assert lib.lora_pool_destroy(h) == 0
    assert lib.lora_pool_create(ctypes.byref(h), ctypes.byref(desc(pages=None))) == LORA_EINVAL
    assert lib.lora_pool_create(ctypes.byref(h), ctypes.byref(desc(h=100))) == LORA_EALIGN
    assert lib.lora_pool_create(ctypes.byref(h), ctypes.byref(desc(pages=fake + 8))) == LORA_EALIGN
    assert lib.lora_pool_create(ctypes.byref(h), ctypes.byref(desc(r_max=257))) == LORA_ETOOBIG
    assert lib.lora_pool_create(ctypes.byref(h), ctypes.byref(desc(num_adapters=0))) == LORA_EINVAL
    # projection widths: multiples of 8, at most LORA_MAX_VEC_PAGES pages
    import numpy as np
    for dims, want in (([256, 64], 0), ([256, 4096], 0), ([100, 256], LORA_EINVAL),
                       ([256, 17 * 256], LORA_ETOOBIG), ([0, 256], LORA_EINVAL)):
        arr = np.asarray(dims, np.int32)
        st = lib.lora_pool_create(ctypes.byref(h), ctypes.byref(desc(proj_dims=arr.ctypes.data)))
        assert st == want, (dims, st)
        if st == 0:
            assert lib.lora_pool_destroy(h) == 0
    assert lib.lora_pool_create(None, ctypes.byref(desc())) == LORA_EINVAL


def test_workspace_size_and_status_strings(lib):
    from heterogeneous_adapters_gb300._binding import LORA_ETOOBIG, lora_pool_desc
    h = ctypes.c_void_p()
    d = lora_pool_desc(1 << 20, 16, 256, 2, 1, 1, 8, 0, 1 << 20, 32, 1 << 20, 1 << 20, 1 << 20)
    assert lib.lora_pool_create(ctypes.byref(h), ctypes.byref(d)) == 0
    n1, n2 = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.lora_workspace_size(h, 64, 64, ctypes.byref(n1)) == 0
    assert lib.lora_workspace_size(h, 100000, 16384, ctypes.byref(n2)) == 0
    assert 256 < n1.value < n2.value and n1.value % 256 == 0
    assert lib.lora_workspace_size(h, 1, 16385, ctypes.byref(n2)) == LORA_ETOOBIG
    lib.lora_pool_destroy(h)
    for s in range(7):
        assert lib.lora_status_string(s)


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "heterogeneous_adapters_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", src, flags=re.M), f
                assert "lora_oracle" not in src, f


def test_stage_pages_host_checks(lib):
    """Staging validates its host-side index arrays before launching anything."""
    import numpy as np

    from heterogeneous_adapters_gb300._binding import LORA_EALIGN, LORA_EINVAL, lora_pool_desc
    h = ctypes.c_void_p()
    pt = np.zeros(32, np.int32)
    d = lora_pool_desc(1 << 20, 16, 256, 2, 1, 1, 8, 0, pt.ctypes.data, 32, 1 << 20, 1 << 20, 1 << 20)
    assert lib.lora_pool_create(ctypes.byref(h), ctypes.byref(d)) == 0
    rows = np.zeros((2, 256), np.uint16)
    good = np.array([3, 4], np.int32)
    bad = np.array([3, 16], np.int32)
    idx = np.array([0, 31], np.int64)
    bad_idx = np.array([0, 32], np.int64)
    pg = np.array([1, 2], np.int32)
    c = lambda a: a.ctypes.data  # noqa: E731
    assert lib.lora_stage_pages(h, c(rows), c(bad), 2, None, None, None, 0, None, None) == LORA_EINVAL
    assert lib.lora_stage_pages(h, c(rows) + 2, c(good), 2, None, None, None, 0, None, None) == LORA_EALIGN
    assert lib.lora_stage_pages(h, None, None, 0, c(pt), c(bad_idx), c(pg), 2, None) == LORA_EINVAL
    other = np.zeros(32, np.int32)
    assert lib.lora_stage_pages(h, None, None, 0, c(other), c(idx), c(pg), 2, None) == LORA_EINVAL
    assert lib.lora_stage_pages(h, None, None, 0, None, None, None, 0, None, None) == 0
    lib.lora_pool_destroy(h)


def test_pool_tuning_defaults_overrides_and_checks(lib):
    """Launch tuning lives in the pool handle (no environment variable is read): the
    defaults, a partial override that keeps the other fields, range checks that leave the
    tuning unchanged, and NULL restoring the defaults."""
    from heterogeneous_adapters_gb300._binding import LORA_EINVAL, lora_tuning, lora_pool_desc
    h = ctypes.c_void_p()
    d = lora_pool_desc(1 << 20, 16, 256, 2, 1, 1, 8, 0, 1 << 20, 32, 1 << 20, 1 << 20, 1 << 20)
    assert lib.lora_pool_create(ctypes.byref(h), ctypes.byref(d)) == 0

    def get():
        t = lora_tuning()
        assert lib.lora_pool_get_tuning(h, ctypes.byref(t)) == 0
        return (t.ring_rows_per_stage, t.split_max_problems, t.mma_min_rows, t.mma_y_stages,
                round(t.fused_ring_speed, 4))

    default = get()
    assert default == (0, 1, -1, 3, 1.22)

    def set_(**kw):
        f = dict(ring_rows_per_stage=0, split_max_problems=-1, mma_min_rows=-1, mma_y_stages=0,
                 fused_ring_speed=0.0)
        f.update(kw)
        t = lora_tuning(**f)
        return lib.lora_pool_set_tuning(h, ctypes.byref(t))

    assert set_(split_max_problems=0, mma_min_rows=64) == 0
    assert get() == (0, 0, 64, 3, 1.22)
    for bad in (dict(ring_rows_per_stage=5), dict(split_max_problems=9), dict(mma_min_rows=1),
                dict(mma_y_stages=5), dict(fused_ring_speed=20.0), dict(reserved=(ctypes.c_int32 * 3)(1, 0, 0))):
        assert set_(**bad) == LORA_EINVAL, bad
        assert get() == (0, 0, 64, 3, 1.22)
    assert lib.lora_pool_set_tuning(h, None) == 0
    assert get() == default
    lib.lora_pool_destroy(h)


def test_mixed_width_pool_ring_speed_default(lib):
    """A pool whose projections differ from h x h defaults the mixed launch's ring-body
    speed to 1.0 (1.22 for h x h pools): the CTA split of the mixed launch as measured on
    the Llama-3-8B step.  An explicit value overrides it and NULL restores it."""
    from heterogeneous_adapters_gb300._binding import lora_tuning, lora_pool_desc
    dims = (ctypes.c_int32 * 4)(256, 256, 256, 128)
    h = ctypes.c_void_p()
    d = lora_pool_desc(1 << 20, 16, 256, 2, 1, 2, 8, 0, 1 << 20, 64, 1 << 20, 1 << 20, 1 << 20,
                       ctypes.cast(dims, ctypes.c_void_p))
    assert lib.lora_pool_create(ctypes.byref(h), ctypes.byref(d)) == 0

    def speed():
        t = lora_tuning()
        assert lib.lora_pool_get_tuning(h, ctypes.byref(t)) == 0
        return round(t.fused_ring_speed, 4)

    assert speed() == 1.0
    t = lora_tuning(0, -1, -1, 0, 0.85)
    assert lib.lora_pool_set_tuning(h, ctypes.byref(t)) == 0
    assert speed() == 0.85
    assert lib.lora_pool_set_tuning(h, None) == 0
    assert speed() == 1.0
    lib.lora_pool_destroy(h)


def test_stage_pages_ce_host_checks(lib):
    """The copy-engine staging validates its index arrays and its staging buffer before
    launching or copying anything (a staging buffer is needed only when the destination
    pages form more than LORA_STAGE_MAX_RUNS runs, and is checked whenever one is given)."""
    import numpy as np

    from heterogeneous_adapters_gb300._binding import LORA_EALIGN, LORA_EINVAL, lora_pool_desc
    h = ctypes.c_void_p()
    pt = np.zeros(32, np.int32)
    d = lora_pool_desc(1 << 20, 16, 256, 2, 1, 1, 8, 0, pt.ctypes.data, 32, 1 << 20, 1 << 20, 1 << 20)
    assert lib.lora_pool_create(ctypes.byref(h), ctypes.byref(d)) == 0
    rows = np.zeros((2, 256), np.uint16)
    good = np.array([3, 4], np.int32)
    c = lambda a: a.ctypes.data  # noqa: E731
    stage = 1 << 20          # a device address stand-in: never used, the checks fail first
    assert lib.lora_stage_pages_ce(h, c(rows), stage, 2 * 512, c(np.array([3, 16], np.int32)), 2,
                                   None, None, None, 0, None, None) == LORA_EINVAL          # page out of range
    assert lib.lora_stage_pages_ce(h, c(rows), stage, 2 * 512 - 16, c(good), 2, None, None, None, 0,
                                   None, None) == LORA_EINVAL                               # staging too small
    # more runs of consecutive pages than LORA_STAGE_MAX_RUNS (every other page): the rows go
    # through the staging buffer, which is then required
    many = np.zeros((65, 256), np.uint16)
    spread = (2 * np.arange(65)).astype(np.int32)
    assert lib.lora_stage_pages_ce(h, c(many), None, 0, c(spread), 65, None, None, None, 0,
                                   None, None) == LORA_EINVAL                               # no staging buffer
    assert lib.lora_stage_pages_ce(h, c(rows), stage + 8, 2 * 512, c(good), 2, None, None, None, 0,
                                   None, None) == LORA_EINVAL                               # misaligned staging
    assert lib.lora_stage_pages_ce(h, c(rows) + 2, stage, 2 * 512, c(good), 2, None, None, None, 0,
                                   None, None) == LORA_EALIGN                               # misaligned rows
    assert lib.lora_stage_pages_ce(h, None, None, 0, None, 0, None, None, None, 0, None, None) == 0
    lib.lora_pool_destroy(h)
