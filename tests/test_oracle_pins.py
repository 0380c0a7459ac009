"""Pins of the fp64 CPU oracle against what the pages and the mathematics fix.

Each test targets a mistake the oracle could plausibly contain (a transposed
operand, a wrong page-table index, a dropped or duplicated term, a wrong scale,
touching base-only rows) and checks it against something other than the
oracle's own formula: the merge identity (a dense library matmul of the merged
weight), the gathered-bmm form printed on the pofe.ai page (a library bmm),
exact invariances, and the pages' flop count.
"""
import itertools

import numpy as np
import pytest

import oracle
from workloads import spec, valuegen as vg
from workloads.materialize import a_param, host_inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def dense_adapter(wl, a, layer, proj):
    """Dense A (r x h) and B (h x r) of adapter a for (layer, proj), generated straight
    from the generator keys of the layout convention -- never through the page table."""
    pool = wl.pool
    r = int(pool.ranks[a])
    h = pool.h
    P = pool.num_proj
    out = []
    for ab, dist, param in ((0, vg.DIST_UNIFORM, a_param(h)),
                            (1, vg.DIST_NORMAL, vg.normal_param(spec.SIGMA_B))):
        local = ((layer * P + proj) * 2 + ab) * r + np.arange(r)
        rows = np.zeros((r, h), np.uint16)
        vg.fill_rows_host(rows, np.arange(r), spec.page_key(a, local), wl.seed, dist, param)
        out.append(vg.bf16_bits_to_f64(rows))
    A, Bcols = out
    return A, Bcols.T  # B is d_out x r: column j is page j


def run_oracle(wl, hi, layer, proj, y0=None, ids=None, want_t=False):
    pool = wl.pool
    x = hi.x[(layer, proj)]
    if y0 is None:
        y0 = vg.bf16_bits_to_f64(hi.y0[(layer, proj)])
    if ids is None:
        ids = wl.batch.token_adapter()
    return oracle.lora_delta(hi.pool, hi.pt, pool.pt_off, pool.ranks, pool.scales,
                             pool.num_layers, pool.num_proj, layer, proj, x, y0, ids,
                             want_t=want_t)


def small_multi(seed=7, h=64, L=2, P=3, N=5, T=24):
    return spec.decode_workload("pin-small", seed, h, L, P, N, [1, 2, 4, 8, 16], T, None,
                                num_pages=None, base_ids=True)


# ----------------------------------------------------------------------------- formula pins

@pytest.mark.parametrize("make", [spec.tiny_decode, small_multi])
def test_merge_identity(make):
    """x (W + s B A)^T == x W^T + s (x A^T) B^T (pofe.ai page, "The bottleneck": the merged
    weight W' = W + gamma B A; fdeinterviews S-LoRA page: the update to W is a low-rank
    product).  Dense library matmuls of the merged weight, per token and per problem."""
    wl = make()
    hi = host_inputs(wl)
    rng = np.random.default_rng(3)
    ids = wl.batch.token_adapter()
    for (l, p) in wl.problems:
        W = rng.normal(0.0, 0.02, size=(wl.h, wl.h))
        xd = vg.bf16_bits_to_f64(hi.x[(l, p)])
        y_ref, _, _ = run_oracle(wl, hi, l, p, y0=xd @ W.T)
        for i, a in enumerate(ids):
            if a < 0:
                merged = W
            else:
                A, B = dense_adapter(wl, a, l, p)
                merged = W + float(wl.pool.scales[a]) * (B @ A)
            want = merged @ xd[i]
            np.testing.assert_allclose(y_ref[i], want, rtol=0, atol=1e-12 * max(1.0, np.abs(want).max()))


def dense_adapter_widths(wl, a, layer, proj):
    """Dense A (r x d_in) and B (d_out x r) of adapter a for (layer, proj) of a pool with
    per-projection widths, from the generator keys of the layout convention: a vector of
    length d takes ceil(d/h) pages, the block of (layer, proj, A or B) lists page kb of every
    vector, then page kb + 1; blocks in (layer, proj, A, B) order.  Never through the page
    table."""
    pool = wl.pool
    r, h, P = int(pool.ranks[a]), pool.h, pool.num_proj
    dims = [tuple(int(v) for v in d) for d in pool.proj_dims]
    npg = [(-(-di // h), -(-do // h)) for di, do in dims]
    layer_units = sum(pi + po for pi, po in npg)
    unit0 = layer * layer_units + sum(pi + po for pi, po in npg[:proj])
    out = []
    for ab, dist, param in ((0, vg.DIST_UNIFORM, a_param(h)),
                            (1, vg.DIST_NORMAL, vg.normal_param(spec.SIGMA_B))):
        d = dims[proj][ab]
        first = unit0 + (npg[proj][0] if ab else 0)
        full = np.zeros((r, npg[proj][ab] * h))
        for kb in range(npg[proj][ab]):
            local = (first + kb) * r + np.arange(r)
            rows = np.zeros((r, h), np.uint16)
            vg.fill_rows_host(rows, np.arange(r), spec.page_key(a, local), wl.seed, dist, param)
            full[:, kb * h:(kb + 1) * h] = vg.bf16_bits_to_f64(rows)
        out.append(full[:, :d])
    A, Bcols = out
    return A, Bcols.T


def test_merge_identity_projection_widths():
    """The merge identity on a pool whose projections are not h x h ("Multi-LoRA serving:
    S-LoRA, Punica and adapter batching", "Worked example": grouped-query k/v narrower than
    h, the MLP wider, every projection adapted): widths below one page, spanning several
    pages, and ending mid-page, for A and B."""
    h = 64
    dims = [(64, 16), (64, 160), (160, 64), (40, 24)]
    wl = spec.decode_workload("pin-widths", 21, h, 2, len(dims), 5, [1, 2, 4, 8, 16], 24, None,
                              base_ids=True, proj_dims=dims)
    hi = host_inputs(wl)
    rng = np.random.default_rng(4)
    ids = wl.batch.token_adapter()
    for (l, p) in wl.problems:
        d_in, d_out = dims[p]
        assert hi.x[(l, p)].shape[1] == d_in
        W = rng.normal(0.0, 0.02, size=(d_out, d_in))
        xd = vg.bf16_bits_to_f64(hi.x[(l, p)])
        y_ref, _, madds = oracle.lora_delta(hi.pool, hi.pt, wl.pool.pt_off, wl.pool.ranks, wl.pool.scales,
                                            wl.pool.num_layers, wl.pool.num_proj, l, p, hi.x[(l, p)],
                                            xd @ W.T, ids, proj_dims=dims)
        assert y_ref.shape == (ids.size, d_out)
        for i, a in enumerate(ids):
            if a < 0:
                merged = W
            else:
                A, B = dense_adapter_widths(wl, a, l, p)
                assert A.shape == (wl.pool.ranks[a], d_in) and B.shape == (d_out, wl.pool.ranks[a])
                merged = W + float(wl.pool.scales[a]) * (B @ A)
            want = merged @ xd[i]
            np.testing.assert_allclose(y_ref[i], want, rtol=0, atol=1e-12 * max(1.0, np.abs(want).max()))
        # flop count: r (d_in + d_out) multiply-adds per adapted token
        r_t = wl.pool.ranks[ids[ids >= 0]].astype(np.int64)
        assert madds == int((r_t * (d_in + d_out)).sum())


def test_gathered_bmm_form():
    """The pofe.ai page's "Implementation sketch" form: v = bmm(A_pool[idx], x), then
    y + scale * bmm(B_pool[idx], v), in float64 torch on CPU, with adapters zero-padded
    to r_max in the dense pools (a library routine, not the oracle's loop)."""
    torch = pytest.importorskip("torch")
    wl = small_multi(seed=11, T=32)
    hi = host_inputs(wl)
    N, h, rmax = wl.pool.num_adapters, wl.h, wl.pool.r_max
    ids = wl.batch.token_adapter()
    for (l, p) in wl.problems:
        A_pool = torch.zeros((N + 1, rmax, h), dtype=torch.float64)   # slot N = zero adapter
        B_pool = torch.zeros((N + 1, h, rmax), dtype=torch.float64)
        scale = torch.zeros(N + 1, dtype=torch.float64)
        for a in range(N):
            A, B = dense_adapter(wl, a, l, p)
            r = A.shape[0]
            A_pool[a, :r] = torch.from_numpy(A)
            B_pool[a, :, :r] = torch.from_numpy(B)
            scale[a] = float(wl.pool.scales[a])
        idx = torch.from_numpy(np.where(ids < 0, N, ids).astype(np.int64))
        x = torch.from_numpy(vg.bf16_bits_to_f64(hi.x[(l, p)]))
        y0 = torch.from_numpy(vg.bf16_bits_to_f64(hi.y0[(l, p)]))
        v = torch.bmm(A_pool[idx], x[:, :, None])
        want = y0 + scale[idx][:, None] * torch.bmm(B_pool[idx], v).squeeze(2)
        got, _, _ = run_oracle(wl, hi, l, p)
        np.testing.assert_allclose(got, want.numpy(), rtol=1e-12, atol=1e-12)


def test_flop_count_matches_pages():
    """Every adapted token costs 2 r (d_in + d_out) extra flops per projection
    (pofe.ai page, "The bottleneck"); the oracle counts its multiply-adds as it runs."""
    wl = small_multi(seed=5, T=40)
    hi = host_inputs(wl)
    ids = wl.batch.token_adapter()
    want = sum(2 * int(wl.pool.ranks[a]) * (wl.h + wl.h) for a in ids if a >= 0)
    for (l, p) in wl.problems:
        _, _, madds = run_oracle(wl, hi, l, p)
        assert 2 * madds == want


def test_shrink_t_matches_dense():
    """t = A x for every adapted token (the shrink alone; orientation of A pinned)."""
    wl = small_multi(seed=13)
    hi = host_inputs(wl)
    ids = wl.batch.token_adapter()
    for (l, p) in wl.problems:
        _, t, _ = run_oracle(wl, hi, l, p, want_t=True)
        xd = vg.bf16_bits_to_f64(hi.x[(l, p)])
        for i, a in enumerate(ids):
            if a < 0:
                assert np.all(t[i] == 0)
                continue
            A, _ = dense_adapter(wl, a, l, p)
            np.testing.assert_allclose(t[i, :A.shape[0]], A @ xd[i], rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------------------- exact special cases

def test_zero_B_gives_zero_delta():
    """Adapters whose B is all zero leave y exactly equal to y0."""
    wl = small_multi(seed=17)
    hi = host_inputs(wl)
    ent = np.concatenate([wl.pool.block_entries(a, l, p, 1)
                          for a in range(wl.pool.num_adapters) for (l, p) in wl.problems])
    hi.pool[hi.pt[ent]] = 0
    for (l, p) in wl.problems:
        y0 = vg.bf16_bits_to_f64(hi.y0[(l, p)])
        got, _, _ = run_oracle(wl, hi, l, p, y0=y0)
        assert np.array_equal(got, y0)


def test_base_only_rows_untouched():
    wl = small_multi(seed=19, T=48)
    hi = host_inputs(wl)
    ids = wl.batch.token_adapter()
    assert (ids == -1).any() and (ids >= 0).any()
    for (l, p) in wl.problems:
        y0 = vg.bf16_bits_to_f64(hi.y0[(l, p)])
        got, _, _ = run_oracle(wl, hi, l, p, y0=y0)
        assert np.array_equal(got[ids == -1], y0[ids == -1])
        assert not np.array_equal(got[ids >= 0], y0[ids >= 0])


def test_rank_r_equals_zero_padded_rmax():
    """Mixed ranks need no padding: each adapter re-laid out at rank r_max with zero
    A rows and zero B columns beyond r gives the identical result (scale unchanged)."""
    wl = small_multi(seed=23)
    hi = host_inputs(wl)
    pool = wl.pool
    N, L, P, rmax, h = pool.num_adapters, pool.num_layers, pool.num_proj, pool.r_max, pool.h
    sizes = np.full(N, L * P * 2 * rmax, dtype=np.int64)
    off2 = np.concatenate([[0], np.cumsum(sizes)[:-1]])
    pages2 = [np.zeros(h, np.uint16)]  # page 0 = zeros
    pt2 = np.zeros(int(sizes.sum()), dtype=np.int32)
    for a in range(N):
        r = int(pool.ranks[a])
        for (l, p) in [(l, p) for l in range(L) for p in range(P)]:
            for ab in (0, 1):
                src = hi.pt[pool.block_entries(a, l, p, ab)]
                base = off2[a] + ((l * P + p) * 2 + ab) * rmax
                for j in range(rmax):
                    if j < r and src[j] >= 0:
                        pages2.append(hi.pool[src[j]])
                        pt2[base + j] = len(pages2) - 1
    pool2 = np.stack(pages2)
    ranks2 = np.full(N, rmax, np.int32)
    for (l, p) in wl.problems:
        got, _, _ = run_oracle(wl, hi, l, p)
        y0 = vg.bf16_bits_to_f64(hi.y0[(l, p)])
        pad, _, _ = oracle.lora_delta(pool2, pt2, off2, ranks2, pool.scales, L, P, l, p,
                                      hi.x[(l, p)], y0, wl.batch.token_adapter())
        assert np.array_equal(got, pad)


def test_page_placement_invariance():
    """Moving every page to another slot of the pool (and rewriting the page table)
    changes nothing, bit for bit."""
    wl = small_multi(seed=29)
    hi = host_inputs(wl)
    rng = np.random.default_rng(0)
    n = hi.pool.shape[0]
    perm = rng.permutation(n)            # new slot of old page q is perm[q]
    pool2 = np.empty_like(hi.pool)
    pool2[perm] = hi.pool
    pt2 = np.where(hi.pt >= 0, perm[np.maximum(hi.pt, 0)], -1).astype(np.int32)
    for (l, p) in wl.problems:
        a, _, _ = run_oracle(wl, hi, l, p)
        y0 = vg.bf16_bits_to_f64(hi.y0[(l, p)])
        b, _, _ = oracle.lora_delta(pool2, pt2, wl.pool.pt_off, wl.pool.ranks, wl.pool.scales,
                                    wl.pool.num_layers, wl.pool.num_proj, l, p, hi.x[(l, p)],
                                    y0, wl.batch.token_adapter())
        assert np.array_equal(a, b)


def test_batch_order_invariance():
    """Permuting the tokens of the batch permutes the results, bit for bit."""
    wl = small_multi(seed=31, T=30)
    hi = host_inputs(wl)
    ids = wl.batch.token_adapter()
    perm = np.random.default_rng(1).permutation(ids.size)
    for (l, p) in wl.problems:
        a, _, _ = run_oracle(wl, hi, l, p)
        y0 = vg.bf16_bits_to_f64(hi.y0[(l, p)])
        b, _, _ = oracle.lora_delta(hi.pool, hi.pt, wl.pool.pt_off, wl.pool.ranks,
                                    wl.pool.scales, wl.pool.num_layers, wl.pool.num_proj, l, p,
                                    hi.x[(l, p)][perm], y0[perm], ids[perm])
        assert np.array_equal(a[perm], b)


def test_oracle_rejects_bad_inputs():
    wl = spec.tiny_decode()
    hi = host_inputs(wl)
    ids = wl.batch.token_adapter().copy()
    ids[0] = wl.pool.num_adapters
    with pytest.raises(oracle.OracleError, match="adapter"):
        run_oracle(wl, hi, 0, 0, ids=ids)
    ids[0] = -2
    with pytest.raises(oracle.OracleError, match="adapter"):
        run_oracle(wl, hi, 0, 0, ids=ids)
    ids = wl.batch.token_adapter()
    a = int(ids[ids >= 0][0])
    bad = hi.pt.copy()
    bad[wl.pool.block_entries(a, 0, 0, 1)[0]] = hi.pool.shape[0]
    with pytest.raises(oracle.OracleError, match="page"):
        oracle.lora_delta(hi.pool, bad, wl.pool.pt_off, wl.pool.ranks, wl.pool.scales, 1, 1, 0, 0,
                          hi.x[(0, 0)], vg.bf16_bits_to_f64(hi.y0[(0, 0)]), ids)


# ----------------------------------------------------------------------------- integer steps

def _brute_group(ids):
    """Enumerate every arrangement of the adapted tokens; keep the one sorted by
    (adapter id, batch position).  Exponential: tiny inputs only."""
    adapted = [i for i, a in enumerate(ids) if a >= 0]
    best = None
    for cand in itertools.permutations(adapted):
        keys = [(ids[i], i) for i in cand]
        if all(keys[k] < keys[k + 1] for k in range(len(keys) - 1)):
            assert best is None
            best = cand
    return list(best) if best is not None else []


@pytest.mark.parametrize("seed", range(12))
def test_group_tokens_brute_force(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(0, 8))
    ids = rng.integers(-1, 3, size=T).astype(np.int32)
    perm, gs, ga = oracle.group_tokens(ids)
    assert list(perm) == _brute_group(list(ids))
    # groups: one per distinct adapter present, ascending, covering perm exactly
    distinct = sorted(set(int(a) for a in ids if a >= 0))
    assert list(ga) == distinct
    assert gs[0] == 0 and gs[-1] == perm.size and np.all(np.diff(gs) > 0)
    for g, a in enumerate(ga):
        assert np.all(ids[perm[gs[g]:gs[g + 1]]] == a)


def test_page_list_walks_the_layout():
    """Every page the oracle lists for (adapter, layer, proj) holds exactly the
    generator stream of that adapter's A row j / B column j (keys fixed at build time)."""
    wl = small_multi(seed=37)
    pool = wl.pool
    key_of = dict(zip(pool.page_ids.tolist(), pool.page_keys.tolist()))
    _, _, ga = oracle.group_tokens(wl.batch.token_adapter())
    for (l, p) in wl.problems:
        pages = oracle.page_list(pool.pt, pool.pt_off, pool.ranks, pool.num_proj, l, p, ga)
        pos = 0
        for a in ga:
            r = int(pool.ranks[a])
            for ab in (0, 1):
                for j in range(r):
                    local = ((l * pool.num_proj + p) * 2 + ab) * r + j
                    assert key_of[int(pages[pos])] == int(spec.page_key(a, local))
                    pos += 1
        assert pos == pages.size


def test_page_list_walks_the_layout_with_widths():
    """Projections of other widths: the oracle's page list for (layer, proj) is, per group,
    page kb of every A row for kb < ceil(d_in/h), then page q of every B column for
    q < ceil(d_out/h), at the entries the layout fixes (U = sum of the projections' page
    blocks, A block at r (l U + pre(p)), B block ceil(d_in/h) r later)."""
    h, L = 256, 2
    dims = [(256, 64), (256, 640), (640, 256), (1032, 8)]
    rng = np.random.default_rng(38)
    ranks = rng.choice(np.asarray([1, 3, 8], np.int32), size=5)
    pool = spec.make_pool_all_resident(rng, h, L, len(dims), ranks, proj_dims=dims)
    ids = rng.integers(-1, 5, size=30).astype(np.int32)
    key_of = dict(zip(pool.page_ids.tolist(), pool.page_keys.tolist()))
    _, _, ga = oracle.group_tokens(ids)
    pv = [(-(-di // h), -(-do // h)) for di, do in dims]
    U = sum(a + b for a, b in pv)
    for l in range(L):
        for p in range(len(dims)):
            pre = sum(a + b for a, b in pv[:p])
            pages = oracle.page_list(pool.pt, pool.pt_off, pool.ranks, pool.num_proj, l, p, ga,
                                     h=h, proj_dims=pool.proj_dims)
            pos = 0
            for a in ga:
                r = int(pool.ranks[a])
                a0 = r * (l * U + pre)
                for ab, nblk in ((0, pv[p][0]), (1, pv[p][1])):
                    base = a0 + ab * pv[p][0] * r
                    for kb in range(nblk):
                        for j in range(r):
                            assert key_of[int(pages[pos])] == int(spec.page_key(a, base + kb * r + j))
                            pos += 1
            assert pos == pages.size


# ----------------------------------------------------------------------------- generator sanity

def test_generator_moments():
    h = 4096
    rows = np.zeros((64, h), np.uint16)
    keys = spec.row_key(spec.KIND_X, 0, 0, np.arange(64))
    vg.fill_rows_host(rows, np.arange(64), keys, 1234, vg.DIST_NORMAL, vg.normal_param(1.0))
    v = vg.bf16_bits_to_f64(rows)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01 and np.abs(v).max() <= 3.47
    vg.fill_rows_host(rows, np.arange(64), keys, 1234, vg.DIST_UNIFORM, a_param(h))
    u = vg.bf16_bits_to_f64(rows)
    b = 1 / np.sqrt(h)
    assert np.abs(u).max() <= b * (1 + 2 ** -8) and abs(u.mean()) < 0.01 * b
    assert abs(u.std() - b / np.sqrt(3)) < 0.01 * b


def test_zipf_batches_match_pages_simulation():
    """pofe.ai page, "How many adapters are actually in a batch?": 1,000 adapters with
    Zipf popularity, batches of 64 hold 33 to 62 distinct adapters; with 64 LRU slots
    at Zipf 1.0 about half of arrivals miss."""
    import collections
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "worked_example_8b.json")))["simulation"]
    rng = np.random.default_rng(0)
    p = spec.zipf_probs(g["adapters"], 1.0)
    draws = rng.choice(g["adapters"], size=(2000, g["batch"]), p=p)
    distinct = np.array([np.unique(b).size for b in draws])
    lo, hi = g["distinct_per_batch_range"]
    assert lo <= distinct.mean() <= hi
    arrivals = rng.choice(g["adapters"], size=200_000, p=p)
    lru = collections.OrderedDict()
    misses = 0
    for k, a in enumerate(arrivals):
        if a in lru:
            lru.move_to_end(a)
        else:
            if k >= 20_000:
                misses += 1
            lru[a] = True
            if len(lru) > g["slots"]:
                lru.popitem(last=False)
    frac = misses / (arrivals.size - 20_000)
    assert abs(frac - g["miss_fraction_at_64_slots_zipf_1"]) < 0.08


# ----------------------------------------------------------------------------- the expand step alone

def test_expand_matches_dense_B():
    """The expand alone: y0 + s B t with B assembled from the generator keys (not through
    the page table), for t = the oracle's shrink; B's orientation and page walk pinned."""
    wl = small_multi(seed=23)
    hi = host_inputs(wl)
    ids = wl.batch.token_adapter()
    p = wl.pool
    for (l, pj) in wl.problems:
        y0 = vg.bf16_bits_to_f64(hi.y0[(l, pj)])
        _, t, _ = run_oracle(wl, hi, l, pj, want_t=True)
        got = oracle.lora_expand(hi.pool, hi.pt, p.pt_off, p.ranks, p.scales, p.num_layers, p.num_proj,
                                 l, pj, t, y0, ids)
        for i, a in enumerate(ids):
            if a < 0:
                assert np.array_equal(got[i], y0[i])
                continue
            _, B = dense_adapter(wl, a, l, pj)
            want = y0[i] + float(p.scales[a]) * (B @ t[i, :B.shape[1]])
            np.testing.assert_allclose(got[i], want, rtol=1e-13, atol=1e-13)


def test_shrink_then_expand_is_the_delta():
    """The two steps composed (shrink of the C oracle, expand of the Python one) give the
    whole delta of the C oracle; the expand is linear in t."""
    wl = small_multi(seed=29)
    hi = host_inputs(wl)
    ids = wl.batch.token_adapter()
    p = wl.pool
    rng = np.random.default_rng(3)
    for (l, pj) in wl.problems:
        y0 = vg.bf16_bits_to_f64(hi.y0[(l, pj)])
        y_ref, t, _ = run_oracle(wl, hi, l, pj, want_t=True)
        args = (hi.pool, hi.pt, p.pt_off, p.ranks, p.scales, p.num_layers, p.num_proj, l, pj)
        np.testing.assert_allclose(oracle.lora_expand(*args, t, y0, ids), y_ref, rtol=1e-12, atol=1e-12)
        t2 = rng.standard_normal(t.shape)
        lhs = oracle.lora_expand(*args, t + t2, y0, ids)
        rhs = oracle.lora_expand(*args, t, y0, ids) + oracle.lora_expand(*args, t2, np.zeros_like(y0), ids)
        np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("n_shards", [2, 4])
def test_tensor_parallel_partition_identity(n_shards):
    """"S-LoRA: Serving Thousands of Concurrent LoRA Adapters", "Kernels and tensor
    parallelism": the adapters partitioned as the base model is.  Shard k holds columns
    [k h/N, (k+1) h/N) of every page: the sum over shards of their shrinks (each over its
    input columns) is the whole shrink, and each shard's expand with that sum gives its
    output columns of the whole delta."""
    from heterogeneous_adapters_gb300 import tp
    wl = small_multi(seed=31, h=64)
    hi = host_inputs(wl)
    ids = wl.batch.token_adapter()
    p = wl.pool
    h = p.h
    for (l, pj) in wl.problems:
        y0 = vg.bf16_bits_to_f64(hi.y0[(l, pj)])
        y_ref, t_ref, _ = run_oracle(wl, hi, l, pj, want_t=True)
        parts = []
        for k in range(n_shards):
            lo, hi_ = tp.shard_range(h, n_shards, k)
            _, tk, _ = oracle.lora_delta(np.ascontiguousarray(hi.pool[:, lo:hi_]), hi.pt, p.pt_off, p.ranks,
                                         p.scales, p.num_layers, p.num_proj, l, pj,
                                         np.ascontiguousarray(hi.x[(l, pj)][:, lo:hi_]),
                                         np.zeros((ids.size, hi_ - lo)), ids, want_t=True)
            parts.append(tk)
        t_sum = np.sum(parts, axis=0)
        np.testing.assert_allclose(t_sum, t_ref, rtol=1e-12, atol=1e-12)
        for k in range(n_shards):
            lo, hi_ = tp.shard_range(h, n_shards, k)
            yk = oracle.lora_expand(np.ascontiguousarray(hi.pool[:, lo:hi_]), hi.pt, p.pt_off, p.ranks, p.scales,
                                    p.num_layers, p.num_proj, l, pj, t_sum, y0[:, lo:hi_], ids)
            np.testing.assert_allclose(yk, y_ref[:, lo:hi_], rtol=1e-12, atol=1e-12)
