"""Seeded synthetic workloads shaped like the multi-LoRA serving pages' examples.

Only metadata and keys live here (adapter ranks, per-token adapter ids, segment
lengths, page placement, page tables, row keys for the value generator); bulk
values come from the counter-based generator in valuegen.  Nothing in this
module computes any part of the LoRA delta.

Conventions, shared by every consumer of a workload:
  * adapter a has rank r_a, scale s_a = ALPHA / r_a (ALPHA = 16), and a block of
    L*P*2*r_a page-table entries starting at pt_off[a];
  * entry ((l*P + p)*2 + ab)*r_a + j of that block is the page holding row j of
    A_a (ab = 0) or column j of B_a (ab = 1) for layer l, projection p;
  * A_a is r_a x d_in, B_a is d_out x r_a, d_in = d_out = h = one page;
  * token adapter id -1 means base only (no delta).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np

ALPHA = 16.0
KIND_PAGE = 1
KIND_X = 2
KIND_Y = 3
SIGMA_X = 1.0       # x ~ N(0, 1)
SIGMA_Y = 1.0       # y0 ~ N(0, 1)
SIGMA_B = 0.02      # B ~ N(0, 0.02)


def page_key(owner, local):
    """Generator key of adapter page `local` of the block owned by `owner`."""
    owner = np.asarray(owner, dtype=np.uint64)
    local = np.asarray(local, dtype=np.uint64)
    return (np.uint64(KIND_PAGE) << np.uint64(56)) | (owner << np.uint64(24)) | local


def row_key(kind: int, layer, proj, row):
    """Generator key of row `row` of the x (KIND_X) or y0 (KIND_Y) buffer of (layer, proj)."""
    layer = np.asarray(layer, dtype=np.uint64)
    proj = np.asarray(proj, dtype=np.uint64)
    row = np.asarray(row, dtype=np.uint64)
    return ((np.uint64(kind) << np.uint64(56)) | (layer << np.uint64(40)) |
            (proj << np.uint64(32)) | row)


def zipf_probs(n: int, s: float) -> np.ndarray:
    """Finite Zipf popularity p_k proportional to k^-s, k = 1..n (adapter id k-1)."""
    w = np.arange(1, n + 1, dtype=np.float64) ** (-s)
    return w / w.sum()


@dataclass
class Pool:
    """Unified paged pool description: one page = h bf16 values."""
    h: int
    num_layers: int
    num_proj: int
    ranks: np.ndarray            # int32 [N]
    pt_off: np.ndarray           # int64 [N]
    pt: np.ndarray               # int32 [pt_len]; -1 = page not resident
    num_pages: int
    # pages that hold adapter values: physical page id, generator key, A (0) or B (1)
    page_ids: np.ndarray         # int64 [n_filled]
    page_keys: np.ndarray        # uint64 [n_filled]
    page_ab: np.ndarray          # uint8 [n_filled]
    r_max: int = 0
    # (d_in, d_out) of every projection, int32 [P, 2]; None: all h x h.  A vector of
    # length d takes ceil(d / h) pages; an adapter's block for (layer, proj, A or B) holds
    # r * pages-per-vector entries, page block by page block (page kb of every row or
    # column, then page kb + 1), blocks in (layer, proj, A, B) order.
    proj_dims: np.ndarray | None = None

    @property
    def num_adapters(self) -> int:
        return int(self.ranks.size)

    @property
    def scales(self) -> np.ndarray:
        return (ALPHA / self.ranks.astype(np.float64)).astype(np.float32)

    def dims(self, proj: int):
        """(d_in, d_out) of projection proj."""
        if self.proj_dims is None:
            return self.h, self.h
        return int(self.proj_dims[proj][0]), int(self.proj_dims[proj][1])

    def layout_units(self):
        """(units of one layer, units before each projection, pages per A row and per B
        column of each projection); one unit = r_a page-table entries."""
        return layout_units(self.h, self.num_proj, self.proj_dims)

    def block_entries(self, adapter: int, layer: int, proj: int, ab: int) -> np.ndarray:
        """Indices into pt of the pages of A (ab=0) or B (ab=1) for (adapter, layer, proj):
        r_a * pages-per-vector entries, page block by page block."""
        r = int(self.ranks[adapter])
        U, pre, pv_in, pv_out = self.layout_units()
        base = int(self.pt_off[adapter]) + r * (layer * U + pre[proj] + (pv_in[proj] if ab else 0))
        n = r * (pv_out[proj] if ab else pv_in[proj])
        return np.arange(base, base + n, dtype=np.int64)


@dataclass
class Batch:
    """Token batch: prefill segments first (rows seg_start[s]..seg_start[s+1]),
    then decode tokens (one row each).  Decode-only batches have no segments."""
    seg_start: np.ndarray        # int32 [S+1] (S may be 0: then [0])
    seg_adapter: np.ndarray      # int32 [S]
    dec_adapter: np.ndarray      # int32 [Td]

    @property
    def num_segments(self) -> int:
        return int(self.seg_adapter.size)

    @property
    def num_decode(self) -> int:
        return int(self.dec_adapter.size)

    @property
    def num_tokens(self) -> int:
        return int(self.seg_start[-1]) + self.num_decode

    def token_adapter(self) -> np.ndarray:
        """Per-token adapter id (int32 [T])."""
        lens = np.diff(self.seg_start.astype(np.int64))
        pre = np.repeat(self.seg_adapter.astype(np.int32), lens)
        return np.concatenate([pre, self.dec_adapter.astype(np.int32)]).astype(np.int32)

    @property
    def kind(self) -> str:
        if self.num_segments == 0:
            return "decode"
        if self.num_decode == 0:
            return "prefill"
        return "mixed"


@dataclass
class Workload:
    name: str
    seed: int
    pool: Pool
    batch: Batch
    problems: list = field(default_factory=list)   # [(layer, proj)] of one step
    notes: str = ""
    # q, k and v (projections 0, 1, 2) of a layer read one input x, as in a transformer
    shared_x: bool = False

    @property
    def h(self) -> int:
        return self.pool.h

    def x_source(self, l: int, p: int):
        """The (layer, projection) whose x buffer problem (l, p) reads."""
        return (l, 0) if self.shared_x and p < 3 else (l, p)


# ----------------------------------------------------------------------------- pool layouts

def layout_units(h: int, P: int, proj_dims=None):
    """Page-table layout in units of r_a entries: (units of one layer, units before each
    projection, pages per A row and per B column of each projection)."""
    dims = [(h, h)] * P if proj_dims is None else [(int(a), int(b)) for a, b in np.asarray(proj_dims)]
    pv = lambda d: -(-d // h)   # noqa: E731
    pre, acc = [], 0
    for d_in, d_out in dims:
        pre.append(acc)
        acc += pv(d_in) + pv(d_out)
    return acc, pre, [pv(d[0]) for d in dims], [pv(d[1]) for d in dims]


def _block_sizes(ranks: np.ndarray, L: int, P: int, h: int = 1, proj_dims=None) -> np.ndarray:
    U = layout_units(h, P, proj_dims)[0]
    return (L * U) * ranks.astype(np.int64)


def _entry_owner_local(ranks: np.ndarray, pt_off: np.ndarray, sizes: np.ndarray, h: int = 1,
                       P: int = 1, proj_dims=None):
    owner = np.repeat(np.arange(ranks.size, dtype=np.int64), sizes)
    local = np.arange(int(sizes.sum()), dtype=np.int64) - pt_off[owner]
    U, _, pv_in, pv_out = layout_units(h, P, proj_dims)
    unit_ab = np.concatenate([[0] * a + [1] * b for a, b in zip(pv_in, pv_out)]).astype(np.uint8)
    ab = unit_ab[(local // ranks[owner].astype(np.int64)) % U]
    return owner, local, ab


def make_pool_all_resident(rng: np.random.Generator, h: int, L: int, P: int, ranks: np.ndarray,
                           num_pages: int | None = None, proj_dims=None) -> Pool:
    """Every adapter page resident, placed at shuffled page indices of the pool."""
    ranks = ranks.astype(np.int32)
    sizes = _block_sizes(ranks, L, P, h, proj_dims)
    pt_off = np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64)
    pt_len = int(sizes.sum())
    if num_pages is None:
        num_pages = pt_len
    assert num_pages >= pt_len
    placement = rng.permutation(num_pages)[:pt_len].astype(np.int64)
    owner, local, ab = _entry_owner_local(ranks, pt_off, sizes, h, P, proj_dims)
    return Pool(h=h, num_layers=L, num_proj=P, ranks=ranks, pt_off=pt_off,
                pt=placement.astype(np.int32), num_pages=num_pages, page_ids=placement,
                page_keys=page_key(owner, local), page_ab=ab, r_max=int(ranks.max()),
                proj_dims=None if proj_dims is None else np.asarray(proj_dims, np.int32).reshape(P, 2))


def make_pool_subset_resident(rng: np.random.Generator, h: int, L: int, P: int,
                              ranks: np.ndarray, resident: np.ndarray, num_pages: int) -> Pool:
    """Only the adapters in `resident` have pages (at shuffled indices of a pool of
    num_pages); the page-table entries of the others are -1 (not resident)."""
    ranks = ranks.astype(np.int32)
    sizes = _block_sizes(ranks, L, P)
    pt_off = np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64)
    pt_len = int(sizes.sum())
    owner, local, ab = _entry_owner_local(ranks, pt_off, sizes)
    is_res = np.zeros(ranks.size, dtype=bool)
    is_res[np.asarray(resident, dtype=np.int64)] = True
    sel = np.nonzero(is_res[owner])[0]
    assert sel.size <= num_pages
    placement = rng.permutation(num_pages)[:sel.size].astype(np.int64)
    pt = np.full(pt_len, -1, dtype=np.int32)
    pt[sel] = placement
    return Pool(h=h, num_layers=L, num_proj=P, ranks=ranks, pt_off=pt_off, pt=pt,
                num_pages=num_pages, page_ids=placement, page_keys=page_key(owner[sel], local[sel]),
                page_ab=ab[sel], r_max=int(ranks.max()))


def make_pool_layer_slices(rng: np.random.Generator, h: int, L: int, P: int, ranks: np.ndarray,
                           num_pages: int) -> Pool:
    """Each adapter owns ONE layer's worth of pages (P*2*r_a, its "slice"), placed
    at random among num_pages pool pages (the rest stand for KV-cache pages).
    Layer l of adapter a reads the slice of pi_l(a), where pi_0 is the identity
    and pi_l (l >= 1) is a seeded permutation of the adapters within each rank
    class, so consecutive layers read different physical pages."""
    ranks = ranks.astype(np.int32)
    N = ranks.size
    slice_sizes = (P * 2) * ranks.astype(np.int64)
    slice_off = np.concatenate([[0], np.cumsum(slice_sizes)[:-1]]).astype(np.int64)
    n_slice = int(slice_sizes.sum())
    assert n_slice <= num_pages
    slice_pages = rng.permutation(num_pages)[:n_slice].astype(np.int64)
    owner_s, local_s, ab_s = _entry_owner_local(ranks, slice_off, slice_sizes // 1)
    # layer permutations within rank classes
    perms = np.empty((L, N), dtype=np.int64)
    perms[0] = np.arange(N)
    for l in range(1, L):
        p = np.arange(N)
        for r in np.unique(ranks):
            idx = np.nonzero(ranks == r)[0]
            p[idx] = idx[rng.permutation(idx.size)]
        perms[l] = p
    sizes = _block_sizes(ranks, L, P)
    pt_off = np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64)
    pt = np.empty(int(sizes.sum()), dtype=np.int32)
    for a in range(N):
        r = int(ranks[a])
        per_layer = P * 2 * r
        for l in range(L):
            src = perms[l, a]
            pt[pt_off[a] + l * per_layer: pt_off[a] + (l + 1) * per_layer] = \
                slice_pages[slice_off[src]: slice_off[src] + per_layer]
    return Pool(h=h, num_layers=L, num_proj=P, ranks=ranks, pt_off=pt_off, pt=pt,
                num_pages=num_pages, page_ids=slice_pages, page_keys=page_key(owner_s, local_s),
                page_ab=ab_s, r_max=int(ranks.max()))


# ----------------------------------------------------------------------------- builders

def all_problems(L: int, P: int) -> list:
    return [(l, p) for l in range(L) for p in range(P)]


def decode_workload(name: str, seed: int, h: int, L: int, P: int, num_adapters: int,
                    rank_choices, T: int, zipf_s: float | None, num_pages: int | None = None,
                    base_ids: bool = False, distinct: bool = False, layer_slices: bool = False,
                    notes: str = "", proj_dims=None) -> Workload:
    """Decode batch of T one-token requests.  Adapter ids: Zipf(zipf_s) over the
    adapters, or uniform over {-1..N-1} when base_ids, or distinct (sampled
    without replacement) when distinct."""
    rng = np.random.default_rng(seed)
    ranks = rng.choice(np.asarray(rank_choices, dtype=np.int32), size=num_adapters)
    if base_ids:
        ids = rng.integers(-1, num_adapters, size=T)
    elif distinct:
        ids = rng.choice(num_adapters, size=T, replace=False)
    else:
        ids = rng.choice(num_adapters, size=T, p=zipf_probs(num_adapters, zipf_s))
    if layer_slices:
        assert proj_dims is None
        pool = make_pool_layer_slices(rng, h, L, P, ranks, num_pages)
    else:
        pool = make_pool_all_resident(rng, h, L, P, ranks, num_pages, proj_dims)
    batch = Batch(seg_start=np.zeros(1, np.int32), seg_adapter=np.zeros(0, np.int32),
                  dec_adapter=ids.astype(np.int32))
    return Workload(name, seed, pool, batch, all_problems(L, P), notes)


def prefill_workload(name: str, seed: int, h: int, L: int, P: int, num_adapters: int,
                     rank_choices, num_requests: int, len_lo: int, len_hi: int,
                     zipf_s: float, notes: str = "") -> Workload:
    """Prefill batch: num_requests prompts of lengths uniform in [len_lo, len_hi]
    (inclusive) packed contiguously, one Zipf(zipf_s) adapter per request."""
    rng = np.random.default_rng(seed)
    ranks = rng.choice(np.asarray(rank_choices, dtype=np.int32), size=num_adapters)
    lens = rng.integers(len_lo, len_hi + 1, size=num_requests)
    ids = rng.choice(num_adapters, size=num_requests, p=zipf_probs(num_adapters, zipf_s))
    pool = make_pool_all_resident(rng, h, L, P, ranks)
    seg_start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    batch = Batch(seg_start=seg_start, seg_adapter=ids.astype(np.int32),
                  dec_adapter=np.zeros(0, np.int32))
    return Workload(name, seed, pool, batch, all_problems(L, P), notes)


def mixed_workload(name: str, seed: int, h: int, L: int, P: int, num_adapters: int,
                   rank_choices, num_prefill: int, len_lo: int, len_hi: int, num_decode: int,
                   num_base_requests: int, zipf_s: float, pool_pages: int,
                   notes: str = "") -> Workload:
    """Continuous-batching step: prefill segments then decode tokens.  Exactly
    num_base_requests of the requests (sampled without replacement) are
    base-only.  Only adapters referenced by the batch are resident, at shuffled
    indices of a pool of pool_pages pages."""
    rng = np.random.default_rng(seed)
    ranks = rng.choice(np.asarray(rank_choices, dtype=np.int32), size=num_adapters)
    lens = rng.integers(len_lo, len_hi + 1, size=num_prefill)
    n_req = num_prefill + num_decode
    ids = rng.choice(num_adapters, size=n_req, p=zipf_probs(num_adapters, zipf_s))
    base = rng.choice(n_req, size=num_base_requests, replace=False)
    ids[base] = -1
    resident = np.unique(ids[ids >= 0])
    pool = make_pool_subset_resident(rng, h, L, P, ranks, resident, pool_pages)
    seg_start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    batch = Batch(seg_start=seg_start, seg_adapter=ids[:num_prefill].astype(np.int32),
                  dec_adapter=ids[num_prefill:].astype(np.int32))
    return Workload(name, seed, pool, batch, all_problems(L, P), notes)


# ----------------------------------------------------------------------------- named workloads

def tiny_decode() -> Workload:
    """Tiny check: h=256, 1 layer x 1 projection, ranks {4,8,8,16}, 16 tokens with
    ids uniform in {-1..3}, 256-page pool with the 72 adapter pages shuffled in."""
    rng = np.random.default_rng(1000)
    ranks = np.array([4, 8, 8, 16], dtype=np.int32)
    ids = rng.integers(-1, 4, size=16).astype(np.int32)
    pool = make_pool_all_resident(rng, 256, 1, 1, ranks, num_pages=256)
    batch = Batch(np.zeros(1, np.int32), np.zeros(0, np.int32), ids)
    return Workload("tiny-h256-r4-16-t16", 1000, pool, batch, [(0, 0)])


def llama7b_decode() -> Workload:
    """Llama-7B decode: 64 one-token requests, Zipf(1.0) over 2,000 adapters of ranks
    {8..64}, 32 layers x q/k/v/o, every adapter resident."""
    return decode_workload("llama7b-decode-bgmv-h4096-t64-a2000", 1001, 4096, 32, 4, 2000,
                           [8, 16, 32, 64], 64, 1.0)


def llama7b_prefill() -> Workload:
    """Llama-7B prefill: 32 prompts of lengths uniform in [64, 1024], Zipf(1.0) over 1,000
    adapters of ranks {8..64}, 32 layers x q/k/v/o."""
    return prefill_workload("llama7b-prefill-sgmv-h4096-s32-a1000", 1002, 4096, 32, 4, 1000,
                            [8, 16, 32, 64], 32, 64, 1024, 1.0)


def mixed_13b() -> Workload:
    """13B continuous-batching step: 8 prefill prompts of [128, 2048] tokens and 192 decode
    tokens, 20 of the 200 requests base-only, Zipf(0.8) over 2,000 adapters of ranks
    {8..128}, 40 layers x q/k/v/o, only the referenced adapters resident."""
    return mixed_workload("13b-mixed-h5120-p8-d192-a2000", 1003, 5120, 40, 4, 2000,
                          [8, 16, 32, 64, 128], 8, 128, 2048, 192, 20, 0.8,
                          pool_pages=1 << 22)


def pool_stress(variant: str = "distinct") -> Workload:
    """Unified-pool stress: 256 decode tokens with distinct adapters (or Zipf(1.2)) from
    2,000, in a 2^20-page pool holding one layer's slice of each adapter."""
    assert variant in ("distinct", "zipf")
    return decode_workload(f"unified-pool-stress-{variant}-h4096-t256-a2000",
                           1004 if variant == "distinct" else 1014, 4096, 32, 4, 2000,
                           [8, 16, 32, 64], 256, 1.2 if variant == "zipf" else None,
                           num_pages=1 << 20, distinct=(variant == "distinct"),
                           layer_slices=True)


# Llama-3-8B (h 4096, 8 KV heads of 128, MLP 14336): q, k, v, o, gate, up, down
LLAMA3_8B_DIMS = [(4096, 4096), (4096, 1024), (4096, 1024), (4096, 4096),
                  (4096, 14336), (4096, 14336), (14336, 4096)]


def llama3_8b_decode(layers: int = 32) -> Workload:
    """Decode batch of 64 tokens over 600 adapters of ranks {8..64} on a Llama-3-8B base,
    every projection of every layer adapted at its own widths (about 105 GB of pool at
    32 layers)."""
    return decode_workload(f"llama3-8b-decode-bgmv-h4096-t64-a600-7proj-l{layers}", 1008, 4096,
                           layers, 7, 600, [8, 16, 32, 64], 64, 1.0,
                           proj_dims=LLAMA3_8B_DIMS)


def llama3_8b_prefill(layers: int = 4) -> Workload:
    """Prefill batch of 32 prompts of lengths uniform in [64, 1024] over 600 adapters of
    ranks {8..64} (Zipf 1.0) on a Llama-3-8B base, every projection adapted at its own
    widths.  Four layers by default: every projection's x and y buffers are allocated at
    the widest projection's width, so all 32 layers would not fit beside the pool."""
    rng = np.random.default_rng(1009)
    P = len(LLAMA3_8B_DIMS)
    ranks = rng.choice(np.asarray([8, 16, 32, 64], np.int32), size=600)
    lens = rng.integers(64, 1025, size=32)
    ids = rng.choice(600, size=32, p=zipf_probs(600, 1.0))
    pool = make_pool_all_resident(rng, 4096, layers, P, ranks, proj_dims=LLAMA3_8B_DIMS)
    seg_start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    batch = Batch(seg_start=seg_start, seg_adapter=ids.astype(np.int32),
                  dec_adapter=np.zeros(0, np.int32))
    return Workload(f"llama3-8b-prefill-sgmv-h4096-s32-a600-7proj-l{layers}", 1009, pool, batch,
                    all_problems(layers, P))


def llama3_8b_mixed(layers: int = 4) -> Workload:
    """Continuous-batching step on a Llama-3-8B base: 8 prefill prompts of [128, 2048] tokens
    and 192 decode tokens, 20 of the 200 requests base-only, Zipf(0.8) over 600 adapters of
    ranks {8..64}, every projection adapted at its own widths, 4 layers by default."""
    rng = np.random.default_rng(1010)
    P = len(LLAMA3_8B_DIMS)
    ranks = rng.choice(np.asarray([8, 16, 32, 64], np.int32), size=600)
    lens = rng.integers(128, 2049, size=8)
    ids = rng.choice(600, size=200, p=zipf_probs(600, 0.8))
    ids[rng.choice(200, size=20, replace=False)] = -1
    pool = make_pool_all_resident(rng, 4096, layers, P, ranks, proj_dims=LLAMA3_8B_DIMS)
    seg_start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    batch = Batch(seg_start=seg_start, seg_adapter=ids[:8].astype(np.int32),
                  dec_adapter=ids[8:].astype(np.int32))
    return Workload(f"llama3-8b-mixed-h4096-p8-d192-a600-7proj-l{layers}", 1010, pool, batch,
                    all_problems(layers, P))


WORKLOADS = {
    "tiny": tiny_decode,
    "decode": llama7b_decode,
    "prefill": llama7b_prefill,
    "mixed": mixed_13b,
    "stress-distinct": lambda: pool_stress("distinct"),
    "stress-zipf": lambda: pool_stress("zipf"),
    "llama3-decode": llama3_8b_decode,
    "llama3-prefill": llama3_8b_prefill,
    "llama3-mixed": llama3_8b_mixed,
}


def shrink_problems(wl: Workload, problems: list) -> Workload:
    """Same workload restricted to a list of (layer, proj) problems."""
    return dataclasses.replace(wl, problems=list(problems))
