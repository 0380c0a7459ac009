"""Shared test harness: run the GPU path through the C ABI on a seeded workload and
compare with the fp64 CPU oracle on the same inputs (regenerated on the host by
the shared generator; nothing the oracle sees comes from the GPU path)."""
from __future__ import annotations

import numpy as np

import oracle
from workloads import valuegen as vg
from workloads.materialize import device_inputs, host_inputs

# Parity gate: |y_gpu - y_ref| <= GATE_ABS + GATE_REL * |y_ref| elementwise.
GATE_ABS = 1e-2
GATE_REL = 1e-2
# Delta-only check (y0 = 0): bf16 rounding of the stored result (half an ulp is at
# most 2^-8 of the value) plus the fp32 accumulation error, bounded by DELTA_ACC
# times the magnitude sum s * sum_j (|t_j| + T_ACC * S_j) |B_jn|.
BF16_HALF_ULP_REL = 2.0 ** -8
DELTA_ACC = 1e-4
# Shrink check: |t_gpu - t_ref| <= T_ACC * S_j with S_j = sum_k |x_k A_jk| (an fp32
# dot product of length h errs by well under 2e-5 of that sum in practice; a dropped
# or duplicated term errs by O(1) of it).
T_ACC = 2e-5


class GpuCase:
    """Device buffers, pool handle and workspace of one workload."""

    def __init__(self, wl, problems=None, y0_zero=False, nan_dummies=True, device="cuda:0",
                 tuning=None):
        """tuning: lora_pool_set_tuning fields for the pool (kernel choice, stage shapes)."""
        import torch
        import heterogeneous_adapters_gb300 as lora
        self.torch = torch
        self.lora = lora
        self.wl = wl
        self.device = device
        self.dev = device_inputs(wl, problems, device=device, nan_dummies=nan_dummies)
        self.y0_zero = y0_zero
        if y0_zero:
            self.dev.y.zero_()
        self.y_init = self.dev.y.clone() if self.dev.y.numel() * 2 < (8 << 30) else None
        p = wl.pool
        self.pool = lora.Pool(self.dev.pool, p.num_pages, p.h, self.dev.pt, p.pt.size,
                              self.dev.pt_off, self.dev.ranks, self.dev.scales, p.num_adapters,
                              p.num_layers, p.num_proj, p.r_max, p.proj_dims)
        if tuning:
            self.pool.set_tuning(**tuning)
        b = wl.batch
        self.T = b.num_tokens
        self.nseg = b.num_segments + b.num_decode
        self.ws_bytes = lora.workspace_size(self.pool, self.T, self.nseg)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.stream = torch.cuda.current_stream(device).cuda_stream
        lora.workspace_init(self.ws, self.ws_bytes, self.stream)

    def problems(self):
        ldx, ldy = self.dev.x.shape[2], self.dev.y.shape[2]
        return [(self.dev.x[self.dev.x_src[i]], self.dev.y[i], ldx, ldy, l, p)
                for i, (l, p) in enumerate(self.dev.problems)]

    def run(self, mode=None):
        b, d, lora = self.wl.batch, self.dev, self.lora
        mode = mode or b.kind
        if mode == "decode":
            lora.bgmv(self.pool, self.problems(), d.token_adapter, self.T, self.ws, self.ws_bytes,
                      self.stream)
        elif mode == "prefill":
            lora.sgmv(self.pool, self.problems(), d.seg_start, d.seg_adapter, b.num_segments,
                      self.T, self.ws, self.ws_bytes, self.stream)
        else:
            lora.apply_mixed(self.pool, self.problems(), d.seg_start, d.seg_adapter,
                             b.num_segments, d.dec_adapter, b.num_decode, self.T, self.ws,
                             self.ws_bytes, self.stream)
        return self.error_bits()

    def error_bits(self) -> int:
        return self.lora.get_device_error(self.ws, self.stream)

    def y_bits(self, idx) -> np.ndarray:
        """y rows of problem idx, its d_out columns."""
        d_out = self.wl.pool.dims(self.dev.problems[idx][1])[1]
        return self.dev.y[idx, :, :d_out].contiguous().view(self.torch.int16).cpu().numpy().view(np.uint16)

    def y_f64(self, idx) -> np.ndarray:
        return vg.bf16_bits_to_f64(self.y_bits(idx))

    def close(self):
        self.pool.close()
        del self.dev, self.ws, self.y_init
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()


def oracle_problem(wl, hi, l, p, y0_zero=False, ids=None, want_t=False):
    pool = wl.pool
    d_out = pool.dims(p)[1]
    y0 = np.zeros((wl.batch.num_tokens, d_out)) if y0_zero else vg.bf16_bits_to_f64(hi.y0[(l, p)])
    ids = wl.batch.token_adapter() if ids is None else ids
    y_ref, t_ref, _ = oracle.lora_delta(hi.pool, hi.pt, pool.pt_off, pool.ranks, pool.scales,
                                        pool.num_layers, pool.num_proj, l, p, hi.x[(l, p)], y0,
                                        ids, want_t=want_t, proj_dims=pool.proj_dims)
    return y_ref, t_ref, y0


def block_values(wl, hi, a, l, p, ab):
    """A rows (ab=0, [r, d_in]) or B columns (ab=1, [r, d_out]) of adapter a for (l, p),
    float64, assembled from their pages (page kb of every vector, then page kb + 1)."""
    pool = wl.pool
    r = int(pool.ranks[a])
    d = pool.dims(p)[ab]
    pages = vg.bf16_bits_to_f64(hi.pool[hi.pt[pool.block_entries(a, l, p, ab)]])   # [pv * r, h]
    pv = pages.shape[0] // r
    return pages.reshape(pv, r, pool.h).transpose(1, 0, 2).reshape(r, pv * pool.h)[:, :d]


def magnitude_sums(wl, hi, l, p):
    """S[i, j] = sum_k |x_ik A_jk| and M[i, n] = s * sum_j (|t_ij| + T_ACC S_ij) |B_nj|
    per adapted row (float64), for the accumulation-error bounds above."""
    pool = wl.pool
    ids = wl.batch.token_adapter()
    xa = np.abs(vg.bf16_bits_to_f64(hi.x[(l, p)]))
    T = xa.shape[0]
    S = np.zeros((T, pool.r_max))
    M = np.zeros((T, pool.dims(p)[1]))
    for a in np.unique(ids[ids >= 0]):
        rows = np.nonzero(ids == a)[0]
        A = block_values(wl, hi, a, l, p, 0)
        B = np.abs(block_values(wl, hi, a, l, p, 1))
        Xa = vg.bf16_bits_to_f64(hi.x[(l, p)])[rows]
        r = A.shape[0]
        S[rows, :r] = xa[rows] @ np.abs(A).T
        tabs = np.abs(Xa @ A.T)
        M[rows] = float(pool.scales[a]) * ((tabs + T_ACC * S[rows, :r]) @ B)
    return S, M


def check_gate(y_gpu, y_ref, what=""):
    err = np.abs(y_gpu - y_ref)
    bound = GATE_ABS + GATE_REL * np.abs(y_ref)
    bad = ~(err <= bound)
    assert not bad.any(), (f"{what}: {bad.sum()} elements outside the gate, worst "
                           f"{(err - bound)[bad].max():.3g} over; max err {np.nanmax(err):.3g}")


def check_delta_only(y_gpu, y_ref, M, ids, what=""):
    rows = ids >= 0
    err = np.abs(y_gpu[rows] - y_ref[rows])
    bound = BF16_HALF_ULP_REL * np.abs(y_ref[rows]) + DELTA_ACC * M[rows] + 1e-30
    bad = ~(err <= bound)
    assert not bad.any(), f"{what}: {bad.sum()} delta elements outside the strict bound"


def check_base_rows_untouched(case, idx, hi_y0_bits, ids, what=""):
    got = case.y_bits(idx)
    base = ids == -1
    if case.y0_zero:
        want = np.zeros_like(got[base])
    else:
        want = hi_y0_bits[base]
    assert np.array_equal(got[base], want), f"{what}: a base-only row changed"


def full_check(wl, case, problem_idx, y0_zero=None, strict=True):
    """Oracle comparison of the listed problems of a GpuCase (all their elements)."""
    y0_zero = case.y0_zero if y0_zero is None else y0_zero
    probs = [case.dev.problems[i] for i in problem_idx]
    hi = host_inputs(wl, problems=probs)
    ids = wl.batch.token_adapter()
    for i, (l, p) in zip(problem_idx, probs):
        y_ref, _, _ = oracle_problem(wl, hi, l, p, y0_zero=y0_zero)
        y_gpu = case.y_f64(i)
        check_gate(y_gpu, y_ref, f"{wl.name} problem {(l, p)}")
        check_base_rows_untouched(case, i, hi.y0[(l, p)], ids, f"{wl.name} {(l, p)}")
        if strict and y0_zero:
            _, M = magnitude_sums(wl, hi, l, p)
            check_delta_only(y_gpu, y_ref, M, ids, f"{wl.name} {(l, p)}")
    return hi
