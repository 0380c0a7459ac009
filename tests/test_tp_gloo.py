"""Tensor-parallel LoRA across world_size-2 gloo ranks on CPU (no GPU): each rank holds its
column shard of every pool page, computes its partial shrink, the ranks sum the partial t
with the module's all-reduce, and each expands its output columns.  The shrink and expand
steps are the fp64 oracle's here (the GPU kernels need a GPU); what is under test is the
partition and the exchange of heterogeneous_adapters_gb300.tp, against the oracle's
unsharded delta."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _case():
    from workloads import spec
    return spec.decode_workload("tp-gloo", 37, 128, 2, 2, 6, [2, 4, 8, 16], 20, None, base_ids=True)


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from heterogeneous_adapters_gb300 import tp
        from workloads import valuegen as vg
        from workloads.materialize import host_inputs

        wl = _case()
        hi = host_inputs(wl)
        p = wl.pool
        ids = wl.batch.token_adapter()
        lo, hi_ = tp.shard_range(p.h, world, rank)
        shard_pool = np.ascontiguousarray(hi.pool[:, lo:hi_])
        worst = 0.0
        for (l, pj) in wl.problems:
            x_k = np.ascontiguousarray(hi.x[(l, pj)][:, lo:hi_])
            y0 = vg.bf16_bits_to_f64(hi.y0[(l, pj)])
            y_k = {}

            def shrink(pool, problems, token_adapter, T, ws, ws_bytes, t, stream):
                _, tk, _ = oracle.lora_delta(shard_pool, hi.pt, p.pt_off, p.ranks, p.scales, p.num_layers,
                                             p.num_proj, l, pj, x_k, np.zeros((T, hi_ - lo)), token_adapter,
                                             want_t=True)
                t[0, :, :tk.shape[1]] = torch.from_numpy(tk)

            def expand(pool, problems, T, ws, ws_bytes, t, stream):
                y_k["y"] = oracle.lora_expand(shard_pool, hi.pt, p.pt_off, p.ranks, p.scales, p.num_layers,
                                              p.num_proj, l, pj, t[0].numpy(), y0[:, lo:hi_], ids)

            delta = tp.TensorParallelDelta(None, shrink=shrink, expand=expand)
            t = torch.zeros((1, ids.size, p.r_max), dtype=torch.float64)
            delta.apply([None], ids, ids.size, None, 0, t, None)
            y_ref, _, _ = oracle.lora_delta(hi.pool, hi.pt, p.pt_off, p.ranks, p.scales, p.num_layers,
                                            p.num_proj, l, pj, hi.x[(l, pj)], y0, ids)
            err = np.abs(y_k["y"] - y_ref[:, lo:hi_]) / (np.abs(y_ref[:, lo:hi_]) + 1e-300)
            worst = max(worst, float(np.max(np.where(np.abs(y_ref[:, lo:hi_]) > 0, err, 0))))
        out[rank] = worst
    finally:
        dist.destroy_process_group()


def test_two_rank_tensor_parallel_delta_matches_unsharded():
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for rank, worst in res.items():
        assert worst < 1e-12, (rank, worst)


def test_shard_ranges_and_exchange_volume():
    from heterogeneous_adapters_gb300 import tp
    assert [tp.shard_range(4096, 4, k) for k in range(4)] == [(0, 1024), (1024, 2048), (2048, 3072), (3072, 4096)]
    with pytest.raises(ValueError):
        tp.shard_range(4100, 4, 0)
    with pytest.raises(ValueError):
        tp.shard_range(64, 16, 0)     # 4-column shards
    # a ring all-reduce of T x r: 2 (N-1)/N of it per rank; none for one rank
    assert tp.exchange_values(64, 16, 1) == 0.0
    assert tp.exchange_values(64, 16, 4) == pytest.approx(1.5 * 64 * 16)
