"""Tensor-parallel LoRA delta: N GPUs each hold 1/N of every adapter.

"S-LoRA: Serving Thousands of Concurrent LoRA Adapters", "Kernels and tensor parallelism":
with the base model split across GPUs as Megatron-LM splits it, the adapters are split
alike, and the LoRA terms add to the base model's communication only a small exchange of
the B x r intermediate (r is much smaller than h).

Partition (the reading used here).  For every projection, rank k of N holds input columns
[k d_in / N, (k+1) d_in / N) of every A row and output rows [k d_out / N, (k+1) d_out / N)
of every B column -- for the h x h projections of one unified pool, columns
[k h / N, (k+1) h / N) of every pool page, so each rank's pool is an ordinary pool of
h / N-wide pages under the same page table.  Then, per projection:
  shrink     rank k: t_k = s * x[:, in_k] A[:, in_k]^T          (lora_shrink on its shard)
  exchange   t = sum_k t_k                                        (one all-reduce of T x r)
  expand     rank k: y[:, out_k] += t B[out_k, :]^T               (lora_expand on its shard)
Rank k's x is its column shard of the input and its y the column shard of the output: the
output sharding of a column-parallel base layer (q, k, v, gate, up).  A row-parallel base
layer (o, down) has its input sharded the same way already; its partial base outputs are
summed by the base model's own all-reduce, and this y shard adds the LoRA term to its
columns of that result.  The exchange moves 2 (N - 1) / N * T * r values per projection
with a ring all-reduce.
"""
from __future__ import annotations


def shard_range(d: int, n: int, k: int) -> tuple[int, int]:
    """Columns [lo, hi) of a width-d dimension held by rank k of n (equal contiguous
    shards; each a multiple of 8 columns, as the library's widths must be)."""
    if n < 1 or not 0 <= k < n:
        raise ValueError(f"rank {k} of {n}")
    if d % n != 0 or (d // n) % 8 != 0:
        raise ValueError(f"width {d} does not split into {n} shards of a multiple of 8 columns")
    w = d // n
    return k * w, (k + 1) * w


def exchange_values(tokens: int, rank_max: int, n: int) -> float:
    """Values each rank sends (and receives) for one projection's exchange: a ring
    all-reduce of the T x r_max partial t moves 2 (N - 1) / N of it."""
    return 2.0 * (n - 1) / n * tokens * rank_max


class TensorParallelDelta:
    """The delta of one rank's shard: shrink, sum of the shards' partial t, expand.

    pool: this rank's lora Pool (its column shard of every page).  shrink / expand /
    all_reduce default to the library's lora_shrink and lora_expand and to
    torch.distributed.all_reduce (sum) over `group` on the same device as t; a caller may
    pass others with the same signatures.  Kernels and collective run on the current
    stream of t's device: pass that stream's handle to apply()."""

    def __init__(self, pool, group=None, shrink=None, expand=None, all_reduce=None):
        from . import _binding
        self.pool = pool
        self.group = group
        self._shrink = shrink or _binding.shrink
        self._expand = expand or _binding.expand
        self._all_reduce = all_reduce or self._torch_all_reduce

    def _torch_all_reduce(self, t):
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=self.group)

    def apply(self, problems, token_adapter, T, ws, ws_bytes, t, stream):
        """y of every problem (this rank's output columns) += the whole projection's delta.
        t: fp32 [nprob][T][r_max] scratch, zeroed by the caller (entries a shard does not
        write must add up to zero across the ranks)."""
        self._shrink(self.pool, problems, token_adapter, T, ws, ws_bytes, t, stream)
        self._all_reduce(t)
        self._expand(self.pool, problems, T, ws, ws_bytes, t, stream)
