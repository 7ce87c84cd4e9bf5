"""Data-parallel replicas of the MLP block: micro-batches shared out over ranks,
fp32 gradients summed over ranks with one all-reduce.

Data parallelism distributes the data over processors, which update the
parameters synchronously; the only communication is an all-reduce that sums the
gradients of all processors ("STRONGHOLD: Fast and Affordable Billion-scale Deep
Learning Model Training" slides, items 4-5; MT-NLG's 3D parallelism combines it
with tensor slicing and pipelines: "Using DeepSpeed and Megatron to Train
Megatron-Turing NLG 530B", Summary).  With gradient accumulation (same page, Key
points) a step's k micro-batches are split over the ranks; each rank accumulates
its share in fp32 (mlp_bwd, accumulate = 0 then 1), and the all-reduce sum makes
every rank hold the gradients of all k micro-batches.  Global micro-batch j keeps
token offset j * T on whichever rank runs it, so its dropout mask, and the summed
gradients, do not depend on how the micro-batches were shared out.

The four gradient accumulators of a block are views into one contiguous fp32
buffer, so one collective covers them.  Every step of the block itself runs in
the library's kernels; this module only shares out work and calls the
collective (NCCL on GPU ranks, gloo on CPU ranks).
"""
from __future__ import annotations

from typing import Callable, Optional

import torch


def shard(k_total: int, world: int, rank: int) -> range:
    """The global micro-batch indices rank ``rank`` of ``world`` runs: contiguous
    blocks, the first ``k_total % world`` ranks taking one more."""
    if world <= 0 or not 0 <= rank < world or k_total < 0:
        raise ValueError(f"bad shard request: k_total {k_total}, world {world}, rank {rank}")
    base, extra = divmod(k_total, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def flat_gradients(h: int, ffn: int, device="cuda", dtype=torch.float32):
    """One contiguous buffer holding dA [h, ffn], da [ffn], dB [ffn, h], db [h], in
    that order, and the four views.  Every view starts 16-byte aligned when h and
    ffn are multiples of 8, as the library requires."""
    n_a, n_b = h * ffn, ffn * h
    flat = torch.zeros(n_a + ffn + n_b + h, dtype=dtype, device=device)
    dA = flat[:n_a].view(h, ffn)
    da = flat[n_a:n_a + ffn]
    dB = flat[n_a + ffn:n_a + ffn + n_b].view(ffn, h)
    db = flat[n_a + ffn + n_b:]
    return flat, (dA, da, dB, db)


def allreduce_gradients(flat: torch.Tensor, group=None, stream: Optional[torch.cuda.Stream] = None):
    """Sum ``flat`` over the ranks of ``group`` in place (torch.distributed; NCCL for
    CUDA tensors, ordered after the work already on ``stream``, gloo for CPU
    tensors)."""
    import torch.distributed as dist
    if flat.is_cuda:
        s = stream if stream is not None else torch.cuda.current_stream(flat.device)
        with torch.cuda.stream(s):
            dist.all_reduce(flat, op=dist.ReduceOp.SUM, group=group)
    else:
        dist.all_reduce(flat, op=dist.ReduceOp.SUM, group=group)


def data_parallel_step(k_total: int, rank: int, world: int, run_microbatch: Callable[[int, bool], None],
                       reset: Callable[[], None], flat: torch.Tensor, group=None, stream=None) -> range:
    """This rank's share of one optimizer step, then the gradient all-reduce.

    run_microbatch(j, accumulate): forward + backward of global micro-batch j,
        adding its weight and bias gradients to the accumulators (accumulate=True)
        or writing them (False: this rank's first micro-batch).
    reset(): zero the accumulators; called only on a rank without a micro-batch.
    flat: the contiguous buffer behind the accumulators (flat_gradients).
    Returns the global micro-batch indices this rank ran.  Afterwards every rank
    holds the sum over all k_total micro-batches.
    """
    mine = shard(k_total, world, rank)
    if len(mine) == 0:
        reset()
    for n, j in enumerate(mine):
        run_microbatch(j, n > 0)
    allreduce_gradients(flat, group, stream)
    return mine


def block_runner(wl, weights, microbatch: Callable[[int], tuple], buf, slice_mode="all", stream=None):
    """run_microbatch for the library's block on this GPU: global micro-batch j is
    ``microbatch(j)`` = (X_j, dO_j) with token offset j * tokens."""
    from . import mlp

    def run(j: int, accumulate: bool):
        X, dO = microbatch(j)
        mlp.block_step(wl, weights, X, dO, buf, token_offset=j * wl.tokens, slice_mode=slice_mode, stream=stream,
                       accumulate=accumulate)
    return run
