"""Data-parallel replicas (data_parallel.py): micro-batches shared out over gloo
ranks on the CPU, gradients summed with the all-reduce.

Each rank computes its micro-batches' gradients with the float64 oracle (the CUDA
block needs a GPU) through the same orchestration the GPU ranks use; after the
all-reduce every rank must hold the gradients of all k micro-batches accumulated
in one process, and, by accumulation invariance, those of one batch of k * T
tokens (gradient accumulation: "Using DeepSpeed and Megatron to Train
Megatron-Turing NLG 530B", Key points; data parallelism sums gradients with an
all-reduce: "STRONGHOLD" slides, items 4-5).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import mlp_oracle as orc
from transformer_lm_megatron_gb300 import data_parallel as dp
from transformer_lm_megatron_gb300 import inputs as gin

T, H, FFN, TS, P, SEED = 24, 16, 64, 2, 0.25, 99
NAMES = ("dA", "da", "dB", "db")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _weights64():
    return tuple(orc.bf16_to_f64(gin.bf16_bits(x)) for x in gin.make_weights(H, FFN))


def _microbatch64(j):
    X, dO = gin.make_microbatch(T, H, j)
    return orc.bf16_to_f64(gin.bf16_bits(X)), orc.bf16_to_f64(gin.bf16_bits(dO))


def _oracle_grads(X64, dO64, w64, token_offset):
    A, a, B, b = w64
    fw = orc.mlp_fwd(X64, A, a, B, b, TS, P, SEED, token_offset=token_offset)
    return orc.mlp_bwd(dO64, X64, A, B, fw["U"], fw["Y"], fw["keep"], TS, P)


def _rank_main(rank, world, port, k_total, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w64 = _weights64()
        flat, views = dp.flat_gradients(H, FFN, device="cpu", dtype=torch.float64)
        flat.fill_(float("nan"))        # the first micro-batch must overwrite, not add

        def run(j, accumulate):
            X64, dO64 = _microbatch64(j)
            g = _oracle_grads(X64, dO64, w64, j * T)
            for v, name in zip(views, NAMES):
                if accumulate:
                    v.add_(torch.from_numpy(g[name]))
                else:
                    v.copy_(torch.from_numpy(g[name]))

        mine = dp.data_parallel_step(k_total, rank, world, run, flat.zero_, flat)
        out[rank] = (list(mine), flat.numpy().copy())
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run_ranks(world, k_total):
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, k_total, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    return dict(out)


def test_shard_covers_every_microbatch_once():
    for k in range(0, 12):
        for world in range(1, 6):
            got = [j for r in range(world) for j in dp.shard(k, world, r)]
            assert got == list(range(k))
            sizes = [len(dp.shard(k, world, r)) for r in range(world)]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        dp.shard(4, 2, 2)


def test_flat_gradient_views_are_aligned_and_disjoint():
    flat, (dA, da, dB, db) = dp.flat_gradients(24, 40, device="cpu")
    assert dA.shape == (24, 40) and da.shape == (40,) and dB.shape == (40, 24) and db.shape == (24,)
    base = flat.data_ptr()
    for v in (dA, da, dB, db):
        assert (v.data_ptr() - base) % 16 == 0 and v.is_contiguous()
    for i, v in enumerate((dA, da, dB, db)):
        v.fill_(i + 1)
    assert flat.sum().item() == 1 * 24 * 40 + 2 * 40 + 3 * 40 * 24 + 4 * 24


@pytest.mark.parametrize("world,k_total", [(2, 5), (3, 2), (2, 4)])
def test_allreduced_gradients_equal_one_process_accumulation(world, k_total):
    """(2, 5): uneven shares; (3, 2): a rank without a micro-batch (it zeroes its
    accumulators and still joins the all-reduce)."""
    out = _run_ranks(world, k_total)
    w64 = _weights64()
    # one process, all k micro-batches accumulated
    seq = {n: 0.0 for n in NAMES}
    mbs = [_microbatch64(j) for j in range(k_total)]
    for j, (X64, dO64) in enumerate(mbs):
        g = _oracle_grads(X64, dO64, w64, j * T)
        for n in NAMES:
            seq[n] = seq[n] + g[n]
    ref = np.concatenate([seq["dA"].ravel(), seq["da"], seq["dB"].ravel(), seq["db"]])
    # one batch of k * T tokens at offset 0 (accumulation invariance)
    Xc = np.concatenate([m[0] for m in mbs])
    dOc = np.concatenate([m[1] for m in mbs])
    gc = _oracle_grads(Xc, dOc, w64, 0)
    ref_cat = np.concatenate([gc["dA"].ravel(), gc["da"], gc["dB"].ravel(), gc["db"]])
    np.testing.assert_allclose(ref_cat, ref, rtol=1e-12, atol=1e-12)
    ran = sorted(j for r in range(world) for j in out[r][0])
    assert ran == list(range(k_total))
    for r in range(world):
        np.testing.assert_allclose(out[r][1], ref, rtol=1e-12, atol=1e-13)
