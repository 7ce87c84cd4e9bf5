"""The data-parallel and pipeline orchestration on the GPU, through the C ABI.

Runs on one GPU: the data-parallel step in a one-rank NCCL group (the collective
on real device buffers, the gradient views of one contiguous buffer passed to
mlp_bwd), and the GPipe schedule with every stage in this process on one stream
(stages run one operation at a time, so no kernel waits on another).  Both must
equal the plain runs bit for bit, and the oracle within the usual bars.
"""
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

from oracle import mlp_oracle as orc
from transformer_lm_megatron_gb300 import build as gb_build
from transformer_lm_megatron_gb300 import data_parallel as dp
from transformer_lm_megatron_gb300 import inputs as gin
from transformer_lm_megatron_gb300 import mlp
from transformer_lm_megatron_gb300 import pipeline as pp

from gpu_harness import BF16_TOL, F32_TOL, Shape, bits_f64, make_case, rel_err, run_gpu, run_oracle, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gb_build.build()
    mlp.load()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_data_parallel_step_one_rank_nccl():
    s = Shape(tokens=200, h=256, ffn=1024, t=4, k=3)
    w_dev, mbs_dev, w64, mbs64 = make_case(s)
    _, ref = run_gpu(s, w_dev, mbs_dev)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1)
    try:
        flat, grads = dp.flat_gradients(s.h, s.ffn, device="cuda")
        flat.fill_(float("nan"))
        buf = mlp.BlockBuffers(s.tokens, s.h, s.ffn, s.t, grads=grads)
        run = dp.block_runner(s, w_dev, lambda j: mbs_dev[j], buf)
        mine = dp.data_parallel_step(s.k, 0, 1, run, lambda: mlp.grad_accum_reset(s.h, s.ffn, *grads), flat)
        torch.cuda.synchronize()
        assert list(mine) == [0, 1, 2]
        assert mlp.mlp_sync_status() == mlp.MLP_OK, mlp.last_error()
    finally:
        dist.destroy_process_group()
    for name, g in zip(("dA", "da", "dB", "db"), grads):
        assert torch.equal(g.cpu(), ref[name]), name
    _, r_grads = run_oracle(s, w64, mbs64, mirror=True)
    for name, g in zip(("dA", "da", "dB", "db"), grads):
        assert rel_err(to_f64(g), r_grads[name]) <= F32_TOL, name


def test_gpipe_schedule_on_one_gpu():
    """Three stages (three MLP blocks with their own weights and dropout seeds),
    four micro-batches: the pipelined run equals the same blocks run one after
    another with the backwards in the same order, bit for bit, and the oracle's
    chain of blocks within the bars."""
    S, m = 3, 4
    wl = gin.Workload("pipe", tokens=192, h=256, ffn=1024, t=2, k=m)
    weights = [tuple(x.cuda() for x in gin.make_weights(wl.h, wl.ffn, seed=100 + s)) for s in range(S)]
    mbs = [tuple(x.cuda() for x in gin.make_microbatch(wl.tokens, wl.h, j)) for j in range(m)]

    def stages():
        return [pp.BlockStage(wl, weights[s], m, seed=1234 + s) for s in range(S)]

    piped = stages()
    outs = pp.run_local(S, m, [st.fwd for st in piped], [st.bwd for st in piped], lambda j: mbs[j][0],
                        lambda j: mbs[j][1])
    # the same operations, one stage at a time: every forward, then the backwards m-1 .. 0
    seq = stages()
    seq_outs = {}
    for j in range(m):
        x = mbs[j][0]
        for st in seq:
            x = st.fwd(j, x)
        seq_outs[j] = x
    for n, j in enumerate(reversed(range(m))):
        g = mbs[j][1]
        for st in reversed(seq):
            g = st.bwd(j, g, n > 0)
    torch.cuda.synchronize()
    assert mlp.mlp_sync_status() == mlp.MLP_OK, mlp.last_error()
    for j in range(m):
        assert torch.equal(outs[j], seq_outs[j]), j
    for a, b in zip(piped, seq):
        for x, y in zip((a.dA, a.da, a.dB, a.db), (b.dA, b.da, b.dB, b.db)):
            assert torch.equal(x, y)
    # the oracle's chain of blocks (each block's input is the previous block's
    # output, each block's dO the next block's dX), in both modes.  A stage's
    # gradients pass through the bf16 storage points of every later block (their
    # dX), so the fp32-gradient bar against the mirroring mode is the oracle's own
    # pure-to-mirror distance for that gradient, never below 1e-3 (the bar of one
    # block), as for the attention block.
    W = [tuple(bits_f64(x.cpu()) for x in w) for w in weights]
    acc = {mirror: [{k: 0.0 for k in ("dA", "da", "dB", "db")} for _ in range(S)] for mirror in (True, False)}
    for mirror in (True, False):
        for j in range(m):
            x = bits_f64(mbs[j][0].cpu())
            saved = []
            for s in range(S):
                A, a, B, b = W[s]
                fw = orc.mlp_fwd(x, A, a, B, b, wl.t, wl.p, 1234 + s, token_offset=j * wl.tokens, mirror=mirror)
                saved.append((x, fw))
                x = fw["O"]
            assert rel_err(to_f64(outs[j]), x) <= BF16_TOL, (mirror, j)
            g = bits_f64(mbs[j][1].cpu())
            for s in reversed(range(S)):
                A, a, B, b = W[s]
                xs, fw = saved[s]
                bw = orc.mlp_bwd(g, xs, A, B, fw["U"], fw["Y"], fw["keep"], wl.t, wl.p, mirror=mirror)
                for k in acc[mirror][s]:
                    acc[mirror][s][k] = acc[mirror][s][k] + bw[k]
                g = bw["dX"]
    for s in range(S):
        for k, got in zip(("dA", "da", "dB", "db"), (piped[s].dA, piped[s].da, piped[s].dB, piped[s].db)):
            bar = max(F32_TOL, rel_err(acc[True][s][k], acc[False][s][k]))
            e = rel_err(to_f64(got), acc[True][s][k])
            assert e <= bar, (s, k, e, bar)
            assert rel_err(to_f64(got), acc[False][s][k]) <= BF16_TOL, (s, k)
