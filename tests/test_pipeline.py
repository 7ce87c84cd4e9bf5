"""GPipe micro-batch pipeline (pipeline.py) over a stack of MLP blocks.

The schedule is checked by itself (every stage's operations, the tick timeline
and its bubble), then run with the float64 oracle as each stage's block: in one
process, and as three gloo ranks on the CPU exchanging activations and gradients
point to point.  Either way each stage's accumulated gradients and the last
stage's outputs must equal the plain sequential run of the blocks, micro-batch by
micro-batch (GPipe is synchronous, so pipelining changes when the work runs, not
what it computes: MindSpore podcast page, GPipe segment).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import mlp_oracle as orc
from transformer_lm_megatron_gb300 import inputs as gin
from transformer_lm_megatron_gb300 import pipeline as pp

T, H, FFN, TS, P = 16, 16, 64, 2, 0.2
NAMES = ("dA", "da", "dB", "db")


def test_schedule_runs_every_forward_before_the_backwards():
    s = pp.gpipe_schedule(3, 4)
    assert len(s) == 3
    for ops in s:
        assert ops == [("F", 0), ("F", 1), ("F", 2), ("F", 3), ("B", 3), ("B", 2), ("B", 1), ("B", 0)]
    with pytest.raises(ValueError):
        pp.gpipe_schedule(0, 4)


@pytest.mark.parametrize("S,m", [(1, 1), (1, 5), (3, 4), (4, 8), (5, 2)])
def test_timeline_length_and_bubble(S, m):
    tl = pp.timeline(S, m)
    assert len(tl) == 2 * (m + S - 1)
    for s in range(S):
        busy = [row[s] for row in tl if row[s] is not None]
        assert busy == pp.gpipe_schedule(S, m)[s]           # each stage keeps its order
    idle = sum(row[s] is None for row in tl for s in range(S))
    assert idle == S * 2 * (S - 1)                            # the bubble: (S-1)/(m+S-1) of the time
    # dependencies: F(j) on stage s after F(j) on s-1; B(j) on s after B(j) on s+1
    when = {(op, s): t for t, row in enumerate(tl) for s, op in enumerate(row) if op is not None}
    for (op, s), t in when.items():
        kind, j = op
        if kind == "F" and s > 0:
            assert when[(("F", j), s - 1)] < t
        if kind == "B" and s < S - 1:
            assert when[(("B", j), s + 1)] < t
        if kind == "B" and s == S - 1:
            assert when[(("F", j), s)] < t


def _stage_weights(s):
    return tuple(orc.bf16_to_f64(gin.bf16_bits(x)) for x in gin.make_weights(H, FFN, seed=100 + s))


def _microbatch(j):
    X, dO = gin.make_microbatch(T, H, j)
    return orc.bf16_to_f64(gin.bf16_bits(X)), orc.bf16_to_f64(gin.bf16_bits(dO))


class OracleStage:
    """One stage with the oracle's block (float64 numpy): the reference for what a
    stage computes, with the activations of each micro-batch kept for its backward."""

    def __init__(self, s, mirror):
        self.w = _stage_weights(s)
        self.seed = 1234 + s
        self.mirror = mirror
        self.saved = {}
        self.grads = None

    def fwd(self, j, x):
        x = np.asarray(x)
        A, a, B, b = self.w
        fw = orc.mlp_fwd(x, A, a, B, b, TS, P, self.seed, token_offset=j * T, mirror=self.mirror)
        self.saved[j] = (x, fw)
        return fw["O"]

    def bwd(self, j, dy, accumulate):
        x, fw = self.saved.pop(j)
        A, a, B, b = self.w
        bw = orc.mlp_bwd(np.asarray(dy), x, A, B, fw["U"], fw["Y"], fw["keep"], TS, P, mirror=self.mirror)
        if accumulate:
            for n in NAMES:
                self.grads[n] = self.grads[n] + bw[n]
        else:
            self.grads = {n: bw[n].copy() for n in NAMES}
        return bw["dX"]


def _sequential(S, m, mirror):
    """The blocks one after another: each micro-batch through every stage forward,
    then back, accumulating every stage's gradients in micro-batch order."""
    stages = [OracleStage(s, mirror) for s in range(S)]
    outs = {}
    for j in range(m):
        x, dO = _microbatch(j)
        for st in stages:
            x = st.fwd(j, x)
        outs[j] = x
        g = dO
        for st in reversed(stages):
            g = st.bwd(j, g, j > 0)
    return outs, [st.grads for st in stages]


@pytest.mark.parametrize("mirror", [False, True])
def test_local_pipeline_equals_sequential_blocks(mirror):
    S, m = 3, 4
    stages = [OracleStage(s, mirror) for s in range(S)]
    outs = pp.run_local(S, m, [st.fwd for st in stages], [st.bwd for st in stages],
                        lambda j: _microbatch(j)[0], lambda j: _microbatch(j)[1])
    ref_outs, ref_grads = _sequential(S, m, mirror)
    for j in range(m):
        np.testing.assert_array_equal(outs[j], ref_outs[j])
    for s in range(S):
        for n in NAMES:
            # the same sums in another order (micro-batches m-1 .. 0)
            np.testing.assert_allclose(stages[s].grads[n], ref_grads[s][n], rtol=1e-12, atol=1e-13)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, m, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        st = OracleStage(rank, mirror=True)
        send_t, recv_t = pp.dist_transport(lambda j, kind: torch.empty(T, H, dtype=torch.float64))
        outs = {}

        def fwd(j, x):
            y = st.fwd(j, x.numpy() if torch.is_tensor(x) else x)
            if rank == world - 1:
                outs[j] = y
            return torch.from_numpy(np.ascontiguousarray(y))

        def bwd(j, dy, accumulate):
            return torch.from_numpy(np.ascontiguousarray(st.bwd(j, dy.numpy() if torch.is_tensor(dy) else dy,
                                                                accumulate)))

        pp.run_stage(rank, world, m, fwd, bwd, send_t, recv_t, lambda j: _microbatch(j)[0],
                     lambda j: _microbatch(j)[1])
        out[rank] = ({n: st.grads[n] for n in NAMES}, outs)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_three_gloo_ranks_pipeline_equals_sequential_blocks():
    S, m = 3, 4
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, S, port, m, out)) for r in range(S)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    ref_outs, ref_grads = _sequential(S, m, mirror=True)
    for s in range(S):
        for n in NAMES:
            np.testing.assert_allclose(out[s][0][n], ref_grads[s][n], rtol=1e-12, atol=1e-13)
    last = out[S - 1][1]
    for j in range(m):
        np.testing.assert_array_equal(last[j], ref_outs[j])
