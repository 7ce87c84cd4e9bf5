"""Micro-batch pipeline (GPipe) over a stack of MLP blocks, one stage per rank.

Pipeline (inter-layer) model parallelism puts consecutive sets of layers on
different devices; it needs large batches to keep the devices busy ("STRONGHOLD"
slides, items 5-7).  GPipe splits the batch into micro-batches and streams them
through the stages so that the stages work at the same time; it is fully
synchronous: every micro-batch's forward runs before the backward, the weight
gradients are accumulated over the micro-batches, and the idle time at the start
and end of the schedule is the pipeline "bubble" (MindSpore podcast page, the
GPipe segment; MT-NLG ran 35-way pipelines: jiqizhixin article on MT-NLG).

Reading for this library: stage s holds one MLP block (its own weights A_s, a_s,
B_s, b_s and fp32 gradient accumulators); block s's output O is block s+1's input
X.  For m micro-batches every stage runs F_0 .. F_{m-1}, then B_{m-1} .. B_0 (the
last stage can start the backward of the last micro-batch as soon as its forward
is done).  The first backward a stage runs writes its gradient accumulators, the
later ones add (mlp_bwd accumulate = 0, then 1).  Activations travel forward and
input gradients backward between neighbouring stages; nothing else is exchanged.

The schedule is independent of how a stage computes: ``run_stage`` drives one
stage on its own rank with send/recv callables (torch.distributed point-to-point:
NCCL between GPU ranks, gloo between CPU ranks); ``run_local`` runs every stage in
one process in an order the schedule allows, passing tensors in memory.
``BlockStage`` gives the forward and backward of a stage through the library's
C ABI on this GPU.
"""
from __future__ import annotations

from typing import Callable, Dict, List, Tuple

import torch

Op = Tuple[str, int]   # ("F", j) or ("B", j)


def gpipe_schedule(n_stages: int, n_micro: int) -> List[List[Op]]:
    """Per stage, the ordered list of operations: forwards of micro-batches
    0 .. m-1, then backwards of m-1 .. 0."""
    if n_stages <= 0 or n_micro <= 0:
        raise ValueError(f"need at least one stage and one micro-batch ({n_stages}, {n_micro})")
    ops = [("F", j) for j in range(n_micro)] + [("B", j) for j in reversed(range(n_micro))]
    return [list(ops) for _ in range(n_stages)]


def timeline(n_stages: int, n_micro: int) -> List[List[Op]]:
    """The schedule as clock ticks when every operation takes one tick and a
    stage may run an operation once its input has arrived: entry [tick][stage] is
    the operation run then, or None.  Its length is 2 (m + S - 1) ticks, of which
    each stage is busy 2 m: the rest is the bubble."""
    sched = gpipe_schedule(n_stages, n_micro)
    pos = [0] * n_stages
    done = set()
    ticks = []
    while any(pos[s] < len(sched[s]) for s in range(n_stages)):
        row = [None] * n_stages
        for s in range(n_stages):
            if pos[s] == len(sched[s]):
                continue
            kind, j = sched[s][pos[s]]
            if _ready(kind, j, s, n_stages, done):
                row[s] = (kind, j)
        if not any(row):
            raise RuntimeError("schedule cannot make progress")
        for s, op in enumerate(row):
            if op is not None:
                done.add((op[0], op[1], s))
                pos[s] += 1
        ticks.append(row)
    return ticks


def _ready(kind: str, j: int, s: int, n_stages: int, done) -> bool:
    if kind == "F":
        return s == 0 or ("F", j, s - 1) in done
    return (s == n_stages - 1 and ("F", j, s) in done) or ("B", j, s + 1) in done


def run_stage(stage: int, n_stages: int, n_micro: int, fwd: Callable, bwd: Callable, send: Callable,
              recv: Callable, first_input: Callable, last_grad: Callable):
    """Run stage ``stage`` of the schedule on this rank.

    fwd(j, x) -> y             forward of micro-batch j on this stage's block
    bwd(j, dy, accumulate) -> dx   backward; accumulate False on the stage's first backward
    send(dst_stage, tensor) / recv(src_stage, j, kind) -> tensor   point-to-point transfers
    first_input(j) -> x        micro-batch j's input (stage 0 only)
    last_grad(j) -> dy         gradient of the last stage's output (last stage only)
    """
    first_bwd = True
    for kind, j in gpipe_schedule(n_stages, n_micro)[stage]:
        if kind == "F":
            x = first_input(j) if stage == 0 else recv(stage - 1, j, "F")
            y = fwd(j, x)
            if stage < n_stages - 1:
                send(stage + 1, y)
        else:
            dy = last_grad(j) if stage == n_stages - 1 else recv(stage + 1, j, "B")
            dx = bwd(j, dy, not first_bwd)
            first_bwd = False
            if stage > 0:
                send(stage - 1, dx)


def run_local(n_stages: int, n_micro: int, fwd: List[Callable], bwd: List[Callable], first_input: Callable,
              last_grad: Callable) -> Dict[int, object]:
    """Every stage in this process, operations taken tick by tick from
    ``timeline``; transfers are handed over in memory.  Returns the last stage's
    outputs {j: y}."""
    inbox: Dict[Tuple[str, int, int], object] = {}
    outputs = {}
    first_bwd = [True] * n_stages
    for row in timeline(n_stages, n_micro):
        for s, op in enumerate(row):
            if op is None:
                continue
            kind, j = op
            if kind == "F":
                x = first_input(j) if s == 0 else inbox.pop(("F", j, s))
                y = fwd[s](j, x)
                if s < n_stages - 1:
                    inbox[("F", j, s + 1)] = y
                else:
                    outputs[j] = y
            else:
                dy = last_grad(j) if s == n_stages - 1 else inbox.pop(("B", j, s))
                dx = bwd[s](j, dy, not first_bwd[s])
                first_bwd[s] = False
                if s > 0:
                    inbox[("B", j, s - 1)] = dx
    return outputs


def dist_transport(like: Callable[[int, str], torch.Tensor], group=None):
    """send/recv callables over torch.distributed, stage s being rank s of
    ``group``; ``like(j, kind)`` gives an empty tensor of the received shape."""
    import torch.distributed as dist

    def send(dst: int, t: torch.Tensor):
        dist.send(t.contiguous(), dst=dst, group=group)

    def recv(src: int, j: int, kind: str) -> torch.Tensor:
        t = like(j, kind)
        dist.recv(t, src=src, group=group)
        return t
    return send, recv


class BlockStage:
    """One stage: an MLP block through the library's C ABI on this GPU, with the
    activations of every micro-batch kept for its backward (GPipe stores them
    until the backward of the micro-batch)."""

    def __init__(self, wl, weights, n_micro: int, seed: int, device="cuda", slice_mode="all", stream=None, grads=None):
        from . import mlp
        self.mlp = mlp
        self.wl, self.weights, self.seed = wl, weights, seed
        self.slice_mode, self.stream = slice_mode, stream
        T, h, F, t = wl.tokens, wl.h, wl.ffn, wl.t
        if grads is None:
            f32 = dict(dtype=torch.float32, device=device)
            grads = (torch.zeros(h, F, **f32), torch.zeros(F, **f32), torch.zeros(F, h, **f32), torch.zeros(h, **f32))
        self.dA, self.da, self.dB, self.db = grads
        # per micro-batch: U, Y, O (forward), dZ, dU, dX (backward); one set of gradient accumulators
        self.acts = [mlp.BlockBuffers(T, h, F, t, device=device, grads=grads) for _ in range(n_micro)]
        self.inputs: Dict[int, torch.Tensor] = {}  # the stage input X of each micro-batch until its backward

    def fwd(self, j: int, x: torch.Tensor) -> torch.Tensor:
        wl, (A, a, B, b), buf = self.wl, self.weights, self.acts[j]
        self.inputs[j] = x
        slices = [-1] if self.slice_mode == "all" else list(range(wl.t))
        for i in slices:
            self.mlp.mlp_fwd(wl.h, wl.ffn, wl.t, i, wl.tokens, wl.p, self.seed, j * wl.tokens, x, A, a, B, b, None,
                             buf.U, buf.Y, buf.Zacc, buf.O, self.stream)
        return buf.O

    def bwd(self, j: int, dy: torch.Tensor, accumulate: bool) -> torch.Tensor:
        wl, (A, a, B, b), buf = self.wl, self.weights, self.acts[j]
        x = self.inputs.pop(j)
        slices = [-1] if self.slice_mode == "all" else list(range(wl.t))
        for i in slices:
            self.mlp.mlp_bwd(wl.h, wl.ffn, wl.t, i, wl.tokens, wl.p, self.seed, j * wl.tokens, 1, accumulate, dy, x,
                             A, B, buf.U, buf.Y, buf.dZ, buf.dU, buf.dXacc, buf.dX, self.dA, self.da, self.dB, self.db,
                             self.stream)
        return buf.dX
