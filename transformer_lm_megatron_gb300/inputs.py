"""Seeded synthetic inputs for the tensor-sliced MLP block.

This module only draws random numbers and names the workloads; it holds none of
the block's arithmetic, so both the CUDA path and the CPU oracle can use it.

Recipe (every workload):
  * weights A [h, F], B [F, h] ~ N(0, 0.02); biases a [F], b [h] ~ N(0, 0.02);
    drawn from one torch.Generator seeded ``WEIGHT_SEED`` in the order A, a, B, b;
  * micro-batch j: X_j [T, h] ~ N(0, 1) then dO_j [T, h] ~ N(0, 1), from a
    generator seeded ``1000 + j``;
  * every value is drawn in fp32 and rounded to bf16 (round-to-nearest-even);
  * dropout seed 1234 for every workload, token offset j * T for micro-batch j,
    so the dropout mask of micro-batch j continues the element numbering of the
    micro-batches before it.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

WEIGHT_SEED = 0
DROPOUT_SEED = 1234
WEIGHT_STD = 0.02


@dataclass(frozen=True)
class Workload:
    """One MLP-block workload: T tokens per micro-batch, hidden h, ffn F, t slices, k micro-batches."""
    name: str
    tokens: int
    h: int
    ffn: int
    t: int
    k: int
    p: float = 0.1
    seed: int = DROPOUT_SEED

    @property
    def f(self) -> int:
        return self.ffn // self.t

    def flops_per_microbatch(self) -> int:
        """Algorithmic FLOPs of one forward+backward: six GEMMs of 2*T*h*F each."""
        return 12 * self.tokens * self.h * self.ffn

    def flops_total(self) -> int:
        return self.flops_per_microbatch() * self.k


# The five workloads of the block (tokens = micro-batch x sequence).
WORKLOADS = {
    "tiny": Workload("tiny", tokens=256, h=256, ffn=1024, t=2, k=2),
    "small": Workload("small", tokens=4096, h=768, ffn=3072, t=1, k=8),
    "mid": Workload("mid", tokens=2048, h=4096, ffn=16384, t=1, k=4),
    "mtnlg": Workload("mtnlg", tokens=2048, h=20480, ffn=81920, t=8, k=1),
    "sweep1": Workload("sweep1", tokens=2048, h=8192, ffn=32768, t=4, k=1),
    "sweep4": Workload("sweep4", tokens=2048, h=8192, ffn=32768, t=4, k=4),
    "sweep16": Workload("sweep16", tokens=2048, h=8192, ffn=32768, t=4, k=16),
    "sweep32": Workload("sweep32", tokens=2048, h=8192, ffn=32768, t=4, k=32),
    # one of the MT-NLG layer's eight slices as a block of its own (A_i 20480 x 10240,
    # B_i 10240 x 20480): 2.8 GB on the device, the size used for counter captures
    "mtnlg_slice": Workload("mtnlg_slice", tokens=2048, h=20480, ffn=10240, t=1, k=1),
}


def _normal_bf16(shape, std, gen, device):
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def make_weights(h: int, ffn: int, device="cpu", seed: int = WEIGHT_SEED):
    """A [h, ffn], a [ffn], B [ffn, h], b [h] as bf16 tensors on ``device``."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    A = _normal_bf16((h, ffn), WEIGHT_STD, g, device)
    a = _normal_bf16((ffn,), WEIGHT_STD, g, device)
    B = _normal_bf16((ffn, h), WEIGHT_STD, g, device)
    b = _normal_bf16((h,), WEIGHT_STD, g, device)
    return A, a, B, b


def make_microbatch(tokens: int, h: int, j: int, device="cpu"):
    """X_j [tokens, h] and dO_j [tokens, h] as bf16 tensors on ``device``."""
    g = torch.Generator(device=device)
    g.manual_seed(1000 + j)
    X = _normal_bf16((tokens, h), 1.0, g, device)
    dO = _normal_bf16((tokens, h), 1.0, g, device)
    return X, dO


def bf16_bits(x: torch.Tensor):
    """The raw bf16 bit patterns of a CPU bf16 tensor as a numpy uint16 array."""
    return x.contiguous().cpu().view(torch.int16).numpy().view("uint16")


# The self-attention block at the MT-NLG layer shape: hidden 20480, 128 heads
# (head size 160), 8 slices, one sequence of 2048 tokens.
ATTN_MTNLG = dict(h=20480, nh=128, t=8, seq_len=2048, tokens=2048)
ATTN_SEED = 7


def make_attn_inputs(h: int, tokens: int, device="cpu", seed: int = ATTN_SEED, std: float = WEIGHT_STD):
    """Wqkv [h, 3h], bqkv [3h], Wo [h, h], bo [h] ~ N(0, std), then X [tokens, h]
    and dOut [tokens, h] ~ N(0, 1), all from one generator seeded ``seed`` in that
    order, drawn in fp32 and rounded to bf16."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    Wqkv = _normal_bf16((h, 3 * h), std, g, device)
    bqkv = _normal_bf16((3 * h,), std, g, device)
    Wo = _normal_bf16((h, h), std, g, device)
    bo = _normal_bf16((h,), std, g, device)
    X = _normal_bf16((tokens, h), 1.0, g, device)
    dOut = _normal_bf16((tokens, h), 1.0, g, device)
    return (Wqkv, bqkv, Wo, bo), X, dOut
