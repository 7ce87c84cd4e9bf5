"""Shared helpers of the GPU parity tests: run the block through the C-ABI on the
GPU and the oracle on the CPU on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

from oracle import mlp_oracle as orc
from transformer_lm_megatron_gb300 import inputs as gin
from transformer_lm_megatron_gb300 import mlp

BF16_TOL = 1e-2   # max|gpu - oracle| / max|oracle| for bf16 activations and gradients
F32_TOL = 1e-3    # the same for fp32 accumulated weight and bias gradients


def rel_err(gpu, ref) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    if den == 0:
        return float(np.max(np.abs(gpu)))
    return float(np.max(np.abs(gpu - ref)) / den)


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a bf16 or fp32 tensor."""
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def bits_f64(t: torch.Tensor) -> np.ndarray:
    """Decode a bf16 tensor through its raw bits with the oracle's decoder."""
    return orc.bf16_to_f64(gin.bf16_bits(t.detach().cpu()))


class Shape:
    def __init__(self, tokens, h, ffn, t, k=1, p=0.1, seed=gin.DROPOUT_SEED):
        self.tokens, self.h, self.ffn, self.t, self.k, self.p, self.seed = tokens, h, ffn, t, k, p, seed

    @property
    def f(self):
        return self.ffn // self.t


def run_gpu(shape, weights_dev, microbatches_dev, slice_mode="all", keep_all=False, buf=None, reset=True,
            first_overwrites=False, token_offset0=0):
    """Forward+backward of every micro-batch on the GPU; gradients accumulate.

    reset: zero the accumulators first (grad_accum_reset); first_overwrites: the
    first micro-batch overwrites them instead (accumulate = 0), later ones add.
    Micro-batch j runs at token offset token_offset0 + j * tokens.
    Returns (per-micro-batch outputs, gradients) as CPU tensors."""
    T = microbatches_dev[0][0].shape[0]
    if buf is None:
        buf = mlp.BlockBuffers(T, shape.h, shape.ffn, shape.t)
    if reset:
        mlp.grad_accum_reset(shape.h, shape.ffn, buf.dA, buf.da, buf.dB, buf.db)
    outs = []
    for j, (X, dO) in enumerate(microbatches_dev):
        mlp.block_step(shape, weights_dev, X, dO, buf, token_offset=token_offset0 + j * T, slice_mode=slice_mode,
                       accumulate=not (first_overwrites and j == 0))
        if keep_all or j == len(microbatches_dev) - 1:
            outs.append({k: getattr(buf, k).cpu() for k in ("U", "Y", "O", "dZ", "dU", "dX")})
        else:
            outs.append(None)
    torch.cuda.synchronize()
    rc = mlp.mlp_sync_status()
    assert rc == mlp.MLP_OK, mlp.last_error()
    grads = {k: getattr(buf, k).cpu() for k in ("dA", "da", "dB", "db")}
    return outs, grads


def run_oracle(shape, weights_f64, microbatches_f64, mirror, keep_all=False):
    A, a, B, b = weights_f64
    T = microbatches_f64[0][0].shape[0]
    acc = {k: 0.0 for k in ("dA", "da", "dB", "db")}
    outs = []
    for j, (X, dO) in enumerate(microbatches_f64):
        fw = orc.mlp_fwd(X, A, a, B, b, shape.t, shape.p, shape.seed, token_offset=j * T, mirror=mirror)
        bw = orc.mlp_bwd(dO, X, A, B, fw["U"], fw["Y"], fw["keep"], shape.t, shape.p, mirror=mirror)
        for k in acc:
            acc[k] = acc[k] + bw[k]
        if keep_all or j == len(microbatches_f64) - 1:
            outs.append({**fw, **bw})
        else:
            outs.append(None)
    return outs, acc


def make_case(shape, device_gen="cpu"):
    """Seeded inputs: (weights on GPU, micro-batches on GPU, weights f64, micro-batches f64)."""
    w = gin.make_weights(shape.h, shape.ffn, device=device_gen)
    mbs = [gin.make_microbatch(shape.tokens, shape.h, j, device=device_gen) for j in range(shape.k)]
    w_dev = tuple(x.cuda() for x in w)
    mbs_dev = [(X.cuda(), dO.cuda()) for X, dO in mbs]
    w64 = tuple(bits_f64(x) for x in w)
    mbs64 = [(bits_f64(X), bits_f64(dO)) for X, dO in mbs]
    return w_dev, mbs_dev, w64, mbs64


def compare_full(shape, gpu_outs, gpu_grads, ref_outs, ref_grads, check_grads=True, label=""):
    """Element-by-element comparison; returns {name: rel_err}. Asserts the bars."""
    errs = {}
    for j, (g, r) in enumerate(zip(gpu_outs, ref_outs)):
        if g is None or r is None:
            continue
        for k in ("U", "Y", "O", "dZ", "dU", "dX"):
            e = rel_err(to_f64(g[k]), r[k])
            errs[f"{k}[{j}]"] = e
            assert e <= BF16_TOL, (label, k, j, e)
    if check_grads:
        for k in ("dA", "da", "dB", "db"):
            e = rel_err(to_f64(gpu_grads[k]), ref_grads[k])
            errs[k] = e
            assert e <= F32_TOL, (label, k, e)
    return errs
