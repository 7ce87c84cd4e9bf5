"""GPU parity of the tensor-sliced self-attention block (attn_fwd / attn_bwd)
against the float64 oracle, through the C ABI.

Bars: bf16 tensors (QKV, P, O, out, dQKV, dX) within max|gpu - oracle| /
max|oracle| <= 1e-2 of both oracle modes, as for the MLP block.  fp32 accumulated
gradients (dWqkv, dbqkv, dWo, dbo) within ATTN_F32_TOL = 5e-3 of the
bf16-mirroring mode and 1e-2 of the pure mode: unlike the MLP's weight gradients
(one bf16 storage point, dZ or dU, between the fp32 GEMMs), dWqkv is reached
through four (dZ, dO, dS, dQKV), and the GPU's fp32 sums round to the other side
of a bf16 step than the float64 mirror for a growing fraction of elements at each;
those one-ulp (2^-8 relative) differences, summed over the tokens, measured up to
2.0e-3 of the largest gradient.  Probabilities are exactly zero above the causal
diagonal, and dropped outputs equal the residual exactly.
"""
import numpy as np
import pytest
import torch

from oracle import attn_oracle as ato
from oracle import mlp_oracle as orc
from transformer_lm_megatron_gb300 import build as gb_build
from transformer_lm_megatron_gb300 import mlp

from gpu_harness import BF16_TOL, bits_f64, rel_err, to_f64

pytestmark = pytest.mark.gpu

ATTN_F32_TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gb_build.build()
    mlp.load()


def _weights(h, gen, std=0.02):
    def rnd(*shape, s=std):
        return (torch.randn(*shape, generator=gen) * s).to(torch.bfloat16)
    return rnd(h, 3 * h), rnd(3 * h), rnd(h, h), rnd(h)


@pytest.fixture
def cta_pair_mode(request):
    mlp.mlp_set_cta_pair(request.param)
    yield request.param
    mlp.mlp_set_cta_pair(-1)


@pytest.mark.parametrize("cta_pair_mode", [0, 1], indirect=True, ids=["single", "pair"])
@pytest.mark.parametrize("T,h,nh,t,L,k", [
    (256, 256, 4, 2, 128, 2),     # two sequences, d = 64, two accumulated micro-batches
    (272, 320, 4, 4, 136, 1),     # ragged: d = 80, seq_len 136 (tails in every GEMM)
    (2048, 2048, 16, 8, 1024, 1),  # two sequences of 1024, d = 128, eight slices
    (2048, 256, 2, 2, 2048, 1),    # one sequence of 2048: the longest rows the warp-per-row softmax holds
    (2304, 128, 2, 1, 2304, 1),    # rows past 2048 columns: the CTA-per-row softmax
])
def test_attention_block_full_parity(T, h, nh, t, L, k, cta_pair_mode):
    p, seed = 0.1, 1234
    gen = torch.Generator().manual_seed(21)
    w = _weights(h, gen, std=0.5 / np.sqrt(h))
    mbs = [((torch.randn(T, h, generator=gen)).to(torch.bfloat16), torch.randn(T, h, generator=gen).to(torch.bfloat16))
           for _ in range(k)]
    dev = torch.device("cuda")
    wd = tuple(x.to(dev) for x in w)
    buf = mlp.AttnBuffers(T, h, nh, L, device=dev)
    outs = []
    for j, (X, dOut) in enumerate(mbs):
        mlp.attn_step(h, nh, t, L, p, seed, wd, X.to(dev), dOut.to(dev), buf, token_offset=j * T, accumulate=j > 0)
        outs.append({n: getattr(buf, n).cpu() for n in ("QKV", "P", "O", "out", "dQKV", "dX")})
    torch.cuda.synchronize()
    assert mlp.mlp_sync_status() == mlp.MLP_OK, mlp.last_error()
    grads = {n: to_f64(getattr(buf, n)) for n in ("dWqkv", "dbqkv", "dWo", "dbo")}

    W64 = [bits_f64(x) for x in w]
    for mirror in (True, False):
        acc = {n: 0.0 for n in grads}
        for j, (X, dOut) in enumerate(mbs):
            X64, d64 = bits_f64(X), bits_f64(dOut)
            fw = ato.attn_fwd(X64, W64[0], W64[1], W64[2], W64[3], nh, t, L, p, seed, token_offset=j * T,
                              mirror=mirror)
            bw = ato.attn_bwd(d64, X64, W64[0], W64[2], fw["QKV"], fw["P"], fw["O"], fw["keep"], nh, t, L, p,
                              mirror=mirror)
            g = outs[j]
            ref = {"QKV": fw["QKV"], "P": fw["P"], "O": fw["O"], "out": fw["out"], "dQKV": bw["dQKV"], "dX": bw["dX"]}
            for name, r in ref.items():
                e = rel_err(to_f64(g[name]), r)
                assert e <= BF16_TOL, (mirror, j, name, e)
            if mirror:
                P = to_f64(g["P"])
                assert np.all(np.triu(P, k=1) == 0)
                keep = fw["keep"]
                np.testing.assert_array_equal(to_f64(g["out"])[~keep], X64[~keep])
            for n in acc:
                acc[n] = acc[n] + bw[n]
        for n in grads:
            e = rel_err(grads[n], acc[n])
            assert e <= (ATTN_F32_TOL if mirror else BF16_TOL), (mirror, n, e)


def test_attention_rejects_bad_shapes():
    dev = torch.device("cuda")
    x = torch.empty(64, dtype=torch.bfloat16, device=dev)
    lib = mlp.load()
    ptrs = [x.data_ptr()] * 5
    # head size not a multiple of 8, and tokens not a multiple of seq_len
    assert lib.attn_fwd(96, 16, 1, 64, 32, 0.1, 1, 0, *ptrs, None, *([x.data_ptr()] * 5), None) == mlp.MLP_EINVAL
    assert lib.attn_fwd(128, 4, 1, 60, 32, 0.1, 1, 0, *ptrs, None, *([x.data_ptr()] * 5), None) == mlp.MLP_EINVAL
