"""GPU parity on the five named workloads at their full sizes.

The small workload is compared element by element with the full oracle.  The
mid, MT-NLG-layer and accumulation-sweep workloads are compared on outputs the
oracle computes one by one from their definitions: whole token rows of O, dX,
U, Y, dU (the row loops over the slices like the block does), the whole dZ, db
and selected entries of dA, dB and da (each a sum over all tokens of one column
of Y or dU).  The MT-NLG layer runs in the configuration the benchmark times
(all eight slices per call); the sweep runs one slice per call, in turn.
"""
import numpy as np
import pytest
import torch

from oracle import mlp_oracle as orc
from transformer_lm_megatron_gb300 import build as gb_build
from transformer_lm_megatron_gb300 import inputs as gin
from transformer_lm_megatron_gb300 import mlp

from gpu_harness import (BF16_TOL, F32_TOL, Shape, compare_full, make_case, rel_err, run_gpu, run_oracle, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gb_build.build()
    mlp.load()


def _bits(t):
    return gin.bf16_bits(t.detach().cpu())


def test_small_workload_full_parity():
    """4096 tokens, h 768, ffn 3072, t 1, eight accumulated micro-batches."""
    wl = gin.WORKLOADS["small"]
    s = Shape(wl.tokens, wl.h, wl.ffn, wl.t, wl.k, wl.p, wl.seed)
    w_dev, mbs_dev, w64, mbs64 = make_case(s)
    g_outs, g_grads = run_gpu(s, w_dev, mbs_dev)
    r_outs, r_grads = run_oracle(s, w64, mbs64, mirror=True)
    compare_full(s, g_outs, g_grads, r_outs, r_grads, label="small")


def test_mid_workload_full_parity():
    """2048 tokens, h 4096, ffn 16384, t 1, four accumulated micro-batches, against
    the whole oracle (6.6 TFLOP of float64 host work): every element of the last
    micro-batch's U, Y, O, dZ, dU, dX and of the accumulated dA, da, dB, db."""
    wl = gin.WORKLOADS["mid"]
    s = Shape(wl.tokens, wl.h, wl.ffn, wl.t, wl.k, wl.p, wl.seed)
    w_dev, mbs_dev, w64, mbs64 = make_case(s)
    g_outs, g_grads = run_gpu(s, w_dev, mbs_dev)
    r_outs, r_grads = run_oracle(s, w64, mbs64, mirror=True)
    compare_full(s, g_outs, g_grads, r_outs, r_grads, label="mid")


def _full_da(Xs, dZs, A, a, B, ffn, block=4096):
    """All of da from the oracle: the column sums of every micro-batch's dU, a
    block of columns at a time (so that only slice-sized blocks of A and B are
    decoded to float64)."""
    out = np.zeros(ffn)
    for c0 in range(0, ffn, block):
        cols = np.arange(c0, min(ffn, c0 + block))
        for X, dZ in zip(Xs, dZs):
            out[cols] += orc.columns_dU(cols, X, A, a, B, dZ, mirror=True).sum(axis=0)
    return out


def _sampled_check(wl, slice_mode, n_rows=64, n_entries=256, seed=0, first_overwrites=False, full_da=True):
    """Runs the workload on the GPU (inputs drawn on the GPU with the seeded
    generators) and checks against the oracle: n_rows token rows of U, Y, O, dU
    and dX, the whole of dZ and db, n_entries entries each of dA and dB, and all
    of da (full_da; else da at the sampled dA columns).  first_overwrites: no
    reset; the first micro-batch overwrites the accumulators (which start as
    NaN), as the benchmark runs it."""
    dev = torch.device("cuda")
    w = gin.make_weights(wl.h, wl.ffn, device=dev)
    mbs = [gin.make_microbatch(wl.tokens, wl.h, j, device=dev) for j in range(wl.k)]
    buf = mlp.BlockBuffers(wl.tokens, wl.h, wl.ffn, wl.t, device=dev)
    if first_overwrites:
        for k in ("dA", "da", "dB", "db"):
            getattr(buf, k).fill_(float("nan"))
    else:
        mlp.grad_accum_reset(wl.h, wl.ffn, buf.dA, buf.da, buf.dB, buf.db)
    for j, (X, dO) in enumerate(mbs):
        mlp.block_step(wl, w, X, dO, buf, token_offset=j * wl.tokens, slice_mode=slice_mode,
                       accumulate=not (first_overwrites and j == 0))
    torch.cuda.synchronize()
    assert mlp.mlp_sync_status() == mlp.MLP_OK, mlp.last_error()

    rng = np.random.default_rng(seed)
    T, h, F = wl.tokens, wl.h, wl.ffn
    last = wl.k - 1
    rows = np.unique(np.concatenate([[0, 127, 128, T - 1], rng.integers(0, T, n_rows - 4)]))
    A = orc.Bf16Matrix(_bits(w[0]))
    a = orc.bf16_to_f64(_bits(w[1]))
    B = orc.Bf16Matrix(_bits(w[2]))
    b = orc.bf16_to_f64(_bits(w[3]))
    Xs = [orc.bf16_to_f64(_bits(X)) for X, _ in mbs]
    dOs = [orc.bf16_to_f64(_bits(dO)) for _, dO in mbs]

    # rows of the last micro-batch: O, dX, U, Y, dU
    ref = orc.rows_fwd_bwd(rows, Xs[last], dOs[last], A, a, B, b, wl.t, wl.p, wl.seed,
                           token_offset=last * T, mirror=True)
    rows_t = torch.from_numpy(rows).to(dev)
    errs = {}
    for key, tensor in (("O", buf.O), ("dX", buf.dX), ("U", buf.U), ("Y", buf.Y), ("dU", buf.dU)):
        got = to_f64(tensor.index_select(0, rows_t))
        errs[key] = rel_err(got, ref[key])
        assert errs[key] <= BF16_TOL, (wl.name, key, errs[key])
    # the whole dZ of the last micro-batch, and the dropout decisions it encodes
    dZ_last = orc.full_dZ(dOs[last], wl.p, wl.seed, token_offset=last * T, mirror=True)
    errs["dZ"] = rel_err(to_f64(buf.dZ), dZ_last)
    assert errs["dZ"] <= BF16_TOL
    keep = orc.dropout_keep(T, h, wl.p, wl.seed, last * T, rows=rows)
    np.testing.assert_array_equal(to_f64(buf.O.index_select(0, rows_t))[~keep], Xs[last][rows][~keep])

    # accumulated gradients: db whole; dA, dB, da at sampled entries (summed over micro-batches)
    dZs = [orc.full_dZ(dOs[j], wl.p, wl.seed, token_offset=j * T, mirror=True) for j in range(wl.k)]
    ref_db = sum(dZ.sum(axis=0) for dZ in dZs)
    errs["db"] = rel_err(to_f64(buf.db), ref_db)
    assert errs["db"] <= F32_TOL, errs
    rB = np.concatenate([[0, F - 1], rng.integers(0, F, n_entries - 2)])
    cB = np.concatenate([[0, h - 1], rng.integers(0, h, n_entries - 2)])
    ref_dB = sum(orc.wgrad_dB_entries(rB, cB, Xs[j], A, a, dZs[j], mirror=True) for j in range(wl.k))
    got_dB = to_f64(buf.dB[torch.from_numpy(rB).to(dev), torch.from_numpy(cB).to(dev)])
    rA = np.concatenate([[0, h - 1], rng.integers(0, h, n_entries - 2)])
    cA = np.concatenate([[0, F - 1], rng.integers(0, F, n_entries - 2)])
    ref_dA = sum(orc.wgrad_dA_entries(rA, cA, Xs[j], A, a, B, dZs[j], mirror=True) for j in range(wl.k))
    got_dA = to_f64(buf.dA[torch.from_numpy(rA).to(dev), torch.from_numpy(cA).to(dev)])
    if full_da:
        ref_da = _full_da(Xs, dZs, A, a, B, F)
        got_da = to_f64(buf.da)
    else:
        ca = np.unique(cA)
        ref_da = sum(orc.columns_dU(ca, Xs[j], A, a, B, dZs[j], mirror=True).sum(axis=0) for j in range(wl.k))
        got_da = to_f64(buf.da[torch.from_numpy(ca).to(dev)])
    # the relative-to-max bar, with the max taken over the sampled reference entries
    errs["dB"] = rel_err(got_dB, ref_dB)
    errs["dA"] = rel_err(got_dA, ref_dA)
    errs["da"] = rel_err(got_da, ref_da)
    for key in ("dB", "dA", "da"):
        assert errs[key] <= F32_TOL, (wl.name, key, errs[key])
    return errs


def test_mid_workload_sampled_parity():
    """2048 tokens, h 4096, ffn 16384, t 1, four accumulated micro-batches."""
    _sampled_check(gin.WORKLOADS["mid"], "all")


def test_mtnlg_layer_sampled_parity():
    """2048 tokens, h 20480, ffn 81920, t 8: all slices per call, the first (only)
    micro-batch writing the gradients, as benchmarked."""
    _sampled_check(gin.WORKLOADS["mtnlg"], "all", first_overwrites=True)


def test_mtnlg_layer_one_slice_calls_sampled_parity():
    """The MT-NLG layer with its eight slices as eight calls in turn (fp32 partial
    sums in HBM)."""
    _sampled_check(gin.WORKLOADS["mtnlg"], "each", seed=1)


@pytest.mark.parametrize("name,first_overwrites", [("sweep1", True), ("sweep4", False), ("sweep16", True),
                                                   ("sweep32", False)])
def test_accumulation_sweep_sampled_parity(name, first_overwrites):
    """h 8192, ffn 32768, t 4, one slice per call in turn, micro-batches accumulated.
    All of da is checked up to 4 micro-batches; at 16 and 32 (35 and 70 TFLOP of
    float64 host work for it) at the 256 sampled dA columns."""
    wl = gin.WORKLOADS[name]
    _sampled_check(wl, "each", first_overwrites=first_overwrites, full_da=wl.k <= 4)
