"""GPU parity of the tensor-sliced MLP block against the CPU oracle, through the C ABI.

Bars: the dropout mask bit-exact; bf16 activations and gradients within
max|gpu - oracle| / max|oracle| <= 1e-2 of both oracle modes; fp32 accumulated
weight and bias gradients within 1e-3 of the oracle's bf16-mirroring mode.
"""
import numpy as np
import pytest
import torch

from oracle import mlp_oracle as orc
from transformer_lm_megatron_gb300 import build as gb_build
from transformer_lm_megatron_gb300 import mlp

from gpu_harness import (BF16_TOL, F32_TOL, Shape, bits_f64, compare_full, make_case, rel_err, run_gpu,
                         run_oracle, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gb_build.build()
    mlp.load()
    torch.cuda.synchronize()


def test_gelu_device_functions_exhaustive_bf16():
    """Every finite bf16 value as a pre-activation: GeLU and GeLU' against fp64."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x64 = orc.bf16_to_f64(bits)
    x64 = x64[np.isfinite(x64)]
    x = torch.from_numpy(x64.astype(np.float32)).cuda()
    y = torch.empty_like(x)
    dy = torch.empty_like(x)
    mlp.mlp_gelu_probe(x, y, dy)
    torch.cuda.synchronize()
    ref_y = orc.gelu(x64)
    ref_dy = orc.gelu_prime(x64)
    gy = y.cpu().numpy().astype(np.float64)
    gdy = dy.cpu().numpy().astype(np.float64)
    # fp32 evaluation: error relative to max(|value|, 1) stays at a few fp32 ulps
    ey = np.abs(gy - ref_y) / np.maximum(np.abs(ref_y), 1.0)
    edy = np.abs(gdy - ref_dy) / np.maximum(np.abs(ref_dy), 1.0)
    assert np.all(np.isfinite(gy)) and np.all(np.isfinite(gdy))
    assert ey.max() < 2e-6, ey.max()
    assert edy.max() < 2e-6, edy.max()


@pytest.mark.parametrize("h,tokens,p,seed,off", [(64, 100, 0.1, 1234, 0), (768, 33, 0.5, 7, 4096),
                                                   (20480, 8, 0.1, 1234, 2**40), (136, 5, 0.0, 1, 3)])
def test_dropout_mask_bit_exact(h, tokens, p, seed, off):
    m = torch.empty(tokens, h, dtype=torch.uint8, device="cuda")
    mlp.mlp_dropout_mask(h, tokens, p, seed, off, m)
    ref = orc.dropout_keep(tokens, h, p, seed, off)
    np.testing.assert_array_equal(m.cpu().numpy().astype(bool), ref)


TINY = Shape(tokens=256, h=256, ffn=1024, t=2, k=2)


def test_tiny_workload_full_parity():
    """The tiny workload (256 tokens, h 256, ffn 1024, t 2, two micro-batches)."""
    w_dev, mbs_dev, w64, mbs64 = make_case(TINY)
    g_outs, g_grads = run_gpu(TINY, w_dev, mbs_dev, keep_all=True)
    for mirror in (True, False):
        r_outs, r_grads = run_oracle(TINY, w64, mbs64, mirror=mirror, keep_all=True)
        compare_full(TINY, g_outs, g_grads, r_outs, r_grads, check_grads=mirror, label=f"mirror={mirror}")
        # the mask decides exactly: dropped outputs equal the residual, dropped dZ are zero
        for j in range(TINY.k):
            keep = orc.dropout_keep(TINY.tokens, TINY.h, TINY.p, TINY.seed, j * TINY.tokens)
            O = to_f64(g_outs[j]["O"])
            X = mbs64[j][0]
            np.testing.assert_array_equal(O[~keep], X[~keep])
            assert np.all(to_f64(g_outs[j]["dZ"])[~keep] == 0)


@pytest.fixture
def cta_pair_mode(request):
    mlp.mlp_set_cta_pair(request.param)
    yield request.param
    mlp.mlp_set_cta_pair(-1)


@pytest.mark.parametrize("cta_pair_mode", [0, 1, -1], indirect=True, ids=["single", "pair", "auto"])
@pytest.mark.parametrize("tokens,h,ffn,t", [
    (200, 136, 656, 2),     # ragged M, N and K tails (none a multiple of the 128/256/64 tiles)
    (1, 64, 128, 1),        # a single token
    (130, 8, 64, 4),        # h = 8: one partial k-block, f = 16
    (384, 320, 1280, 1),    # several M tiles, N tail of 64
    (520, 264, 1040, 2),    # M tail of 8 rows past two CTA-pair tiles
])
def test_ragged_shapes_full_parity(tokens, h, ffn, t, cta_pair_mode):
    s = Shape(tokens=tokens, h=h, ffn=ffn, t=t, k=2, p=0.1)
    w_dev, mbs_dev, w64, mbs64 = make_case(s)
    g_outs, g_grads = run_gpu(s, w_dev, mbs_dev)
    for mirror in (True, False):
        r_outs, r_grads = run_oracle(s, w64, mbs64, mirror=mirror)
        compare_full(s, g_outs, g_grads, r_outs, r_grads, check_grads=mirror,
                     label=f"pair mode {cta_pair_mode}, mirror={mirror}")


@pytest.mark.parametrize("t", [2, 4, 8])
def test_one_slice_calls_full_parity(t):
    """One call per slice in order (fp32 partial sums through Zacc / dXacc in HBM),
    two accumulated micro-batches, against the oracle."""
    s = Shape(tokens=200, h=256, ffn=2048, t=t, k=2)
    w_dev, mbs_dev, w64, mbs64 = make_case(s)
    g_outs, g_grads = run_gpu(s, w_dev, mbs_dev, slice_mode="each")
    for mirror in (True, False):
        r_outs, r_grads = run_oracle(s, w64, mbs64, mirror=mirror)
        compare_full(s, g_outs, g_grads, r_outs, r_grads, check_grads=mirror, label=f"each t={t}, mirror={mirror}")


def test_slice_invariance():
    """t = 1, 2, 4, 8 and both call forms agree within tolerance with identical
    dropped positions (the special case t = 1 is the plain dense block)."""
    base = None
    for t in (1, 2, 4, 8):
        s = Shape(tokens=256, h=256, ffn=2048, t=t, k=1)
        w_dev, mbs_dev, w64, mbs64 = make_case(s)
        for mode in ("all", "each"):
            outs, grads = run_gpu(s, w_dev, mbs_dev, slice_mode=mode)
            if base is None:
                base = (outs, grads)
                continue
            for k in ("O", "dX", "U", "Y", "dU", "dZ"):
                assert rel_err(to_f64(outs[0][k]), to_f64(base[0][0][k])) <= BF16_TOL, (t, mode, k)
            for k in grads:
                assert rel_err(to_f64(grads[k]), to_f64(base[1][k])) <= F32_TOL, (t, mode, k)
            O = to_f64(outs[0]["O"])
            X = mbs64[0][0]
            keep = orc.dropout_keep(s.tokens, s.h, s.p, s.seed, 0)
            np.testing.assert_array_equal(O[~keep], X[~keep])
            np.testing.assert_array_equal(to_f64(outs[0]["U"]), to_f64(base[0][0]["U"]))


def test_exact_invariants():
    """Power-of-two scaling of dO scales every gradient exactly; zero second layer
    gives O == X exactly; reset + one micro-batch equals a fresh run bit for bit."""
    s = Shape(tokens=192, h=128, ffn=512, t=2, k=1)
    w_dev, mbs_dev, _, _ = make_case(s)
    outs1, g1 = run_gpu(s, w_dev, mbs_dev)
    X, dO = mbs_dev[0]
    outs2, g2 = run_gpu(s, w_dev, [(X, dO * 2)])
    for k in g1:
        assert torch.equal(g2[k], g1[k] * 2), k
    assert torch.equal(outs2[0]["dX"].float(), outs1[0]["dX"].float() * 2)
    # checkpoint/restore of the accumulators: accumulate, copy, continue == uninterrupted
    buf = mlp.BlockBuffers(s.tokens, s.h, s.ffn, s.t)
    run_gpu(s, w_dev, mbs_dev, buf=buf)
    saved = {k: getattr(buf, k).clone() for k in ("dA", "da", "dB", "db")}
    _, g_cont = run_gpu(s, w_dev, mbs_dev, buf=buf, reset=False)
    buf2 = mlp.BlockBuffers(s.tokens, s.h, s.ffn, s.t)
    for k, v in saved.items():
        getattr(buf2, k).copy_(v)
    _, g_rest = run_gpu(s, w_dev, mbs_dev, buf=buf2, reset=False)
    for k in g_cont:
        assert torch.equal(g_cont[k], g_rest[k]), k
    # reset then one micro-batch equals the fresh result
    _, g_reset = run_gpu(s, w_dev, mbs_dev, buf=buf)
    for k in g1:
        assert torch.equal(g_reset[k], g1[k]), k
    # B = 0, b = 0: O = X + dropout(0) = X exactly
    A, a, B, b = w_dev
    outs0, _ = run_gpu(s, (A, a, torch.zeros_like(B), torch.zeros_like(b)), mbs_dev)
    assert torch.equal(outs0[0]["O"], X.cpu())


@pytest.mark.parametrize("mode", ["all", "each"])
def test_first_microbatch_overwrite_equals_reset_then_accumulate(mode):
    """accumulate = 0 on the first micro-batch (accumulators left holding NaN)
    gives bit for bit what grad_accum_reset + accumulate = 1 gives."""
    s = Shape(tokens=200, h=256, ffn=1024, t=4, k=3)
    w_dev, mbs_dev, w64, mbs64 = make_case(s)
    _, g_ref = run_gpu(s, w_dev, mbs_dev, slice_mode=mode)
    buf = mlp.BlockBuffers(s.tokens, s.h, s.ffn, s.t)
    for k in ("dA", "da", "dB", "db"):
        getattr(buf, k).fill_(float("nan"))
    _, g_new = run_gpu(s, w_dev, mbs_dev, slice_mode=mode, buf=buf, reset=False, first_overwrites=True)
    for k in g_ref:
        assert torch.equal(g_new[k], g_ref[k]), k
    r_outs, r_grads = run_oracle(s, w64, mbs64, mirror=True)
    for k in ("dA", "da", "dB", "db"):
        assert rel_err(to_f64(g_new[k]), r_grads[k]) <= F32_TOL, k


@pytest.mark.parametrize("mode", ["all", "each"])
def test_accumulation_invariance_and_sum_of_singles(mode):
    """Gradient accumulation (MT-NLG summary page, Key points): k micro-batches of
    T tokens accumulated with token offsets j T give the gradients of one batch of
    k T tokens at offset 0, up to fp32 summation order (1e-3, relative to max), with
    the same dropout mask, so every output row is bit-identical; and they equal
    the sum, in float64, of the k micro-batches' gradients computed one at a time,
    up to the fp32 rounding of the running sum (1e-6)."""
    s = Shape(tokens=256, h=256, ffn=1024, t=2, k=3)
    w_dev, mbs_dev, _, _ = make_case(s)
    outs_acc, g_acc = run_gpu(s, w_dev, mbs_dev, slice_mode=mode, keep_all=True)
    # one batch of k T tokens
    Xc = torch.cat([X for X, _ in mbs_dev])
    dOc = torch.cat([dO for _, dO in mbs_dev])
    sc = Shape(tokens=s.k * s.tokens, h=s.h, ffn=s.ffn, t=s.t, k=1)
    outs_cat, g_cat = run_gpu(sc, w_dev, [(Xc, dOc)], slice_mode=mode)
    for key in ("U", "Y", "O", "dZ", "dU", "dX"):
        got = torch.cat([outs_acc[j][key] for j in range(s.k)])
        assert torch.equal(got, outs_cat[0][key]), key
    for key in g_acc:
        e = rel_err(to_f64(g_acc[key]), to_f64(g_cat[key]))
        assert e <= F32_TOL, (key, e)
    # the sum of single micro-batches
    singles = {key: 0.0 for key in g_acc}
    for j in range(s.k):
        _, g_j = run_gpu(s, w_dev, [mbs_dev[j]], slice_mode=mode, first_overwrites=True, token_offset0=j * s.tokens)
        for key in singles:
            singles[key] = singles[key] + to_f64(g_j[key])
    for key in g_acc:
        e = rel_err(to_f64(g_acc[key]), singles[key])
        assert e <= 1e-6, (key, e)


def test_bounded_wait_reports_timeout():
    assert mlp.mlp_sync_status() == mlp.MLP_OK
    mlp.mlp_wait_timeout_probe(1000000)   # 1 ms
    assert mlp.mlp_sync_status() == mlp.MLP_ETIMEOUT
    assert "bounded wait" in mlp.last_error()
    assert mlp.mlp_sync_status() == mlp.MLP_OK  # the word is cleared, the context still works
    x = torch.ones(16, device="cuda")
    assert float(x.sum()) == 16.0


def test_trace_reports_every_launch_in_order():
    s = Shape(tokens=256, h=128, ffn=512, t=2, k=1)
    w_dev, mbs_dev, _, _ = make_case(s)
    buf = mlp.BlockBuffers(s.tokens, s.h, s.ffn, s.t)
    tr = mlp.Trace(capacity=64)
    tr.start()
    mlp.block_step(s, w_dev, *mbs_dev[0], buf, accumulate=False)
    torch.cuda.synchronize()
    entries = tr.stop()
    kinds = [k for k, _, _ in entries]
    # forward F1, F2; backward B1, B2, da column sum, B5, B3, B4
    assert kinds == [0, 1, 10, 2, 11, 5, 3, 4]
    mnk = [m for _, m, _ in entries]
    assert mnk[0] == (s.tokens, s.ffn, s.h) and mnk[3] == (s.tokens, s.ffn, s.h)
    assert mnk[5] == (s.tokens, s.h, s.ffn)
    assert mnk[6] == (s.ffn, s.h, s.tokens) and mnk[7] == (s.h, s.ffn, s.tokens)
    assert all(t_ms > 0 for _, _, t_ms in entries)
    with pytest.raises(mlp.MLPError):
        tr.stop()                                    # no trace running


def test_launch_counter_counts_kernels():
    s = Shape(tokens=128, h=64, ffn=256, t=2, k=1)
    w_dev, mbs_dev, _, _ = make_case(s)
    buf = mlp.BlockBuffers(s.tokens, s.h, s.ffn, s.t)
    n0 = mlp.mlp_launch_count()
    mlp.block_step(s, w_dev, *mbs_dev[0], buf)
    torch.cuda.synchronize()
    # all slices per call: forward 2 GEMMs; backward dropout + 4 GEMMs + 1 column sum
    assert mlp.mlp_launch_count() - n0 == 2 + 1 + 5
    n1 = mlp.mlp_launch_count()
    mlp.block_step(s, w_dev, *mbs_dev[0], buf, slice_mode="each")
    torch.cuda.synchronize()
    # one call per slice: 2 GEMMs per slice forward; 1 + 5 per slice backward
    assert mlp.mlp_launch_count() - n1 == 2 * s.t + 1 + 5 * s.t


@pytest.mark.parametrize("mode", ["all", "each"])
def test_dependent_launch_changes_no_bit(mode):
    """Programmatic dependent launch only lets a kernel's prologue overlap the
    previous kernel: outputs and gradients are bit-identical with it on and off.
    Both call modes are deterministic: no atomics, fixed-order column sums, and
    each fp32 reduction in HBM adds one tile per launch, launches in slice order."""
    s = Shape(tokens=1000, h=384, ffn=1536, t=4, k=3)
    w_dev, mbs_dev, _, _ = make_case(s)
    try:
        mlp.mlp_set_dependent_launch(False)
        o_off, g_off = run_gpu(s, w_dev, mbs_dev, slice_mode=mode)
        mlp.mlp_set_dependent_launch(True)
        o_on, g_on = run_gpu(s, w_dev, mbs_dev, slice_mode=mode)
    finally:
        mlp.mlp_set_dependent_launch(True)
    for k in o_off[-1]:
        assert torch.equal(o_on[-1][k], o_off[-1][k]), k
    for k in g_off:
        assert torch.equal(g_on[k], g_off[k]), k


@pytest.mark.parametrize("cta_pair_mode", [0, 1], indirect=True, ids=["single", "pair"])
@pytest.mark.parametrize("tokens,h,ffn,t", [
    (512, 1280, 2048, 1),   # every GEMM with a bf16 epilogue has fewer tiles than half the CTA pairs
    (456, 1288, 1552, 2),   # the same with ragged M, N and K (K of F2/B5 not a multiple of 64)
])
def test_split_tail_full_parity(tokens, h, ffn, t, cta_pair_mode):
    """GEMMs whose last wave is at most half full run their tail tiles as two
    half-reductions (split tail).  These shapes put F1, F2, B2 and B5 entirely in
    the tail: full parity with the oracle, bit-identical repeats (the two partial
    sums commute), and agreement with the unsplit kernel to fp32 rounding."""
    s = Shape(tokens=tokens, h=h, ffn=ffn, t=t, k=2, p=0.1)
    w_dev, mbs_dev, w64, mbs64 = make_case(s)
    g_outs, g_grads = run_gpu(s, w_dev, mbs_dev, keep_all=True)
    for mirror in (True, False):
        r_outs, r_grads = run_oracle(s, w64, mbs64, mirror=mirror, keep_all=True)
        compare_full(s, g_outs, g_grads, r_outs, r_grads, check_grads=mirror,
                     label=f"split tail, pair mode {cta_pair_mode}, mirror={mirror}")
    again_outs, again_grads = run_gpu(s, w_dev, mbs_dev, keep_all=True)
    for j in range(s.k):
        for k in g_outs[j]:
            assert torch.equal(again_outs[j][k], g_outs[j][k]), (j, k)
    try:
        mlp.mlp_set_split_tail(False)
        u_outs, u_grads = run_gpu(s, w_dev, mbs_dev, keep_all=True)
    finally:
        mlp.mlp_set_split_tail(True)
    for j in range(s.k):
        for k in ("U", "Y", "O", "dX"):
            a, b = to_f64(g_outs[j][k]), to_f64(u_outs[j][k])
            # the same fp32 sum in two orders, then one bf16 rounding: at most one bf16 step apart
            assert np.max(np.abs(a - b)) <= 2.0 ** -7 * np.max(np.abs(b)) + 1e-30, (j, k)


def test_split_tail_on_concurrent_streams():
    """Two blocks whose GEMMs split their tail run at the same time on two streams:
    each stream has its own workspace region, so both match their one-stream runs
    bit for bit."""
    shapes = [Shape(tokens=512, h=1280, ffn=2048, t=1, k=2, p=0.1),
              Shape(tokens=512, h=1280, ffn=2048, t=1, k=2, p=0.1, seed=99)]  # another dropout mask
    s = shapes[0]
    cases = [make_case(sh) for sh in shapes]
    ref = []
    for sh, (w_dev, mbs_dev, _, _) in zip(shapes, cases):
        outs, grads = run_gpu(sh, w_dev, mbs_dev, keep_all=True)
        ref.append((outs, grads))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    bufs = [mlp.BlockBuffers(s.tokens, s.h, s.ffn, s.t) for _ in cases]
    torch.cuda.synchronize()
    for rep in range(3):
        for j in range(s.k):
            for c, (w_dev, mbs_dev, _, _) in enumerate(cases):
                X, dO = mbs_dev[j]
                mlp.block_step(shapes[c], w_dev, X, dO, bufs[c], token_offset=j * s.tokens, stream=streams[c],
                               accumulate=j > 0)
        torch.cuda.synchronize()
        assert mlp.mlp_sync_status() == mlp.MLP_OK, mlp.last_error()
        for c in range(2):
            for k in ("U", "Y", "O", "dZ", "dU", "dX"):
                assert torch.equal(getattr(bufs[c], k).cpu(), ref[c][0][-1][k]), (rep, c, k)
            for k in ("dA", "da", "dB", "db"):
                assert torch.equal(getattr(bufs[c], k).cpu(), ref[c][1][k]), (rep, c, k)


@pytest.mark.parametrize("tokens,h,ffn,t,mode", [
    (200, 136, 656, 2, "all"),      # ragged M, N and K tails, all slices per call
    (200, 136, 656, 2, "each"),     # the same, one slice per call
    (256, 512, 2048, 4, "each"),    # accumulation-sweep-like: four slices, one per call
    (512, 1280, 2048, 1, "all"),    # split tail of F2 (dropout + residual) and B5 (input gradient)
])
def test_explicit_residual_and_no_residual_gradient(tokens, h, ffn, t, mode):
    """mlp_fwd with a residual R that is not X, and mlp_bwd with residual_grad = 0
    (dX = sum_i dU_i A_i^T, no dO term), against oracle.mlp_fwd(..., R=R) and
    oracle.mlp_bwd(..., residual_is_input=False) in both modes, over two
    accumulated micro-batches."""
    s = Shape(tokens=tokens, h=h, ffn=ffn, t=t, k=2, p=0.1)
    w_dev, mbs_dev, w64, mbs64 = make_case(s)
    gen = torch.Generator().manual_seed(77)
    Rs = [torch.randn(tokens, h, generator=gen).to(torch.bfloat16) for _ in range(s.k)]
    buf = mlp.BlockBuffers(tokens, h, ffn, t)
    A, a, B, b = w_dev
    slices = [-1] if mode == "all" else list(range(t))
    outs = []
    for j, (X, dO) in enumerate(mbs_dev):
        R = Rs[j].cuda()
        for i in slices:
            mlp.mlp_fwd(h, ffn, t, i, tokens, s.p, s.seed, j * tokens, X, A, a, B, b, R, buf.U, buf.Y, buf.Zacc,
                        buf.O)
        for i in slices:
            mlp.mlp_bwd(h, ffn, t, i, tokens, s.p, s.seed, j * tokens, 0, j > 0, dO, X, A, B, buf.U, buf.Y, buf.dZ,
                        buf.dU, buf.dXacc, buf.dX, buf.dA, buf.da, buf.dB, buf.db)
        outs.append({k: getattr(buf, k).cpu() for k in ("U", "Y", "O", "dZ", "dU", "dX")})
    torch.cuda.synchronize()
    assert mlp.mlp_sync_status() == mlp.MLP_OK, mlp.last_error()
    grads = {k: getattr(buf, k).cpu() for k in ("dA", "da", "dB", "db")}
    Aw, aw, Bw, bw = w64
    for mirror in (True, False):
        acc = {k: 0.0 for k in grads}
        for j, (X64, dO64) in enumerate(mbs64):
            R64 = bits_f64(Rs[j])
            fw = orc.mlp_fwd(X64, Aw, aw, Bw, bw, t, s.p, s.seed, token_offset=j * tokens, R=R64, mirror=mirror)
            bwd = orc.mlp_bwd(dO64, X64, Aw, Bw, fw["U"], fw["Y"], fw["keep"], t, s.p, mirror=mirror,
                              residual_is_input=False)
            ref = {**fw, **bwd}
            for k in ("U", "Y", "O", "dZ", "dU", "dX"):
                e = rel_err(to_f64(outs[j][k]), ref[k])
                assert e <= BF16_TOL, (mirror, j, k, e)
            # dropped outputs are the residual R exactly
            O = to_f64(outs[j]["O"])
            np.testing.assert_array_equal(O[~fw["keep"]], R64[~fw["keep"]])
            for k in acc:
                acc[k] = acc[k] + bwd[k]
        if mirror:
            for k in grads:
                e = rel_err(to_f64(grads[k]), acc[k])
                assert e <= F32_TOL, (k, e)


@pytest.fixture
def tile_scheduler():
    yield
    mlp.mlp_set_tile_scheduler(-1)


@pytest.mark.parametrize("cta_pair_mode", [0, 1], indirect=True, ids=["single", "pair"])
@pytest.mark.parametrize("tokens,h,ffn,t,mode", [
    (1000, 384, 1536, 4, "all"),     # several waves per GEMM
    (1000, 384, 1536, 4, "each"),    # one-slice calls: fp32 partial sums through Zacc / dXacc
    (512, 1280, 2048, 1, "all"),     # split tail (two half-reductions per tail tile)
    (2304, 768, 3072, 1, "all"),     # many waves, ragged tails
])
def test_tile_scheduler_changes_no_bit(tokens, h, ffn, t, mode, cta_pair_mode, tile_scheduler):
    """The dynamic tile order (a counter in global memory hands out the tiles) and
    the static round-robin order give bit-identical results: a tile's arithmetic
    does not depend on which CTA computes it.  Three accumulated micro-batches, so
    the counters must come back to zero after every launch."""
    s = Shape(tokens=tokens, h=h, ffn=ffn, t=t, k=3)
    w_dev, mbs_dev, w64, mbs64 = make_case(s)
    mlp.mlp_set_tile_scheduler(0)
    o_st, g_st = run_gpu(s, w_dev, mbs_dev, slice_mode=mode, keep_all=True)
    mlp.mlp_set_tile_scheduler(1)
    o_dy, g_dy = run_gpu(s, w_dev, mbs_dev, slice_mode=mode, keep_all=True)
    o_dy2, g_dy2 = run_gpu(s, w_dev, mbs_dev, slice_mode=mode, keep_all=True)
    for j in range(s.k):
        for k in o_st[j]:
            assert torch.equal(o_dy[j][k], o_st[j][k]), (j, k)
            assert torch.equal(o_dy2[j][k], o_st[j][k]), (j, k)
    for k in g_st:
        assert torch.equal(g_dy[k], g_st[k]), k
        assert torch.equal(g_dy2[k], g_st[k]), k
    r_outs, r_grads = run_oracle(s, w64, mbs64, mirror=True)
    compare_full(s, [o_dy[-1]], g_dy, [r_outs[-1]], r_grads, label="dynamic tile order")


@pytest.fixture
def wgrad_transpose():
    yield
    mlp.mlp_set_wgrad_transpose(-1)


@pytest.mark.parametrize("tokens,h,ffn,t", [
    (1024, 256, 1024, 1),     # whole 64 x 64 tiles of the copies
    (1000, 264, 1056, 1),     # ragged copy tiles along both dimensions
    (1000, 384, 1536, 4),     # every slice in one call, t = 4
    (1004, 256, 1024, 1),     # tokens % 8 != 0: no copies (their tensor maps need 16-byte rows)
])
def test_wgrad_transposed_operands_change_no_bit(tokens, h, ffn, t, wgrad_transpose):
    """B3 and B4 reading transposed copies of dZ and X (K-major operands held in
    dXacc) give, bit for bit, what they give reading dZ and X as MN-major
    operands: the same products, reduced in the same order.  The copy launch runs
    once per micro-batch when asked for and the shape allows it, and never
    otherwise.  Two micro-batches, so the second adds its gradients (reduce-add
    epilogues) to the first's."""
    s = Shape(tokens=tokens, h=h, ffn=ffn, t=t, k=2)
    w_dev, mbs_dev, w64, mbs64 = make_case(s)
    runs = {}
    for mode in (0, 1):
        mlp.mlp_set_wgrad_transpose(mode)
        tr = mlp.Trace(capacity=256)
        tr.start()
        runs[mode] = run_gpu(s, w_dev, mbs_dev, slice_mode="all", keep_all=True)
        tr.stop()
        copies = sum(1 for kind, _, _ in tr.entries if kind == 15)
        assert copies == (s.k if mode == 1 and tokens % 8 == 0 else 0), (mode, copies)
    (o_mn, g_mn), (o_k, g_k) = runs[0], runs[1]
    for j in range(s.k):
        for k in o_mn[j]:
            assert torch.equal(o_k[j][k], o_mn[j][k]), (j, k)
    for k in g_mn:
        assert torch.equal(g_k[k], g_mn[k]), k
    r_outs, r_grads = run_oracle(s, w64, mbs64, mirror=True)
    compare_full(s, [o_k[-1]], g_k, [r_outs[-1]], r_grads, label="transposed weight-gradient operands")


@pytest.mark.parametrize("mode", ["all", "each"])
def test_cuda_graph_replay_equals_eager(mode):
    """A step captured in a CUDA graph and replayed gives, bit for bit, what the
    eager calls give, replay after replay: the library keeps no per-call host state
    that a replay would miss, and its device-side counters (split tail, tile order)
    return to zero after every kernel."""
    s = Shape(tokens=512, h=1280, ffn=2048, t=2, k=2)     # F2 and B5 split their tail
    w_dev, mbs_dev, _, _ = make_case(s)
    o_ref, g_ref = run_gpu(s, w_dev, mbs_dev, slice_mode=mode, reset=False, first_overwrites=True)
    buf = mlp.BlockBuffers(s.tokens, s.h, s.ffn, s.t)

    def step():
        for j, (X, dO) in enumerate(mbs_dev):
            mlp.block_step(s, w_dev, X, dO, buf, token_offset=j * s.tokens, slice_mode=mode, accumulate=j > 0)

    step()                                    # first calls on this shape happen outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(3):
        for k in ("dA", "da", "dB", "db", "O", "dX"):
            getattr(buf, k).fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert mlp.mlp_sync_status() == mlp.MLP_OK, mlp.last_error()
        for k in ("O", "dX", "U", "Y", "dU", "dZ"):
            assert torch.equal(getattr(buf, k).cpu(), o_ref[-1][k]), k
        for k in ("dA", "da", "dB", "db"):
            assert torch.equal(getattr(buf, k).cpu(), g_ref[k]), k
