"""GPU parity of the tensor-sliced self-attention block (attn_fwd / attn_bwd)
against the float64 oracle, through the C ABI.

Bars, with g the oracle's own distance between its pure and bf16-mirroring modes
for the tensor on the same inputs (max|mirror - pure| / max|pure|; it comes from
the oracle alone):
  * against the bf16-mirroring mode: bf16 tensors (QKV, P, O, out, dQKV, dX)
    within max|gpu - oracle| / max|oracle| <= 1e-2, as for the MLP block; fp32
    accumulated gradients (dWqkv, dbqkv, dWo, dbo) within max(1e-3, g).  The
    mirroring mode rounds to bf16 at the block's storage points from exact values;
    the block rounds at the same points from fp32 values, so it can land on the
    other side of a bf16 step wherever the exact value is within fp32 error of a
    rounding boundary.  g measures the whole effect of those storage roundings on
    the gradient (every element rounded, through every point: QKV, P, O, dZ, dO,
    dS, dQKV for dWqkv), so a result no farther from the mirror than the mirror is
    from the exact value is what the storage precisions allow (g is 2.8e-3 to
    3.7e-3 for dWqkv on the small shapes below).
  * against the pure mode: the mirror bar plus g, which is what the triangle
    inequality leaves for a result within the mirror bar.  At the MT-NLG shape
    with N(0, 0.02) weights the scores have a standard deviation of about 8, so
    the bf16 storage of Q and K alone moves the probabilities by about 1 %, and g
    for O is about 1.6e-2: no implementation that stores QKV in bf16 can be within
    1e-2 of the exact-arithmetic block there.
  * Probabilities are exactly zero above the causal diagonal, and dropped outputs
    equal the residual exactly.
"""
import numpy as np
import pytest
import torch

from oracle import attn_oracle as ato
from oracle import mlp_oracle as orc
from transformer_lm_megatron_gb300 import build as gb_build
from transformer_lm_megatron_gb300 import inputs as gin
from transformer_lm_megatron_gb300 import mlp

from gpu_harness import BF16_TOL, F32_TOL, bits_f64, rel_err, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gb_build.build()
    mlp.load()


def _weights(h, gen, std=0.02):
    def rnd(*shape, s=std):
        return (torch.randn(*shape, generator=gen) * s).to(torch.bfloat16)
    return rnd(h, 3 * h), rnd(3 * h), rnd(h, h), rnd(h)


def f32_bar(pure, mirror) -> float:
    """The fp32-gradient bar against the mirroring mode: the oracle's own
    pure-to-mirror distance for the tensor, never below 1e-3."""
    return max(F32_TOL, rel_err(mirror, pure))


def pure_bar(mirror_bar, pure, mirror) -> float:
    """The bar against the pure mode for a tensor held to ``mirror_bar`` against
    the mirroring mode: that bar plus the oracle's pure-to-mirror distance."""
    return mirror_bar + rel_err(mirror, pure)


@pytest.fixture
def cta_pair_mode(request):
    mlp.mlp_set_cta_pair(request.param)
    yield request.param
    mlp.mlp_set_cta_pair(-1)


@pytest.fixture
def attn_core(request):
    mlp.mlp_set_attn_fused(request.param == "fused")
    yield request.param
    mlp.mlp_set_attn_fused(True)


@pytest.mark.parametrize("attn_core", ["fused", "unfused"], indirect=True)
@pytest.mark.parametrize("cta_pair_mode", [0, 1], indirect=True, ids=["single", "pair"])
@pytest.mark.parametrize("T,h,nh,t,L,k", [
    (256, 256, 4, 2, 128, 2),     # two sequences, d = 64, two accumulated micro-batches
    (272, 320, 4, 4, 136, 1),     # ragged: d = 80, seq_len 136 (tails in every GEMM)
    (2048, 2048, 16, 8, 1024, 1),  # two sequences of 1024, d = 128, eight slices
    (2048, 256, 2, 2, 2048, 1),    # one sequence of 2048: the longest rows the warp-per-row softmax holds
    (2304, 128, 2, 1, 2304, 1),    # rows past 2048 columns: the CTA-per-row softmax
])
def test_attention_block_full_parity(T, h, nh, t, L, k, cta_pair_mode, attn_core):
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
    acc = {m: {n: 0.0 for n in grads} for m in (True, False)}
    for j, (X, dOut) in enumerate(mbs):
        X64, d64 = bits_f64(X), bits_f64(dOut)
        ref = {}
        for mirror in (True, False):
            fw = ato.attn_fwd(X64, W64[0], W64[1], W64[2], W64[3], nh, t, L, p, seed, token_offset=j * T,
                              mirror=mirror)
            bw = ato.attn_bwd(d64, X64, W64[0], W64[2], fw["QKV"], fw["P"], fw["O"], fw["keep"], nh, t, L, p,
                              mirror=mirror)
            ref[mirror] = {"QKV": fw["QKV"], "P": fw["P"], "O": fw["O"], "out": fw["out"], "dQKV": bw["dQKV"],
                           "dX": bw["dX"], "keep": fw["keep"]}
            for n in grads:
                acc[mirror][n] = acc[mirror][n] + bw[n]
        g = outs[j]
        for name in ("QKV", "P", "O", "out", "dQKV", "dX"):
            got = to_f64(g[name])
            e = rel_err(got, ref[True][name])
            assert e <= BF16_TOL, ("mirror", j, name, e)
            e = rel_err(got, ref[False][name])
            assert e <= pure_bar(BF16_TOL, ref[False][name], ref[True][name]), ("pure", j, name, e)
        P = to_f64(g["P"])
        assert np.all(np.triu(P, k=1) == 0)
        keep = ref[True]["keep"]
        np.testing.assert_array_equal(to_f64(g["out"])[~keep], X64[~keep])
    for n in grads:
        bar = f32_bar(acc[False][n], acc[True][n])
        e = rel_err(grads[n], acc[True][n])
        assert e <= bar, ("mirror", n, e, bar)
        e = rel_err(grads[n], acc[False][n])
        assert e <= pure_bar(bar, acc[False][n], acc[True][n]), ("pure", n, e)


def _bits(t):
    return gin.bf16_bits(t.detach().cpu())


def test_attention_block_mtnlg_shape_sampled_parity():
    """The benchmarked shape: h 20480, 128 heads (d = 160), t 8, one sequence of
    2048 tokens, weights N(0, 0.02), the same seeded inputs the benchmark uses.
    Checked at sampled positions, each computed by the oracle from its definition
    (attn_sampled): token rows of QKV, O, out, dQKV, dX; the probability rows of
    three heads at those tokens; 256 entries each of dWqkv and dWo; all of dbqkv
    and dbo."""
    c = gin.ATTN_MTNLG
    h, nh, t, L, T = c["h"], c["nh"], c["t"], c["seq_len"], c["tokens"]
    p, seed = 0.1, gin.DROPOUT_SEED
    dev = torch.device("cuda")
    w, X, dOut = gin.make_attn_inputs(h, T, device=dev)
    buf = mlp.AttnBuffers(T, h, nh, L, device=dev)
    mlp.attn_step(h, nh, t, L, p, seed, w, X, dOut, buf, accumulate=False)
    torch.cuda.synchronize()
    assert mlp.mlp_sync_status() == mlp.MLP_OK, mlp.last_error()

    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 1023, T - 1], rng.integers(0, T, 58)]))
    heads = [0, 61, nh - 1]
    n_e = 256
    rq = np.concatenate([[0, h - 1], rng.integers(0, h, n_e - 2)])
    cq = np.concatenate([[0, 3 * h - 1], rng.integers(0, 3 * h, n_e - 2)])
    ro = np.concatenate([[0, h - 1], rng.integers(0, h, n_e - 2)])
    co = np.concatenate([[0, h - 1], rng.integers(0, h, n_e - 2)])
    ridx = torch.from_numpy(rows).to(dev)
    got = {"QKV": to_f64(buf.QKV.index_select(0, ridx)), "O": to_f64(buf.O.index_select(0, ridx)),
           "out": to_f64(buf.out.index_select(0, ridx)), "dQKV": to_f64(buf.dQKV.index_select(0, ridx)),
           "dX": to_f64(buf.dX.index_select(0, ridx)),
           "dWqkv": to_f64(buf.dWqkv[torch.from_numpy(rq).to(dev), torch.from_numpy(cq).to(dev)]),
           "dWo": to_f64(buf.dWo[torch.from_numpy(ro).to(dev), torch.from_numpy(co).to(dev)]),
           "dbqkv": to_f64(buf.dbqkv), "dbo": to_f64(buf.dbo)}
    P_got = {j: to_f64(buf.P[0, j].index_select(0, ridx)) for j in heads}

    Wqkv = orc.Bf16Matrix(_bits(w[0]))
    Wo = orc.Bf16Matrix(_bits(w[2]))
    bqkv, bo = orc.bf16_to_f64(_bits(w[1])), orc.bf16_to_f64(_bits(w[3]))
    X64, d64 = orc.bf16_to_f64(_bits(X)), orc.bf16_to_f64(_bits(dOut))
    del buf, w
    ref = {mirror: ato.attn_sampled(X64, d64, Wqkv, bqkv, Wo, bo, nh, t, L, p, seed, rows, heads, (rq, cq), (ro, co),
                                    mirror=mirror)
           for mirror in (True, False)}
    gaps, errs = {}, {}
    for name in ("QKV", "O", "out", "dQKV", "dX"):
        e = rel_err(got[name], ref[True][name])
        errs[name] = e
        assert e <= BF16_TOL, ("mirror", name, e)
        e = rel_err(got[name], ref[False][name])
        gaps[name] = rel_err(ref[True][name], ref[False][name])
        assert e <= pure_bar(BF16_TOL, ref[False][name], ref[True][name]), ("pure", name, e, gaps[name])
    for j in heads:
        e = rel_err(P_got[j], ref[True]["P"][j])
        assert e <= BF16_TOL, ("mirror", "P", j, e)
        e = rel_err(P_got[j], ref[False]["P"][j])
        assert e <= pure_bar(BF16_TOL, ref[False]["P"][j], ref[True]["P"][j]), ("pure", "P", j, e)
    # causal: nothing above the diagonal; dropped outputs are the residual exactly
    for j in heads:
        for q, row in enumerate(rows):
            assert np.all(P_got[j][q, row + 1:] == 0), (j, row)
    keep = ref[True]["keep"]
    np.testing.assert_array_equal(got["out"][~keep], X64[rows][~keep])
    for name in ("dWqkv", "dWo", "dbqkv", "dbo"):
        bar = f32_bar(ref[False][name], ref[True][name])
        e = rel_err(got[name], ref[True][name])
        errs[name] = e
        gaps[name] = rel_err(ref[True][name], ref[False][name])
        assert e <= bar, ("mirror", name, e, bar)
        e = rel_err(got[name], ref[False][name])
        assert e <= pure_bar(bar, ref[False][name], ref[True][name]), ("pure", name, e)
    print("mtnlg-shape attention, max rel err vs mirror:", {k: f"{v:.2e}" for k, v in errs.items()},
          "oracle pure-vs-mirror:", {k: f"{v:.2e}" for k, v in gaps.items()})


def test_attention_rejects_bad_shapes():
    dev = torch.device("cuda")
    x = torch.empty(64, dtype=torch.bfloat16, device=dev)
    lib = mlp.load()
    ptrs = [x.data_ptr()] * 5
    # head size not a multiple of 8, and tokens not a multiple of seq_len
    assert lib.attn_fwd(96, 16, 1, 64, 32, 0.1, 1, 0, *ptrs, None, *([x.data_ptr()] * 5), None) == mlp.MLP_EINVAL
    assert lib.attn_fwd(128, 4, 1, 60, 32, 0.1, 1, 0, *ptrs, None, *([x.data_ptr()] * 5), None) == mlp.MLP_EINVAL


def test_attention_tile_scheduler_changes_no_bit():
    """The batched attention products skip the tiles above the causal diagonal, so
    the work per tile varies; the dynamic tile order balances it.  Results are
    bit-identical to the static order."""
    T, h, nh, t, L = 2048, 2048, 16, 8, 1024
    gen = torch.Generator().manual_seed(5)
    w = tuple(x.cuda() for x in _weights(h, gen, std=0.5 / np.sqrt(h)))
    X = torch.randn(T, h, generator=gen).to(torch.bfloat16).cuda()
    dOut = torch.randn(T, h, generator=gen).to(torch.bfloat16).cuda()
    res = []
    try:
        for mode in (0, 1, -1):
            mlp.mlp_set_tile_scheduler(mode)
            buf = mlp.AttnBuffers(T, h, nh, L)
            mlp.attn_step(h, nh, t, L, 0.1, 1234, w, X, dOut, buf, accumulate=False)
            torch.cuda.synchronize()
            assert mlp.mlp_sync_status() == mlp.MLP_OK, mlp.last_error()
            res.append({n: getattr(buf, n).clone() for n in ("QKV", "P", "O", "out", "dQKV", "dX", "dWqkv", "dbqkv",
                                                              "dWo", "dbo")})
    finally:
        mlp.mlp_set_tile_scheduler(-1)
    for r in res[1:]:
        for n in r:
            assert torch.equal(r[n], res[0][n]), n


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "unfused"])
def test_attention_wgrad_transposed_operands_change_no_bit(fused):
    """dWo and dWqkv reading transposed copies of dZ and X (K-major operands held in
    the dS workspace, before the core writes it and after the products read it)
    give, bit for bit, what they give reading dZ and X as MN-major operands; with
    either attention core.  The copies run only when asked for."""
    T, h, nh, t, L = 2048, 2048, 16, 8, 1024
    gen = torch.Generator().manual_seed(6)
    w = tuple(x.cuda() for x in _weights(h, gen, std=0.5 / np.sqrt(h)))
    X = torch.randn(T, h, generator=gen).to(torch.bfloat16).cuda()
    dOut = torch.randn(T, h, generator=gen).to(torch.bfloat16).cuda()
    res = []
    try:
        mlp.mlp_set_attn_fused(fused)
        for mode in (0, 1):
            mlp.mlp_set_wgrad_transpose(mode)
            buf = mlp.AttnBuffers(T, h, nh, L)
            tr = mlp.Trace(capacity=64)
            tr.start()
            mlp.attn_step(h, nh, t, L, 0.1, 1234, w, X, dOut, buf, accumulate=False)
            torch.cuda.synchronize()
            tr.stop()
            assert mlp.mlp_sync_status() == mlp.MLP_OK, mlp.last_error()
            copies = sum(1 for kind, _, _ in tr.entries if kind == 15)
            assert copies == (2 if mode == 1 else 0), (mode, copies)
            res.append({n: getattr(buf, n).clone() for n in ("out", "dQKV", "dX", "dWqkv", "dbqkv", "dWo", "dbo")})
    finally:
        mlp.mlp_set_wgrad_transpose(-1)
        mlp.mlp_set_attn_fused(True)
    for n in res[0]:
        assert torch.equal(res[1][n], res[0][n]), n


@pytest.mark.parametrize("T,h,nh,L", [
    (2048, 2048, 16, 1024),   # d = 128, two sequences
    (1088, 640, 4, 136),      # d = 160 (three 64-column atoms, the last half used), ragged 136-token sequences
    (384, 640, 8, 384),       # d = 80: a head size that is not a multiple of 64
])
def test_fused_core_agrees_with_unfused(T, h, nh, L):
    """The fused core (S on chip, two passes) and the three-launch core compute the
    same P and O: P within one bf16 step (its softmax sums run in another order),
    O, the block output and dQKV within the bf16 bar; P is exactly zero above the
    diagonal.  (Both cores are compared with the oracle in the parity tests.)"""
    gen = torch.Generator().manual_seed(9)
    w = tuple(x.cuda() for x in _weights(h, gen, std=0.5 / np.sqrt(h)))
    X = torch.randn(T, h, generator=gen).to(torch.bfloat16).cuda()
    dOut = torch.randn(T, h, generator=gen).to(torch.bfloat16).cuda()
    res = {}
    try:
        for fused in (False, True):
            mlp.mlp_set_attn_fused(fused)
            buf = mlp.AttnBuffers(T, h, nh, L)
            buf.P.fill_(float("nan"))       # the fused core must write every entry, zeros included
            mlp.attn_step(h, nh, 1, L, 0.1, 1234, w, X, dOut, buf, accumulate=False)
            torch.cuda.synchronize()
            assert mlp.mlp_sync_status() == mlp.MLP_OK, mlp.last_error()
            res[fused] = {n: to_f64(getattr(buf, n)) for n in ("P", "O", "out", "dQKV")}
    finally:
        mlp.mlp_set_attn_fused(True)
    Pf, Pu = res[True]["P"], res[False]["P"]
    assert np.all(np.isfinite(Pf))
    # one bf16 step of a value x is 2^(floor(log2|x|) - 7), at most 2^-7 |x|
    steps = np.abs(Pf - Pu) / (2.0 ** -7 * np.maximum(np.abs(Pu), np.abs(Pf)) + 1e-38)
    assert steps.max() <= 1.0, steps.max()
    for i in range(Pf.shape[0]):
        for j in range(Pf.shape[1]):
            assert np.all(np.triu(Pf[i, j], k=1) == 0)
    for n in ("O", "out", "dQKV"):
        assert rel_err(res[True][n], res[False][n]) <= BF16_TOL, n
