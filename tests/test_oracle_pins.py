"""Pins of the CPU oracle against facts that do not come from the oracle itself.

* bf16 rounding against torch's fp32->bf16 conversion (round-to-nearest-even);
* GeLU against its closed-form identities and torch's tanh-approximate GeLU;
* the dropout mask against an independent big-int SplitMix64 stream and the
  generator's published test vector (tests/golden/);
* the whole block (t = 1) against torch fp64 modules with autograd, a library
  special case of the tensor-sliced block;
* slice invariance (the g / f sums over row-split partial products, STRONGHOLD
  slides items 7-8), accumulation invariance (gradient accumulation over
  micro-batches, MT-NLG summary page, Key points), central finite differences,
  and agreement of the sampled evaluators with the full oracle.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import mlp_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
M64 = (1 << 64) - 1


def _rand(shape, std, rng):
    return orc.round_bf16(rng.standard_normal(shape) * std)


def _block_inputs(T, h, F, rng, std_w=0.02):
    X = _rand((T, h), 1.0, rng)
    A = _rand((h, F), std_w, rng)
    a = _rand((F,), std_w, rng)
    B = _rand((F, h), std_w, rng)
    b = _rand((h,), std_w, rng)
    dO = _rand((T, h), 1.0, rng)
    return X, A, a, B, b, dO


# --------------------------------------------------------------------------- bf16
def test_round_bf16_matches_torch_rne():
    rng = np.random.default_rng(1)
    x32 = (rng.standard_normal(200000) * 10.0 ** rng.integers(-30, 30, 200000)).astype(np.float32)
    # exact ties: bf16 values plus half a bf16 ulp (low 16 bits = 0x8000)
    ties = ((rng.integers(0, 0x7F00, 5000, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    x32 = np.concatenate([x32, ties, -ties, np.float32([0.0, 1.0, -2.5, 1e-40, -3e-39])])
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.f64_to_bf16_bits(x32.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_bf16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = orc.bf16_to_f64(bits)
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    # every finite pattern survives a round trip
    np.testing.assert_array_equal(orc.f64_to_bf16_bits(got[finite]) & 0x7FFF, bits[finite] & 0x7FFF)


# --------------------------------------------------------------------------- GeLU
def test_gelu_identities():
    x = np.linspace(-12, 12, 10001)
    assert orc.gelu(0.0) == 0.0
    assert orc.gelu_prime(0.0) == 0.5
    # tanh is odd, so gelu(x) - gelu(-x) = x
    np.testing.assert_allclose(orc.gelu(x) - orc.gelu(-x), x, rtol=0, atol=1e-14)
    # limits: gelu(x) -> x for large x, -> 0 for very negative x
    assert abs(orc.gelu(12.0) - 12.0) < 1e-12 and abs(orc.gelu(-12.0)) < 1e-12
    # the tanh form approximates x * Phi(x) (erf GeLU) closely
    erf_gelu = np.array([0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0))) for v in x])
    assert np.max(np.abs(orc.gelu(x) - erf_gelu)) < 1e-3


def test_gelu_matches_torch_tanh_gelu():
    x = np.linspace(-20, 20, 40001)
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    np.testing.assert_allclose(orc.gelu(x), ref, rtol=1e-14, atol=1e-15)
    xt = torch.from_numpy(x).requires_grad_(True)
    torch.nn.functional.gelu(xt, approximate="tanh").sum().backward()
    np.testing.assert_allclose(orc.gelu_prime(x), xt.grad.numpy(), rtol=1e-13, atol=1e-14)


def test_gelu_prime_central_difference():
    x = np.linspace(-8, 8, 3201)
    eps = 1e-5
    fd = (orc.gelu(x + eps) - orc.gelu(x - eps)) / (2 * eps)
    np.testing.assert_allclose(orc.gelu_prime(x), fd, rtol=0, atol=1e-9)


# --------------------------------------------------------------------------- mask
def _bigint_splitmix_stream(seed, n):
    """Independent restatement: a stateful stream, big-int arithmetic mod 2^64."""
    s = seed & M64
    out = []
    for _ in range(n):
        s = (s + 0x9E3779B97F4A7C15) & M64
        z = s
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        out.append(z ^ (z >> 31))
    return out


def test_splitmix64_published_vector():
    rows = []
    with open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt")) as fh:
        for line in fh:
            if line.strip() and not line.startswith("#"):
                rows.append(tuple(int(v) for v in line.split()))
    assert len(rows) == 5
    for seed, n, val in rows:
        assert int(orc.splitmix64(seed, np.array([n]))[0]) == val
        assert _bigint_splitmix_stream(seed, n + 1)[n] == val


@pytest.mark.parametrize("seed", [0, 1234, 2**63 + 12345, M64])
def test_splitmix64_matches_bigint_stream(seed):
    n = 3000
    ref = _bigint_splitmix_stream(seed, n)
    got = orc.splitmix64(seed, np.arange(n))
    assert [int(v) for v in got] == ref


def test_dropout_mask_definition_and_statistics():
    T, h, p, seed, off = 37, 24, 0.1, 1234, 5
    keep = orc.dropout_keep(T, h, p, seed, off)
    thr = orc.keep_threshold(p)
    assert thr == 429496736                       # 0.1f * 2^32 is exactly this integer
    stream = _bigint_splitmix_stream(seed, (off + T) * h)
    for tok in range(T):
        for c in range(h):
            e = (off + tok) * h + c
            assert keep[tok, c] == ((stream[e] >> 32) >= thr)
    # kept fraction within 5 sigma of 1 - p on a large mask
    big = orc.dropout_keep(4096, 1024, p, seed)
    n = big.size
    assert abs(big.mean() - (1 - p)) < 5 * math.sqrt(p * (1 - p) / n)
    assert orc.dropout_keep(64, 64, 0.0, seed).all()
    # rows= selects the same entries as the full mask
    np.testing.assert_array_equal(orc.dropout_keep(T, h, p, seed, off, rows=[3, 30]), keep[[3, 30]])


# --------------------------------------------------------------------------- block
def _torch_block(X, A, a, B, b, keep, p, dO):
    """The t = 1 block written with torch fp64 library modules, gradients by autograd."""
    tX = torch.from_numpy(X).requires_grad_(True)
    tA = torch.from_numpy(A).requires_grad_(True)
    ta = torch.from_numpy(a).requires_grad_(True)
    tB = torch.from_numpy(B).requires_grad_(True)
    tb = torch.from_numpy(b).requires_grad_(True)
    lin1 = torch.nn.functional.linear(tX, tA.t(), ta)
    y = torch.nn.functional.gelu(lin1, approximate="tanh")
    z = torch.nn.functional.linear(y, tB.t(), tb)
    m = torch.from_numpy(keep.astype(np.float64)) / (1.0 - float(np.float32(p)))
    o = tX + z * m
    o.backward(torch.from_numpy(dO))
    return {"O": o.detach().numpy(), "dX": tX.grad.numpy(), "dA": tA.grad.numpy(),
            "da": ta.grad.numpy(), "dB": tB.grad.numpy(), "db": tb.grad.numpy()}


@pytest.mark.parametrize("t", [1, 2, 4])
def test_block_matches_torch_autograd(t):
    rng = np.random.default_rng(7)
    T, h, F, p = 19, 16, 64, 0.25
    X, A, a, B, b, dO = _block_inputs(T, h, F, rng, std_w=0.3)
    fw = orc.mlp_fwd(X, A, a, B, b, t, p, seed=99, token_offset=3)
    bw = orc.mlp_bwd(dO, X, A, B, fw["U"], fw["Y"], fw["keep"], t, p)
    ref = _torch_block(X, A, a, B, b, fw["keep"], p, dO)
    for key in ("O",):
        np.testing.assert_allclose(fw[key], ref[key], rtol=1e-12, atol=1e-12)
    for key in ("dX", "dA", "da", "dB", "db"):
        np.testing.assert_allclose(bw[key], ref[key], rtol=1e-12, atol=1e-12)


def test_slice_invariance():
    rng = np.random.default_rng(3)
    T, h, F = 33, 32, 128
    X, A, a, B, b, dO = _block_inputs(T, h, F, rng, std_w=0.2)
    outs = []
    for t in (1, 2, 4, 8):
        fw = orc.mlp_fwd(X, A, a, B, b, t, 0.1, 1234)
        bw = orc.mlp_bwd(dO, X, A, B, fw["U"], fw["Y"], fw["keep"], t, 0.1)
        outs.append((fw, bw))
    f1, b1 = outs[0]
    for fw, bw in outs[1:]:
        np.testing.assert_array_equal(fw["keep"], f1["keep"])
        for key in ("Z", "O"):
            np.testing.assert_allclose(fw[key], f1[key], rtol=1e-12, atol=1e-13)
        for key in ("dX", "dA", "da", "dB", "db"):
            np.testing.assert_allclose(bw[key], b1[key], rtol=1e-12, atol=1e-13)


def test_accumulation_invariance():
    rng = np.random.default_rng(5)
    T, h, F, t, k, p = 16, 16, 64, 2, 3, 0.2
    X, A, a, B, b, _ = _block_inputs(T * k, h, F, rng, std_w=0.2)
    dO = _rand((T * k, h), 1.0, rng)
    whole_f = orc.mlp_fwd(X, A, a, B, b, t, p, 1234, token_offset=0)
    whole = orc.mlp_bwd(dO, X, A, B, whole_f["U"], whole_f["Y"], whole_f["keep"], t, p)
    acc = {key: 0.0 for key in ("dA", "da", "dB", "db")}
    for j in range(k):
        rows = slice(j * T, (j + 1) * T)
        fw = orc.mlp_fwd(X[rows], A, a, B, b, t, p, 1234, token_offset=j * T)
        np.testing.assert_allclose(fw["O"], whole_f["O"][rows], rtol=1e-13, atol=1e-14)
        bw = orc.mlp_bwd(dO[rows], X[rows], A, B, fw["U"], fw["Y"], fw["keep"], t, p)
        np.testing.assert_allclose(bw["dX"], whole["dX"][rows], rtol=1e-13, atol=1e-14)
        for key in acc:
            acc[key] = acc[key] + bw[key]
    for key in acc:
        np.testing.assert_allclose(acc[key], whole[key], rtol=1e-12, atol=1e-13)


def test_finite_differences():
    """Central differences of L = sum(O * G) with the mask held fixed."""
    rng = np.random.default_rng(11)
    T, h, F, t, p, seed = 4, 8, 32, 2, 0.25, 77
    X, A, a, B, b, G = _block_inputs(T, h, F, rng, std_w=0.5)

    def loss(X_, A_, a_, B_, b_):
        return float(np.sum(orc.mlp_fwd(X_, A_, a_, B_, b_, t, p, seed)["O"] * G))

    fw = orc.mlp_fwd(X, A, a, B, b, t, p, seed)
    assert 0 < fw["keep"].sum() < fw["keep"].size      # both kept and dropped entries
    bw = orc.mlp_bwd(G, X, A, B, fw["U"], fw["Y"], fw["keep"], t, p)
    args = [X, A, a, B, b]
    names = ["dX", "dA", "da", "dB", "db"]
    eps = 1e-6
    for which, name in enumerate(names):
        base = args[which]
        num = np.empty_like(base)
        for idx in np.ndindex(base.shape):
            plus = [v.copy() for v in args]
            minus = [v.copy() for v in args]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            num[idx] = (loss(*plus) - loss(*minus)) / (2 * eps)
        err = np.max(np.abs(num - bw[name])) / max(np.max(np.abs(bw[name])), 1e-30)
        assert err <= 1e-6, (name, err)


def test_mirror_mode_rounds_at_storage_points():
    rng = np.random.default_rng(9)
    T, h, F, t, p = 32, 32, 128, 2, 0.1
    X, A, a, B, b, dO = _block_inputs(T, h, F, rng)
    fp = orc.mlp_fwd(X, A, a, B, b, t, p, 1234)
    fm = orc.mlp_fwd(X, A, a, B, b, t, p, 1234, mirror=True)
    bm = orc.mlp_bwd(dO, X, A, B, fm["U"], fm["Y"], fm["keep"], t, p, mirror=True)
    for arr in (fm["U"], fm["Y"], fm["O"], bm["dZ"], bm["dU"], bm["dX"]):
        np.testing.assert_array_equal(orc.round_bf16(arr), arr)
    # Y is the rounded GeLU of the unrounded pre-activation, not of the rounded U
    np.testing.assert_array_equal(fm["Y"], orc.round_bf16(orc.gelu(fp["U"])))
    for key in ("O",):
        rel = np.max(np.abs(fm[key] - fp[key])) / np.max(np.abs(fp[key]))
        assert rel < 1e-2


def test_sampled_evaluators_match_full_oracle():
    rng = np.random.default_rng(13)
    T, h, F, t, p, off = 40, 24, 96, 3, 0.1, 7
    X, A, a, B, b, dO = _block_inputs(T, h, F, rng)
    for mirror in (False, True):
        fw = orc.mlp_fwd(X, A, a, B, b, t, p, 1234, token_offset=off, mirror=mirror)
        bw = orc.mlp_bwd(dO, X, A, B, fw["U"], fw["Y"], fw["keep"], t, p, mirror=mirror)
        rows = [0, 5, 39]
        for tt in (1, t):
            r = orc.rows_fwd_bwd(rows, X, dO, A, a, B, b, tt, p, 1234, token_offset=off, mirror=mirror)
            np.testing.assert_allclose(r["O"], fw["O"][rows], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(r["dX"], bw["dX"][rows], rtol=1e-12, atol=1e-12)
            for key in ("dU", "U", "Y"):
                src = bw if key == "dU" else fw
                np.testing.assert_allclose(r[key], src[key][rows], rtol=1e-12, atol=1e-12)
        # the lazily decoded bf16 form gives identical values
        Ab = orc.Bf16Matrix(orc.f64_to_bf16_bits(A))
        Bb = orc.Bf16Matrix(orc.f64_to_bf16_bits(B))
        r2 = orc.rows_fwd_bwd(rows, X, dO, Ab, a, Bb, b, t, p, 1234, token_offset=off, mirror=mirror)
        np.testing.assert_array_equal(r2["O"], r["O"])
        np.testing.assert_array_equal(r2["dX"], r["dX"])
        dZ = orc.full_dZ(dO, p, 1234, token_offset=off, mirror=mirror)
        np.testing.assert_array_equal(dZ, bw["dZ"])
        ri = np.array([0, 95, 50, 7])
        ci = np.array([0, 23, 11, 7])
        np.testing.assert_allclose(orc.wgrad_dB_entries(ri, ci, X, A, a, dZ, mirror),
                                   bw["dB"][ri, ci], rtol=1e-12, atol=1e-13)
        ri2 = np.array([0, 23, 11, 5])
        ci2 = np.array([0, 95, 50, 31])
        np.testing.assert_allclose(orc.wgrad_dA_entries(ri2, ci2, X, A, a, B, dZ, mirror),
                                   bw["dA"][ri2, ci2], rtol=1e-12, atol=1e-13)
        dUc = orc.columns_dU(np.array([3, 60]), X, A, a, B, dZ, mirror)
        np.testing.assert_allclose(dUc.sum(axis=0), bw["da"][[3, 60]], rtol=1e-12, atol=1e-13)


def test_planted_mistakes_are_caught():
    """A dropped bias, a wrong GeLU' sign or a transposed operand breaks the autograd pin."""
    rng = np.random.default_rng(17)
    T, h, F, p = 8, 8, 32, 0.2
    X, A, a, B, b, dO = _block_inputs(T, h, F, rng, std_w=0.3)
    fw = orc.mlp_fwd(X, A, a, B, b, 1, p, 5)
    ref = _torch_block(X, A, a, B, b, fw["keep"], p, dO)
    # dropped bias b
    bad_O = X + np.where(fw["keep"], fw["Z"] * orc.dropout_scale(p), 0.0)
    assert np.max(np.abs(bad_O - ref["O"])) > 1e-6
    # wrong sign in GeLU'
    th = np.tanh(orc.SQRT_2_OVER_PI * (fw["U"] + orc.GELU_CUBIC * fw["U"] ** 3))
    bad_gp = 0.5 * (1 + th) - 0.5 * fw["U"] * (1 - th * th) * orc.SQRT_2_OVER_PI
    dZ = np.where(fw["keep"], dO * orc.dropout_scale(p), 0.0)
    bad_dA = X.T @ ((dZ @ B.T) * bad_gp)
    assert np.max(np.abs(bad_dA - ref["dA"])) > 1e-6
    # transposed operand in dB
    bad_dB = (dZ.T @ fw["Y"]).T if F == h else fw["Y"].T @ dZ[::-1]
    assert np.max(np.abs(bad_dB - ref["dB"])) > 1e-6
