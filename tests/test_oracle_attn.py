"""Pins of the attention-block oracle: torch's causal scaled_dot_product_attention
with autograd in float64 (a library routine), slice invariance over the head split,
and central finite differences."""
import numpy as np
import pytest
import torch

from oracle import attn_oracle as ato
from oracle import mlp_oracle as orc


def _inputs(T, h, rng, std=0.3):
    X = orc.round_bf16(rng.standard_normal((T, h)))
    Wqkv = orc.round_bf16(rng.standard_normal((h, 3 * h)) * std)
    bqkv = orc.round_bf16(rng.standard_normal(3 * h) * std)
    Wo = orc.round_bf16(rng.standard_normal((h, h)) * std)
    bo = orc.round_bf16(rng.standard_normal(h) * std)
    dOut = orc.round_bf16(rng.standard_normal((T, h)))
    return X, Wqkv, bqkv, Wo, bo, dOut


def _torch_block(X, Wqkv, bqkv, Wo, bo, keep, p, dOut, nh, seq_len):
    T, h = X.shape
    d = h // nh
    n_seq = T // seq_len
    ts = [torch.from_numpy(a.copy()).requires_grad_(True) for a in (X, Wqkv, bqkv, Wo, bo)]
    tX, tW, tb, tWo, tbo = ts
    qkv = torch.nn.functional.linear(tX, tW.t(), tb)

    def heads(x):
        return x.reshape(n_seq, seq_len, nh, d).transpose(1, 2)

    q, k, v = heads(qkv[:, :h]), heads(qkv[:, h:2 * h]), heads(qkv[:, 2 * h:])
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    o = o.transpose(1, 2).reshape(T, h)
    z = torch.nn.functional.linear(o, tWo.t(), tbo)
    m = torch.from_numpy(keep.astype(np.float64)) / (1.0 - float(np.float32(p)))
    out = tX + z * m
    out.backward(torch.from_numpy(dOut))
    return {"out": out.detach().numpy(), "O": o.detach().numpy(), "dX": tX.grad.numpy(), "dWqkv": tW.grad.numpy(),
            "dbqkv": tb.grad.numpy(), "dWo": tWo.grad.numpy(), "dbo": tbo.grad.numpy()}


@pytest.mark.parametrize("t", [1, 2, 4])
def test_block_matches_torch_sdpa_autograd(t):
    rng = np.random.default_rng(3)
    T, h, nh, seq_len, p = 24, 16, 4, 12, 0.25
    X, Wqkv, bqkv, Wo, bo, dOut = _inputs(T, h, rng)
    fw = ato.attn_fwd(X, Wqkv, bqkv, Wo, bo, nh, t, seq_len, p, seed=5, token_offset=2)
    bw = ato.attn_bwd(dOut, X, Wqkv, Wo, fw["QKV"], fw["P"], fw["O"], fw["keep"], nh, t, seq_len, p)
    ref = _torch_block(X, Wqkv, bqkv, Wo, bo, fw["keep"], p, dOut, nh, seq_len)
    np.testing.assert_allclose(fw["O"], ref["O"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(fw["out"], ref["out"], rtol=1e-11, atol=1e-12)
    for key in ("dX", "dWqkv", "dbqkv", "dWo", "dbo"):
        np.testing.assert_allclose(bw[key], ref[key], rtol=1e-10, atol=1e-11)


def test_probabilities_are_causal_and_normalised():
    rng = np.random.default_rng(4)
    X, Wqkv, bqkv, Wo, bo, _ = _inputs(16, 8, rng)
    fw = ato.attn_fwd(X, Wqkv, bqkv, Wo, bo, 2, 1, 8, 0.1, 1)
    P = fw["P"]
    np.testing.assert_allclose(P.sum(axis=-1), 1.0, rtol=1e-13)
    assert np.all(np.triu(P, k=1) == 0)
    assert np.all(P[..., 0, 0] == 1.0)               # the first query sees only itself


def test_finite_differences():
    rng = np.random.default_rng(8)
    T, h, nh, t, seq_len, p, seed = 6, 4, 2, 2, 3, 0.25, 11
    X, Wqkv, bqkv, Wo, bo, G = _inputs(T, h, rng, std=0.5)

    def loss(X_, W_, b_, Wo_, bo_):
        return float(np.sum(ato.attn_fwd(X_, W_, b_, Wo_, bo_, nh, t, seq_len, p, seed)["out"] * G))

    fw = ato.attn_fwd(X, Wqkv, bqkv, Wo, bo, nh, t, seq_len, p, seed)
    assert 0 < fw["keep"].sum() < fw["keep"].size
    bw = ato.attn_bwd(G, X, Wqkv, Wo, fw["QKV"], fw["P"], fw["O"], fw["keep"], nh, t, seq_len, p)
    args = [X, Wqkv, bqkv, Wo, bo]
    names = ["dX", "dWqkv", "dbqkv", "dWo", "dbo"]
    eps = 1e-6
    for which, name in enumerate(names):
        num = np.empty_like(args[which])
        for idx in np.ndindex(args[which].shape):
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            num[idx] = (loss(*plus) - loss(*minus)) / (2 * eps)
        err = np.max(np.abs(num - bw[name])) / max(np.max(np.abs(bw[name])), 1e-30)
        assert err <= 1e-6, (name, err)


def test_mirror_mode_rounds_at_storage_points():
    rng = np.random.default_rng(9)
    X, Wqkv, bqkv, Wo, bo, dOut = _inputs(16, 16, rng)
    fm = ato.attn_fwd(X, Wqkv, bqkv, Wo, bo, 4, 2, 8, 0.1, 1, mirror=True)
    bm = ato.attn_bwd(dOut, X, Wqkv, Wo, fm["QKV"], fm["P"], fm["O"], fm["keep"], 4, 2, 8, 0.1, mirror=True)
    for arr in (fm["QKV"], fm["P"], fm["O"], fm["out"], bm["dZ"], bm["dO"], bm["dQKV"], bm["dX"]):
        np.testing.assert_array_equal(orc.round_bf16(arr), arr)


def test_planted_mistakes_are_caught():
    """A dropped 1/sqrt(d), a causal mask one key too wide, a sign error in the
    softmax gradient or Q/K taken from the wrong block all break the torch pin."""
    rng = np.random.default_rng(23)
    T, h, nh, t, L, p, seed = 16, 8, 2, 1, 8, 0.2, 3
    X, Wqkv, bqkv, Wo, bo, dOut = _inputs(T, h, rng, std=0.5)
    fw = ato.attn_fwd(X, Wqkv, bqkv, Wo, bo, nh, t, L, p, seed)
    ref = _torch_block(X, Wqkv, bqkv, Wo, bo, fw["keep"], p, dOut, nh, L)
    d = h // nh
    QKV = fw["QKV"]

    def head_out(scale, wide, q_block=0, k_block=1):
        O = np.zeros((T, h))
        for s in range(T // L):
            rows = slice(s * L, (s + 1) * L)
            for j in range(nh):
                q = QKV[rows, q_block * h + j * d:q_block * h + (j + 1) * d]
                k = QKV[rows, k_block * h + j * d:k_block * h + (j + 1) * d]
                v = QKV[rows, 2 * h + j * d:2 * h + (j + 1) * d]
                mask = np.tril(np.ones((L, L), dtype=bool), k=1 if wide else 0)
                sc = np.where(mask, (q @ k.T) * scale, -np.inf)
                e = np.exp(sc - sc.max(axis=1, keepdims=True))
                O[rows, j * d:(j + 1) * d] = (e / e.sum(axis=1, keepdims=True)) @ v
        return O

    np.testing.assert_allclose(head_out(1 / np.sqrt(d), False), ref["O"], rtol=1e-10, atol=1e-12)
    assert np.max(np.abs(head_out(1.0, False) - ref["O"])) > 1e-6             # dropped 1/sqrt(d)
    assert np.max(np.abs(head_out(1 / np.sqrt(d), True) - ref["O"])) > 1e-6   # mask one key too wide
    assert np.max(np.abs(head_out(1 / np.sqrt(d), False, 1, 0) - ref["O"])) > 1e-6  # Q and K swapped
    # softmax gradient with the sign of the row sum flipped
    bw = ato.attn_bwd(dOut, X, Wqkv, Wo, QKV, fw["P"], fw["O"], fw["keep"], nh, t, L, p)
    np.testing.assert_allclose(bw["dWqkv"], ref["dWqkv"], rtol=1e-10, atol=1e-11)
    dQ = np.zeros((T, h))
    for s in range(T // L):
        rows = slice(s * L, (s + 1) * L)
        for j in range(nh):
            pr = fw["P"][s, j]
            do = bw["dO"][rows, j * d:(j + 1) * d]
            dp = do @ QKV[rows, 2 * h + j * d:2 * h + (j + 1) * d].T
            ds = pr * (dp + (dp * pr).sum(axis=1, keepdims=True)) / np.sqrt(d)
            dQ[rows, j * d:(j + 1) * d] = ds @ QKV[rows, h + j * d:h + (j + 1) * d]
    bad_dWq = X.T @ dQ
    assert np.max(np.abs(bad_dWq - ref["dWqkv"][:, :h])) > 1e-6


@pytest.mark.parametrize("mirror", [False, True])
def test_sampled_evaluator_matches_full_oracle(mirror):
    """attn_sampled (column-blocked weights, sampled entries) equals attn_fwd +
    attn_bwd at every sampled position, also with the weights given as raw bf16
    bits (Bf16Matrix), on a shape with two sequences and two slices."""
    rng = np.random.default_rng(5)
    T, h, nh, t, L, p = 48, 32, 4, 2, 24, 0.2
    X, Wqkv, bqkv, Wo, bo, dOut = _inputs(T, h, rng)
    fw = ato.attn_fwd(X, Wqkv, bqkv, Wo, bo, nh, t, L, p, 9, token_offset=3, mirror=mirror)
    bw = ato.attn_bwd(dOut, X, Wqkv, Wo, fw["QKV"], fw["P"], fw["O"], fw["keep"], nh, t, L, p, mirror=mirror)
    rows = np.array([0, 5, 23, 24, 47])
    heads = [0, 3]
    rq, cq = np.array([0, 31, 7]), np.array([0, 95, 50])
    ro, co = np.array([1, 31]), np.array([0, 31])
    for wq, wo in ((Wqkv, Wo), (orc.Bf16Matrix(orc.f64_to_bf16_bits(Wqkv)), orc.Bf16Matrix(orc.f64_to_bf16_bits(Wo)))):
        s = ato.attn_sampled(X, dOut, wq, bqkv, wo, bo, nh, t, L, p, 9, rows, heads, (rq, cq), (ro, co),
                             token_offset=3, mirror=mirror, col_block=5)
        ref = {"QKV": fw["QKV"][rows], "O": fw["O"][rows], "out": fw["out"][rows], "dQKV": bw["dQKV"][rows],
               "dX": bw["dX"][rows], "dWqkv": bw["dWqkv"][rq, cq], "dWo": bw["dWo"][ro, co], "dbqkv": bw["dbqkv"],
               "dbo": bw["dbo"]}
        for key, r in ref.items():
            np.testing.assert_allclose(s[key], r, rtol=1e-12, atol=1e-12, err_msg=key)
        np.testing.assert_array_equal(s["keep"], fw["keep"][rows])
        for j in heads:
            np.testing.assert_allclose(s["P"][j], fw["P"][rows // L, j, rows % L], rtol=1e-12, atol=1e-14)
