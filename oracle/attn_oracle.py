"""CPU oracle of the tensor-sliced self-attention block (test infrastructure only).

The pages describe the MT-NLG model as a left-to-right transformer decoder with 128
attention heads, hidden size 20480, trained with Megatron "tensor slicing" inside a
node (jiqizhixin article on MT-NLG; "Using DeepSpeed and Megatron to Train
Megatron-Turing NLG 530B", Summary).  They give the split only for the MLP (A
column-wise, B row-wise, operators f and g: "STRONGHOLD ..." slides, items 7-8).
Reading for attention, mirroring that split: the fused QKV projection is split
column-wise by heads (slice i owns heads [i*nh/t, (i+1)*nh/t) and the matching
columns of the Q, K and V blocks), each head's attention is local to its slice,
and the output projection Wo is split row-wise with the partial products summed
over slices (operator g), followed by bias, dropout and residual as in the MLP
block.  Attention is causal (left-to-right decoder) within each sequence of
``seq_len`` tokens; no dropout is applied to the attention probabilities (the pages
name dropout only on the block output).

Layouts: X [T, h]; Wqkv [h, 3h] = [Wq | Wk | Wv] with head j of each block at
columns j*d .. (j+1)*d (d = h / nh); bqkv [3h]; Wo [h, h] (rows j*d .. belong to
head j); bo [h].  T = n_seq * seq_len tokens, sequence s = rows s*seq_len ...

Forward (float64; ``mirror`` additionally rounds to bf16 where the GPU stores bf16:
QKV, P, O, out, and in the backward dZ, dO, dS, dQKV, dX):
    QKV_i = X Wqkv[:, cols_i] + bqkv[cols_i]              (column split by heads)
    per sequence and head:  S = Q K^T / sqrt(d), masked to keys <= query
                            P = softmax(S),  O_head = P V
    Z = sum_i O[:, rows_i] Wo[rows_i, :]                  (row split, operator g)
    out = R + dropout(Z + bo)            (the MLP block's mask and scaling)
Backward (loss L = sum out * dOut):
    dZ = dOut m / (1-p);  dbo = sum dZ;  dWo = O^T dZ;  dO = dZ Wo^T
    per sequence and head:  dV = P^T dO;  dP = dO V^T;
                            dS = P (dP - rowsum(dP P)) / sqrt(d)
                            dQ = dS K;  dK = dS^T Q
    dWqkv = X^T dQKV;  dbqkv = sum dQKV;  dX = dOut + dQKV Wqkv^T   (operator f)

Pinned by tests/test_oracle_attn.py against torch's scaled_dot_product_attention
and autograd (float64), slice invariance and central finite differences.
"""
from __future__ import annotations

import math

import numpy as np

from .mlp_oracle import dropout_keep, dropout_scale, round_bf16


def _rb(x, mirror):
    return round_bf16(x) if mirror else x


def _slice_cols(h, t, i):
    """Columns of slice i within one of the Q, K, V blocks (and rows of Wo)."""
    w = h // t
    return slice(i * w, (i + 1) * w)


def attn_fwd(X, Wqkv, bqkv, Wo, bo, nh, t, seq_len, p, seed, token_offset=0, R=None, mirror=False):
    T, h = X.shape
    assert h % nh == 0 and nh % t == 0 and T % seq_len == 0
    d = h // nh
    n_seq = T // seq_len
    R = X if R is None else R
    QKV = np.empty((T, 3 * h))
    for i in range(t):                              # column split of the QKV projection
        for blk in range(3):
            cs = _slice_cols(h, t, i)
            cols = slice(blk * h + cs.start, blk * h + cs.stop)
            QKV[:, cols] = _rb(X @ Wqkv[:, cols] + bqkv[cols], mirror)
    P = np.zeros((n_seq, nh, seq_len, seq_len))
    O = np.empty((T, h))
    causal = np.tril(np.ones((seq_len, seq_len), dtype=bool))
    for s in range(n_seq):
        rows = slice(s * seq_len, (s + 1) * seq_len)
        for j in range(nh):
            q = QKV[rows, j * d:(j + 1) * d]
            k = QKV[rows, h + j * d:h + (j + 1) * d]
            v = QKV[rows, 2 * h + j * d:2 * h + (j + 1) * d]
            sc = np.where(causal, (q @ k.T) / math.sqrt(d), -np.inf)
            e = np.exp(sc - sc.max(axis=1, keepdims=True))
            pr = _rb(e / e.sum(axis=1, keepdims=True), mirror)
            P[s, j] = pr
            O[rows, j * d:(j + 1) * d] = pr @ v
    O = _rb(O, mirror)
    Z = np.zeros((T, h))
    for i in range(t):                              # row split of Wo, summed over slices
        rs = _slice_cols(h, t, i)
        Z += O[:, rs] @ Wo[rs, :]
    keep = dropout_keep(T, h, p, seed, token_offset)
    out = R + np.where(keep, (Z + bo) * dropout_scale(p), 0.0)
    return {"QKV": QKV, "P": P, "O": O, "Z": Z, "keep": keep, "out": _rb(out, mirror)}


def attn_bwd(dOut, X, Wqkv, Wo, QKV, P, O, keep, nh, t, seq_len, p, mirror=False, residual_is_input=True):
    T, h = X.shape
    d = h // nh
    n_seq = T // seq_len
    dZ = _rb(np.where(keep, dOut * dropout_scale(p), 0.0), mirror)
    dbo = dZ.sum(axis=0)
    dWo = np.empty_like(Wo)
    dO = np.zeros((T, h))
    for i in range(t):
        rs = _slice_cols(h, t, i)
        dWo[rs, :] = O[:, rs].T @ dZ
        dO[:, rs] = dZ @ Wo[rs, :].T
    dO = _rb(dO, mirror)
    dQKV = np.empty((T, 3 * h))
    for s in range(n_seq):
        rows = slice(s * seq_len, (s + 1) * seq_len)
        for j in range(nh):
            qc = slice(j * d, (j + 1) * d)
            kc = slice(h + j * d, h + (j + 1) * d)
            vc = slice(2 * h + j * d, 2 * h + (j + 1) * d)
            pr = P[s, j]
            do = dO[rows, qc]
            dQKV[rows, vc] = pr.T @ do
            dp = do @ QKV[rows, vc].T
            delta = (dp * pr).sum(axis=1, keepdims=True)
            ds = _rb(pr * (dp - delta) / math.sqrt(d), mirror)
            dQKV[rows, qc] = ds @ QKV[rows, kc]
            dQKV[rows, kc] = ds.T @ QKV[rows, qc]
    dQKV = _rb(dQKV, mirror)
    dWqkv = X.T @ dQKV
    dbqkv = dQKV.sum(axis=0)
    dX = _rb((dOut if residual_is_input else 0.0) + dQKV @ Wqkv.T, mirror)
    return {"dZ": dZ, "dO": dO, "dQKV": dQKV, "dX": dX, "dWqkv": dWqkv, "dbqkv": dbqkv, "dWo": dWo, "dbo": dbo}


# ----------------------------------------------------------------------------
# Sampled evaluation for shapes whose full float64 weight gradients do not fit in
# host memory (the MT-NLG layer shape: dWqkv alone would be 10 GB).  The same
# steps as attn_fwd / attn_bwd, in the same order and roundings; the weights are
# read a column (or row) block at a time, so they may be given as
# mlp_oracle.Bf16Matrix, and only the requested entries of the weight gradients
# are formed.  Every token's Q, K, V and every head's attention are still
# computed, because an output row of the block depends on all of them.
# ----------------------------------------------------------------------------
def attn_sampled(X, dOut, Wqkv, bqkv, Wo, bo, nh, t, seq_len, p, seed, rows, heads, wqkv_idx, wo_idx,
                 token_offset=0, mirror=False, col_block=2560):
    """Outputs of one forward + backward at sampled positions (residual R = X).

    rows      token rows (global indices) of QKV, O, out, dQKV, dX, and of P
    heads     heads whose probability rows P[seq(row), head, row, :] are returned
    wqkv_idx  (r, c) index arrays of the dWqkv entries to form; wo_idx likewise for dWo
    Returns a dict: QKV, O, out, dQKV, dX [len(rows), ...]; P {head: [len(rows), seq_len]};
    dWqkv, dWo (the requested entries); dbqkv, dbo (whole); keep [len(rows), h].
    """
    T, h = X.shape
    assert h % nh == 0 and nh % t == 0 and T % seq_len == 0
    d = h // nh
    n_seq = T // seq_len
    rows = np.asarray(rows)
    # forward projection, every token: slice i's columns of the Q, K and V blocks
    QKV = np.empty((T, 3 * h))
    for i in range(t):
        cs = _slice_cols(h, t, i)
        for blk in range(3):
            for c0 in range(cs.start, cs.stop, col_block):
                cols = slice(blk * h + c0, blk * h + min(c0 + col_block, cs.stop))
                QKV[:, cols] = _rb(X @ Wqkv[:, cols] + bqkv[cols], mirror)
    # output gradient of the block and the gradient reaching O (row split of Wo)
    keep_all = dropout_keep(T, h, p, seed, token_offset)
    dZ = _rb(np.where(keep_all, dOut * dropout_scale(p), 0.0), mirror)
    dO = np.zeros((T, h))
    for i in range(t):
        rs = _slice_cols(h, t, i)
        dO[:, rs] = dZ @ Wo[rs, :].T
    dO = _rb(dO, mirror)
    # per sequence and head: the forward attention and its backward
    O = np.empty((T, h))
    dQKV = np.empty((T, 3 * h))
    P_rows = {j: np.zeros((len(rows), seq_len)) for j in heads}
    causal = np.tril(np.ones((seq_len, seq_len), dtype=bool))
    for s in range(n_seq):
        rsl = slice(s * seq_len, (s + 1) * seq_len)
        in_seq = np.nonzero((rows >= s * seq_len) & (rows < (s + 1) * seq_len))[0]
        for j in range(nh):
            qc = slice(j * d, (j + 1) * d)
            kc = slice(h + j * d, h + (j + 1) * d)
            vc = slice(2 * h + j * d, 2 * h + (j + 1) * d)
            q, k, v = QKV[rsl, qc], QKV[rsl, kc], QKV[rsl, vc]
            sc = np.where(causal, (q @ k.T) / math.sqrt(d), -np.inf)
            e = np.exp(sc - sc.max(axis=1, keepdims=True))
            pr = _rb(e / e.sum(axis=1, keepdims=True), mirror)
            O[rsl, qc] = pr @ v
            if j in P_rows:
                P_rows[j][in_seq] = pr[rows[in_seq] - s * seq_len]
            do = dO[rsl, qc]
            dQKV[rsl, vc] = pr.T @ do
            dp = do @ v.T
            delta = (dp * pr).sum(axis=1, keepdims=True)
            ds = _rb(pr * (dp - delta) / math.sqrt(d), mirror)
            dQKV[rsl, qc] = ds @ k
            dQKV[rsl, kc] = ds.T @ q
    O = _rb(O, mirror)
    dQKV = _rb(dQKV, mirror)
    # block output rows: row split of Wo summed over slices, bias, dropout, residual
    Zr = np.zeros((len(rows), h))
    for i in range(t):
        rs = _slice_cols(h, t, i)
        Zr += O[rows][:, rs] @ Wo[rs, :]
    keep = keep_all[rows]
    out = _rb(X[rows] + np.where(keep, (Zr + bo) * dropout_scale(p), 0.0), mirror)
    # input-gradient rows (operator f: sum over every column block of Wqkv)
    dXs = np.zeros((len(rows), h))
    for c0 in range(0, 3 * h, col_block):
        cols = slice(c0, min(c0 + col_block, 3 * h))
        dXs += dQKV[rows][:, cols] @ Wqkv[:, cols].T
    dX = _rb(dOut[rows] + dXs, mirror)
    r_q, c_q = (np.asarray(a) for a in wqkv_idx)
    r_o, c_o = (np.asarray(a) for a in wo_idx)
    dWqkv = np.array([X[:, r] @ dQKV[:, c] for r, c in zip(r_q, c_q)])
    dWo = np.array([O[:, r] @ dZ[:, c] for r, c in zip(r_o, c_o)])
    return {"QKV": QKV[rows], "O": O[rows], "out": out, "dQKV": dQKV[rows], "dX": dX, "P": P_rows,
            "dWqkv": dWqkv, "dWo": dWo, "dbqkv": dQKV.sum(axis=0), "dbo": dZ.sum(axis=0), "keep": keep}
