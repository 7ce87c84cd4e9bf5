"""CPU oracle of the tensor-sliced transformer MLP block (test infrastructure).

This is NOT part of the product.  Only the tests, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it.  It shares no code with the
CUDA library and is written for a reader to check against the pages by eye:
float64 numpy, one library matmul per product, no blocking or fusion.

What it computes (one micro-batch, T tokens, hidden h, ffn F, t slices, f = F/t):

  Forward, following the Megatron tensor-parallel MLP of "STRONGHOLD: Fast and
  Affordable Billion-scale Deep Learning Model Training" (slides, items 7-8):
    A is split column-wise, A = [A_1 .. A_t];   U_i = X A_i + a_i,  Y_i = GeLU(U_i)
    B is split row-wise,    B = [B_1; .. ; B_t]; Z = sum_i Y_i B_i   (operator g)
    O = R + Dropout(Z + b)
  Backward (operator f sums the input gradient over slices):
    dZ = dO * m / (1 - p);  db = sum_tok dZ
    dY_i = dZ B_i^T;  dU_i = dY_i * GeLU'(U_i);  da_i = sum_tok dU_i
    dB_i = Y_i^T dZ;  dA_i = X^T dU_i
    dX = dO + sum_i dU_i A_i^T
  Weight gradients of successive micro-batches are summed (gradient accumulation:
  "Using DeepSpeed and Megatron to Train Megatron-Turing NLG 530B", Key points).

Readings where the pages are silent (the pages give neither bias, residual, GeLU
form, dropout scaling nor mask generator):
  * biases: a is split with A's columns and added before GeLU; b is added once,
    after the sum over slices;
  * residual: O = R + dropout(Z + b), R = X when no residual is given;
  * GeLU: tanh form 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)));
  * dropout: inverted dropout, kept values scaled by 1/(1-p);
  * mask: element e = (token_offset + token) * h + column of the [T, h] output;
    r = SplitMix64 finaliser of (seed + (e+1) * 0x9E3779B97F4A7C15 mod 2^64)
    (Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
    OOPSLA 2014); keep  <=>  (r >> 32) >= round(p * 2^32).

Two modes:
  * ``mirror=False`` (pure): float64 everywhere after the bf16 inputs.
  * ``mirror=True``: additionally rounds to bf16 (nearest-even) at the points
    where the block stores bf16 tensors: U, Y, O, dZ, dU, dX.  GeLU reads the
    unrounded pre-activation, GeLU' reads the stored (rounded) U.

Every function is pinned by tests under ``tests/`` (closed forms, identities,
finite differences, a library-routine special case, brute force).
"""
from __future__ import annotations

import math

import numpy as np

SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
GELU_CUBIC = 0.044715

MASK64 = (1 << 64) - 1
SPLITMIX_GAMMA = 0x9E3779B97F4A7C15
SPLITMIX_M1 = 0xBF58476D1CE4E5B9
SPLITMIX_M2 = 0x94D049BB133111EB


# ----------------------------------------------------------------------------
# bf16 <-> float64
# ----------------------------------------------------------------------------
def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of raw bf16 bit patterns (uint16) as float64."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even (float64 out).

    bf16 keeps 8 significant bits; below 2^-126 its spacing is fixed at 2^-133.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)
    q = np.ldexp(1.0, e - 8)                 # spacing of bf16 values near x
    return np.rint(x / q) * q                # rint: round half to even


def f64_to_bf16_bits(x) -> np.ndarray:
    """Raw bf16 bit patterns of float64 values (rounded to nearest-even)."""
    r = round_bf16(x).astype(np.float32)     # exact: r has 8 significant bits
    return (r.view(np.uint32) >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------
# GeLU (tanh form) and its derivative
# ----------------------------------------------------------------------------
def gelu(x):
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(SQRT_2_OVER_PI * (x + GELU_CUBIC * x ** 3)))


def gelu_prime(x):
    """d/dx of ``gelu``: product rule on 0.5 x (1 + tanh(s(x)))."""
    x = np.asarray(x, dtype=np.float64)
    th = np.tanh(SQRT_2_OVER_PI * (x + GELU_CUBIC * x ** 3))
    ds = SQRT_2_OVER_PI * (1.0 + 3.0 * GELU_CUBIC * x * x)
    return 0.5 * (1.0 + th) + 0.5 * x * (1.0 - th * th) * ds


# ----------------------------------------------------------------------------
# Dropout mask: counter-hashed SplitMix64
# ----------------------------------------------------------------------------
def keep_threshold(p: float) -> int:
    """Integer threshold on the high 32 hash bits: round(p_f32 * 2^32), halves up."""
    pf = float(np.float32(p))
    return int(math.floor(pf * 4294967296.0 + 0.5))


def splitmix64(seed: int, idx) -> np.ndarray:
    """Output number ``idx`` (0-based) of a SplitMix64 stream seeded with ``seed``."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        x = np.uint64(seed & MASK64) + (idx + np.uint64(1)) * np.uint64(SPLITMIX_GAMMA)
        z = (x ^ (x >> np.uint64(30))) * np.uint64(SPLITMIX_M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(SPLITMIX_M2)
        return z ^ (z >> np.uint64(31))


def dropout_keep(tokens: int, h: int, p: float, seed: int, token_offset: int = 0,
                 rows=None) -> np.ndarray:
    """Boolean keep mask [len(rows), h] for the given token rows (default: all)."""
    rows = np.arange(tokens, dtype=np.uint64) if rows is None else np.asarray(rows, dtype=np.uint64)
    e = (np.uint64(token_offset) + rows)[:, None] * np.uint64(h) + np.arange(h, dtype=np.uint64)[None, :]
    r = splitmix64(seed, e)
    return (r >> np.uint64(32)) >= np.uint64(keep_threshold(p))


def dropout_scale(p: float) -> float:
    return 1.0 / (1.0 - float(np.float32(p)))


# ----------------------------------------------------------------------------
# The block
# ----------------------------------------------------------------------------
def _rb(x, mirror):
    return round_bf16(x) if mirror else x


def mlp_fwd(X, A, a, B, b, t, p, seed, token_offset=0, R=None, mirror=False):
    """Forward of one micro-batch.  All array inputs are float64 (decoded bf16).

    Returns a dict with U, Y [T, F] (as stored), Z [T, h] (sum over slices),
    keep [T, h] and O [T, h].
    """
    T, h = X.shape
    F = A.shape[1]
    assert F % t == 0
    f = F // t
    R = X if R is None else R
    U = np.empty((T, F))
    Y = np.empty((T, F))
    Z = np.zeros((T, h))
    for i in range(t):                        # slice i: columns of A, rows of B
        cols = slice(i * f, (i + 1) * f)
        Ui = X @ A[:, cols] + a[cols]
        Yi = gelu(Ui)
        U[:, cols] = _rb(Ui, mirror)
        Y[:, cols] = _rb(Yi, mirror)
        Z += Y[:, cols] @ B[cols, :]          # partial product of slice i, summed
    keep = dropout_keep(T, h, p, seed, token_offset)
    O = R + np.where(keep, (Z + b) * dropout_scale(p), 0.0)
    return {"U": U, "Y": Y, "Z": Z, "keep": keep, "O": _rb(O, mirror)}


def mlp_bwd(dO, X, A, B, U, Y, keep, t, p, mirror=False, residual_is_input=True):
    """Backward of one micro-batch given the stored U, Y and the keep mask.

    Returns dZ, dU, dX and this micro-batch's gradients dA, da, dB, db.
    ``residual_is_input``: the residual R is X itself, so dO flows into dX.
    """
    T, h = X.shape
    F = A.shape[1]
    f = F // t
    dZ = _rb(np.where(keep, dO * dropout_scale(p), 0.0), mirror)
    db = dZ.sum(axis=0)
    dU = np.empty((T, F))
    dA = np.empty_like(A)
    da = np.empty(F)
    dB = np.empty_like(B)
    dXs = np.zeros((T, h))
    for i in range(t):
        cols = slice(i * f, (i + 1) * f)
        dYi = dZ @ B[cols, :].T
        dUi = _rb(dYi * gelu_prime(U[:, cols]), mirror)
        dU[:, cols] = dUi
        da[cols] = dUi.sum(axis=0)
        dB[cols, :] = Y[:, cols].T @ dZ
        dA[:, cols] = X.T @ dUi
        dXs += dUi @ A[:, cols].T             # partial input gradient of slice i, summed
    dX = _rb((dO if residual_is_input else 0.0) + dXs, mirror)
    return {"dZ": dZ, "dU": dU, "dX": dX, "dA": dA, "da": da, "dB": dB, "db": db}


# ----------------------------------------------------------------------------
# Sampled evaluation for workloads too large for the full oracle.  Each output
# is computed from its definition alone: a token row of O / dX (the row loops over
# the slices exactly as the block does), or a weight-gradient entry as a sum over
# all tokens of one column of Y or dU.
# ----------------------------------------------------------------------------
class Bf16Matrix:
    """A bf16 matrix kept as raw bits; indexing returns the exact float64 values of
    the selected block only (so a 3 GB weight never needs a 13 GB float64 copy)."""

    def __init__(self, bits):
        self.bits = np.asarray(bits, dtype=np.uint16)
        self.shape = self.bits.shape

    def __getitem__(self, idx):
        return bf16_to_f64(self.bits[idx])


def rows_fwd_bwd(rows, X, dO, A, a, B, b, t, p, seed, token_offset=0, mirror=False):
    """O, dX, U, Y, dU, dZ rows for the given token rows (residual R = X).

    X, dO, A, B may be float64 arrays or ``Bf16Matrix``; only slice-sized blocks
    of A and B are decoded at a time."""
    rows = np.asarray(rows)
    h = X.shape[1]
    F = A.shape[1]
    f = F // t
    Xr = X[rows]
    dOr = dO[rows]
    keep = dropout_keep(X.shape[0], h, p, seed, token_offset, rows=rows)
    s = dropout_scale(p)
    dZr = _rb(np.where(keep, dOr * s, 0.0), mirror)
    Zr = np.zeros((len(rows), h))
    dXs = np.zeros((len(rows), h))
    Ur_all = np.empty((len(rows), F))
    Yr_all = np.empty((len(rows), F))
    dUr_all = np.empty((len(rows), F))
    for i in range(t):
        cols = slice(i * f, (i + 1) * f)
        A_i = A[:, cols]
        B_i = B[cols, :]
        Ur = Xr @ A_i + a[cols]
        Yr = _rb(gelu(Ur), mirror)
        Urs = _rb(Ur, mirror)
        Zr += Yr @ B_i
        dUr = _rb((dZr @ B_i.T) * gelu_prime(Urs), mirror)
        dXs += dUr @ A_i.T
        Ur_all[:, cols] = Urs
        Yr_all[:, cols] = Yr
        dUr_all[:, cols] = dUr
    Or = _rb(Xr + np.where(keep, (Zr + b) * s, 0.0), mirror)
    dXr = _rb(dOr + dXs, mirror)
    return {"O": Or, "dX": dXr, "U": Ur_all, "Y": Yr_all, "dU": dUr_all, "dZ": dZr, "keep": keep}


def full_dZ(dO, p, seed, token_offset=0, mirror=False):
    T, h = dO.shape
    keep = dropout_keep(T, h, p, seed, token_offset)
    return _rb(np.where(keep, dO * dropout_scale(p), 0.0), mirror)


def columns_U(cols, X, A, a, mirror=False):
    """U[:, cols] over all tokens (as stored) and the unrounded pre-activation."""
    cols = np.asarray(cols)
    Uc = X @ A[:, cols] + a[cols]
    return _rb(Uc, mirror), Uc


def wgrad_dB_entries(r_idx, c_idx, X, A, a, dZ, mirror=False):
    """dB[r, c] = sum_tok Y[tok, r] dZ[tok, c] for paired index arrays."""
    r_idx = np.asarray(r_idx)
    c_idx = np.asarray(c_idx)
    ur = np.unique(r_idx)
    _, Uraw = columns_U(ur, X, A, a, mirror)
    Yc = _rb(gelu(Uraw), mirror)
    pos = {int(v): k for k, v in enumerate(ur)}
    return np.array([Yc[:, pos[int(r)]] @ dZ[:, int(c)] for r, c in zip(r_idx, c_idx)])


def columns_dU(cols, X, A, a, B, dZ, mirror=False):
    """dU[:, cols] over all tokens."""
    cols = np.asarray(cols)
    Us, _ = columns_U(cols, X, A, a, mirror)
    return _rb((dZ @ B[cols, :].T) * gelu_prime(Us), mirror)


def wgrad_dA_entries(r_idx, c_idx, X, A, a, B, dZ, mirror=False):
    """dA[r, c] = sum_tok X[tok, r] dU[tok, c] for paired index arrays."""
    r_idx = np.asarray(r_idx)
    c_idx = np.asarray(c_idx)
    uc = np.unique(c_idx)
    dUc = columns_dU(uc, X, A, a, B, dZ, mirror)
    pos = {int(v): k for k, v in enumerate(uc)}
    return np.array([X[:, int(r)] @ dUc[:, pos[int(c)]] for r, c in zip(r_idx, c_idx)])
