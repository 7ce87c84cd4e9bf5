"""Python binding of the C-ABI library ``libgb_mlp.so`` (argument marshalling only).

Every function takes torch tensors (CUDA, contiguous) and forwards their device
pointers and the current CUDA stream to the entry point of the same name; all
arithmetic runs in the library's kernels.  The library must be built
(``transformer_lm_megatron_gb300.build``); there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

MLP_OK = 0
MLP_EINVAL = -1
MLP_EALIGN = -2
MLP_EUNSUPPORTED = -3
MLP_ECUDA = -4
MLP_ETIMEOUT = -5

_lib = None

_vp = ctypes.c_void_p
_i32 = ctypes.c_int
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64
_f32 = ctypes.c_float

_SIGNATURES = {
    "mlp_fwd": (_i32, [_i32, _i32, _i32, _i32, _i64, _f32, _u64, _u64] + [_vp] * 6 + [_vp, _vp, _vp, _vp, _vp]),
    "mlp_bwd": (_i32, [_i32, _i32, _i32, _i32, _i64, _f32, _u64, _u64, _i32, _i32] + [_vp] * 6 + [_vp] * 4
                + [_vp] * 4 + [_vp]),
    "grad_accum_reset": (_i32, [_i32, _i32, _vp, _vp, _vp, _vp, _vp]),
    "mlp_sync_status": (_i32, [_vp]),
    "mlp_last_error": (ctypes.c_char_p, []),
    "mlp_dropout_mask": (_i32, [_i32, _i64, _f32, _u64, _u64, _vp, _vp]),
    "mlp_gelu_probe": (_i32, [_vp, _i64, _vp, _vp, _vp]),
    "mlp_wait_timeout_probe": (_i32, [_u64, _vp]),
    "mlp_launch_count": (_u64, []),
    "mlp_set_cta_pair": (_i32, [_i32]),
    "mlp_set_dependent_launch": (_i32, [_i32]),
    "mlp_set_split_tail": (_i32, [_i32]),
    "mlp_set_tile_scheduler": (_i32, [_i32]),
    "mlp_set_wgrad_transpose": (_i32, [_i32]),
    "mlp_set_attn_fused": (_i32, [_i32]),
    "adam_step": (_i32, [_i64, _vp, _f32, _vp, _vp, _vp, _vp, _f32, _f32, _f32, _f32, _f32, _i32, _vp]),
    "attn_fwd": (_i32, [_i32, _i32, _i32, _i64, _i32, _f32, _u64, _u64] + [_vp] * 11 + [_vp]),
    "attn_bwd": (_i32, [_i32, _i32, _i32, _i64, _i32, _f32, _u64, _u64, _i32, _i32] + [_vp] * 17 + [_vp]),
    "mlp_fwd_static_scratch": (_i32, [_i32, _i32, _i32, _i32, _i64, _f32, _u64, _u64] + [_vp] * 6 + [_vp, _vp, _vp, _vp]),
    "mlp_trace_begin": (_i32, [_i32]),
    "mlp_trace_end": (_i32, [_i32, _vp, _vp, _vp]),
}


class MLPError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{msg} (code {code})")
        self.code = code


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load (once) and return the ctypes handle of the library."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} (run transformer_lm_megatron_gb300.build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def last_error() -> str:
    return load().mlp_last_error().decode()


def _check(rc: int):
    if rc != MLP_OK:
        raise MLPError(rc, last_error())


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def mlp_fwd(h, ffn, t, slice_, tokens, p, seed, token_offset, X, A, a, B, b, R, U, Y, Zacc, O, stream=None):
    _check(load().mlp_fwd(h, ffn, t, slice_, tokens, p, seed, token_offset, _ptr(X), _ptr(A), _ptr(a), _ptr(B),
                          _ptr(b), _ptr(R), _ptr(U), _ptr(Y), _ptr(Zacc), _ptr(O), _stream(stream)))


def mlp_bwd(h, ffn, t, slice_, tokens, p, seed, token_offset, residual_grad, accumulate, dO, X, A, B, U, Y, dZ, dU,
            dXacc, dX, dA, da, dB, db, stream=None):
    _check(load().mlp_bwd(h, ffn, t, slice_, tokens, p, seed, token_offset, int(residual_grad), int(accumulate),
                          _ptr(dO), _ptr(X),
                          _ptr(A), _ptr(B), _ptr(U), _ptr(Y), _ptr(dZ), _ptr(dU), _ptr(dXacc), _ptr(dX), _ptr(dA),
                          _ptr(da), _ptr(dB), _ptr(db), _stream(stream)))


def mlp_fwd_static_scratch(h, ffn, t, slice_, tokens, p, seed, token_offset, X, A, a, B, b, R, U, Y, O,
                           stream=None):
    """mlp_fwd for callers that cannot allocate: the fp32 slice workspace is the
    library's own fixed 16 MiB array (tokens * h <= 4,194,304); see the header."""
    _check(load().mlp_fwd_static_scratch(h, ffn, t, slice_, tokens, p, seed, token_offset, _ptr(X), _ptr(A), _ptr(a),
                                         _ptr(B), _ptr(b), _ptr(R), _ptr(U), _ptr(Y), _ptr(O), _stream(stream)))


def grad_accum_reset(h, ffn, dA, da, dB, db, stream=None):
    _check(load().grad_accum_reset(h, ffn, _ptr(dA), _ptr(da), _ptr(dB), _ptr(db), _stream(stream)))


def adam_step(grad, master, m, v, weight, lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0, step=1,
              grad_scale=1.0, stream=None):
    """One mixed-precision Adam update of a parameter tensor (see include/gb_mlp.h)."""
    n = grad.numel()
    for t in (master, m, v, weight):
        if t.numel() != n:
            raise ValueError("adam_step: all tensors need the same number of elements")
    _check(load().adam_step(n, _ptr(grad), grad_scale, _ptr(master), _ptr(m), _ptr(v), _ptr(weight), lr, beta1,
                            beta2, eps, weight_decay, step, _stream(stream)))


def attn_fwd(h, nh, t, tokens, seq_len, p, seed, token_offset, X, Wqkv, bqkv, Wo, bo, R, QKV, S, P, O, out,
             stream=None):
    _check(load().attn_fwd(h, nh, t, tokens, seq_len, p, seed, token_offset, _ptr(X), _ptr(Wqkv), _ptr(bqkv),
                           _ptr(Wo), _ptr(bo), _ptr(R), _ptr(QKV), _ptr(S), _ptr(P), _ptr(O), _ptr(out),
                           _stream(stream)))


def attn_bwd(h, nh, t, tokens, seq_len, p, seed, token_offset, residual_grad, accumulate, dOut, X, Wqkv, Wo, QKV, P,
             O, dZ, dO, dP, dS, dQKV, dX, dWqkv, dbqkv, dWo, dbo, stream=None):
    _check(load().attn_bwd(h, nh, t, tokens, seq_len, p, seed, token_offset, int(residual_grad), int(accumulate),
                           _ptr(dOut), _ptr(X), _ptr(Wqkv), _ptr(Wo), _ptr(QKV), _ptr(P), _ptr(O), _ptr(dZ), _ptr(dO),
                           _ptr(dP), _ptr(dS), _ptr(dQKV), _ptr(dX), _ptr(dWqkv), _ptr(dbqkv), _ptr(dWo), _ptr(dbo),
                           _stream(stream)))


class AttnBuffers:
    """Saved activations, workspaces and fp32 gradients of the attention block."""

    def __init__(self, tokens: int, h: int, nh: int, seq_len: int, device="cuda"):
        n_seq = tokens // seq_len
        bf = dict(dtype=torch.bfloat16, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        pshape = (n_seq, nh, seq_len, seq_len)
        self.QKV = torch.empty(tokens, 3 * h, **bf)
        self.S = torch.empty(pshape, **f32)
        self.P = torch.empty(pshape, **bf)
        self.O = torch.empty(tokens, h, **bf)
        self.out = torch.empty(tokens, h, **bf)
        self.dZ = torch.empty(tokens, h, **bf)
        self.dO = torch.empty(tokens, h, **bf)
        self.dP = self.S          # the scores are dead once P exists; the backward reuses them
        self.dS = torch.empty(pshape, **bf)
        self.dQKV = torch.empty(tokens, 3 * h, **bf)
        self.dX = torch.empty(tokens, h, **bf)
        self.dWqkv = torch.zeros(h, 3 * h, **f32)
        self.dbqkv = torch.zeros(3 * h, **f32)
        self.dWo = torch.zeros(h, h, **f32)
        self.dbo = torch.zeros(h, **f32)


def attn_step(h, nh, t, seq_len, p, seed, weights, X, dOut, buf: AttnBuffers, token_offset=0, accumulate=True,
              stream=None):
    """One forward + backward of the attention block on one micro-batch."""
    Wqkv, bqkv, Wo, bo = weights
    T = X.shape[0]
    attn_fwd(h, nh, t, T, seq_len, p, seed, token_offset, X, Wqkv, bqkv, Wo, bo, None, buf.QKV, buf.S, buf.P, buf.O,
             buf.out, stream)
    attn_bwd(h, nh, t, T, seq_len, p, seed, token_offset, 1, accumulate, dOut, X, Wqkv, Wo, buf.QKV, buf.P, buf.O,
             buf.dZ, buf.dO, buf.dP, buf.dS, buf.dQKV, buf.dX, buf.dWqkv, buf.dbqkv, buf.dWo, buf.dbo, stream)


def mlp_sync_status(stream=None) -> int:
    return load().mlp_sync_status(_stream(stream))


def mlp_dropout_mask(h, tokens, p, seed, token_offset, m, stream=None):
    _check(load().mlp_dropout_mask(h, tokens, p, seed, token_offset, _ptr(m), _stream(stream)))


def mlp_gelu_probe(x, y, dy, stream=None):
    _check(load().mlp_gelu_probe(_ptr(x), x.numel(), _ptr(y), _ptr(dy), _stream(stream)))


def mlp_wait_timeout_probe(limit_ns, stream=None):
    _check(load().mlp_wait_timeout_probe(limit_ns, _stream(stream)))


def mlp_launch_count() -> int:
    return int(load().mlp_launch_count())


def mlp_set_cta_pair(mode: int):
    _check(load().mlp_set_cta_pair(mode))


def mlp_set_dependent_launch(enable: bool):
    _check(load().mlp_set_dependent_launch(1 if enable else 0))


def mlp_set_split_tail(enable: bool):
    _check(load().mlp_set_split_tail(1 if enable else 0))


def mlp_set_attn_fused(enable: bool):
    _check(load().mlp_set_attn_fused(1 if enable else 0))


def mlp_set_tile_scheduler(mode: int):
    """1 dynamic tile order for every GEMM, 0 static for every GEMM, -1 (default)
    dynamic for the batched attention products only."""
    _check(load().mlp_set_tile_scheduler(int(mode)))


def mlp_set_wgrad_transpose(mode: int):
    """1 the weight-gradient GEMMs read transposed copies of X and dZ (held in dXacc)
    whenever they can, 0 never, -1 (default) when the GEMMs are large enough."""
    _check(load().mlp_set_wgrad_transpose(int(mode)))


TRACE_NAMES = {0: "F1 gemm X.A_i +a, GeLU", 1: "F2 gemm Y_i.B_i (+dropout,+residual)", 2: "B2 gemm dZ.B_i^T *GeLU'",
               3: "B3 gemm Y_i^T.dZ (+= dB)", 4: "B4 gemm X^T.dU_i (+= dA)", 5: "B5 gemm dU_i.A_i^T (+dO)",
               10: "dropout backward + db", 11: "column sum da", 12: "accumulator reset", 14: "adam step",
               15: "transposed copies X^T, dZ^T",
               20: "attention GEMM", 21: "softmax, softmax-grad row sums", 22: "fused attention core"}
GEMM_KINDS = (0, 1, 2, 3, 4, 5)


class Trace:
    """Per-launch device times of this library's kernels (CUDA event pairs on the launch stream)."""

    def __init__(self, capacity: int):
        self.capacity = capacity
        self.entries = []

    def start(self):
        _check(load().mlp_trace_begin(self.capacity))

    def stop(self):
        import numpy as np
        kinds = np.zeros(self.capacity, dtype=np.int32)
        mnk = np.zeros(3 * self.capacity, dtype=np.int64)
        ms = np.zeros(self.capacity, dtype=np.float32)
        n = load().mlp_trace_end(self.capacity, kinds.ctypes.data, mnk.ctypes.data, ms.ctypes.data)
        if n < 0:
            _check(n)
        self.entries = [(int(kinds[i]), tuple(int(v) for v in mnk[3 * i:3 * i + 3]), float(ms[i])) for i in range(n)]
        return self.entries

    def summary(self):
        """{kind: (launches, total ms, flops)} with GEMM flops 2*M*N*K."""
        out = {}
        for kind, (m, n, k), t in self.entries:
            c, tot, fl = out.get(kind, (0, 0.0, 0))
            out[kind] = (c + 1, tot + t, fl + (2 * m * n * k if kind in GEMM_KINDS else 0))
        return out

    def roofline(self, peak, peak_kind):
        """The dominant kernel (the tcgen05 GEMM, all six contractions) against the bf16
        tensor peak ``peak`` (TFLOP/s), described by ``peak_kind``."""
        summ = self.summary()
        g_launch = sum(summ[k][0] for k in GEMM_KINDS if k in summ)
        g_ms = sum(summ[k][1] for k in GEMM_KINDS if k in summ)
        g_flops = sum(summ[k][2] for k in GEMM_KINDS if k in summ)
        all_ms = sum(v[1] for v in summ.values())
        if g_launch == 0 or g_ms <= 0:
            return None
        achieved = (g_flops / g_launch) / (g_ms / g_launch / 1e3) / 1e12
        kernels = {TRACE_NAMES.get(k, str(k)): {"launches": v[0], "ms": round(v[1], 4),
                                                 "share": round(v[1] / all_ms, 4)} for k, v in sorted(summ.items())}
        return {"bound": "tensor", "kernel": "k_gemm_bf16_tc (tcgen05, all six GEMMs)", "achieved": achieved,
                "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_kind": peak_kind, "traffic": None,
                "flops_per_launch": g_flops / g_launch, "avg_launch_ms": g_ms / g_launch,
                "gemm_share_of_kernel_time": g_ms / all_ms if all_ms else None, "kernels": kernels}


# ---------------------------------------------------------------------------
# Buffers of one block, allocated with torch (the library allocates nothing).
# ---------------------------------------------------------------------------
class BlockBuffers:
    """Activations, workspaces and fp32 gradient accumulators for one workload."""

    def __init__(self, tokens: int, h: int, ffn: int, t: int, device="cuda", grads=None):
        """grads: optional (dA, da, dB, db) fp32 accumulators to use instead of new
        ones, e.g. the views of one contiguous buffer (data_parallel.flat_gradients)."""
        bf = dict(dtype=torch.bfloat16, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        self.U = torch.empty(tokens, ffn, **bf)
        self.Y = torch.empty(tokens, ffn, **bf)
        self.O = torch.empty(tokens, h, **bf)
        self.dZ = torch.empty(tokens, h, **bf)
        self.dU = torch.empty(tokens, ffn, **bf)
        self.dX = torch.empty(tokens, h, **bf)
        self.Zacc = torch.empty(tokens, h, **f32) if t > 1 else None
        # the one-slice calls' sum over slices; otherwise scratch for the transposed
        # operands of the weight-gradient GEMMs
        self.dXacc = torch.empty(tokens, h, **f32)
        if grads is None:
            grads = (torch.zeros(h, ffn, **f32), torch.zeros(ffn, **f32), torch.zeros(ffn, h, **f32),
                     torch.zeros(h, **f32))
        self.dA, self.da, self.dB, self.db = grads


def block_step(wl, weights, X, dO, buf: BlockBuffers, token_offset=0, slice_mode="all", stream=None,
               accumulate=True):
    """One micro-batch forward + backward of workload ``wl``.

    slice_mode "all": one call each with slice = -1; "each": t calls per pass, in order.
    accumulate: add this micro-batch's weight/bias gradients to buf's accumulators
    (True) or overwrite them (False: the first micro-batch of a step).
    """
    A, a, B, b = weights
    T = X.shape[0]
    slices = [-1] if slice_mode == "all" else list(range(wl.t))
    for i in slices:
        mlp_fwd(wl.h, wl.ffn, wl.t, i, T, wl.p, wl.seed, token_offset, X, A, a, B, b, None, buf.U, buf.Y, buf.Zacc,
                buf.O, stream)
    for i in slices:
        mlp_bwd(wl.h, wl.ffn, wl.t, i, T, wl.p, wl.seed, token_offset, 1, accumulate, dO, X, A, B, buf.U, buf.Y,
                buf.dZ, buf.dU, buf.dXacc, buf.dX, buf.dA, buf.da, buf.dB, buf.db, stream)
