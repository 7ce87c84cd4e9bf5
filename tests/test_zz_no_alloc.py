"""mlp_fwd_static_scratch: the forward for callers that cannot allocate device memory.

Such callers (a plugin inside a host application that owns all device memory
through its own pool, or a serving loop that must not call cudaMalloc once it
runs) cannot pass the fp32 workspace that one-slice forward calls need.  This
entry point uses a fixed array in the library's own device memory instead.  The
test checks it against mlp_fwd with a caller-owned workspace, through the C ABI,
on two forward passes in a row (so a pass that found the array holding the
previous pass's contents must still be right), and that sizes beyond the array
are refused.  It runs on its own in a fresh process as well as after the others.
"""
import pytest
import torch

from transformer_lm_megatron_gb300 import build as gb_build
from transformer_lm_megatron_gb300 import inputs as gin
from transformer_lm_megatron_gb300 import mlp

from gpu_harness import BF16_TOL, rel_err, to_f64

pytestmark = pytest.mark.gpu

SCRATCH_FLOATS = 4 << 20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gb_build.build()
    mlp.load()


def _forward(use_static, h, ffn, t, T, j, w, X):
    A, a, B, b = w
    dev = X.device
    U = torch.empty(T, ffn, dtype=torch.bfloat16, device=dev)
    Y = torch.empty_like(U)
    O = torch.empty(T, h, dtype=torch.bfloat16, device=dev)
    Zacc = None if use_static else torch.empty(T, h, dtype=torch.float32, device=dev)
    for i in range(t):  # one call per slice, in order
        if use_static:
            mlp.mlp_fwd_static_scratch(h, ffn, t, i, T, 0.1, 1234, j * T, X, A, a, B, b, None, U, Y, O)
        else:
            mlp.mlp_fwd(h, ffn, t, i, T, 0.1, 1234, j * T, X, A, a, B, b, None, U, Y, Zacc, O)
    torch.cuda.synchronize()
    assert mlp.mlp_sync_status() == mlp.MLP_OK, mlp.last_error()
    return U, Y, O


@pytest.mark.parametrize("T,h,ffn,t", [(200, 256, 1024, 4), (2048, 2048, 8192, 8)])
def test_static_scratch_forward_matches_caller_workspace(T, h, ffn, t):
    dev = torch.device("cuda")
    w = tuple(x.to(dev) for x in gin.make_weights(h, ffn))
    for j in range(2):  # two calls in a row; the second starts with the first's leftovers
        X, _ = gin.make_microbatch(T, h, j)
        X = X.to(dev)
        ref = _forward(False, h, ffn, t, T, j, w, X)
        got = _forward(True, h, ffn, t, T, j, w, X)
        for name, r, g in zip(("U", "Y", "O"), ref, got):
            err = rel_err(to_f64(g), to_f64(r))
            assert err <= BF16_TOL, (j, name, err)


def test_static_scratch_refuses_sizes_beyond_the_array():
    dev = torch.device("cuda")
    h, T = 4096, SCRATCH_FLOATS // 4096 + 8
    dummy = torch.empty(16, dtype=torch.bfloat16, device=dev)
    rc = mlp.load().mlp_fwd_static_scratch(h, 4 * h, 2, 0, T, 0.1, 1234, 0, *([dummy.data_ptr()] * 6), None,
                                           *([dummy.data_ptr()] * 3), None)
    assert rc == mlp.MLP_EINVAL
    assert "exceeds" in mlp.last_error()
