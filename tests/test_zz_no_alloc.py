"""mlp_fwd_static_scratch: the forward for callers that cannot allocate device memory.

Such callers (a plugin inside a host application that owns all device memory
through its own pool, or a serving loop that must not call cudaMalloc once it
runs) cannot pass the fp32 workspace that one-slice forward calls need.  This
entry point uses a fixed array in the library's own device memory instead.

The test checks it against mlp_fwd with a caller-owned workspace, through the C
ABI, on two forward passes in a row, so that a pass which finds the array holding
the previous pass's contents must still be right.  Both entry points run the same
kernels in the same order on the same inputs, so U, Y and O must agree bit for
bit: a partly stale workspace would show up as a difference.  O is also compared
with the oracle.  Sizes beyond the array are refused.  The file runs after every
other test file (its name sorts last); one test runs the comparison again in a
fresh Python process, where the library's first call on the device is this entry
point's.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from oracle import mlp_oracle as orc
from transformer_lm_megatron_gb300 import build as gb_build
from transformer_lm_megatron_gb300 import inputs as gin
from transformer_lm_megatron_gb300 import mlp

from gpu_harness import BF16_TOL, bits_f64, rel_err, to_f64

pytestmark = pytest.mark.gpu

SCRATCH_FLOATS = 4 << 20
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gb_build.build()
    mlp.load()


def _forward(use_static, h, ffn, t, T, j, w, X, static_first=False):
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
    w_host = gin.make_weights(h, ffn)
    w = tuple(x.to(dev) for x in w_host)
    for j in range(2):  # two passes in a row; the second starts with the first's leftovers
        X_host, _ = gin.make_microbatch(T, h, j)
        X = X_host.to(dev)
        # the static-scratch pass first, so that in a fresh process it is the
        # library's first call on the device
        got = _forward(True, h, ffn, t, T, j, w, X)
        ref = _forward(False, h, ffn, t, T, j, w, X)
        for name, r, g in zip(("U", "Y", "O"), ref, got):
            assert torch.equal(g, r), (j, name)
        if T * ffn <= 1 << 20:
            # O against the float64 oracle (bf16-mirroring and pure modes)
            w64 = tuple(bits_f64(x) for x in w_host)
            for mirror in (True, False):
                fw = orc.mlp_fwd(bits_f64(X_host), *w64, t, 0.1, 1234, token_offset=j * T, mirror=mirror)
                err = rel_err(to_f64(got[2]), fw["O"])
                assert err <= BF16_TOL, (j, mirror, err)


def test_static_scratch_refuses_sizes_beyond_the_array():
    dev = torch.device("cuda")
    h, T = 4096, SCRATCH_FLOATS // 4096 + 8
    d = torch.empty(16, dtype=torch.bfloat16, device=dev).data_ptr()
    # h, ffn, t, slice, tokens, p, seed, token_offset, X, A, a, B, b, R, U, Y, O, stream
    rc = mlp.load().mlp_fwd_static_scratch(h, 4 * h, 2, 0, T, 0.1, 1234, 0, d, d, d, d, d, None, d, d, d, None)
    assert rc == mlp.MLP_EINVAL
    assert "exceeds" in mlp.last_error()


def test_static_scratch_in_a_fresh_process():
    """The comparison again in a new interpreter, where the set-up of the array's
    device address happens on that process's first call."""
    if os.environ.get("GB_NO_ALLOC_CHILD"):
        pytest.skip("already the fresh process")
    env = dict(os.environ, GB_NO_ALLOC_CHILD="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_zz_no_alloc.py"), "-k", "matches_caller_workspace"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "2 passed" in r.stdout, r.stdout[-2000:]
