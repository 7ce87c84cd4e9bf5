"""Host-side checks of the C-ABI library: it builds for sm_103a, loads without a
GPU, exports every entry point the header declares, and rejects bad arguments
before touching the device."""
import ctypes
import os
import re

import pytest

from transformer_lm_megatron_gb300 import build as gb_build
from transformer_lm_megatron_gb300 import mlp

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gb_mlp.h")


@pytest.fixture(scope="module")
def lib():
    gb_build.build()
    return mlp.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:int|uint64_t|const char\s*\*)\s*(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = set(_declared_functions())
    for required in ("mlp_fwd", "mlp_bwd", "grad_accum_reset", "mlp_sync_status", "mlp_last_error",
                     "mlp_dropout_mask", "mlp_gelu_probe", "mlp_wait_timeout_probe", "mlp_launch_count"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    handle = ctypes.CDLL(mlp.library_path())
    for name in _declared_functions():
        assert hasattr(handle, name), name


def test_binding_covers_every_declared_symbol():
    assert set(_declared_functions()) == set(mlp._SIGNATURES)


P = None  # null pointer
GOOD = 4096  # a 16-byte aligned fake address: never dereferenced, validation fails first


def _fwd(lib, h=64, ffn=256, t=2, slice_=-1, tokens=16, p=0.1, ptr=GOOD, R=None, Zacc=GOOD):
    return lib.mlp_fwd(h, ffn, t, slice_, tokens, p, 1234, 0, ptr, ptr, ptr, ptr, ptr, R, ptr, ptr, Zacc, ptr, None)


@pytest.mark.parametrize("kw,code", [
    (dict(h=0), mlp.MLP_EINVAL),
    (dict(h=12), mlp.MLP_EINVAL),                 # h % 8 != 0
    (dict(ffn=260, t=2), mlp.MLP_EINVAL),         # f = 130, not a multiple of 8
    (dict(ffn=256, t=3), mlp.MLP_EINVAL),         # ffn % t != 0
    (dict(t=0), mlp.MLP_EINVAL),
    (dict(tokens=0), mlp.MLP_EINVAL),
    (dict(tokens=1 << 31), mlp.MLP_EINVAL),
    (dict(p=1.0), mlp.MLP_EINVAL),
    (dict(p=-0.1), mlp.MLP_EINVAL),
    (dict(p=float("nan")), mlp.MLP_EINVAL),
    (dict(slice_=2), mlp.MLP_EINVAL),
    (dict(slice_=-2), mlp.MLP_EINVAL),
    (dict(ptr=None), mlp.MLP_EINVAL),
    (dict(ptr=GOOD + 2), mlp.MLP_EALIGN),
    (dict(R=GOOD + 8), mlp.MLP_EALIGN),
    (dict(Zacc=None, slice_=0), mlp.MLP_EINVAL),   # one-slice calls with t > 1 need the fp32 workspace
])
def test_fwd_rejects_bad_arguments(lib, kw, code):
    assert _fwd(lib, **kw) == code
    assert mlp.last_error()


def test_bwd_rejects_bad_arguments(lib):
    g = GOOD
    args = [64, 256, 2, -1, 16, 0.1, 1234, 0, 1, 1] + [g] * 8 + [g, g] + [g] * 4 + [None]
    bad = list(args)
    bad[0] = 20
    assert lib.mlp_bwd(*bad) == mlp.MLP_EINVAL
    bad = list(args)
    bad[3] = 0                                       # one-slice call with t > 1 ...
    bad[18] = None                                   # ... needs the dXacc workspace
    assert lib.mlp_bwd(*bad) == mlp.MLP_EINVAL
    bad = list(args)
    bad[10] = g + 4                                  # dO misaligned
    assert lib.mlp_bwd(*bad) == mlp.MLP_EALIGN


def test_reset_and_helpers_reject_bad_arguments(lib):
    assert lib.grad_accum_reset(12, 256, GOOD, GOOD, GOOD, GOOD, None) == mlp.MLP_EINVAL
    assert lib.grad_accum_reset(64, 256, GOOD, None, GOOD, GOOD, None) == mlp.MLP_EINVAL
    assert lib.mlp_dropout_mask(64, 0, 0.1, 1, 0, GOOD, None) == mlp.MLP_EINVAL
    assert lib.mlp_wait_timeout_probe(5 * 10**9, None) == mlp.MLP_EINVAL


def test_valid_call_without_gpu_reports_unsupported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _fwd(lib) == mlp.MLP_EUNSUPPORTED
    assert _fwd(lib, Zacc=None) == mlp.MLP_EUNSUPPORTED   # all-slices calls need no workspace
    assert mlp.mlp_launch_count() == 0


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(8, 8)
    with pytest.raises(ValueError):
        mlp._ptr(x) if not torch.cuda.is_available() else (_ for _ in ()).throw(ValueError())


def test_switches_reject_bad_values(lib):
    assert lib.mlp_set_cta_pair(2) == mlp.MLP_EINVAL
    assert lib.mlp_set_dependent_launch(2) == mlp.MLP_EINVAL
    assert lib.mlp_set_split_tail(-1) == mlp.MLP_EINVAL
    assert lib.mlp_set_tile_scheduler(2) == mlp.MLP_EINVAL
    assert lib.mlp_set_attn_fused(2) == mlp.MLP_EINVAL
    assert lib.mlp_set_attn_fused(1) == mlp.MLP_OK
    assert lib.mlp_set_wgrad_transpose(2) == mlp.MLP_EINVAL
    assert lib.mlp_set_wgrad_transpose(-2) == mlp.MLP_EINVAL
    for mode in (0, 1, -1):
        assert lib.mlp_set_wgrad_transpose(mode) == mlp.MLP_OK
    assert lib.mlp_set_tile_scheduler(-1) == mlp.MLP_OK
    for fn in (lib.mlp_set_cta_pair, lib.mlp_set_dependent_launch, lib.mlp_set_split_tail, lib.mlp_set_tile_scheduler):
        assert fn(1) == mlp.MLP_OK
    assert lib.mlp_set_cta_pair(-1) == mlp.MLP_OK
    assert lib.mlp_set_tile_scheduler(-1) == mlp.MLP_OK


def test_adam_rejects_bad_arguments(lib):
    def call(**kw):
        a = dict(n=1024, grad=GOOD, grad_scale=1.0, master=GOOD, m=GOOD, v=GOOD, weight=GOOD, lr=1e-3, beta1=0.9,
                 beta2=0.95, eps=1e-8, weight_decay=0.0, step=1)
        a.update(kw)
        return lib.adam_step(a["n"], a["grad"], a["grad_scale"], a["master"], a["m"], a["v"], a["weight"], a["lr"],
                             a["beta1"], a["beta2"], a["eps"], a["weight_decay"], a["step"], None)
    assert call(n=0) == mlp.MLP_EINVAL
    assert call(step=0) == mlp.MLP_EINVAL
    assert call(beta1=1.0) == mlp.MLP_EINVAL
    assert call(eps=0.0) == mlp.MLP_EINVAL
    assert call(m=None) == mlp.MLP_EINVAL
    assert call(weight=GOOD + 2) == mlp.MLP_EALIGN


def test_attention_rejects_bad_shapes_without_a_gpu(lib):
    ptrs = [GOOD] * 5
    outs = [GOOD] * 5
    # h, nh, t, tokens, seq_len, p, seed, token_offset, X, Wqkv, bqkv, Wo, bo, R, QKV, S, P, O, out, stream
    assert lib.attn_fwd(96, 16, 1, 64, 32, 0.1, 1, 0, *ptrs, None, *outs, None) == mlp.MLP_EINVAL   # d = 6
    assert lib.attn_fwd(128, 4, 1, 60, 32, 0.1, 1, 0, *ptrs, None, *outs, None) == mlp.MLP_EINVAL   # 60 % 32
    assert lib.attn_fwd(128, 4, 3, 64, 32, 0.1, 1, 0, *ptrs, None, *outs, None) == mlp.MLP_EINVAL   # t does not divide nh
    assert lib.attn_fwd(128, 4, 1, 64, 32, 1.0, 1, 0, *ptrs, None, *outs, None) == mlp.MLP_EINVAL   # p = 1
