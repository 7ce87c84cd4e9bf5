"""Pins of the Adam-step oracle: torch.optim.AdamW in float64 (a library routine
implementing the published algorithm), and closed forms of special cases."""
import numpy as np
import pytest
import torch

from oracle import adam_oracle as ado
from oracle import mlp_oracle as orc


def _state(n, rng):
    master = rng.standard_normal(n) * 0.02
    m = rng.standard_normal(n) * 1e-3
    v = np.abs(rng.standard_normal(n)) * 1e-6
    grad = rng.standard_normal(n) * 3.0
    return grad, master, m, v


@pytest.mark.parametrize("wd,scale", [(0.0, 1.0), (0.1, 0.25)])
def test_matches_torch_adamw_over_several_steps(wd, scale):
    rng = np.random.default_rng(0)
    n = 4096
    _, master, _, _ = _state(n, rng)
    p = torch.nn.Parameter(torch.from_numpy(master.copy()))
    opt = torch.optim.AdamW([p], lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=wd)
    w, m, v = master.copy(), np.zeros(n), np.zeros(n)
    for step in range(1, 6):
        grad = rng.standard_normal(n) * 2.0
        p.grad = torch.from_numpy(grad * scale)
        opt.step()
        w, m, v, wb = ado.adam_step(grad, w, m, v, step, 1e-3, 0.9, 0.95, 1e-8, wd, grad_scale=scale)
        st = opt.state[p]
        np.testing.assert_allclose(w, p.detach().numpy(), rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=1e-12, atol=1e-18)
        np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-12, atol=1e-20)
        np.testing.assert_array_equal(wb, orc.round_bf16(w))


def test_first_step_is_a_signed_learning_rate():
    """From m = v = 0 the bias-corrected update is lr * g / (|g| + eps)."""
    rng = np.random.default_rng(1)
    grad, master, _, _ = _state(1000, rng)
    lr = 3e-4
    w, m, v, _ = ado.adam_step(grad, master, np.zeros_like(grad), np.zeros_like(grad), 1, lr, 0.9, 0.95, 1e-8)
    np.testing.assert_allclose(master - w, lr * grad / (np.abs(grad) + 1e-8), rtol=1e-12)
    np.testing.assert_allclose(m, 0.1 * grad, rtol=1e-15)
    np.testing.assert_allclose(v, 0.05 * grad * grad, rtol=1e-14)


def test_zero_gradient_only_decays():
    rng = np.random.default_rng(2)
    _, master, _, _ = _state(1000, rng)
    z = np.zeros_like(master)
    w, m, v, _ = ado.adam_step(z, master, z, z, 7, 1e-3, 0.9, 0.95, 1e-8, weight_decay=0.1)
    np.testing.assert_array_equal(m, 0.0)
    np.testing.assert_array_equal(v, 0.0)
    np.testing.assert_allclose(w, master * (1 - 1e-4), rtol=1e-15)


def test_planted_mistakes_are_caught():
    """No bias correction, eps inside the square root, or weight decay coupled into
    the gradient (L2 instead of decoupled) all break the AdamW pin."""
    rng = np.random.default_rng(5)
    n = 2048
    grad, master, m, v = _state(n, rng)
    lr, b1, b2, eps, wd, step = 1e-3, 0.9, 0.95, 1e-8, 0.1, 3
    p = torch.nn.Parameter(torch.from_numpy(master.copy()))
    opt = torch.optim.AdamW([p], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd)
    opt.state[p] = {"step": torch.tensor(float(step - 1)), "exp_avg": torch.from_numpy(m.copy()),
                    "exp_avg_sq": torch.from_numpy(v.copy())}
    p.grad = torch.from_numpy(grad.copy())
    opt.step()
    ref = p.detach().numpy()
    w, _, _, _ = ado.adam_step(grad, master, m, v, step, lr, b1, b2, eps, wd)
    np.testing.assert_allclose(w, ref, rtol=1e-12, atol=1e-15)
    m1 = b1 * m + (1 - b1) * grad
    v1 = b2 * v + (1 - b2) * grad * grad
    no_bias_corr = master - lr * wd * master - lr * m1 / (np.sqrt(v1) + eps)
    eps_inside = master - lr * wd * master - (lr / (1 - b1 ** step)) * m1 / np.sqrt(v1 / (1 - b2 ** step) + eps)
    g2 = grad + wd * master
    m2 = b1 * m + (1 - b1) * g2
    v2 = b2 * v + (1 - b2) * g2 * g2
    coupled = master - (lr / (1 - b1 ** step)) * m2 / (np.sqrt(v2 / (1 - b2 ** step)) + eps)
    for bad in (no_bias_corr, eps_inside, coupled):
        assert not np.allclose(bad, ref, rtol=1e-12, atol=1e-15)  # the pin's tolerance
