"""CPU oracle of the mixed-precision Adam step (test infrastructure only).

The pages state the cost of mixed-precision Adam, about 20 bytes of training
state per parameter ("Using DeepSpeed and Megatron to Train Megatron-Turing NLG
530B", summary page, Key points), but not the update itself.  The update is the
published Adam algorithm with decoupled weight decay (Kingma & Ba, "Adam: A Method
for Stochastic Optimization", 2015, Algorithm 1; Loshchilov & Hutter, "Decoupled
Weight Decay Regularization", 2019).  Reading of the state: bf16 model weights (2 B),
the fp32 gradient accumulator of the block (4 B), fp32 master weights (4 B) and the
fp32 moments m and v (4 B each): 18 B per parameter.

One step t (t = 1, 2, ...) on every parameter, in float64:
    g  = grad * grad_scale                      (e.g. 1 / micro-batches)
    m  = beta1 m + (1 - beta1) g
    v  = beta2 v + (1 - beta2) g^2
    m_hat = m / (1 - beta1^t),   v_hat = v / (1 - beta2^t)
    w  = w - lr * weight_decay * w - lr * m_hat / (sqrt(v_hat) + eps)
    weight_bf16 = round_to_bf16(w)
The bias-corrected form is written as step_size = lr / (1 - beta1^t) times
m / (sqrt(v) / sqrt(1 - beta2^t) + eps), which equals the expression above.

Pinned by tests/test_oracle_adam.py against torch.optim.AdamW (float64) and closed
forms (first step, zero gradient).
"""
from __future__ import annotations

import math

import numpy as np

from .mlp_oracle import round_bf16


def adam_step(grad, master, m, v, step, lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0, grad_scale=1.0):
    """Returns (master, m, v, weight_bf16_values) after step number ``step`` (>= 1).

    All arrays float64 (the fp32 state decoded exactly); inputs are not modified."""
    g = np.asarray(grad, dtype=np.float64) * grad_scale
    m_new = beta1 * np.asarray(m, dtype=np.float64) + (1.0 - beta1) * g
    v_new = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g * g
    bc1 = 1.0 - beta1 ** step
    bc2 = 1.0 - beta2 ** step
    denom = np.sqrt(v_new) / math.sqrt(bc2) + eps
    w = np.asarray(master, dtype=np.float64)
    w_new = w - lr * weight_decay * w - (lr / bc1) * m_new / denom
    return w_new, m_new, v_new, round_bf16(w_new)
