"""Training-step tail after the backward, in float64: microbatch averaging, global
gradient-norm clipping and the AdamW update.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[BP] § Ackumulation över mikrobatcher: the backward of every microbatch adds into the
gradient buffers; the sum is scaled by 1 / n_microbatches before one optimizer step, and
the buffers are zeroed for the next step.
[BP] § Parningsdisciplinen names the helper kernels of gradient clipping (a partial and a
final gradient-norm reduction, then a gradient scale).
[BP] § Optimiser-tillståndet: AdamW keeps two extra buffers per weight, the first moment m
and the second moment v.

Readings (the pages give no formulas): the clipping is global-norm clipping over every
gradient tensor, g ← g · min(1, max_norm / (‖g‖₂ + 1e-6)), applied to the averaged
gradients (max_norm ≤ 0 disables it); AdamW is Adam with decoupled weight decay, bias
corrected with the step count t ≥ 1:
    m ← β₁ m + (1 − β₁) g,   v ← β₂ v + (1 − β₂) g²,
    m̂ = m / (1 − β₁ᵗ),        v̂ = v / (1 − β₂ᵗ),
    θ ← θ (1 − lr·λ) − lr · m̂ / (√v̂ + ε).
"""
from __future__ import annotations

import math

import numpy as np


def f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def global_grad_norm(grads, scale=1.0):
    """‖scale · g‖₂ over every element of every tensor in `grads` (a list)."""
    s = 0.0
    for g in grads:
        s += float(np.sum((f64(g) * scale) ** 2))
    return math.sqrt(s)


def clip_coefficient(norm, max_norm):
    """min(1, max_norm / (norm + 1e-6)); 1 when clipping is off (max_norm ≤ 0)."""
    if max_norm <= 0:
        return 1.0
    return min(1.0, max_norm / (norm + 1e-6))


def adamw_tensor(p, g, m, v, step, lr, beta1, beta2, eps, weight_decay):
    """AdamW on one tensor with its (already scaled and clipped) gradient g.  Returns
    (new θ, new m, new v)."""
    g = f64(g)
    m = beta1 * f64(m) + (1.0 - beta1) * g
    v = beta2 * f64(v) + (1.0 - beta2) * g * g
    mhat = m / (1.0 - beta1 ** step)
    vhat = v / (1.0 - beta2 ** step)
    p = f64(p) * (1.0 - lr * weight_decay) - lr * mhat / (np.sqrt(vhat) + eps)
    return p, m, v


def adamw_step(params, grads, m, v, step, lr, beta1, beta2, eps, weight_decay, max_norm=0.0, grad_scale=1.0):
    """One optimizer step over lists of tensors.  The gradients are first scaled by
    grad_scale (1 / n_microbatches), then clipped to the global norm max_norm, then AdamW
    updates each tensor.  Returns (new params, new m, new v, the norm before clipping)."""
    norm = global_grad_norm(grads, grad_scale)
    c = clip_coefficient(norm, max_norm)
    out_p, out_m, out_v = [], [], []
    for p, g, mm, vv in zip(params, grads, m, v):
        p, mm, vv = adamw_tensor(p, f64(g) * grad_scale * c, mm, vv, step, lr, beta1, beta2, eps, weight_decay)
        out_p.append(p)
        out_m.append(mm)
        out_v.append(vv)
    return out_p, out_m, out_v, norm
