"""Central finite differences: the page's grad-check harness, in float64.

[AE] § 验证方法: scalar loss L = Σ W∘out with a fixed random W (so dL/dout = W);
each input's analytic gradient is compared with (L(x+ε) − L(x−ε)) / 2ε.
The page's ε and tolerances (1e-2 / 2e-2 linear, 1e-3 / 3e-2 / atol 1e-3
non-linear) are for float32 on a GPU; in float64 ε = 1e-6 leaves an O(ε²)
truncation error far below the 1e-6 relative bound the oracle tests use.
"""
from __future__ import annotations

import numpy as np


def numeric_grad(f, x, eps=1e-6, idx=None):
    """∂f/∂x by central differences; f maps an array to a float.  `idx` limits the
    entries probed (flat indices); the others are returned as NaN."""
    x = np.array(x, dtype=np.float64, copy=True)
    g = np.full(x.size, np.nan)
    flat = x.reshape(-1)
    probe = range(x.size) if idx is None else idx
    for i in probe:
        old = flat[i]
        flat[i] = old + eps
        fp = f(x)
        flat[i] = old - eps
        fm = f(x)
        flat[i] = old
        g[i] = (fp - fm) / (2.0 * eps)
    return g.reshape(x.shape)


def weighted_loss(W):
    """L(out) = Σ W∘out and its gradient dL/dout = W."""
    W = np.asarray(W, dtype=np.float64)
    return (lambda out: float(np.sum(W * out))), W


def max_rel_err(a, b, floor=1e-6):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    mask = ~np.isnan(b)
    den = np.maximum(np.abs(b[mask]), floor * max(np.max(np.abs(b[mask])), 1e-300))
    return float(np.max(np.abs(a[mask] - b[mask]) / den)) if mask.any() else 0.0
