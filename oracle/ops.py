"""Forward and analytic backward of every op on the hot path, in float64.

Each function is the plain definition written out; no blocking, fusion or
reordering.  Arrays are row-major; "rows" are the leading dims, "cols" the last.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf as _erf


def f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------------------
# Linear / elementwise ops — [AE] § Key Design Decisions, op backward table
# ---------------------------------------------------------------------------------------

def matmul_fwd(A, B):
    """C = A @ B.  [AE] op table row `matmul`."""
    return f64(A) @ f64(B)


def matmul_bwd(d, A, B):
    """dA = d @ Bᵀ, dB = Aᵀ @ d (transposes act on the last two axes when batched).
    [AE] op table row `matmul`."""
    d, A, B = f64(d), f64(A), f64(B)
    return d @ np.swapaxes(B, -1, -2), np.swapaxes(A, -1, -2) @ d


def add_fwd(a, b):
    """a + b.  [AE] op table row `add`."""
    return f64(a) + f64(b)


def add_bwd(d):
    """da = d, db = d.  [AE] op table row `add`."""
    d = f64(d)
    return d.copy(), d.copy()


def mul_fwd(a, b):
    """a ∘ b.  [AE] op table row `mul`."""
    return f64(a) * f64(b)


def mul_bwd(d, a, b):
    """da = d ∘ b, db = d ∘ a.  [AE] op table row `mul`."""
    d = f64(d)
    return d * f64(b), d * f64(a)


def scale_fwd(x, alpha):
    """x · α.  [AE] op table row `scale`."""
    return f64(x) * alpha


def scale_bwd(d, alpha):
    """dx = d · α.  [AE] op table row `scale`."""
    return f64(d) * alpha


def sum_fwd(x):
    """Full sum to a scalar: the reduction behind the validation loss L = Σ W∘out
    ([AE] § 验证方法)."""
    return np.sum(f64(x))


def sum_bwd(g, shape):
    """dx = g broadcast to the input shape."""
    return np.full(shape, float(g))


def add_bias_fwd(x, bias):
    """y[r,c] = x[r,c] + bias[c].  [AE] op table row `add_bias`."""
    return f64(x) + f64(bias)[None, :]


def add_bias_bwd(d):
    """dx = d; dbias[c] = Σ_r d[r,c] (sum along the broadcast dim).  [AE] op table row `add_bias`."""
    d = f64(d)
    return d.copy(), d.sum(axis=0)


# ---------------------------------------------------------------------------------------
# Activations
# ---------------------------------------------------------------------------------------

def sigmoid(x):
    x = f64(x)
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-x[pos]))
    ex = np.exp(x[~pos])
    out[~pos] = ex / (1.0 + ex)
    return out


def silu_fwd(x):
    """y = x·σ(x).  [AE] op table row `silu`."""
    x = f64(x)
    return x * sigmoid(x)


def silu_bwd(d, x):
    """dx = d·(σ + x·σ·(1−σ)).  [AE] op table row `silu`."""
    x = f64(x)
    s = sigmoid(x)
    return f64(d) * (s + x * s * (1.0 - s))


def swiglu_fwd(g, u):
    """y = silu(g) ∘ u.  [AE] op table row `swiglu` (g is the gate projection)."""
    return silu_fwd(g) * f64(u)


def swiglu_bwd(d, g, u):
    """Backward by composition of silu and mul, as [AE] op table row `swiglu` states:
    with a = silu(g), y = a∘u ⇒ da = d∘u, du = d∘a, dg = silu_bwd(da, g)."""
    d, u = f64(d), f64(u)
    a = silu_fwd(g)
    da, du = mul_bwd(d, a, u)
    return silu_bwd(da, g), du


def gelu_fwd(x):
    """Exact GELU y = x·Φ(x) = ½x(1 + erf(x/√2)).

    [BP] § Varje Forward-op Får En Backward-tvilling (k_mlp_fwd: MLP with GELU) names
    GELU without its variant; the definition (erf form) is taken.
    """
    x = f64(x)
    return 0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)))


def gelu_bwd(d, x):
    """dx = d·(Φ(x) + x·φ(x)); the saved tensor is the pre-activation x
    ([BP] § Sparade tensorer: k_mlp_bwd needs the GELU pre-activation)."""
    x = f64(x)
    Phi = 0.5 * (1.0 + _erf(x / math.sqrt(2.0)))
    phi = np.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)
    return f64(d) * (Phi + x * phi)


# ---------------------------------------------------------------------------------------
# Norms
# ---------------------------------------------------------------------------------------

def rms_norm_fwd(x, gamma, eps):
    """ir = 1/√(mean_c x² + eps); y = x·ir·γ; returns (y, ir).  [AE] § RMSNorm."""
    x = f64(x)
    ir = 1.0 / np.sqrt(np.mean(x * x, axis=-1) + eps)
    return x * ir[..., None] * f64(gamma), ir


def rms_norm_bwd(d, x, gamma, ir):
    """g = d∘γ, n = cols:
    dx = ir·g − x·ir³/n·Σ_c g·x ;  dγ[c] = Σ_r d·x·ir.  [AE] § RMSNorm."""
    d, x, gamma, ir = f64(d), f64(x), f64(gamma), f64(ir)
    n = x.shape[-1]
    g = d * gamma
    s = np.sum(g * x, axis=-1)
    dx = ir[..., None] * g - x * (ir ** 3 / n * s)[..., None]
    dgamma = np.sum((d * x * ir[..., None]).reshape(-1, n), axis=0)
    return dx, dgamma


def layernorm_fwd(x, gamma, beta, eps):
    """μ = mean x; var = mean (x−μ)² (biased); rstd = 1/√(var+eps);
    x̂ = (x−μ)·rstd; y = x̂·γ + β; returns (y, μ, rstd).

    [BP] § Varje Forward-op Får En Backward-tvilling (k_layernorm_fwd) and § Sparade
    tensorer (mean and variance saved for k_layernorm_bwd) name LayerNorm without its
    formula; the standard definition is taken, saving rstd as the variance encoding.
    """
    x = f64(x)
    mu = np.mean(x, axis=-1)
    xc = x - mu[..., None]
    var = np.mean(xc * xc, axis=-1)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = xc * rstd[..., None]
    return xhat * f64(gamma) + f64(beta), mu, rstd


def layernorm_bwd(d, x, gamma, mu, rstd):
    """g = d∘γ: dx = rstd·(g − mean g − x̂·mean(g∘x̂)); dγ = Σ_r d∘x̂; dβ = Σ_r d."""
    d, x, gamma, mu, rstd = f64(d), f64(x), f64(gamma), f64(mu), f64(rstd)
    n = x.shape[-1]
    xhat = (x - mu[..., None]) * rstd[..., None]
    g = d * gamma
    dx = rstd[..., None] * (g - np.mean(g, axis=-1, keepdims=True)
                            - xhat * np.mean(g * xhat, axis=-1, keepdims=True))
    dgamma = np.sum((d * xhat).reshape(-1, n), axis=0)
    dbeta = np.sum(d.reshape(-1, n), axis=0)
    return dx, dgamma, dbeta


# ---------------------------------------------------------------------------------------
# RoPE — [AE] op table row `rope` and § RoPE 反向推导
# ---------------------------------------------------------------------------------------

def rope_angles(positions, hd, base):
    """θ[s, i] = pos_s · base^(−2i/hd) for i < hd/2, in float64.

    The pages state the rotation (rotate-half pairs (i, i+h)) but not the frequency
    schedule; the standard schedule with `base` is taken.
    """
    pos = f64(positions)
    i = np.arange(hd // 2, dtype=np.float64)
    inv = base ** (-2.0 * i / hd)
    return pos[..., None] * inv


def rope_fwd(x, positions, base):
    """x[..., S, hd] with positions[S]: per pair (i, i+h), h = hd/2:
    y_i = x_i cos θ − x_{i+h} sin θ ;  y_{i+h} = x_{i+h} cos θ + x_i sin θ.

    The forward is the rotation whose transpose [AE] § RoPE 反向推导 prints as the backward.
    """
    x = f64(x)
    hd = x.shape[-1]
    h = hd // 2
    th = rope_angles(positions, hd, base)
    c, s = np.cos(th), np.sin(th)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_bwd(d, positions, base):
    """dx_i = d_i cos + d_{i+h} sin ;  dx_{i+h} = d_{i+h} cos − d_i sin.  [AE] § RoPE 反向推导."""
    d = f64(d)
    hd = d.shape[-1]
    h = hd // 2
    th = rope_angles(positions, hd, base)
    c, s = np.cos(th), np.sin(th)
    d1, d2 = d[..., :h], d[..., h:]
    return np.concatenate([d1 * c + d2 * s, d2 * c - d1 * s], axis=-1)


# ---------------------------------------------------------------------------------------
# Softmax — [AE] op table row `softmax` and § Softmax 反向推导
# ---------------------------------------------------------------------------------------

def causal_mask(q_len, k_len):
    """True where key c is visible from query s (c ≤ s)."""
    s = np.arange(q_len)[:, None]
    c = np.arange(k_len)[None, :]
    return c <= s


def softmax_fwd(x, causal=False):
    """Row-wise safe softmax y = exp(x − max)/Σ exp(x − max) over the visible columns.

    With causal=True, x is [..., S_q, S_k] and column c of row s is masked when
    c > s; masked entries get y = 0 and take no part in the max or the sum.
    """
    x = f64(x)
    if causal:
        vis = causal_mask(x.shape[-2], x.shape[-1])
        xm = np.where(vis, x, -np.inf)
    else:
        xm = x
    m = np.max(xm, axis=-1, keepdims=True)
    e = np.exp(xm - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def softmax_bwd(d, y):
    """dx = y ∘ (d − Σ_c d∘y)."""
    d, y = f64(d), f64(y)
    return y * (d - np.sum(d * y, axis=-1, keepdims=True))


# ---------------------------------------------------------------------------------------
# Cross-entropy — [AE] op table row `cross_entropy` and § Cross-entropy 反向推导
# ---------------------------------------------------------------------------------------

def logsumexp_rows(x):
    x = f64(x)
    m = np.max(x, axis=-1)
    return m + np.log(np.sum(np.exp(x - m[:, None]), axis=-1))


def cross_entropy_fwd(x, targets):
    """loss = (1/R) Σ_r (lse(x_r) − x_r[t_r]); returns (loss, lse[R])."""
    x = f64(x)
    t = np.asarray(targets, dtype=np.int64)
    R = x.shape[0]
    if np.any(t < 0) or np.any(t >= x.shape[1]):
        raise ValueError("target out of range")
    lse = logsumexp_rows(x)
    return float(np.mean(lse - x[np.arange(R), t])), lse


def cross_entropy_bwd(x, targets, lse, upstream):
    """dx = upstream·(softmax(x_r) − onehot(t_r))/R."""
    x = f64(x)
    t = np.asarray(targets, dtype=np.int64)
    R = x.shape[0]
    p = np.exp(x - f64(lse)[:, None])
    p[np.arange(R), t] -= 1.0
    return p * (float(upstream) / R)


# ---------------------------------------------------------------------------------------
# Embedding — [BP] § Varje Forward-op Får En Backward-tvilling (k_embed_fwd/bwd),
# § Var gradienter lever i minnet (token and position embeddings)
# ---------------------------------------------------------------------------------------

def embedding_fwd(ids, E, P=None, S=None):
    """h[t] = E[id[t]] (+ P[t mod S] when learned positions are used)."""
    ids = np.asarray(ids, dtype=np.int64)
    E = f64(E)
    if np.any(ids < 0) or np.any(ids >= E.shape[0]):
        raise ValueError("token id out of range")
    h = E[ids].copy()
    if P is not None:
        h += f64(P)[np.arange(len(ids)) % S]
    return h


def embedding_bwd(ids, dh, V, S=None, with_pos=False):
    """dE[v] = Σ_{t: id[t]=v} dh[t], summed in ascending t;  dP[s] = Σ_b dh[b·S + s]."""
    ids = np.asarray(ids, dtype=np.int64)
    dh = f64(dh)
    dE = np.zeros((V, dh.shape[1]))
    for t in range(len(ids)):
        dE[ids[t]] += dh[t]
    dP = None
    if with_pos:
        dP = dh.reshape(-1, S, dh.shape[1]).sum(axis=0)
    return dE, dP


# ---------------------------------------------------------------------------------------
# Composed attention — [AE] § Attention 用组合
# ---------------------------------------------------------------------------------------

def attention_fwd(q, k, v, causal=True):
    """Per (batch, head): scores = (Q Kᵀ)·(1/√hd); P = softmax(scores); O = P V.

    q, k, v are [B, H, S, hd].  The page's 1/√d is read as 1/√head_dim.
    Returns (O, P).
    """
    q, k, v = f64(q), f64(k), f64(v)
    hd = q.shape[-1]
    scores = np.einsum("bhsd,bhtd->bhst", q, k) * (1.0 / math.sqrt(hd))
    P = softmax_fwd(scores, causal=causal)
    return np.einsum("bhst,bhtd->bhsd", P, v), P


def attention_lse(q, k, causal=True):
    """Per (batch, head, query s): the natural-log normaliser of the attention softmax,
    lse[s] = log Σ_c exp(scores[s, c]) over the visible keys c, scores = (Q Kᵀ)/√hd — the
    quantity the safe softmax divides by, so that P = exp(scores − lse).  [B, H, S]."""
    q, k = f64(q), f64(k)
    hd = q.shape[-1]
    scores = np.einsum("bhsd,bhtd->bhst", q, k) * (1.0 / math.sqrt(hd))
    if causal:
        scores = np.where(causal_mask(scores.shape[-2], scores.shape[-1]), scores, -np.inf)
    m = np.max(scores, axis=-1, keepdims=True)
    return (m + np.log(np.sum(np.exp(scores - m), axis=-1, keepdims=True)))[..., 0]


def attention_bwd(dO, q, k, v, P):
    """Backward of the composition matmul → scale → softmax → matmul, step by step."""
    dO, q, k, v, P = f64(dO), f64(q), f64(k), f64(v), f64(P)
    hd = q.shape[-1]
    dP = np.einsum("bhsd,bhtd->bhst", dO, v)            # dP = dO Vᵀ
    dV = np.einsum("bhst,bhsd->bhtd", P, dO)            # dV = Pᵀ dO
    dS = softmax_bwd(dP, P)
    dS = scale_bwd(dS, 1.0 / math.sqrt(hd))
    dQ = np.einsum("bhst,bhtd->bhsd", dS, k)            # dQ = dS K
    dK = np.einsum("bhst,bhsd->bhtd", dS, q)            # dK = dSᵀ Q
    return dQ, dK, dV
