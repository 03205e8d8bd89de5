"""Pins of the oracle's per-op definitions against things other than themselves:
central finite differences of the oracle's own forward (so a wrong backward fails),
closed forms, invariants of the mathematics, and library routines on special cases.
"""
import math

import numpy as np
import pytest
from scipy.special import erf, logsumexp
from scipy.stats import norm as normal_dist

from oracle import fd
from oracle import ops as O

RTOL = 1e-6


def rng(s=0):
    return np.random.default_rng(s)


def fd_check(fwd, grads, inputs, W, eps=1e-6, tol=RTOL):
    """grads: analytic gradients of L = Σ W∘fwd(*inputs) w.r.t. each input."""
    L, _ = fd.weighted_loss(W)
    for k, (x, g) in enumerate(zip(inputs, grads)):
        def f(xk, k=k):
            args = list(inputs)
            args[k] = xk
            return L(fwd(*args))
        num = fd.numeric_grad(f, x, eps)
        # FD round-off is ~1e-16·|L|/ε: entries below 1e-3·max|grad| are held to an
        # absolute bound of tol·1e-3·max|grad| instead of a relative one.
        err = fd.max_rel_err(g, num, floor=1e-3)
        assert err < tol, f"input {k}: rel err {err}"


# ----------------------------------------------------------------------------- linear


def test_matmul_fd_and_library():
    r = rng(1)
    A, B = r.normal(size=(5, 7)), r.normal(size=(7, 3))
    W = r.normal(size=(5, 3))
    dA, dB = O.matmul_bwd(W, A, B)
    fd_check(O.matmul_fwd, [dA, dB], [A, B], W)
    # special case: the definition equals the textbook triple loop
    C = np.zeros((5, 3))
    for i in range(5):
        for j in range(3):
            C[i, j] = sum(A[i, k] * B[k, j] for k in range(7))
    assert np.allclose(O.matmul_fwd(A, B), C, rtol=1e-13, atol=1e-13)


def test_matmul_square_fd():
    """Square operands, so a transposed operand in the backward still has valid shapes."""
    r = rng(15)
    A, B = r.normal(size=(6, 6)), r.normal(size=(6, 6))
    W = r.normal(size=(6, 6))
    dA, dB = O.matmul_bwd(W, A, B)
    fd_check(O.matmul_fwd, [dA, dB], [A, B], W)


def test_add_mul_scale_sum():
    r = rng(2)
    a, b = r.normal(size=(4, 6)), r.normal(size=(4, 6))
    W = r.normal(size=(4, 6))
    fd_check(O.add_fwd, list(O.add_bwd(W)), [a, b], W)
    fd_check(O.mul_fwd, list(O.mul_bwd(W, a, b)), [a, b], W)
    fd_check(lambda x: O.scale_fwd(x, 0.37), [O.scale_bwd(W, 0.37)], [a], W)
    # mul(x, x) contributes twice: d/dx Σ W∘x∘x = 2 W x
    da, db = O.mul_bwd(W, a, a)
    assert np.allclose(da + db, 2 * W * a)
    assert O.sum_fwd(a) == pytest.approx(float(np.sum(a)))
    assert np.all(O.sum_bwd(1.5, (2, 3)) == 1.5)


def test_add_bias():
    r = rng(3)
    x, b = r.normal(size=(9, 5)), r.normal(size=5)
    W = r.normal(size=(9, 5))
    dx, db = O.add_bias_bwd(W)
    fd_check(O.add_bias_fwd, [dx, db], [x, b], W)
    # dbias is the column sum, element by element in a loop
    for c in range(5):
        assert db[c] == pytest.approx(sum(W[r_, c] for r_ in range(9)), rel=1e-14)


# ----------------------------------------------------------------------------- activations


def test_silu():
    r = rng(4)
    x = r.normal(size=(3, 8)) * 3
    W = r.normal(size=(3, 8))
    fd_check(O.silu_fwd, [O.silu_bwd(W, x)], [x], W)
    assert O.silu_fwd(np.array([0.0]))[0] == 0.0
    assert O.silu_bwd(np.array([1.0]), np.array([0.0]))[0] == pytest.approx(0.5)
    # large |x|: silu(x) → x for x → +∞, → 0 for x → −∞ (no overflow)
    assert O.silu_fwd(np.array([800.0]))[0] == pytest.approx(800.0)
    assert abs(O.silu_fwd(np.array([-800.0]))[0]) < 1e-300


def test_swiglu_equals_composition():
    r = rng(5)
    g, u = r.normal(size=(4, 6)) * 2, r.normal(size=(4, 6))
    W = r.normal(size=(4, 6))
    dg, du = O.swiglu_bwd(W, g, u)
    fd_check(O.swiglu_fwd, [dg, du], [g, u], W)
    # exact equality with silu then mul
    assert np.array_equal(O.swiglu_fwd(g, u), O.mul_fwd(O.silu_fwd(g), u))


def test_gelu():
    r = rng(6)
    x = r.normal(size=(3, 7)) * 2
    W = r.normal(size=(3, 7))
    fd_check(O.gelu_fwd, [O.gelu_bwd(W, x)], [x], W)
    assert O.gelu_fwd(np.array([0.0]))[0] == 0.0
    assert O.gelu_bwd(np.array([1.0]), np.array([0.0]))[0] == pytest.approx(0.5)
    # Φ from the normal distribution's CDF (a different library routine than erf)
    xs = np.linspace(-4, 4, 17)
    assert np.allclose(O.gelu_fwd(xs), xs * normal_dist.cdf(xs), rtol=1e-12, atol=1e-15)
    # math.erf on scalars
    for v in (-2.5, -0.3, 0.7, 3.1):
        assert O.gelu_fwd(np.array([v]))[0] == pytest.approx(0.5 * v * (1 + math.erf(v / math.sqrt(2))), rel=1e-13)


# ----------------------------------------------------------------------------- norms


def test_rms_norm():
    r = rng(7)
    x = r.normal(size=(5, 12))
    gamma = 1 + 0.1 * r.normal(size=12)
    W = r.normal(size=(5, 12))
    eps = 1e-5
    y, ir = O.rms_norm_fwd(x, gamma, eps)
    dx, dg = O.rms_norm_bwd(W, x, gamma, ir)
    fd_check(lambda a, b: O.rms_norm_fwd(a, b, eps)[0], [dx, dg], [x, gamma], W)
    # inv_rms from its definition, row by row
    for i in range(5):
        assert ir[i] == pytest.approx(1 / math.sqrt(sum(v * v for v in x[i]) / 12 + eps), rel=1e-14)
    # invariant: Σ_c x·dx = eps·ir³·Σ_c g·x  (g = d∘γ)
    lhs = np.sum(x * dx, axis=1)
    rhs = eps * ir ** 3 * np.sum(W * gamma * x, axis=1)
    assert np.allclose(lhs, rhs, rtol=1e-6, atol=1e-12)
    # constant row c·1 with γ = 1 ⇒ y ≈ sign(c)·1
    yc, _ = O.rms_norm_fwd(np.full((1, 8), 3.0), np.ones(8), 0.0)
    assert np.allclose(yc, 1.0)


def test_layernorm():
    r = rng(8)
    x = r.normal(size=(4, 10)) * 2 + 0.5
    gamma, beta = 1 + 0.1 * r.normal(size=10), 0.1 * r.normal(size=10)
    W = r.normal(size=(4, 10))
    eps = 1e-5
    y, mu, rstd = O.layernorm_fwd(x, gamma, beta, eps)
    dx, dg, db = O.layernorm_bwd(W, x, gamma, mu, rstd)
    fd_check(lambda a, g, b: O.layernorm_fwd(a, g, b, eps)[0], [dx, dg, db], [x, gamma, beta], W)
    # exact invariants: Σ_c dx = 0 and Σ_c dx·x̂ = eps·rstd³·Σ_c g·x̂ (→ 0 as eps → 0)
    xhat = (x - mu[:, None]) * rstd[:, None]
    assert np.allclose(dx.sum(1), 0, atol=1e-12)
    want = eps * rstd ** 3 * np.sum(W * gamma * xhat, axis=1)
    assert np.allclose((dx * xhat).sum(1), want, rtol=1e-6, atol=1e-13)
    # library: numpy's biased variance
    assert np.allclose(rstd, 1 / np.sqrt(np.var(x, axis=1) + eps), rtol=1e-14)


# ----------------------------------------------------------------------------- rope


def test_rope_identities():
    r = rng(9)
    B, H, S, hd = 2, 3, 7, 8
    x = r.normal(size=(B, H, S, hd))
    pos = np.arange(S)
    y = O.rope_fwd(x, pos, 10000.0)
    # position 0 is the identity, forward and backward
    assert np.array_equal(y[:, :, 0], x[:, :, 0])
    assert np.array_equal(O.rope_bwd(x, pos, 10000.0)[:, :, 0], x[:, :, 0])
    # backward is the transpose (inverse) rotation: bwd(fwd(x)) = x
    assert np.allclose(O.rope_bwd(y, pos, 10000.0), x, atol=1e-13)
    # per-pair norm preserved
    h = hd // 2
    n0 = x[..., :h] ** 2 + x[..., h:] ** 2
    n1 = y[..., :h] ** 2 + y[..., h:] ** 2
    assert np.allclose(n0, n1, rtol=1e-13)
    # bwd == fwd with −θ (negated positions)
    assert np.allclose(O.rope_bwd(x, pos, 10000.0), O.rope_fwd(x, -pos, 10000.0), atol=1e-14)
    # FD
    W = r.normal(size=x.shape)
    fd_check(lambda a: O.rope_fwd(a, pos, 10000.0), [O.rope_bwd(W, pos, 10000.0)], [x], W)
    # textbook complex form: (x_i + i x_{i+h}) · e^{iθ}
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * O.rope_angles(pos, hd, 10000.0))
    assert np.allclose(y[..., :h], z.real) and np.allclose(y[..., h:], z.imag)
    # frequency schedule for pair i at position s: s·base^(−2i/hd)
    th = O.rope_angles(np.array([5]), 8, 100.0)
    assert np.allclose(th[0], [5.0, 5 * 100 ** -0.25, 5 * 100 ** -0.5, 5 * 100 ** -0.75])


# ----------------------------------------------------------------------------- softmax


def test_softmax():
    r = rng(10)
    x = r.normal(size=(6, 9)) * 3
    y = O.softmax_fwd(x)
    assert np.allclose(y.sum(1), 1, atol=1e-14)
    # library routine
    assert np.allclose(y, np.exp(x - logsumexp(x, axis=1, keepdims=True)), rtol=1e-13)
    W = r.normal(size=x.shape)
    dx = O.softmax_bwd(W, y)
    assert np.allclose(dx.sum(1), 0, atol=1e-14)          # Jacobian rows sum to zero
    fd_check(O.softmax_fwd, [dx], [x], W)
    # constant row ⇒ uniform
    assert np.allclose(O.softmax_fwd(np.full((1, 5), 7.0)), 0.2)
    # shift invariance and large inputs (safe softmax)
    assert np.allclose(O.softmax_fwd(x + 1000.0), y, rtol=1e-12)


def test_softmax_causal():
    r = rng(11)
    x = r.normal(size=(2, 5, 5))
    y = O.softmax_fwd(x, causal=True)
    assert np.array_equal(y[:, 0], np.tile([1.0, 0, 0, 0, 0], (2, 1)))
    assert np.all(y[:, np.triu_indices(5, 1)[0], np.triu_indices(5, 1)[1]] == 0)
    for s in range(5):   # each row is the plain softmax of its visible prefix
        assert np.allclose(y[:, s, : s + 1], O.softmax_fwd(x[:, s, : s + 1]), rtol=1e-14)
    W = r.normal(size=x.shape)
    fd_check(lambda a: O.softmax_fwd(a, causal=True), [O.softmax_bwd(W, y)], [x], W)


# ----------------------------------------------------------------------------- cross-entropy


def test_cross_entropy():
    r = rng(12)
    R, V = 7, 11
    x = r.normal(size=(R, V)) * 2
    t = r.integers(0, V, size=R)
    loss, lse = O.cross_entropy_fwd(x, t)
    # library: logsumexp, and the loop definition of mean NLL
    assert np.allclose(lse, logsumexp(x, axis=1), rtol=1e-14)
    nll = [-math.log(math.exp(x[i, t[i]]) / sum(math.exp(v) for v in x[i])) for i in range(R)]
    assert loss == pytest.approx(sum(nll) / R, rel=1e-12)
    dx = O.cross_entropy_bwd(x, t, lse, 1.0)
    assert np.allclose(dx.sum(1), 0, atol=1e-15)
    num = fd.numeric_grad(lambda a: O.cross_entropy_fwd(a, t)[0], x)
    assert fd.max_rel_err(dx, num, floor=1e-3) < RTOL
    # upstream scaling
    assert np.allclose(O.cross_entropy_bwd(x, t, lse, 2.5), 2.5 * dx)
    # constant row ⇒ loss = ln V
    l2, _ = O.cross_entropy_fwd(np.zeros((3, V)), np.array([0, 4, 10]))
    assert l2 == pytest.approx(math.log(V), rel=1e-14)
    with pytest.raises(ValueError):
        O.cross_entropy_fwd(x, np.full(R, V))


# ----------------------------------------------------------------------------- embedding


def test_embedding():
    r = rng(13)
    V, d, B, S = 10, 4, 3, 5
    E, P = r.normal(size=(V, d)), r.normal(size=(S, d))
    ids = r.integers(0, V, size=B * S)
    h = O.embedding_fwd(ids, E, P, S)
    for tkn in range(B * S):
        assert np.array_equal(h[tkn], E[ids[tkn]] + P[tkn % S])
    dh = r.normal(size=(B * S, d))
    dE, dP = O.embedding_bwd(ids, dh, V, S, with_pos=True)
    assert np.allclose(dE.sum(0), dh.sum(0))               # Σ_v dE[v] = Σ_t dh[t]
    # one-hot matmul form: dE = onehotᵀ dh
    oh = np.zeros((B * S, V))
    oh[np.arange(B * S), ids] = 1
    assert np.allclose(dE, oh.T @ dh, rtol=1e-14)
    W = r.normal(size=h.shape)
    dE2, dP2 = O.embedding_bwd(ids, W, V, S, with_pos=True)
    fd_check(lambda e, p: O.embedding_fwd(ids, e, p, S), [dE2, dP2], [E, P], W)
    with pytest.raises(ValueError):
        O.embedding_fwd(np.array([V]), E)


# ----------------------------------------------------------------------------- attention


def test_attention_composed():
    r = rng(14)
    B, H, S, hd = 1, 2, 5, 4
    q, k, v = (r.normal(size=(B, H, S, hd)) for _ in range(3))
    O_, P = O.attention_fwd(q, k, v, causal=True)
    W = r.normal(size=O_.shape)
    dQ, dK, dV = O.attention_bwd(W, q, k, v, P)
    fd_check(lambda a, b, c: O.attention_fwd(a, b, c, True)[0], [dQ, dK, dV], [q, k, v], W)
    # S = 1 ⇒ O = V ; causal row 0 ⇒ O[0] = V[0]
    O1, _ = O.attention_fwd(q[:, :, :1], k[:, :, :1], v[:, :, :1])
    assert np.allclose(O1, v[:, :, :1])
    assert np.allclose(O_[:, :, 0], v[:, :, 0])


def test_attention_lse():
    """The softmax normaliser: closed forms (zero queries ⇒ log of the visible-key count;
    causal row 0 ⇒ its single score) and brute force by loops with the library logsumexp."""
    r = rng(15)
    B, H, S, hd = 2, 2, 6, 4
    q, k = r.normal(size=(B, H, S, hd)), r.normal(size=(B, H, S, hd))
    lse = O.attention_lse(q, k, causal=True)
    assert np.allclose(O.attention_lse(np.zeros_like(q), k, causal=True), np.log(np.arange(1, S + 1)), rtol=1e-14)
    assert np.allclose(O.attention_lse(np.zeros_like(q), k, causal=False), np.log(S), rtol=1e-14)
    assert np.allclose(lse[:, :, 0], np.sum(q[:, :, 0] * k[:, :, 0], axis=-1) / 2.0, rtol=1e-14)
    for b in range(B):
        for h in range(H):
            for s_ in range(S):
                sc = [sum(q[b, h, s_, i] * k[b, h, c, i] for i in range(hd)) / math.sqrt(hd) for c in range(s_ + 1)]
                assert abs(lse[b, h, s_] - logsumexp(sc)) <= 1e-13 * max(1.0, abs(lse[b, h, s_]))
    # P = exp(scores − lse) is the oracle's own softmax
    _, P = O.attention_fwd(q, k, k, causal=True)
    sc = np.einsum("bhsd,bhtd->bhst", q, k) / math.sqrt(hd)
    vis = np.tril(np.ones((S, S), dtype=bool))
    assert np.allclose(np.where(vis, np.exp(sc - lse[..., None]), 0.0), P, rtol=1e-12, atol=1e-15)
