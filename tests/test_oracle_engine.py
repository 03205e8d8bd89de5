"""Pins of the oracle's engines: the Var tape against the arena engine and against
closed forms, the page's fan-out identity, dual numbers against printed values,
and the dropout RNG against the published SplitMix64 sequence and its invariants."""
import math
import os

import numpy as np
import pytest

from oracle import arena as A
from oracle import dropout as D
from oracle import dual
from oracle import fd
from oracle import ops as O
from oracle import tape as t

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name), encoding="utf-8"):
        line = line.split("#", 1)[0].strip()
        if line:
            rows.append(line.split())
    return rows


# ----------------------------------------------------------------------------- tape


def test_fanout_four_x():
    """[AE] § 梯度累加: y = x∘x + x∘x ⇒ dL/dx = 4x with L = Σ y."""
    x0 = np.random.default_rng(0).normal(size=(3, 4))
    x = t.leaf(x0)
    y = t.add(t.mul(x, x), t.mul(x, x))
    t.backward(t.sum_all(y))
    assert np.allclose(x.grad, 4 * x0, rtol=0, atol=0)


def test_same_var_twice_visited_once():
    x = t.leaf(np.array([1.5, -2.0]))
    y = t.mul(x, x)
    order = t.topo_order(t.sum_all(y))
    assert sum(1 for n in order if n is x) == 1
    t.backward(t.sum_all(y))
    assert np.array_equal(x.grad, 2 * x.value)


def test_backward_requires_scalar():
    with pytest.raises(ValueError):
        t.backward(t.leaf(np.ones(3)))


def test_tape_matches_arena_engine():
    """Both engines on the same scalar expressions must agree exactly (float64)."""
    vals = {"a": 0.7, "b": -1.3, "c": 2.1}
    # f = sigmoid(a·b) + tanh(b) · exp(c·a) + a·a, with fan-out on a and b
    ar = A.Arena()
    a, b, c = ar.var(vals["a"]), ar.var(vals["b"]), ar.var(vals["c"])
    out = ar.add(ar.add(ar.sigmoid(ar.mul(a, b)), ar.mul(ar.tanh(b), ar.exp(ar.mul(c, a)))), ar.mul(a, a))
    fa = ar.forward(out)
    ar.backward(out)

    # the same expression through the tape (array ops on 0-d values)
    ta, tb, tc = (t.leaf(np.array(vals[k])) for k in "abc")
    ab = t.mul(ta, tb)
    sg = t.Var(O.sigmoid(ab.value), [ab], lambda g, ps: t.push_grad(ps[0], g * O.sigmoid(ps[0].value) * (1 - O.sigmoid(ps[0].value))))
    th = t.Var(np.tanh(tb.value), [tb], lambda g, ps: t.push_grad(ps[0], g * (1 - np.tanh(ps[0].value) ** 2)))
    ca = t.mul(tc, ta)
    ex = t.Var(np.exp(ca.value), [ca], lambda g, ps: t.push_grad(ps[0], g * np.exp(ps[0].value)))
    f = t.add(t.add(sg, t.mul(th, ex)), t.mul(ta, ta))
    t.backward(f)
    assert float(f.value) == pytest.approx(fa, rel=1e-15)
    for v, i in ((ta, a), (tb, b), (tc, c)):
        assert float(v.grad) == pytest.approx(ar.gradient(i), rel=1e-14)
    # and against closed-form partials
    sa = 1 / (1 + math.exp(-vals["a"] * vals["b"]))
    dfa = sa * (1 - sa) * vals["b"] + math.tanh(vals["b"]) * math.exp(vals["c"] * vals["a"]) * vals["c"] + 2 * vals["a"]
    assert ar.gradient(a) == pytest.approx(dfa, rel=1e-14)


def test_arena_tanh_uses_output():
    """The printed engine's tanh backward uses the input; the oracle uses tanh's output."""
    ar = A.Arena()
    x = ar.var(0.8)
    y = ar.tanh(x)
    ar.forward(y)
    ar.backward(y)
    assert ar.gradient(x) == pytest.approx(1 - math.tanh(0.8) ** 2, rel=1e-15)


def test_composed_attention_tape_fd():
    """[AE] § Attention 用组合: end-to-end grad-check of dQ, dK, dV through the tape."""
    r = np.random.default_rng(3)
    q0, k0, v0 = (r.normal(size=(1, 1, 6, 4)) for _ in range(3))
    W = r.normal(size=(1, 1, 6, 4))

    def loss(qa, ka, va):
        q, k, v = t.leaf(qa), t.leaf(ka), t.leaf(va)
        out = t.attention(q, k, v, causal=True)
        L = t.sum_all(t.mul(out, t.leaf(W)))
        return L, (q, k, v)

    L, (q, k, v) = loss(q0, k0, v0)
    t.backward(L)
    for idx, (leafv, x0) in enumerate(((q, q0), (k, k0), (v, v0))):
        def f(x, idx=idx):
            args = [q0, k0, v0]
            args[idx] = x
            return float(loss(*args)[0].value)
        num = fd.numeric_grad(f, x0, eps=1e-5)
        assert fd.max_rel_err(leafv.grad, num) < 1e-6
    # the tape composition equals the oracle's direct attention backward
    _, P = O.attention_fwd(q0, k0, v0, True)
    dQ, dK, dV = O.attention_bwd(W, q0, k0, v0, P)
    assert np.allclose(q.grad, dQ, rtol=1e-12, atol=1e-14)
    assert np.allclose(k.grad, dK, rtol=1e-12, atol=1e-14)
    assert np.allclose(v.grad, dV, rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------------------- dual numbers


def test_dual_printed_values():
    rows = {r[0]: r for r in _read_table("dual_numbers.txt")}
    x = dual.Dual.variable(2.0)
    f = x * x + x * 3.0
    assert f.val == float(rows["f_x2_plus_3x"][2]) and f.deriv == float(rows["f_x2_plus_3x"][3])
    x = dual.Dual.variable(1.5)
    g = (x * x).sin()
    assert g.val == pytest.approx(float(rows["g_sin_x2"][2]), abs=5e-7)
    assert g.deriv == pytest.approx(float(rows["g_sin_x2"][3]), abs=5e-7)
    assert abs(g.deriv - (-2.05756)) > 0.1     # the page's printed derivative is wrong


def test_hyperdual_printed_values():
    rows = {r[0]: (float(r[1]), float(r[2])) for r in _read_table("hyperdual.txt")}
    x, y = dual.HyperDual.var1(2.0), dual.HyperDual.var2(3.0)
    f = x * x * y + x.sin() + y * y * y
    for key, got in (("value", f.val), ("df_dx", f.g1), ("df_dy", f.g2), ("d2f_dxdy", f.h)):
        want, tol = rows[key]
        assert abs(got - want) <= tol, key


def test_dual_checks_op_derivatives():
    """Forward-mode derivatives of silu, gelu and sigmoid equal the oracle's analytic backward."""
    for v in (-3.2, -0.4, 0.0, 0.9, 2.7):
        x = dual.Dual.variable(v)
        s = x.sigmoid()
        assert O.silu_bwd(np.array([1.0]), np.array([v]))[0] == pytest.approx((x * s).deriv, rel=1e-13, abs=1e-15)
        ge = x * 0.5 * ((x / math.sqrt(2.0)).erf() + 1.0)
        assert O.gelu_bwd(np.array([1.0]), np.array([v]))[0] == pytest.approx(ge.deriv, rel=1e-13, abs=1e-15)
        assert O.gelu_fwd(np.array([v]))[0] == pytest.approx(ge.val, rel=1e-13, abs=1e-15)
        # RMS of a 1-vector chain: d/dx [x / sqrt(x² + eps)]
        eps = 1e-5
        r_ = x / (x * x + eps).sqrt()
        _, ir = O.rms_norm_fwd(np.array([[v]]), np.ones(1), eps)
        dx, _ = O.rms_norm_bwd(np.array([[1.0]]), np.array([[v]]), np.ones(1), ir)
        assert dx[0, 0] == pytest.approx(r_.deriv, rel=1e-10, abs=1e-12)


# ----------------------------------------------------------------------------- dropout RNG


def test_splitmix64_published_sequence():
    """SplitMix64 (Steele, Lea & Flood 2014; reference C code by S. Vigna) seeded with 0
    emits 0xe220a8397b1dcdaf, 0x6e789e6aa1b965f4, 0x06c45d188009454f: output k is the
    mixer applied to k·γ, i.e. splitmix64(state) with state = (k−1)·γ."""
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    states = np.array([0, 0x9E3779B97F4A7C15, (2 * 0x9E3779B97F4A7C15) & (2**64 - 1)], dtype=np.uint64)
    got = [int(v) for v in D.splitmix64(states)]
    assert got == want


def test_dropout_uniform_definition_small():
    """u_i from the page's formula evaluated with Python integers, element by element."""
    M = 2**64 - 1
    seed = 0x5EED ^ 0xA77

    def mix(z):
        z = (z + 0x9E3779B97F4A7C15) & M
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M
        return z ^ (z >> 31)

    u = D.uniforms(64, seed)
    for i in range(64):
        h = mix(seed ^ ((i * 0x9E3779B97F4A7C15) & M))
        assert float(u[i]) == (h >> 40) / 2.0**24


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_dropout_keep_fraction(p):
    n = 1 << 20
    keep = D.keep_mask(n, p, 0x5EED)
    sigma = math.sqrt(n * p * (1 - p))
    assert abs(keep.sum() - n * (1 - p)) < 5 * sigma


def test_dropout_expectation_and_identities():
    x = np.random.default_rng(1).normal(size=(64, 32)).astype(np.float32)
    p = 0.3
    acc = np.zeros_like(x, dtype=np.float64)
    K = 400
    for s in range(K):
        acc += D.dropout_fwd(x, p, 1000 + s)
    mean = acc / K
    # E[out] = x; per-element std of the mean is |x|·sqrt(p/(1-p))/sqrt(K)
    z = np.abs(mean - x) / (np.abs(x) * math.sqrt(p / (1 - p)) / math.sqrt(K) + 1e-12)
    assert np.mean(z) < 1.2 and np.max(z) < 6
    # p = 0 and eval are exact identities
    assert np.array_equal(D.dropout_fwd(x, 0.0, 7), x)
    assert np.array_equal(D.dropout_fwd(x, 0.5, 7, training=False), x)
    # backward applies the forward's mask
    out = D.dropout_fwd(np.ones_like(x), p, 7)
    dx = D.dropout_bwd(np.ones_like(x), p, 7)
    assert np.array_equal(out != 0, dx != 0)
    # the mask is the same for f32 and bf16 storage
    xb = D.dropout_fwd(x, p, 7, dtype="bf16")
    assert np.array_equal(xb != 0, D.dropout_fwd(x, p, 7) != 0)
    # kept values are x·scale
    keep = D.keep_mask(x.size, p, 7).reshape(x.shape)
    assert np.array_equal(D.dropout_fwd(x, p, 7)[keep], (x * D.scale_f32(p))[keep])
    with pytest.raises(ValueError):
        D.dropout_fwd(x, 1.0, 7)


def test_dropout_fixed_seed_gradcheck():
    """[DO] § 验证方法 gate 1: with a fixed seed the mask does not move under ±ε."""
    r = np.random.default_rng(2)
    x0 = r.normal(size=(8, 16))
    W = r.normal(size=(8, 16))

    def f(x):
        return float(np.sum(W * t.dropout(t.leaf(x), 0.25, 99).value))

    xv = t.leaf(x0)
    t.backward(t.sum_all(t.mul(t.dropout(xv, 0.25, 99), t.leaf(W))))
    num = fd.numeric_grad(f, x0)
    assert fd.max_rel_err(xv.grad, num) < 1e-6


def test_site_seeds():
    assert D.site_seed(0x5EED, 0, D.SITE_ATTN) == 0x5EED ^ 0xA77
    assert D.site_seed(0x5EED, 3, D.SITE_FFN) == 0x5EED ^ 3 ^ 0xF70
    assert D.site_seed(1, 0, D.SITE_ATTN) != D.site_seed(1, 0, D.SITE_FFN)


def test_dropout_keep_boundary():
    """keep = (u ≥ p): with p equal to one element's u (a multiple of 2⁻²⁴, exact in float32)
    that element is kept, and with p one float32 step above it, dropped."""
    seed = 0x5EED ^ 0xF70
    u = D.uniforms(4096, seed)
    j = int(np.argmin(np.abs(u - np.float32(0.37))))
    assert D.keep_mask(4096, float(u[j]), seed)[j]
    assert not D.keep_mask(4096, float(np.nextafter(u[j], np.float32(1.0))), seed)[j]
