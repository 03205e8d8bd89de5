"""Pins of the optimizer-step oracle (microbatch average, global-norm clipping, AdamW)
against things other than itself: PyTorch's own AdamW and gradient-norm clipping run on the
CPU in float64 (independent library implementations), the first-step closed form, the
microbatch-average identity and the clipped-norm invariant."""
import math

import numpy as np
import pytest

from oracle import optim as OP

torch = pytest.importorskip("torch")

HP = dict(lr=3e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def tensors(seed, shapes=((7, 5), (13,), (3, 4, 2))):
    rng = np.random.default_rng(seed)
    return [rng.normal(size=s) for s in shapes]


def test_adamw_matches_torch_over_steps():
    """Five steps of the oracle against torch.optim.AdamW (float64, CPU, same hyperparameters)."""
    p0 = tensors(1)
    tp = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in p0]
    opt = torch.optim.AdamW(tp, lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=HP["weight_decay"])
    p = [x.copy() for x in p0]
    m = [np.zeros_like(x) for x in p0]
    v = [np.zeros_like(x) for x in p0]
    for step in range(1, 6):
        g = tensors(100 + step)
        for t, gg in zip(tp, g):
            t.grad = torch.tensor(gg, dtype=torch.float64)
        opt.step()
        p, m, v, _ = OP.adamw_step(p, g, m, v, step, **HP)
        for t, x in zip(tp, p):
            assert np.allclose(t.detach().numpy(), x, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("max_norm", [0.5, 1e3])
def test_clip_matches_torch(max_norm):
    """Global-norm clipping against torch.nn.utils.clip_grad_norm_ (float64, CPU): the norm it
    reports and the clipped gradients the update sees (through a step with lr·λ = 0, β₁ = 0,
    β₂ → v̂ = g², so the update is the clipped g over |g| + ε)."""
    g = tensors(7)
    tg = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in g]
    for t, x in zip(tg, g):
        t.grad = torch.tensor(x, dtype=torch.float64)
    tnorm = float(torch.nn.utils.clip_grad_norm_(tg, max_norm))
    assert math.isclose(OP.global_grad_norm(g), tnorm, rel_tol=1e-12)
    c = OP.clip_coefficient(OP.global_grad_norm(g), max_norm)
    for t, x in zip(tg, g):
        assert np.allclose(t.grad.numpy(), x * c, rtol=1e-12, atol=0)


def test_first_step_closed_form():
    """At t = 1, m̂ = g and v̂ = g², so θ₁ = θ₀(1 − lr·λ) − lr·g / (|g| + ε)."""
    p0, g = tensors(2), tensors(3)
    z = [np.zeros_like(x) for x in p0]
    p1, m1, v1, _ = OP.adamw_step(p0, g, z, z, 1, **HP)
    for a, b, gg in zip(p1, p0, g):
        want = b * (1 - HP["lr"] * HP["weight_decay"]) - HP["lr"] * gg / (np.abs(gg) + HP["eps"])
        assert np.allclose(a, want, rtol=1e-12, atol=1e-15)
    for mm, vv, gg in zip(m1, v1, g):
        assert np.allclose(mm, 0.1 * gg) and np.allclose(vv, 0.05 * gg * gg)


@pytest.mark.parametrize("n", [2, 4])
def test_microbatch_average_identity(n):
    """[BP] § Ackumulation över mikrobatcher: n identical microbatches summed into the buffers
    and scaled by 1/n give the same step as one microbatch (exact for n a power of two)."""
    p0, g = tensors(4), tensors(5)
    z = [np.zeros_like(x) for x in p0]
    one = OP.adamw_step(p0, g, z, z, 3, **HP, max_norm=1.0)
    many = OP.adamw_step(p0, [n * x for x in g], z, z, 3, **HP, max_norm=1.0, grad_scale=1.0 / n)
    assert one[3] == many[3]
    for a, b in zip(one[0], many[0]):
        assert np.array_equal(a, b)


def test_clipped_norm_is_max_norm():
    """With the norm above max_norm, the gradients AdamW sees have norm max_norm·‖g‖/(‖g‖+1e-6);
    below it they are untouched."""
    g = tensors(6)
    n = OP.global_grad_norm(g)
    c = OP.clip_coefficient(n, 0.25 * n)
    assert math.isclose(OP.global_grad_norm([x * c for x in g]), 0.25 * n * n / (n + 1e-6), rel_tol=1e-12)
    assert OP.clip_coefficient(n, 2 * n) == 1.0 and OP.clip_coefficient(n, 0.0) == 1.0
