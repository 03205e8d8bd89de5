"""Host logic of the GPU tape, on CPU: which buffer each push lands in.

The tape's arithmetic runs in libxt; here the few kernels these graphs need are replaced by
torch CPU ops (a test-only stand-in, never used by the product), so that the tape's own
decisions — topological order, first push sets / later pushes add, buffer ownership — are
checked without a GPU against the oracle's tape ([AE] § Tape 设计 and § 梯度累加: the first
contribution sets a Var's grad, later ones are added, per Var)."""
import types

import numpy as np
import pytest
import torch

from oracle import tape as OT
from transformer_fwd_bwd_gb300 import tape as T


def _fake_xt():
    def ew(fn):
        def call(*args, **kw):
            fn(*args)
        return call

    def convert(dst, src):
        dst.copy_(src.to(dst.dtype))

    def accumulate(dst, src):
        dst.add_(src.to(dst.dtype))

    def add_fwd(a, b, y):
        torch.add(a, b, out=y)

    def mul_fwd(a, b, y):
        torch.mul(a, b, out=y)

    def mul_bwd(g, a, b, da, db):
        torch.mul(g, b, out=da)
        torch.mul(g, a, out=db)

    def scale_fwd(x, y, alpha):
        torch.mul(x, alpha, out=y)

    def scale_bwd(g, dx, alpha):
        torch.mul(g, alpha, out=dx)

    def sum_fwd(x, y):
        y.copy_(x.to(torch.float64).sum().to(y.dtype).reshape(1))

    def sum_bwd(g, dx):
        dx.fill_(float(g.reshape(-1)[0]))

    def silu_fwd(x, y):
        torch.mul(x, torch.sigmoid(x), out=y)

    def silu_bwd(g, x, dx):
        s = torch.sigmoid(x)
        torch.mul(g, s * (1 + x * (1 - s)), out=dx)

    return types.SimpleNamespace(
        xt_convert=ew(convert), xt_accumulate=ew(accumulate), xt_add_fwd=ew(add_fwd), xt_mul_fwd=ew(mul_fwd),
        xt_mul_bwd=ew(mul_bwd), xt_scale_fwd=ew(scale_fwd), xt_scale_bwd=ew(scale_bwd), xt_sum_fwd=ew(sum_fwd),
        xt_sum_bwd=ew(sum_bwd), xt_silu_fwd=ew(silu_fwd), xt_silu_bwd=ew(silu_bwd))


@pytest.fixture
def cpu_tape(monkeypatch):
    monkeypatch.setattr(T, "xt", _fake_xt())
    return T


def _graphs():
    """Graphs whose reverse walk gives an add's (or a mul's) parents their first push from that
    node and a later push from another consumer: the pattern that exposes a shared buffer."""
    def scale_then_add(lib, x, y):
        # L = Σ(2x) + Σ(x + y): add's backward runs first and sets x and y; scale's adds 2 to x only
        return lib.add(lib.sum_all(lib.scale(x, 2.0)), lib.sum_all(lib.add(x, y)))

    def residual_chain(lib, x, y):
        # u = 3x, v = silu(y), s = u + v; L = Σ(0.5u) + Σ(v∘y) + Σ(s∘s): the s-branch walks first, so
        # u and v take their first push from the add, then one more each from their own consumers
        u, v = lib.scale(x, 3.0), lib.silu(y)
        s = lib.add(u, v)
        other = lib.add(lib.sum_all(lib.scale(u, 0.5)), lib.sum_all(lib.mul(v, y)))
        return lib.add(other, lib.sum_all(lib.mul(s, s)))

    def fan_out_four_x(lib, x, y):
        # [AE] § 梯度累加: y = x∘x + x∘x ⇒ dL/dx = 4x; y takes no part (zero grad is never pushed)
        return lib.add(lib.sum_all(lib.add(lib.mul(x, x), lib.mul(x, x))), lib.sum_all(lib.scale(y, 0.0)))

    return {"scale_then_add": scale_then_add, "residual_chain": residual_chain, "fan_out_four_x": fan_out_four_x}


@pytest.mark.parametrize("name", sorted(_graphs()))
def test_tape_push_matches_oracle_tape(cpu_tape, name):
    build = _graphs()[name]
    rng = np.random.default_rng(90)
    x0, y0 = rng.standard_normal((5, 7)), rng.standard_normal((5, 7))
    x, y = T.leaf(torch.tensor(x0)), T.leaf(torch.tensor(y0))
    T.backward(build(T, x, y))
    rx, ry = OT.leaf(x0), OT.leaf(y0)
    OT.backward(build(OT, rx, ry))
    np.testing.assert_allclose(x.grad.numpy(), rx.grad, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y.grad.numpy(), ry.grad, rtol=1e-12, atol=1e-12)


def test_scale_then_add_closed_form(cpu_tape):
    """L = Σ(2x) + Σ(x + y) ⇒ dL/dx = 3, dL/dy = 1 everywhere (a shared add buffer gave dy = 3)."""
    x, y = T.leaf(torch.zeros(4, 3, dtype=torch.float64)), T.leaf(torch.zeros(4, 3, dtype=torch.float64))
    T.backward(_graphs()["scale_then_add"](T, x, y))
    assert torch.equal(x.grad, torch.full((4, 3), 3.0, dtype=torch.float64))
    assert torch.equal(y.grad, torch.ones(4, 3, dtype=torch.float64))


def test_no_two_vars_share_a_grad_buffer(cpu_tape):
    rng = np.random.default_rng(91)
    x, y = (T.leaf(torch.tensor(rng.standard_normal((3, 4)))) for _ in range(2))
    u, v = T.scale(x, 3.0), T.silu(y)
    s = T.add(u, v)
    T.backward(T.add(T.sum_all(T.mul(s, s)), T.sum_all(T.add(u, v))))
    bufs = [t.grad.data_ptr() for t in (x, y, u, v, s)]
    assert len(set(bufs)) == len(bufs)
