"""Reverse-mode tape over libxt's per-op kernels (define-by-run).

[AE] § Key Design Decisions / Tape 设计 and § 梯度累加:
  * a Var holds a value (device tensor), an optional grad, its parents and an optional
    backward closure (None marks a leaf);
  * backward(loss): post-order DFS from the loss, de-duplicated by object identity; the loss
    must be a scalar and its grad is seeded with 1; nodes are walked in reverse order and
    each closure receives the node's accumulated grad and its parents;
  * every gradient push goes through push: the first contribution sets the parent's grad,
    later ones are added (xt_accumulate, or the producing kernel's accumulate flag), for
    leaves and interior nodes alike — so fan-out (one tensor consumed several times,
    mul(x, x) included) sums all contributions.

Grads have the value's dtype unless the Var was created with grad_dtype="f32"; a float32
grad buffer then sums bf16 contributions in float32 (the fan-out of large-vocab logits needs
this: the cross-entropy term is ~1e-9 per element against O(1) terms).  All arithmetic runs
in libxt; torch provides buffers and the stream.
"""
from __future__ import annotations

import math

import torch

from . import xt

_F32, _BF16 = torch.float32, torch.bfloat16


class Var:
    __slots__ = ("value", "grad", "parents", "backward_fn", "grad_dtype", "name")

    def __init__(self, value, parents=(), backward_fn=None, grad_dtype=None, name=None):
        self.value = value
        self.grad = None
        self.parents = list(parents)
        self.backward_fn = backward_fn
        self.grad_dtype = grad_dtype or value.dtype
        self.name = name


def leaf(value: torch.Tensor, grad_dtype=None, name=None) -> Var:
    return Var(value, grad_dtype=grad_dtype, name=name)


def push(v: Var, g: torch.Tensor, owned: bool = False):
    """Adds contribution g to v.grad (first push sets it).

    A first push stores g itself only when the caller hands over a buffer nobody else holds
    (owned=True: a gradient the closure has just written).  Any other g (the node's own grad
    passed through by add / add_bias, or a buffer also pushed to a sibling) is copied into a
    buffer of v's own, so a later accumulate into v can never change another Var's grad."""
    if v.grad is None:
        if owned and g.dtype == v.grad_dtype:
            v.grad = g
        else:
            v.grad = torch.empty(g.shape, dtype=v.grad_dtype, device=g.device)
            xt.xt_convert(v.grad, g)
    else:
        xt.xt_accumulate(v.grad, g)


def topo_order(root: Var):
    order, seen = [], set()
    stack = [(root, False)]
    while stack:
        node, expanded = stack.pop()
        if expanded:
            order.append(node)
            continue
        if id(node) in seen:
            continue
        seen.add(id(node))
        stack.append((node, True))
        for p in reversed(node.parents):
            if id(p) not in seen:
                stack.append((p, False))
    return order


# The seed tensor of the backward pass in progress (the loss's grad, exactly 1): a closure that
# receives it knows its node is the root with upstream 1.
_seed = [None]


def backward(loss: Var):
    if loss.value.numel() != 1:
        raise ValueError("backward() needs a scalar loss")
    order = topo_order(loss)
    seed = torch.empty(1, dtype=_F32, device=loss.value.device)
    one = torch.ones(1, dtype=_F32, device=loss.value.device)
    xt.xt_convert(seed, one)
    seed = seed if loss.value.dtype == _F32 else _cast(seed, loss.value.dtype)
    push(loss, seed, owned=True)
    _seed[0] = seed
    try:
        for node in reversed(order):
            if node.backward_fn is not None and node.grad is not None:
                node.backward_fn(node.grad, node.parents)
    finally:
        _seed[0] = None


def _empty_like(t, dtype=None):
    return torch.empty(t.shape, dtype=dtype or t.dtype, device=t.device)


def _cast(t, dtype):
    if t.dtype == dtype:
        return t
    out = torch.empty(t.shape, dtype=dtype, device=t.device)
    xt.xt_convert(out, t)
    return out


def _as(g, ref):
    """Upstream grad g in the dtype of the kernel's inputs `ref` (cast when they differ)."""
    return _cast(g, ref.dtype)


# ------------------------------------------------------------------------------ op nodes


def add(a: Var, b: Var) -> Var:
    y = _empty_like(a.value)
    xt.xt_add_fwd(a.value, b.value, y)

    def bw(g, ps):
        push(ps[0], g)
        push(ps[1], g)
    return Var(y, [a, b], bw)


def mul(a: Var, b: Var) -> Var:
    y = _empty_like(a.value)
    xt.xt_mul_fwd(a.value, b.value, y)

    def bw(g, ps):
        g = _as(g, ps[0].value)
        da, db = _empty_like(ps[0].value), _empty_like(ps[1].value)
        xt.xt_mul_bwd(g, ps[0].value, ps[1].value, da, db)
        push(ps[0], da, owned=True)
        push(ps[1], db, owned=True)
    return Var(y, [a, b], bw)


def scale(x: Var, alpha: float) -> Var:
    y = _empty_like(x.value)
    xt.xt_scale_fwd(x.value, y, alpha)

    def bw(g, ps):
        g = _as(g, ps[0].value)
        dx = _empty_like(g)
        xt.xt_scale_bwd(g, dx, alpha)
        push(ps[0], dx, owned=True)
    return Var(y, [x], bw)


def sum_all(x: Var) -> Var:
    y = torch.empty(1, dtype=_F32, device=x.value.device)
    xt.xt_sum_fwd(x.value, y)

    def bw(g, ps):
        dx = _empty_like(ps[0].value)
        xt.xt_sum_bwd(_cast(g, _F32), dx)
        push(ps[0], dx, owned=True)
    return Var(y, [x], bw)


def matmul(a: Var, b: Var, trans_b: bool = False) -> Var:
    """C = A @ B (or A @ Bᵀ with trans_b), 2-D, on the tensor cores; C in A's dtype."""
    A, B = a.value, b.value
    M, K = A.shape
    N = B.shape[0] if trans_b else B.shape[1]
    dab = xt.dt(A)
    d = xt.matmul_desc(M, N, K, trans_b=int(trans_b), lda=K, ldb=K if trans_b else N, ldc=N, dtype_ab=dab,
                       dtype_c=dab)
    y = torch.empty((M, N), dtype=A.dtype, device=A.device)
    xt.xt_matmul_fwd(d, A, B, y)

    def bw(g, ps):
        g = _as(g, ps[0].value)
        dA, dB = _empty_like(ps[0].value), _empty_like(ps[1].value)
        xt.xt_matmul_bwd(d, ps[0].value, ps[1].value, g, dA, dB)
        push(ps[0], dA, owned=True)
        push(ps[1], dB, owned=True)
    return Var(y, [a, b], bw)


def add_bias(x: Var, b: Var) -> Var:
    y = _empty_like(x.value)
    xt.xt_add_bias_fwd(x.value, b.value, y)

    def bw(g, ps):
        g = _as(g, ps[0].value)
        db = _empty_like(ps[1].value, _F32)
        xt.xt_add_bias_bwd(g, None, db)
        push(ps[0], g)
        push(ps[1], _cast(db, ps[1].grad_dtype), owned=True)
    return Var(y, [x, b], bw)


def silu(x: Var) -> Var:
    y = _empty_like(x.value)
    xt.xt_silu_fwd(x.value, y)

    def bw(g, ps):
        g = _as(g, ps[0].value)
        dx = _empty_like(g)
        xt.xt_silu_bwd(g, ps[0].value, dx)
        push(ps[0], dx, owned=True)
    return Var(y, [x], bw)


def gelu(x: Var) -> Var:
    y = _empty_like(x.value)
    xt.xt_gelu_fwd(x.value, y)

    def bw(g, ps):
        g = _as(g, ps[0].value)
        dx = _empty_like(g)
        xt.xt_gelu_bwd(g, ps[0].value, dx)
        push(ps[0], dx, owned=True)
    return Var(y, [x], bw)


def swiglu(gate: Var, up: Var) -> Var:
    y = _empty_like(gate.value)
    xt.xt_swiglu_fwd(gate.value, up.value, y)

    def bw(g, ps):
        g = _as(g, ps[0].value)
        dg, du = _empty_like(ps[0].value), _empty_like(ps[1].value)
        xt.xt_swiglu_bwd(g, ps[0].value, ps[1].value, dg, du)
        push(ps[0], dg, owned=True)
        push(ps[1], du, owned=True)
    return Var(y, [gate, up], bw)


def rms_norm(x: Var, gamma: Var, eps: float) -> Var:
    rows = x.value.shape[0]
    y = _empty_like(x.value)
    ir = torch.empty(rows, dtype=_F32, device=x.value.device)
    xt.xt_rms_norm_fwd(x.value, gamma.value, y, ir, eps)

    def bw(g, ps):
        g = _as(g, ps[0].value)
        dx, dg = _empty_like(ps[0].value), _empty_like(ps[1].value, _F32)
        xt.xt_rms_norm_bwd(g, ps[0].value, ps[1].value, ir, dx, dg)
        push(ps[0], dx, owned=True)
        push(ps[1], _cast(dg, ps[1].grad_dtype), owned=True)
    return Var(y, [x, gamma], bw)


def layernorm(x: Var, gamma: Var, beta: Var, eps: float) -> Var:
    rows = x.value.shape[0]
    y = _empty_like(x.value)
    mu = torch.empty(rows, dtype=_F32, device=x.value.device)
    rs = torch.empty(rows, dtype=_F32, device=x.value.device)
    xt.xt_layernorm_fwd(x.value, gamma.value, beta.value, y, mu, rs, eps)

    def bw(g, ps):
        g = _as(g, ps[0].value)
        dx = _empty_like(ps[0].value)
        dg, db = _empty_like(ps[1].value, _F32), _empty_like(ps[2].value, _F32)
        xt.xt_layernorm_bwd(g, ps[0].value, ps[1].value, mu, rs, dx, dg, db)
        push(ps[0], dx, owned=True)
        push(ps[1], _cast(dg, ps[1].grad_dtype), owned=True)
        push(ps[2], _cast(db, ps[2].grad_dtype), owned=True)
    return Var(y, [x, gamma, beta], bw)


def softmax(x: Var, causal: bool = False) -> Var:
    """Row softmax over the last axis; with causal, x is [..., S, S] and c > s is masked."""
    S = x.value.shape[-1]
    y = _empty_like(x.value)
    xt.xt_softmax_fwd(x.value, y, causal=1 if causal else 0, q_len=x.value.shape[-2] if causal else 0)

    def bw(g, ps):
        g = _as(g, y)
        dx = _empty_like(y)
        xt.xt_softmax_bwd(g, y, dx, causal=1 if causal else 0, q_len=ps[0].value.shape[-2] if causal else 0)
        push(ps[0], dx, owned=True)
    del S
    return Var(y, [x], bw)


def cross_entropy(x: Var, targets: torch.Tensor) -> Var:
    rows, V = x.value.shape
    lse = torch.empty(rows, dtype=_F32, device=x.value.device)
    loss = torch.empty(1, dtype=_F32, device=x.value.device)
    xt.xt_cross_entropy_fwd(x.value, targets, lse, loss)

    def bw(g, ps):
        up = _cast(g, _F32)
        p = ps[0]
        if p.grad is None:   # first push: write the gradient in the grad dtype directly
            p.grad = torch.empty(p.value.shape, dtype=p.grad_dtype, device=p.value.device)
            xt.xt_cross_entropy_bwd(p.value, targets, lse, up, p.grad, acc=0)
        else:                # later push: accumulate in place (no intermediate buffer)
            xt.xt_cross_entropy_bwd(p.value, targets, lse, up, p.grad, acc=1)
    return Var(loss, [x], bw)


def cross_entropy_fanout(x: Var, targets: torch.Tensor, c_lin: float, c_sq: float) -> Var:
    """L = cross_entropy(x) + c_lin·Σx + c_sq·Σ(x∘x) as one node: the three consumers of x of
    [AE] § 梯度累加's fan-out example fused, forward and backward in one pass over x (each row
    held on chip while its lse and gradient are formed).  The forward already writes
    dL/dx for upstream 1 into a float32 buffer the node owns; when the node is the backward's
    root (its upstream is the seed, exactly 1) that buffer is pushed as x's gradient, otherwise
    the backward runs the pass again scaled by the upstream.  Value: the float32 scalar L, a
    view of a 3-element tensor (Σx, Σx², L)."""
    rows, V = x.value.shape
    dev = x.value.device
    lse = torch.empty(rows, dtype=_F32, device=dev)
    loss = torch.empty(1, dtype=_F32, device=dev)
    sums = torch.empty(3, dtype=_F32, device=dev)
    gbuf = torch.empty((rows, V), dtype=_F32, device=dev)
    xt.xt_cross_entropy_fanout_fwd_bwd(x.value, targets, c_lin, c_sq, lse, loss, sums, gbuf)
    state = {"g": gbuf}

    def bw(g, ps):
        p = ps[0]
        buf = state.pop("g")
        if g is _seed[0]:
            push(p, buf, owned=True)
            return
        del buf
        up = _cast(g, _F32)
        if p.grad is None:
            out = torch.empty(p.value.shape, dtype=_F32, device=dev)
            xt.xt_cross_entropy_fanout_fwd_bwd(p.value, targets, c_lin, c_sq, lse, loss, sums, out, upstream=up)
            push(p, out, owned=True)
        elif p.grad.dtype == _F32:
            xt.xt_cross_entropy_fanout_fwd_bwd(p.value, targets, c_lin, c_sq, lse, loss, sums, p.grad, upstream=up,
                                               acc=1)
        else:
            out = torch.empty(p.value.shape, dtype=_F32, device=dev)
            xt.xt_cross_entropy_fanout_fwd_bwd(p.value, targets, c_lin, c_sq, lse, loss, sums, out, upstream=up)
            push(p, out)
    node = Var(sums[2:3], [x], bw)
    node.name = "cross_entropy_fanout"
    return node


def dropout(x: Var, p: float, seed: int, training: bool = True) -> Var:
    """p == 0 or eval returns x itself: no node ([DO] § train / eval 开关)."""
    if p == 0.0 or not training:
        return x
    y = _empty_like(x.value)
    xt.xt_dropout_fwd(x.value, y, p, seed)

    def bw(g, ps):
        g = _as(g, ps[0].value)
        dx = _empty_like(g)
        xt.xt_dropout_bwd(g, dx, p, seed)
        push(ps[0], dx, owned=True)
    return Var(y, [x], bw)


def attention(q: Var, k: Var, v: Var, causal: bool = True) -> Var:
    """Composed attention ([AE] § Attention 用组合) on [B·H, S, hd] blocks: scores = q kᵀ·(1/√hd),
    P = softmax(scores), out = P v — each step a node, so the backward is the composition."""
    BH, S, hd = q.value.shape
    scores = _bmm(q, k, trans_b=True, alpha=1.0 / math.sqrt(hd))
    probs = softmax(scores, causal=causal)
    return _bmm(probs, v, trans_b=False, alpha=1.0)


def _bmm(a: Var, b: Var, trans_b: bool, alpha: float) -> Var:
    """Batched C[z] = alpha·A[z] @ op(B[z]) over contiguous [Z, ·, ·] operands."""
    A, B = a.value, b.value
    Z, M, K = A.shape
    N = B.shape[1] if trans_b else B.shape[2]
    dab = xt.dt(A)
    d = xt.matmul_desc(M, N, K, trans_b=int(trans_b), lda=K, ldb=K if trans_b else N, ldc=N, batch_inner=Z,
                       dtype_ab=dab, dtype_c=dab, alpha=alpha,
                       strides=(0, M * K, 0, B.shape[1] * B.shape[2], 0, M * N))
    y = torch.empty((Z, M, N), dtype=A.dtype, device=A.device)
    xt.xt_matmul_fwd(d, A, B, y)

    def bw(g, ps):
        g = _as(g, ps[0].value)
        dA, dB = _empty_like(ps[0].value), _empty_like(ps[1].value)
        xt.xt_matmul_bwd(d, ps[0].value, ps[1].value, g, dA, dB)
        push(ps[0], dA, owned=True)
        push(ps[1], dB, owned=True)
    return Var(y, [a, b], bw)
