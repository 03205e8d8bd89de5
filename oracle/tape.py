"""Tape-based reverse-mode engine (define-by-run), in float64.

[AE] § Key Design Decisions / Tape 设计 and § 梯度累加:
  * a Var holds a value, an optional grad, its parents and an optional backward
    closure (None marks a leaf);
  * backward(): (1) post-order DFS from the loss builds a topological order,
    de-duplicated by node identity; (2) the loss must be a scalar and its grad is
    seeded with 1; (3) nodes are walked in reverse order and each closure receives
    the node's accumulated grad and its parents;
  * push_grad: the first contribution sets the grad, later ones are summed (fan-out),
    for leaves and interior nodes alike; the same Var used twice by one node
    (mul(x, x)) receives both contributions.
The fan-out summation order is the order of the pushes (reverse topological order).
"""
from __future__ import annotations

import math

import numpy as np

from . import dropout as _dropout
from . import ops as _ops


class Var:
    __slots__ = ("value", "grad", "parents", "backward_fn", "name")

    def __init__(self, value, parents=(), backward_fn=None, name=None):
        self.value = np.asarray(value, dtype=np.float64) if not isinstance(value, np.ndarray) \
            else value.astype(np.float64, copy=False)
        self.grad = None
        self.parents = list(parents)
        self.backward_fn = backward_fn
        self.name = name

    @property
    def is_leaf(self):
        return self.backward_fn is None


def push_grad(v: Var, g) -> None:
    g = np.asarray(g, dtype=np.float64)
    if v.grad is None:
        v.grad = g.copy()
    else:
        v.grad = v.grad + g


def topo_order(root: Var):
    """Post-order DFS, de-duplicated by object identity (iterative)."""
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


def backward(loss: Var) -> None:
    if loss.value.size != 1:
        raise ValueError("backward() needs a scalar loss")
    order = topo_order(loss)
    loss.grad = np.ones_like(loss.value)
    for node in reversed(order):
        if node.backward_fn is not None and node.grad is not None:
            node.backward_fn(node.grad, node.parents)


# ---------------------------------------------------------------------------------------
# Op node constructors ([AE] op table); each closure captures what its backward needs.
# ---------------------------------------------------------------------------------------

def leaf(value, name=None) -> Var:
    return Var(value, name=name)


def matmul(a: Var, b: Var) -> Var:
    def bw(g, ps):
        da, db = _ops.matmul_bwd(g, ps[0].value, ps[1].value)
        push_grad(ps[0], da)
        push_grad(ps[1], db)
    return Var(_ops.matmul_fwd(a.value, b.value), [a, b], bw)


def transpose(a: Var) -> Var:
    """Last-two-axes transpose node (the page wraps Kᵀ in an ad-hoc node in its test)."""
    def bw(g, ps):
        push_grad(ps[0], np.swapaxes(g, -1, -2))
    return Var(np.swapaxes(a.value, -1, -2), [a], bw)


def add(a: Var, b: Var) -> Var:
    def bw(g, ps):
        da, db = _ops.add_bwd(g)
        push_grad(ps[0], da)
        push_grad(ps[1], db)
    return Var(_ops.add_fwd(a.value, b.value), [a, b], bw)


def mul(a: Var, b: Var) -> Var:
    def bw(g, ps):
        da, db = _ops.mul_bwd(g, ps[0].value, ps[1].value)
        push_grad(ps[0], da)
        push_grad(ps[1], db)
    return Var(_ops.mul_fwd(a.value, b.value), [a, b], bw)


def scale(a: Var, alpha: float) -> Var:
    def bw(g, ps):
        push_grad(ps[0], _ops.scale_bwd(g, alpha))
    return Var(_ops.scale_fwd(a.value, alpha), [a], bw)


def sum_all(a: Var) -> Var:
    shape = a.value.shape

    def bw(g, ps):
        push_grad(ps[0], _ops.sum_bwd(g, shape))
    return Var(_ops.sum_fwd(a.value), [a], bw)


def add_bias(x: Var, b: Var) -> Var:
    def bw(g, ps):
        dx, db = _ops.add_bias_bwd(g)
        push_grad(ps[0], dx)
        push_grad(ps[1], db)
    return Var(_ops.add_bias_fwd(x.value, b.value), [x, b], bw)


def silu(x: Var) -> Var:
    def bw(g, ps):
        push_grad(ps[0], _ops.silu_bwd(g, ps[0].value))
    return Var(_ops.silu_fwd(x.value), [x], bw)


def swiglu(gate: Var, up: Var) -> Var:
    def bw(g, ps):
        dg, du = _ops.swiglu_bwd(g, ps[0].value, ps[1].value)
        push_grad(ps[0], dg)
        push_grad(ps[1], du)
    return Var(_ops.swiglu_fwd(gate.value, up.value), [gate, up], bw)


def gelu(x: Var) -> Var:
    def bw(g, ps):
        push_grad(ps[0], _ops.gelu_bwd(g, ps[0].value))
    return Var(_ops.gelu_fwd(x.value), [x], bw)


def rms_norm(x: Var, gamma: Var, eps: float) -> Var:
    y, ir = _ops.rms_norm_fwd(x.value, gamma.value, eps)

    def bw(g, ps):
        dx, dg = _ops.rms_norm_bwd(g, ps[0].value, ps[1].value, ir)
        push_grad(ps[0], dx)
        push_grad(ps[1], dg)
    return Var(y, [x, gamma], bw)


def layernorm(x: Var, gamma: Var, beta: Var, eps: float) -> Var:
    y, mu, rstd = _ops.layernorm_fwd(x.value, gamma.value, beta.value, eps)

    def bw(g, ps):
        dx, dg, db = _ops.layernorm_bwd(g, ps[0].value, ps[1].value, mu, rstd)
        push_grad(ps[0], dx)
        push_grad(ps[1], dg)
        push_grad(ps[2], db)
    return Var(y, [x, gamma, beta], bw)


def rope(x: Var, positions, base: float) -> Var:
    def bw(g, ps):
        push_grad(ps[0], _ops.rope_bwd(g, positions, base))
    return Var(_ops.rope_fwd(x.value, positions, base), [x], bw)


def softmax(x: Var, causal: bool = False) -> Var:
    y = _ops.softmax_fwd(x.value, causal=causal)

    def bw(g, ps):
        push_grad(ps[0], _ops.softmax_bwd(g, y))
    return Var(y, [x], bw)


def cross_entropy(x: Var, targets) -> Var:
    loss, lse = _ops.cross_entropy_fwd(x.value, targets)

    def bw(g, ps):
        push_grad(ps[0], _ops.cross_entropy_bwd(ps[0].value, targets, lse, float(g)))
    return Var(np.float64(loss), [x], bw)


def dropout(x: Var, p: float, seed: int, training: bool = True) -> Var:
    """p == 0 (or eval) returns x itself: no node is created ([DO] § train / eval 开关)."""
    if p == 0.0 or not training:
        return x
    keep = _dropout.keep_mask(x.value.size, p, seed).reshape(x.value.shape)
    sc = float(_dropout.scale_f32(p))

    def bw(g, ps):
        push_grad(ps[0], np.where(keep, g * sc, 0.0))
    return Var(np.where(keep, x.value * sc, 0.0), [x], bw)


def embedding(ids, E: Var, P: Var = None, S: int = None) -> Var:
    parents = [E] + ([P] if P is not None else [])
    V = E.value.shape[0]

    def bw(g, ps):
        dE, dP = _ops.embedding_bwd(ids, g, V, S, with_pos=P is not None)
        push_grad(ps[0], dE)
        if P is not None:
            push_grad(ps[1], dP)
    return Var(_ops.embedding_fwd(ids, E.value, None if P is None else P.value, S), parents, bw)


def reshape(x: Var, shape) -> Var:
    old = x.value.shape

    def bw(g, ps):
        push_grad(ps[0], np.reshape(g, old))
    return Var(np.reshape(x.value, shape), [x], bw)


def split_heads(x: Var, B: int, S: int, H: int, hd: int) -> Var:
    """[T, H·hd] → [B, H, S, hd] view (pure re-indexing node)."""
    def bw(g, ps):
        push_grad(ps[0], np.transpose(g, (0, 2, 1, 3)).reshape(B * S, H * hd))
    return Var(np.transpose(x.value.reshape(B, S, H, hd), (0, 2, 1, 3)), [x], bw)


def merge_heads(x: Var) -> Var:
    B, H, S, hd = x.value.shape

    def bw(g, ps):
        push_grad(ps[0], np.transpose(g.reshape(B, S, H, hd), (0, 2, 1, 3)))
    return Var(np.transpose(x.value, (0, 2, 1, 3)).reshape(B * S, H * hd), [x], bw)


def attention(q: Var, k: Var, v: Var, causal: bool = True) -> Var:
    """Composed attention ([AE] § Attention 用组合): every step is a node, so the
    backward follows matmul → softmax → scale → matmul without a fused kernel."""
    hd = q.value.shape[-1]
    scores = scale(matmul(q, transpose(k)), 1.0 / math.sqrt(hd))
    probs = softmax(scores, causal=causal)
    return matmul(probs, v)
