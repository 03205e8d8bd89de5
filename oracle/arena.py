"""Second reverse-mode engine: an index arena over scalar nodes.

[AD] § 3.1 计算图构建 and § 3.3 反向传播: nodes live in a vector in creation order,
which is already a topological order; backward zeroes every grad, seeds the
output with 1 and walks ids from the output down to 0, adding each node's local
partials into its inputs (+=).

Two defects of the printed engine are not carried over:
  * its recursive evaluator re-evaluates shared sub-graphs (the page itself says a
    visited mark is needed) — here the forward is one pass in creation order;
  * its Tanh backward uses the INPUT value where tanh's output belongs
    (1 − x² instead of 1 − tanh²(x)) — here the node's own output is used.

This engine exists to cross-check the Var tape: both must give identical float64
gradients on the same scalar expressions.
"""
from __future__ import annotations

import math


class Arena:
    def __init__(self):
        self.op = []      # (name, param)
        self.inp = []     # list of input ids
        self.out = []     # forward values
        self.grad = []

    def _node(self, name, inputs, param=None):
        self.op.append((name, param))
        self.inp.append(list(inputs))
        self.out.append(0.0)
        self.grad.append(0.0)
        return len(self.op) - 1

    def const(self, v):
        return self._node("const", [], float(v))

    var = const

    def add(self, a, b): return self._node("add", [a, b])
    def sub(self, a, b): return self._node("sub", [a, b])
    def mul(self, a, b): return self._node("mul", [a, b])
    def div(self, a, b): return self._node("div", [a, b])
    def neg(self, a): return self._node("neg", [a])
    def exp(self, a): return self._node("exp", [a])
    def ln(self, a): return self._node("ln", [a])
    def sin(self, a): return self._node("sin", [a])
    def cos(self, a): return self._node("cos", [a])
    def tanh(self, a): return self._node("tanh", [a])
    def sigmoid(self, a): return self._node("sigmoid", [a])
    def relu(self, a): return self._node("relu", [a])
    def sqrt(self, a): return self._node("sqrt", [a])
    def powf(self, a, n): return self._node("pow", [a], float(n))

    def forward(self, out_id):
        for i in range(out_id + 1):
            name, prm = self.op[i]
            x = [self.out[j] for j in self.inp[i]]
            if name == "const":
                v = prm
            elif name == "add":
                v = x[0] + x[1]
            elif name == "sub":
                v = x[0] - x[1]
            elif name == "mul":
                v = x[0] * x[1]
            elif name == "div":
                v = x[0] / x[1]
            elif name == "neg":
                v = -x[0]
            elif name == "exp":
                v = math.exp(x[0])
            elif name == "ln":
                v = math.log(x[0])
            elif name == "sin":
                v = math.sin(x[0])
            elif name == "cos":
                v = math.cos(x[0])
            elif name == "tanh":
                v = math.tanh(x[0])
            elif name == "sigmoid":
                v = 1.0 / (1.0 + math.exp(-x[0]))
            elif name == "relu":
                v = x[0] if x[0] > 0.0 else 0.0
            elif name == "sqrt":
                v = math.sqrt(x[0])
            elif name == "pow":
                v = x[0] ** prm
            else:
                raise ValueError(name)
            self.out[i] = v
        return self.out[out_id]

    def backward(self, out_id):
        for i in range(len(self.grad)):
            self.grad[i] = 0.0
        self.grad[out_id] = 1.0
        for i in range(out_id, -1, -1):
            name, prm = self.op[i]
            g = self.grad[i]
            ins = self.inp[i]
            if name == "const":
                continue
            a = self.out[ins[0]]
            if name == "add":
                self.grad[ins[0]] += g
                self.grad[ins[1]] += g
            elif name == "sub":
                self.grad[ins[0]] += g
                self.grad[ins[1]] -= g
            elif name == "mul":
                b = self.out[ins[1]]
                self.grad[ins[0]] += g * b
                self.grad[ins[1]] += g * a
            elif name == "div":
                b = self.out[ins[1]]
                self.grad[ins[0]] += g / b
                self.grad[ins[1]] += g * (-a / (b * b))
            elif name == "neg":
                self.grad[ins[0]] -= g
            elif name == "exp":
                self.grad[ins[0]] += g * self.out[i]
            elif name == "ln":
                self.grad[ins[0]] += g / a
            elif name == "sin":
                self.grad[ins[0]] += g * math.cos(a)
            elif name == "cos":
                self.grad[ins[0]] -= g * math.sin(a)
            elif name == "tanh":
                t = self.out[i]
                self.grad[ins[0]] += g * (1.0 - t * t)
            elif name == "sigmoid":
                s = self.out[i]
                self.grad[ins[0]] += g * s * (1.0 - s)
            elif name == "relu":
                if a > 0.0:
                    self.grad[ins[0]] += g
            elif name == "sqrt":
                self.grad[ins[0]] += g / (2.0 * self.out[i])
            elif name == "pow":
                self.grad[ins[0]] += g * prm * a ** (prm - 1.0)

    def gradient(self, i):
        return self.grad[i]
