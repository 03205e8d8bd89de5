"""Forward-mode AD on scalar chains: dual numbers and hyper-dual numbers.

[AD] § 二、数学基础：对偶数与微分: a + bε with ε² = 0, so f(a + ε) = f(a) + f'(a)ε;
every primitive carries its derivative by the chain rule.  Used as an independent
check of the analytic per-element derivatives (silu', gelu', σ') on scalars.

[AD] § 五、高阶导数与 Hessian 计算: HyperDual numbers a + b ε₁ + c ε₂ + d ε₁ε₂ carry two
first partials and the mixed second partial.  The page's struct has no sin(); it
is added here (sin(a+…) = sin a + cos a·(b ε₁ + c ε₂) + (cos a·d − sin a·b·c) ε₁ε₂)
because the page's worked example f(x, y) = x²y + sin x + y³ needs it.
"""
from __future__ import annotations

import math


class Dual:
    __slots__ = ("val", "deriv")

    def __init__(self, val, deriv=0.0):
        self.val = float(val)
        self.deriv = float(deriv)

    @staticmethod
    def variable(v):
        return Dual(v, 1.0)

    @staticmethod
    def constant(v):
        return Dual(v, 0.0)

    @staticmethod
    def _lift(o):
        return o if isinstance(o, Dual) else Dual(o, 0.0)

    def __add__(self, o):
        o = Dual._lift(o)
        return Dual(self.val + o.val, self.deriv + o.deriv)

    __radd__ = __add__

    def __sub__(self, o):
        o = Dual._lift(o)
        return Dual(self.val - o.val, self.deriv - o.deriv)

    def __rsub__(self, o):
        return Dual._lift(o) - self

    def __mul__(self, o):
        o = Dual._lift(o)
        return Dual(self.val * o.val, self.deriv * o.val + self.val * o.deriv)

    __rmul__ = __mul__

    def __truediv__(self, o):
        o = Dual._lift(o)
        return Dual(self.val / o.val, (self.deriv * o.val - self.val * o.deriv) / (o.val * o.val))

    def __rtruediv__(self, o):
        return Dual._lift(o) / self

    def __neg__(self):
        return Dual(-self.val, -self.deriv)

    def exp(self):
        v = math.exp(self.val)
        return Dual(v, v * self.deriv)

    def ln(self):
        return Dual(math.log(self.val), self.deriv / self.val)

    def sin(self):
        return Dual(math.sin(self.val), math.cos(self.val) * self.deriv)

    def cos(self):
        return Dual(math.cos(self.val), -math.sin(self.val) * self.deriv)

    def powf(self, n):
        return Dual(self.val ** n, n * self.val ** (n - 1.0) * self.deriv)

    def sqrt(self):
        v = math.sqrt(self.val)
        return Dual(v, self.deriv / (2.0 * v))

    def relu(self):
        return Dual(self.val if self.val > 0 else 0.0, self.deriv if self.val > 0 else 0.0)

    def sigmoid(self):
        v = 1.0 / (1.0 + math.exp(-self.val))
        return Dual(v, v * (1.0 - v) * self.deriv)

    def tanh(self):
        v = math.tanh(self.val)
        return Dual(v, (1.0 - v * v) * self.deriv)

    def erf(self):
        """Extension (not on the page): d/dx erf(x) = 2/√π · e^(−x²)."""
        return Dual(math.erf(self.val),
                    2.0 / math.sqrt(math.pi) * math.exp(-self.val * self.val) * self.deriv)


class HyperDual:
    __slots__ = ("val", "g1", "g2", "h")

    def __init__(self, val, g1=0.0, g2=0.0, h=0.0):
        self.val, self.g1, self.g2, self.h = float(val), float(g1), float(g2), float(h)

    @staticmethod
    def var1(v):
        return HyperDual(v, 1.0, 0.0, 0.0)

    @staticmethod
    def var2(v):
        return HyperDual(v, 0.0, 1.0, 0.0)

    @staticmethod
    def _lift(o):
        return o if isinstance(o, HyperDual) else HyperDual(o)

    def __add__(self, o):
        o = HyperDual._lift(o)
        return HyperDual(self.val + o.val, self.g1 + o.g1, self.g2 + o.g2, self.h + o.h)

    __radd__ = __add__

    def __mul__(self, o):
        o = HyperDual._lift(o)
        return HyperDual(self.val * o.val,
                         self.g1 * o.val + self.val * o.g1,
                         self.g2 * o.val + self.val * o.g2,
                         self.h * o.val + self.g1 * o.g2 + self.g2 * o.g1 + self.val * o.h)

    __rmul__ = __mul__

    def sin(self):
        s, c = math.sin(self.val), math.cos(self.val)
        return HyperDual(s, c * self.g1, c * self.g2, c * self.h - s * self.g1 * self.g2)
