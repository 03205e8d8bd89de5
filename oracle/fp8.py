"""FP8 E4M3 encoding, per-tensor quantization and the FP8 matmul, in exact arithmetic.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[BP] § Vad generiska ramverk kostar (item 4, the mixed-precision pipeline) names an FP8 E4M3
tensor-core path without giving the format's details or a scaling rule.  Readings: the
format is E4M3 as the OCP 8-bit floating-point specification
defines it (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no infinities; exponent
field 0 holds the subnormals m·2⁻⁹; the all-ones code S.1111.111 is NaN; the largest finite
value is 1.75·2⁸ = 448); conversion rounds to nearest, ties to the even code, and saturates
finite values beyond ±448 to ±448.  Quantization is per tensor: scale = 448 / amax (1 when
amax = 0), codes = E4M3(x·scale) with the product formed in float32, and the value a code
stands for is decode(code) / scale.  The FP8 matmul is C = α·(A/sa)(B/sb)ᵀ over the decoded
codes, A [M, K] and B [N, K] both K-contiguous.
"""
from __future__ import annotations

import numpy as np

MAX = 448.0


def decode_code(c: int) -> float:
    """The value of E4M3 code c (0..255) from the format's definition."""
    s = -1.0 if c & 0x80 else 1.0
    e = (c >> 3) & 0xF
    m = c & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


DECODE = np.array([decode_code(c) for c in range(256)], dtype=np.float64)
# the finite non-negative codes in increasing value (0x00 .. 0x7E)
_POS = DECODE[:0x7F]


def encode(x) -> np.ndarray:
    """E4M3 codes (uint8) of the values x: nearest code, ties to the even code, finite values
    beyond ±448 saturated, NaN to 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint8)
    flat, res = x.ravel(), out.ravel()
    for i, v in enumerate(flat):
        if np.isnan(v):
            res[i] = 0x7F
            continue
        sign = 0x80 if (v < 0 or (v == 0 and np.signbit(v))) else 0
        a = min(abs(v), MAX)
        lo = int(np.searchsorted(_POS, a, side="right")) - 1   # largest code with value ≤ a
        if _POS[lo] == a or lo == 0x7E:
            c = lo
        else:
            dl, dh = a - _POS[lo], _POS[lo + 1] - a
            c = lo if dl < dh else lo + 1 if dh < dl else (lo if lo % 2 == 0 else lo + 1)
        res[i] = sign | c
    return out


def decode(codes) -> np.ndarray:
    return DECODE[np.asarray(codes, dtype=np.uint8)]


def quantize(x):
    """Per-tensor quantization: (codes, scale) with scale = 448 / amax as one float32
    division (1 when amax = 0) and the codes of float32(x)·scale formed in float32."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = float(np.max(np.abs(x32))) if x32.size else 0.0
    scale = np.float32(MAX) / np.float32(amax) if amax > 0 else np.float32(1.0)   # one float32 division
    return encode((x32 * scale).astype(np.float32)), float(scale)


def matmul_fp8(a_codes, b_codes, alpha=1.0, inv_scale_a=1.0, inv_scale_b=1.0):
    """C = α · (decode(A)·inv_scale_a) @ (decode(B)·inv_scale_b)ᵀ in float64; A [M, K] and
    B [N, K] hold codes."""
    A = decode(a_codes) * inv_scale_a
    B = decode(b_codes) * inv_scale_b
    return alpha * (A @ B.T)
