"""Counter-based inverted dropout, in exact integer arithmetic.

[DO] § Key Design Decisions / RNG：counter-based: the keep decision of element i
depends only on (seed, i):
    key  = seed XOR (i · 0x9E3779B97F4A7C15)          (mod 2⁶⁴)
    h    = splitmix64(key)
    u    = (h >> 40) / 2²⁴                               (exact in float32)
    keep = u ≥ p                                         (compared in float32)
    out  = keep ? x · (1/(1−p)) : 0
and the backward applies the same mask ([DO] § dropout 节点的 backward).

Readings where the page is silent:
  * "splitmix64" is named but not printed.  The published SplitMix64 generator
    (Steele, Lea & Flood, OOPSLA 2014) advances its state by the golden gamma
    0x9E3779B97F4A7C15 and then mixes; splitmix64(key) here is that step taken
    from state `key`: z = key + γ; z = (z ^ z>>30)·0xBF58476D1CE4E5B9;
    z = (z ^ z>>27)·0x94D049BB133111EB; z ^ z>>31.
  * The scale 1/(1−p) is computed in float64 from float32(p) and rounded once to
    float32; the product x·scale is one float32 multiply.  For bf16 storage the
    float32 product is rounded to bf16 (nearest-even); the mask is decided in
    float32 and is therefore identical for both storage types ([DO] § 与既有特性的组合, bf16).
  * Per-site seeds ([DO] § 每个 dropout 站点的确定性 seed): seed = base ⊕ layer ⊕ site,
    site = 0xA77 (attention) or 0xF70 (FFN; the page's "0xF7N" is garbled, N is
    not a hex digit, and is read as 0xF70).
  * p = 0 or eval ⇒ exact identity ([DO] § train / eval 开关).
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
MIX1 = np.uint64(0xBF58476D1CE4E5B9)
MIX2 = np.uint64(0x94D049BB133111EB)
SITE_ATTN = 0xA77
SITE_FFN = 0xF70

_U = np.uint64


def splitmix64(state):
    """One SplitMix64 output from state `state` (uint64 array; all arithmetic mod 2⁶⁴)."""
    z = np.asarray(state, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = z + GAMMA
        z = (z ^ (z >> _U(30))) * MIX1
        z = (z ^ (z >> _U(27))) * MIX2
    return z ^ (z >> _U(31))


def site_seed(base_seed: int, layer: int, site: int) -> int:
    return (int(base_seed) ^ int(layer) ^ int(site)) & 0xFFFFFFFFFFFFFFFF


def uniforms(n: int, seed: int) -> np.ndarray:
    """u_i for i in [0, n), as float32."""
    i = np.arange(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        key = _U(seed) ^ (i * GAMMA)
    h = splitmix64(key)
    return (h >> _U(40)).astype(np.float32) * np.float32(2.0 ** -24)


def keep_mask(n: int, p: float, seed: int) -> np.ndarray:
    """Boolean keep mask of n elements (True = kept)."""
    return uniforms(n, seed) >= np.float32(p)


def scale_f32(p: float) -> np.float32:
    return np.float32(1.0 / (1.0 - float(np.float32(p))))


def _round_bf16(a32: np.ndarray) -> np.ndarray:
    """float32 → bfloat16 (round to nearest, ties to even), returned as float32 values."""
    u = np.ascontiguousarray(a32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + _U(0x7FFF) + ((u >> _U(16)) & _U(1))) >> _U(16)
    return (r << _U(16)).astype(np.uint32).view(np.float32)


def dropout_fwd(x, p: float, seed: int, training: bool = True, dtype: str = "f32"):
    """Returns out with x's shape (float32 values; bf16-representable when dtype='bf16')."""
    x32 = np.asarray(x, dtype=np.float32)
    if p == 0.0 or not training:
        return x32.copy()
    if not (0.0 <= p < 1.0):
        raise ValueError("p must be in [0, 1)")
    keep = keep_mask(x32.size, p, seed).reshape(x32.shape)
    out = np.where(keep, x32 * scale_f32(p), np.float32(0.0)).astype(np.float32)
    return _round_bf16(out) if dtype == "bf16" else out


def dropout_bwd(d, p: float, seed: int, training: bool = True, dtype: str = "f32"):
    """dx = keep ? d · scale : 0 with the same mask as the forward."""
    return dropout_fwd(d, p, seed, training, dtype)
