"""Helpers for the GPU parity tests: moving synthetic inputs to the device and comparing
device results with the oracle under the tolerances the tests use.

Output buffers carry guard bands that are checked after every GPU test (see empty()).

Tolerances:
  * fp32 row / elementwise ops: max_i |g − r| / max(|r_i|, m_i, 1e-6·max|r|) ≤ 1e-5, where
    m_i is the magnitude of the terms that the defining formula adds for element i (its
    Σ|terms|); where a formula cancels (near a root of silu', a LayerNorm output x̂γ ≈ −β,
    a RoPE rotation, the RMS / softmax backward), float32 evaluation is accurate relative to
    m_i, not to |r_i|;
  * bf16 ops (oracle run on the same bf16-rounded inputs): |g − r| ≤ 1 bf16 ulp of |r_i|
    (2^(⌊log2 |r_i|⌋ − 7)) + 1e-5·max(m_i, 1e-6·max|r|);
  * GEMM paths and whole-block gradients: ‖g − r‖ / ‖r‖ ≤ 2e-2.
"""
import numpy as np
import torch

DEV = "cuda"


def dev(a, dtype="f32"):
    t = torch.tensor(np.ascontiguousarray(a, dtype=np.float32)).contiguous()
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    return t.to(DEV)


def host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


# Guard bands (canaries): every output buffer the tests allocate with empty() is the middle of
# a larger allocation whose 256 bytes before and after hold a fixed bit pattern; after each GPU
# test the bands are read back, and a kernel that wrote outside its output fails the test
# (check_guards, called from conftest.py).  256 bytes keep the output 16-byte aligned.
GUARD_BYTES = 256
_PATTERN = {torch.float32: (torch.int32, 0x7FC0DEAD), torch.bfloat16: (torch.int16, 0x7FDE)}
_guards = []


def empty(shape, dtype="f32", fill=None):
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    shape = tuple(shape) if isinstance(shape, (tuple, list)) else (shape,)
    n = int(np.prod(shape)) if len(shape) else 1
    g = GUARD_BYTES // torch.tensor([], dtype=td).element_size()
    buf = torch.empty(n + 2 * g, dtype=td, device=DEV)
    it, pat = _PATTERN[td]
    bits = buf.view(it)
    bits[:g] = pat
    bits[g + n:] = pat
    out = buf[g:g + n].view(shape)
    if fill is not None:
        out.fill_(fill)
    _guards.append((buf, g, n, it, pat))
    return out


def check_guards():
    """Bands around every empty() buffer since the last call that no longer hold the pattern."""
    bad = []
    for buf, g, n, it, pat in _guards:
        bits = buf.view(it)
        for name, band in (("before", bits[:g]), ("after", bits[g + n:])):
            if not bool((band == pat).all()):
                bad.append(f"{tuple(buf.shape)} {buf.dtype} output: guard band {name} overwritten")
    _guards.clear()
    return bad


def _mag(r, mag):
    a = np.abs(np.asarray(r, np.float64))
    m = a if mag is None else np.maximum(a, np.abs(np.asarray(mag, np.float64)))
    return np.maximum(m, 1e-6 * max(float(np.max(a)) if a.size else 0.0, 1e-30))


def rel_err_floor(g, r, mag=None):
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    return float(np.max(np.abs(g - r) / _mag(r, mag)))


def bf16_ulp_excess(g, r, mag=None):
    """max over elements of |g − r| / (1 ulp(r) + 1e-5·m); ≤ 1 passes."""
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    a = np.abs(r)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1e-300)))
    ulp = np.where(a > 0, 2.0 ** (e - 7), 0.0)
    tol = ulp + 1e-5 * _mag(r, mag)
    return float(np.max(np.abs(g - r) / tol))


def norm_err(g, r):
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    return float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300))


def check(g, r, dtype, what="", mag=None):
    if dtype == "f32":
        e = rel_err_floor(g, r, mag)
        assert e <= 1e-5, f"{what}: fp32 rel err {e:.3e}"
    else:
        e = bf16_ulp_excess(g, r, mag)
        assert e <= 1.0, f"{what}: bf16 error {e:.3f} ulp-units"


def sync():
    torch.cuda.synchronize()
