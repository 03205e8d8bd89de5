"""GPU parity of the fused attention (xt_attention_fwd / xt_attention_bwd) against the oracle's
composed attention ([AE] § Attention 用组合): O, the saved normaliser lse, and dQ, dK, dV, with
q, k, v as column blocks of one [T, 3·H·hd] bf16 buffer (the block's layout).  Normalised error
‖g − r‖/‖r‖ ≤ 2e-2 for O and the gradients (the GEMM-path tolerance), |lse − r| ≤ 1e-3 (fp32
accumulation of exact bf16 products); shapes span several 128-tiles and ragged tails; the full
12-head × 1024 case is checked on sampled heads."""
import numpy as np
import pytest
import torch

import synth
from oracle import ops as O
from tests.gpu_util import empty, host, norm_err

pytestmark = pytest.mark.gpu

xt = pytest.importorskip("transformer_fwd_bwd_gb300.xt")

HD = 64


def heads(x2d, B, S, H):
    """[B·S, H·hd] → [B, H, S, hd]"""
    return x2d.reshape(B, S, H, HD).transpose(0, 2, 1, 3)


def bf16_dev(a):
    return torch.from_numpy(synth.bf16_bits(a).view(np.int16)).view(torch.bfloat16).cuda()


def make(B, S, H, seed, std=1.0):
    d = H * HD
    qkv = synth.normal((B * S, 3 * d), seed, std=std, dtype="bf16")
    dO = synth.normal((B * S, d), seed + 1, dtype="bf16")
    return qkv, dO


def run(B, S, H, causal, qkv, dO, with_lo=True):
    """Forward then backward; with_lo keeps O's bf16 rounding residual for the backward's D."""
    d = H * HD
    Q = bf16_dev(qkv)
    o = empty((B * S, d), "bf16")
    o_lo = empty((B * S, d), "bf16") if with_lo else None
    lse = empty((B, H, S))
    xt.xt_attention_fwd(Q[:, :d], Q[:, d:2 * d], Q[:, 2 * d:], o, lse, B, S, H, HD, causal, o_lo=o_lo)
    dqkv = empty((B * S, 3 * d), "bf16")
    dOd = bf16_dev(dO)
    xt.xt_attention_bwd(Q[:, :d], Q[:, d:2 * d], Q[:, 2 * d:], o, dOd, lse, dqkv[:, :d], dqkv[:, d:2 * d],
                        dqkv[:, 2 * d:], B, S, H, HD, causal, o_lo=o_lo)
    torch.cuda.synchronize()
    assert xt.device_errors() == 0
    if with_lo:   # the residual is at most half a bf16 ulp of O: |o_lo| ≤ 2⁻⁸·|o|
        assert bool(torch.all(o_lo.float().abs() <= o.float().abs() * 2.0 ** -8))
    return host(o), host(lse), host(dqkv)


def oracle(B, S, H, causal, qkv, dO, sel=None):
    """Oracle O, lse, dQ, dK, dV, plus the cancellation-free magnitudes of dQ and dK:
    α·(P∘(|dP| + |D|))·|K| and its transpose with |Q| (D = Σ_c dP∘P), the size of the terms
    whose sum the gradient is (dS = P∘(dP − D) sums to zero over each row)."""
    d = H * HD
    q, k, v = (heads(qkv[:, i * d:(i + 1) * d], B, S, H) for i in range(3))
    g = heads(dO, B, S, H)
    if sel is not None:
        q, k, v, g = (x[sel[0]:sel[0] + 1, sel[1]:sel[1] + 1] for x in (q, k, v, g))
    Ov, P = O.attention_fwd(q, k, v, causal=causal)
    lse = O.attention_lse(q, k, causal=causal)
    dQ, dK, dV = O.attention_bwd(g, q, k, v, P)
    dP = np.einsum("bhsd,bhtd->bhst", g, v)
    Dr = np.sum(dP * P, axis=-1, keepdims=True)
    T = P * (np.abs(dP) + np.abs(Dr)) / np.sqrt(HD)
    mag = {"dQ": np.einsum("bhst,bhtd->bhsd", T, np.abs(k)), "dK": np.einsum("bhst,bhsd->bhtd", T, np.abs(q))}
    return Ov, lse, dQ, dK, dV, mag


def grad_err(g, r, mag=None):
    """‖g − r‖ / max(‖r‖, 0.1·‖mag‖): the plain normalised error unless the exact gradient
    cancels (S = 1 gives dQ = dK = 0 exactly), where it is taken against the terms' size."""
    den = np.linalg.norm(r)
    if mag is not None:
        den = max(den, 0.1 * np.linalg.norm(mag))
    return float(np.linalg.norm(np.asarray(g) - r) / max(den, 1e-300))


def check(B, S, H, causal, seed, std=1.0, with_lo=True):
    qkv, dO = make(B, S, H, seed, std)
    o, lse, dqkv = run(B, S, H, causal, qkv, dO, with_lo)
    d = H * HD
    Ov, rl, dQ, dK, dV, mag = oracle(B, S, H, causal, qkv, dO)
    errs = {"O": norm_err(heads(o, B, S, H), Ov)}
    for i, (name, want) in enumerate((("dQ", dQ), ("dK", dK), ("dV", dV))):
        errs[name] = grad_err(heads(dqkv[:, i * d:(i + 1) * d], B, S, H), want, mag.get(name))
    assert np.max(np.abs(lse - rl)) <= 1e-3, np.max(np.abs(lse - rl))
    for k, e in errs.items():
        assert e <= 2e-2, f"{k}: normalised error {e:.3e}"
    return errs


@pytest.mark.parametrize("B,S,H,causal", [(1, 128, 1, 1), (2, 200, 3, 1), (1, 1, 2, 1), (1, 384, 2, 0),
                                          (2, 300, 2, 1), (1, 129, 1, 0), (3, 64, 2, 1)])
def test_attention_parity(B, S, H, causal):
    check(B, S, H, causal, seed=300 + S + H)


def test_attention_without_residual():
    """The backward also accepts the bf16 O alone (D from the rounded O)."""
    check(2, 200, 3, 1, seed=305, with_lo=False)


def test_attention_large_scores():
    """Scores of several units: the running max rises across key tiles (rescaling O)."""
    check(1, 512, 2, 1, seed=310, std=3.0)


def test_attention_deterministic():
    qkv, dO = make(2, 256, 2, 320)
    a = run(2, 256, 2, 1, qkv, dO)
    b = run(2, 256, 2, 1, qkv, dO)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_attention_full_size_sampled_heads():
    """B 8, S 1024, 12 heads × 64 (the 12-layer stack's attention), checked on sampled heads."""
    B, S, H = 8, 1024, 12
    qkv, dO = make(B, S, H, 330)
    o, lse, dqkv = run(B, S, H, 1, qkv, dO)
    d = H * HD
    for b, h in ((0, 0), (3, 7), (7, 11)):
        Ov, rl, dQ, dK, dV, _ = oracle(B, S, H, 1, qkv, dO, sel=(b, h))
        assert norm_err(heads(o, B, S, H)[b, h], Ov[0, 0]) <= 2e-2
        assert np.max(np.abs(lse[b, h] - rl[0, 0])) <= 1e-3
        for i, want in enumerate((dQ, dK, dV)):
            got = heads(dqkv[:, i * d:(i + 1) * d], B, S, H)[b, h]
            assert norm_err(got, want[0, 0]) <= 2e-2, (b, h, i)


def test_attention_rejects_unsupported():
    q = torch.zeros(128, 3 * 32, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(128, 32, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(xt.XtError):   # head_dim 32
        xt.xt_attention_fwd(q[:, :32], q[:, 32:64], q[:, 64:], o, lse, 1, 128, 1, 32, 1)
    qf = torch.zeros(128, 3 * 64, dtype=torch.float32, device="cuda")
    of = torch.zeros(128, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(xt.XtError):   # fp32
        xt.xt_attention_fwd(qf[:, :64], qf[:, 64:128], qf[:, 128:], of, lse, 1, 128, 1, 64, 1)
