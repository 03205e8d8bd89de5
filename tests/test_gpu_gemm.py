"""GPU parity of the tensor-core matmul against the oracle (NumPy float64 on the same
bf16 / fp32 inputs), through the C ABI.

Bounds: the contract is ‖g − r‖/‖r‖ ≤ 2e-2.  The tests also hold each case to what its
arithmetic allows: bf16 operands are exact in the fp32 products, so only fp32 accumulation
and output rounding remain (≤ 1e-5 normalised for fp32 C, ≤ 4e-3 for bf16 C); tf32 keeps
10 mantissa bits of each operand (≤ 2e-3 normalised).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import ops as O
from tests.gpu_util import check, dev, empty, host, norm_err, sync

pytestmark = pytest.mark.gpu

xt = pytest.importorskip("transformer_fwd_bwd_gb300.xt")


def bound(ab, c):
    if ab == "f32":
        return 2e-3
    return 1e-5 if c == "f32" else 4e-3


def stored(M, N, K, ta, tb, ab, seed):
    A = synth.normal((K, M) if ta else (M, K), seed, dtype=ab)
    B = synth.normal((N, K) if tb else (K, N), seed + 1, dtype=ab)
    return A, B


def op(X, t):
    return X.T if t else X


CASES = [(128, 64, 64), (200, 96, 72), (256, 256, 128), (1000, 776, 328), (64, 40, 16), (384, 512, 1024)]


@pytest.mark.parametrize("ab", ["bf16", "f32"])
@pytest.mark.parametrize("c", ["f32", "bf16"])
@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", CASES)
def test_matmul_fwd(ab, c, ta, tb, M, N, K):
    A, B = stored(M, N, K, ta, tb, ab, 40)
    want = O.matmul_fwd(op(A, ta), op(B, tb)) * 0.5
    C = empty((M, N), c)
    d = xt.matmul_desc(M, N, K, trans_a=ta, trans_b=tb, dtype_ab=xt.XT_BF16 if ab == "bf16" else xt.XT_F32,
                       dtype_c=xt.XT_F32 if c == "f32" else xt.XT_BF16, alpha=0.5)
    xt.xt_matmul_fwd(d, dev(A, ab), dev(B, ab), C); sync()
    e = norm_err(host(C), want)
    assert e <= min(2e-2, bound(ab, c)), f"normalised error {e:.2e}"
    assert xt.device_errors() == 0


@pytest.mark.parametrize("ab", ["bf16", "f32"])
def test_matmul_accumulate_and_k0(ab):
    M, N, K = 300, 136, 200
    A, B = stored(M, N, K, 0, 0, ab, 41)
    C0 = synth.normal((M, N), 43)
    Cd = dev(C0, "f32")
    d = xt.matmul_desc(M, N, K, dtype_ab=xt.XT_BF16 if ab == "bf16" else xt.XT_F32, accumulate=1)
    xt.xt_matmul_fwd(d, dev(A, ab), dev(B, ab), Cd); sync()
    assert norm_err(host(Cd), C0 + A @ B) <= bound(ab, "f32")
    # K = 0: C = 0 without accumulate, unchanged with
    d0 = xt.matmul_desc(M, N, 0, dtype_ab=d.dtype_ab, accumulate=0, lda=8, ldb=N)
    xt.xt_matmul_fwd(d0, dev(A, ab), dev(B, ab), Cd); sync()
    assert np.all(host(Cd) == 0)


@pytest.mark.parametrize("ab", ["bf16", "f32"])
@pytest.mark.parametrize("S,hd", [(256, 64), (200, 64), (16, 16)])
def test_matmul_batched_heads(ab, S, hd):
    """Attention layout: q, k, v are column blocks of a [B·S, 3·H·hd] buffer; per (b, h)
    scores = q kᵀ · scale into [B, H, S, S]; o = P v into [B·S, H·hd]."""
    Bn, H = 2, 3
    dm = H * hd
    qkv = synth.normal((Bn * S, 3 * dm), 44, dtype=ab)
    q = qkv[:, :dm].reshape(Bn, S, H, hd).transpose(0, 2, 1, 3)
    k = qkv[:, dm:2 * dm].reshape(Bn, S, H, hd).transpose(0, 2, 1, 3)
    v = qkv[:, 2 * dm:].reshape(Bn, S, H, hd).transpose(0, 2, 1, 3)
    QKV = dev(qkv, ab)
    dab = xt.XT_BF16 if ab == "bf16" else xt.XT_F32
    e = 2 if ab == "bf16" else 4
    sc = 1.0 / np.sqrt(hd)
    scores = empty((Bn, H, S, S))
    d = xt.matmul_desc(S, S, hd, trans_a=0, trans_b=1, lda=3 * dm, ldb=3 * dm, ldc=S, batch_outer=Bn,
                       batch_inner=H, dtype_ab=dab, dtype_c=xt.XT_F32, alpha=sc,
                       strides=(S * 3 * dm, hd, S * 3 * dm, hd, H * S * S, S * S))
    xt.xt_matmul_fwd(d, QKV, QKV[:, dm:], scores); sync()
    want = np.einsum("bhsd,bhtd->bhst", q, k) * sc
    assert norm_err(host(scores), want) <= bound(ab, "f32")
    # o = P v with P from the oracle, written into the head-interleaved [B·S, H·hd] layout
    P = synth.to_storage(O.softmax_fwd(want, causal=True), ab)
    out = torch.zeros((Bn * S, dm), dtype=torch.float32, device="cuda")
    d2 = xt.matmul_desc(S, hd, S, trans_a=0, trans_b=0, lda=S, ldb=3 * dm, ldc=dm, batch_outer=Bn, batch_inner=H,
                        dtype_ab=dab, dtype_c=xt.XT_F32, strides=(H * S * S, S * S, S * 3 * dm, hd, S * dm, hd))
    xt.xt_matmul_fwd(d2, dev(P, ab), QKV[:, 2 * dm:], out); sync()
    wo = np.einsum("bhst,bhtd->bhsd", P, v).transpose(0, 2, 1, 3).reshape(Bn * S, dm)
    assert norm_err(host(out), wo) <= bound(ab, "f32")
    del e


@pytest.mark.parametrize("S", [384, 200, 1024])
def test_matmul_causal_modes(S):
    """Mode 1 skips output tiles above the diagonal block; mode 2 stops K at the block
    diagonal (probabilities are 0 beyond); mode 3 starts K at the block diagonal."""
    hd = 64
    rng = np.random.default_rng(45)
    q = synth.normal((S, hd), 46, dtype="bf16")
    k = synth.normal((S, hd), 47, dtype="bf16")
    full = q @ k.T
    C = empty((S, S), fill=float("nan"))
    d = xt.matmul_desc(S, S, hd, trans_b=1, causal=1)
    xt.xt_matmul_fwd(d, dev(q, "bf16"), dev(k, "bf16"), C); sync()
    g = host(C)
    s_idx, c_idx = np.meshgrid(np.arange(S), np.arange(S), indexing="ij")
    need = c_idx < np.minimum((s_idx // 128 + 1) * 128, S)   # what the causal softmax reads
    assert norm_err(g[need], full[need]) <= 1e-5
    # mode 2: A is a causal probability block (zero beyond each row's 128-aligned extent)
    P = np.where(c_idx <= s_idx, synth.normal((S, S), 48, dtype="bf16"), 0.0)
    Pd = dev(np.where(need, P, np.nan), "bf16")   # beyond the extent: never read
    v = synth.normal((S, hd), 49, dtype="bf16")
    O2 = empty((S, hd))
    d2 = xt.matmul_desc(S, hd, S, causal=2)
    xt.xt_matmul_fwd(d2, Pd, dev(v, "bf16"), O2); sync()
    assert norm_err(host(O2), P @ v) <= 1e-5
    # mode 3: dV = Pᵀ dO with P stored [S_q, S_k] read transposed
    dO = synth.normal((S, hd), 50, dtype="bf16")
    dV = empty((S, hd))
    d3 = xt.matmul_desc(S, hd, S, trans_a=1, causal=3)
    xt.xt_matmul_fwd(d3, Pd, dev(dO, "bf16"), dV); sync()
    assert norm_err(host(dV), P.T @ dO) <= 1e-5
    del rng


@pytest.mark.parametrize("ab", ["bf16", "f32"])
@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_matmul_bwd(ab, ta, tb):
    M, N, K = 264, 200, 136
    A, B = stored(M, N, K, ta, tb, ab, 51)
    dC = synth.normal((M, N), 53, dtype=ab)
    dA_r, dB_r = O.matmul_bwd(dC, op(A, ta), op(B, tb))
    dA_r, dB_r = op(dA_r, ta) * 2.0, op(dB_r, tb) * 2.0   # back into the stored layouts, alpha = 2
    dab = xt.XT_BF16 if ab == "bf16" else xt.XT_F32
    d = xt.matmul_desc(M, N, K, trans_a=ta, trans_b=tb, dtype_ab=dab, alpha=2.0)
    dA = empty(A.shape)
    dB = torch.ones(B.shape, dtype=torch.float32, device="cuda")
    xt.xt_matmul_bwd(d, dev(A, ab), dev(B, ab), dev(dC, ab), dA, dB, 0, 1); sync()
    assert norm_err(host(dA), dA_r) <= bound(ab, "f32")
    assert norm_err(host(dB), dB_r + 1) <= bound(ab, "f32")


def test_matmul_large_sampled():
    """Transformer-sized projections (QKV of the 12-layer stack: 8192 × 2304 × 768) and the
    tied logits (8192 × 50304 × 768, NT), checked on sampled rows against the oracle."""
    for (M, N, K, tb) in [(8192, 2304, 768, 0), (8192, 50304, 768, 1)]:
        A = synth.normal((M, K), 54, dtype="bf16")
        B = synth.normal((N, K) if tb else (K, N), 55, std=0.02, dtype="bf16")
        C = empty((M, N), "bf16")
        d = xt.matmul_desc(M, N, K, trans_b=tb, dtype_c=xt.XT_BF16)
        xt.xt_matmul_fwd(d, dev(A, "bf16"), dev(B, "bf16"), C); sync()
        rows = np.random.default_rng(0).choice(M, 24, replace=False)
        rows = np.concatenate([rows, [0, 127, 128, M - 1]])
        want = A[rows] @ op(B, tb)
        assert norm_err(host(C[torch.tensor(rows, device="cuda")]), want) <= 4e-3
        assert xt.device_errors() == 0


def test_matmul_alignment_rejected():
    A = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.float32, device="cuda")
    d = xt.matmul_desc(64, 64, 60, lda=60, ldb=64)   # 120-byte rows: not 16-byte aligned
    with pytest.raises(xt.XtError) as ei:
        xt.xt_matmul_fwd(d, A, A, C)
    assert ei.value.code == xt.XT_ERR_ALIGNMENT


@pytest.fixture
def schedule():
    """Sets the GEMM schedule override for one test and restores the model's choice after."""
    yield xt.gemm_set_schedule
    xt.gemm_set_schedule(0)


def schedules_of(fn):
    """Runs fn with GEMM profiling on; the schedule code of each GEMM launch it made
    (causal mode, 10 × K splits, or 1000 for stream-K)."""
    xt.profile_gemm(64)
    try:
        fn()
        sync()
        _, _, sh = xt.profile_gemm_read(shapes=True)
    finally:
        xt.profile_gemm(0)
    return [int(x) for x in sh[:, 7]]


@pytest.mark.parametrize("ab", ["bf16", "f32"])
@pytest.mark.parametrize("c", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", [(768, 768, 8192), (768, 3072, 8192), (200, 136, 4096)])
def test_matmul_split_k(ab, c, M, N, K, schedule):
    """Weight-gradient shapes (small M·N, long K) under the deterministic K split: partial
    tiles in workspace slices, then a fixed-order reduction into C (with += here)."""
    schedule(2)
    A = synth.normal((K, M), 56, dtype=ab)   # stored [K, M]: dW = xᵀ dy layout
    B = synth.normal((K, N), 57, dtype=ab)
    C0 = synth.normal((M, N), 58, dtype=c)
    d = xt.matmul_desc(M, N, K, trans_a=1, dtype_ab=xt.XT_BF16 if ab == "bf16" else xt.XT_F32,
                       dtype_c=xt.XT_F32 if c == "f32" else xt.XT_BF16, accumulate=1, alpha=0.5)
    outs = []
    for _ in range(2):
        Cd = dev(C0, c)
        xt.xt_matmul_fwd(d, dev(A, ab), dev(B, ab), Cd)
        sync()
        outs.append(host(Cd))
    want = C0 + 0.5 * (A.T @ B)
    tol = bound(ab, c) if c == "f32" else 8e-3
    assert norm_err(outs[0], want) <= tol
    assert np.array_equal(outs[0], outs[1]), "K split is not deterministic"
    assert xt.device_errors() == 0


# (M, N, K, trans_a): the weight-gradient layout; ragged M, N and K; a few output tiles over
# a long K, so every CTA holds a piece of one and a tile's first CTA adds many partials; a tile
# count that is not a multiple of the SMs with short K (enough k-blocks for two-way slices).
SK_CASES = [(768, 768, 8192, 1), (200, 136, 4096, 1), (128, 256, 10240, 0), (1000, 776, 656, 0)]


@pytest.mark.parametrize("form", [3, 4])
@pytest.mark.parametrize("ab", ["bf16", "f32"])
@pytest.mark.parametrize("c", ["f32", "bf16"])
@pytest.mark.parametrize("acc", [0, 1])
@pytest.mark.parametrize("M,N,K,ta", SK_CASES)
def test_matmul_stream_k(form, ab, c, acc, M, N, K, ta, schedule):
    """Stream-K schedules (3: equal shares of k-block iterations over every SM; 4: tiles × s
    CTAs, one K slice each): partial tiles pass through workspace slots and flags and are
    summed in CTA order by each tile's first CTA.  Same bound as the whole-tile schedule,
    bit-identical on a rerun."""
    schedule(form)
    A = synth.normal((K, M) if ta else (M, K), 60, dtype=ab)
    B = synth.normal((K, N), 61, dtype=ab)
    C0 = synth.normal((M, N), 62, dtype=c)
    d = xt.matmul_desc(M, N, K, trans_a=ta, dtype_ab=xt.XT_BF16 if ab == "bf16" else xt.XT_F32,
                       dtype_c=xt.XT_F32 if c == "f32" else xt.XT_BF16, accumulate=acc, alpha=0.5)
    Ad, Bd = dev(A, ab), dev(B, ab)
    ws = xt.matmul_workspace(d)
    outs = []
    for _ in range(2):
        Cd = dev(C0, c)
        codes = schedules_of(lambda: xt.xt_matmul_fwd(d, Ad, Bd, Cd, ws=ws))
        assert len(codes) == 1 and (codes[0] == 1000 if form == 3 else codes[0] > 1000), codes
        outs.append(host(Cd))
    want = (C0 if acc else 0) + 0.5 * (op(A, ta) @ B)
    tol = bound(ab, c) if (c == "f32" or not acc) else 8e-3
    assert norm_err(outs[0], want) <= tol
    assert np.array_equal(outs[0], outs[1]), "stream-K is not deterministic"
    assert xt.device_errors() == 0
    # the flag words are left zero for the next call
    assert int(ws[:4096].count_nonzero()) == 0


@pytest.mark.parametrize("form", [3, 4])
def test_matmul_stream_k_batched(form, schedule):
    """Stream-K over batched tiles (outer 2 × inner 3 batches with element strides)."""
    schedule(form)
    Bo, Bi, M, N, K = 2, 3, 200, 96, 2048
    A = synth.normal((Bo, Bi, M, K), 63, dtype="bf16")
    B = synth.normal((Bo, Bi, K, N), 64, dtype="bf16")
    Cd = empty((Bo, Bi, M, N))
    d = xt.matmul_desc(M, N, K, batch_outer=Bo, batch_inner=Bi,
                       strides=(Bi * M * K, M * K, Bi * K * N, K * N, Bi * M * N, M * N))
    codes = schedules_of(lambda: xt.xt_matmul_fwd(d, dev(A, "bf16"), dev(B, "bf16"), Cd))
    assert len(codes) == 1 and (codes[0] == 1000 if form == 3 else codes[0] > 1000), codes
    assert norm_err(host(Cd), A @ B) <= 1e-5
    assert xt.device_errors() == 0


@pytest.mark.parametrize("M,N,K,tb", [(8192, 768, 3072, 0), (3072, 768, 8192, 0), (8192, 768, 2304, 1)])
def test_matmul_model_schedule_full_size(M, N, K, tb):
    """The 12-layer stack's shapes under the time model's own choice (whole tiles, a K split or
    a stream-K form, single or paired CTAs), checked on sampled rows against the oracle product
    of those rows."""
    A = synth.normal((M, K), 65, std=0.5, dtype="bf16")
    B = synth.normal((N, K) if tb else (K, N), 66, std=0.02, dtype="bf16")
    Cm = empty((M, N), "bf16")
    d = xt.matmul_desc(M, N, K, trans_b=tb, dtype_c=xt.XT_BF16)
    Ad, Bd = dev(A, "bf16"), dev(B, "bf16")
    codes = schedules_of(lambda: xt.xt_matmul_fwd(d, Ad, Bd, Cm))
    assert len(codes) == 1, codes
    rows = np.random.default_rng(1).choice(M, 24, replace=False)
    rows = np.concatenate([rows, [0, 127, 128, M - 1]])
    want = A[rows] @ op(B, tb)
    assert norm_err(host(Cm[torch.tensor(rows, device="cuda")]), want) <= 4e-3
    assert xt.device_errors() == 0


def test_gemm_set_schedule_rejects():
    with pytest.raises(xt.XtError):
        xt.gemm_set_schedule(5)


GELU_CASES = [(200, 320, 72), (1000, 768, 328), (256, 3072, 768), (128, 64, 64)]


@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", GELU_CASES)
def test_matmul_gelu_fwd(ta, tb, M, N, K):
    """[BP] MLP up projection + exact GELU from one GEMM: C = α·op(A)@op(B) in bf16, and
    Y = gelu(C) of that rounded C to one bf16 ulp; end to end Y against the oracle's
    gelu(matmul) within the bf16 GEMM bound."""
    A, B = stored(M, N, K, ta, tb, "bf16", 45)
    want_c = O.matmul_fwd(op(A, ta), op(B, tb)) * 0.5
    Cm = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Y = empty((M, N), "bf16")
    d = xt.matmul_desc(M, N, K, trans_a=ta, trans_b=tb, dtype_c=xt.XT_BF16, alpha=0.5)
    xt.xt_matmul_gelu_fwd(d, dev(A, "bf16"), dev(B, "bf16"), Cm, Y); sync()
    assert xt.device_errors() == 0
    c = host(Cm)
    assert norm_err(c, want_c) <= 4e-3
    check(host(Y), O.gelu_fwd(c), "bf16", "gelu of the stored pre-activation")
    assert norm_err(host(Y), O.gelu_fwd(want_c)) <= 4e-3


@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", GELU_CASES)
def test_matmul_gelu_bwd(ta, tb, M, N, K):
    """GELU backward fused after the product: C = (α·op(A)@op(B)) ∘ gelu'(X)."""
    A, B = stored(M, N, K, ta, tb, "bf16", 46)
    X = synth.normal((M, N), 47, dtype="bf16")
    want = O.gelu_bwd(O.matmul_fwd(op(A, ta), op(B, tb)) * 0.5, X)
    Cm = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    d = xt.matmul_desc(M, N, K, trans_a=ta, trans_b=tb, dtype_c=xt.XT_BF16, alpha=0.5)
    xt.xt_matmul_gelu_bwd(d, dev(A, "bf16"), dev(B, "bf16"), dev(X, "bf16"), Cm); sync()
    assert xt.device_errors() == 0
    assert norm_err(host(Cm), want) <= 4e-3


def test_matmul_gelu_rejects():
    A = torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(64, 96, dtype=torch.bfloat16, device="cuda")
    Cm = torch.zeros(128, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(xt.XtError):   # N not a multiple of 64
        xt.xt_matmul_gelu_fwd(xt.matmul_desc(128, 96, 64, dtype_c=xt.XT_BF16), A, B, Cm, Cm)
    C32 = torch.zeros(128, 128, dtype=torch.float32, device="cuda")
    B2 = torch.zeros(64, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(xt.XtError):   # float32 output
        xt.xt_matmul_gelu_fwd(xt.matmul_desc(128, 128, 64, dtype_c=xt.XT_F32), A, B2, C32, C32)
