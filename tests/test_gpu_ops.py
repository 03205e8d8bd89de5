"""GPU parity of every row / elementwise op against the oracle, through the C ABI.

Inputs come from `synth` (seeded), are rounded to the run's dtype, and are fed to both
sides; shapes span several vectors / row groups plus ragged tails and the scalar path.
Column reductions (dγ, dβ, dbias, full sums) are compared with a bound proportional to
the sum of the magnitudes of their terms (the condition of a sum): |g − r| ≤ 1e-5·Σ|terms|
(+ 1 bf16 ulp for bf16 outputs).
"""
import numpy as np
import pytest
import torch
from scipy.special import erf

import synth
from oracle import dropout as OD
from oracle import ops as O
from tests.gpu_util import check, dev, empty, host, sync

pytestmark = pytest.mark.gpu

xt = pytest.importorskip("transformer_fwd_bwd_gb300.xt")

DTYPES = ["f32", "bf16"]
ROWS_COLS = [(37, 768), (6, 1000), (9, 33), (3, 4096), (2, 8192), (300, 64)]


def inputs(shape, seed, dtype, std=1.0, mean=0.0):
    return synth.normal(shape, seed, std=std, mean=mean, dtype=dtype)


def check_sum(g, r, abs_sum, dtype, what=""):
    g, r, a = (np.asarray(v, np.float64) for v in (g, r, abs_sum))
    tol = 1e-5 * np.maximum(a, 1e-30)
    if dtype == "bf16":
        ar = np.abs(r)
        with np.errstate(divide="ignore"):
            e = np.floor(np.log2(np.where(ar > 0, ar, 1e-300)))
        tol = tol + np.where(ar > 0, 2.0 ** (e - 7), 0.0)
    excess = float(np.max(np.abs(g - r) / tol))
    assert excess <= 1.0, f"{what}: column-sum error {excess:.3f}× the bound"


# ----------------------------------------------------------------------------- elementwise


@pytest.mark.parametrize("dtype", DTYPES)
def test_gelu_paired_matches_scalar(dtype):
    """The 16-byte-aligned path evaluates GELU's erfc polynomial two elements per paired FMA; an
    unaligned view takes the one-element path. Each lane of a paired FMA rounds as the scalar FMA
    does, so the two must agree bit for bit."""
    n = 8 * 4101
    a = inputs((n,), 31, dtype) * 3
    d = inputs((n,), 32, dtype)
    A, D = dev(a, dtype), dev(d, dtype)
    y1, y2 = empty((n,), dtype), empty((n,), dtype)
    xt.xt_gelu_fwd(A, y1)
    xt.xt_gelu_fwd(A[1:], y2[1:])
    sync()
    assert torch.equal(y1[1:], y2[1:])
    xt.xt_gelu_bwd(D, A, y1)
    xt.xt_gelu_bwd(D[1:], A[1:], y2[1:])
    sync()
    assert torch.equal(y1[1:], y2[1:])


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [1, 37, 4101, 768 * 1024])
def test_elementwise(dtype, n):
    a = inputs((n,), 1, dtype) * 2
    b = inputs((n,), 2, dtype)
    d = inputs((n,), 3, dtype)
    A, B, D = dev(a, dtype), dev(b, dtype), dev(d, dtype)
    y = empty((n,), dtype)
    xt.xt_add_fwd(A, B, y); sync(); check(host(y), a + b, dtype, "add", mag=np.abs(a) + np.abs(b))
    xt.xt_mul_fwd(A, B, y); sync(); check(host(y), a * b, dtype, "mul")
    xt.xt_scale_fwd(A, y, 0.37); sync(); check(host(y), a * np.float32(0.37), dtype, "scale")
    xt.xt_silu_fwd(A, y); sync(); check(host(y), O.silu_fwd(a), dtype, "silu")
    sg = O.sigmoid(a)
    xt.xt_silu_bwd(D, A, y); sync()
    check(host(y), O.silu_bwd(d, a), dtype, "silu_bwd", mag=np.abs(d) * (sg + np.abs(a) * sg * (1 - sg)))
    xt.xt_gelu_fwd(A, y); sync(); check(host(y), O.gelu_fwd(a), dtype, "gelu")
    Phi, phi = 0.5 * (1 + erf(a / np.sqrt(2))), np.exp(-a * a / 2) / np.sqrt(2 * np.pi)
    xt.xt_gelu_bwd(D, A, y); sync()
    check(host(y), O.gelu_bwd(d, a), dtype, "gelu_bwd", mag=np.abs(d) * (Phi + np.abs(a) * phi))
    da, db = empty((n,), dtype), empty((n,), dtype)
    xt.xt_mul_bwd(D, A, B, da, db); sync()
    ra, rb = O.mul_bwd(d, a, b)
    check(host(da), ra, dtype, "mul_bwd a"); check(host(db), rb, dtype, "mul_bwd b")
    # mul(x, x): both grads pushed into one buffer (accumulate on the second)
    xt.xt_mul_bwd(D, A, A, da, da, 0, 1); sync()
    check(host(da), 2 * d * a, dtype, "mul(x,x) bwd")  # second push adds an equal value: exact
    # add backward copies / accumulates
    xt.xt_add_bwd(D, da, db, 0, 1); sync()
    check(host(da), d, dtype, "add_bwd copy")
    rb_s = synth.to_storage(rb, dtype)
    check(host(db), rb_s + d, dtype, "add_bwd acc", mag=np.abs(rb_s) + np.abs(d))
    # scale backward with accumulate
    z = dev(np.ones(n), dtype)
    xt.xt_scale_bwd(D, z, 2.0, acc=1); sync()
    check(host(z), 1 + 2 * d, dtype, "scale_bwd acc", mag=1 + 2 * np.abs(d))


def test_accumulate_mixed_dtypes():
    n = 10007
    base = inputs((n,), 4, "f32")
    src = inputs((n,), 5, "bf16")
    dst = dev(base, "f32")
    xt.xt_accumulate(dst, dev(src, "bf16")); sync()
    check(host(dst), base + src, "f32", "f32 += bf16", mag=np.abs(base) + np.abs(src))
    dstb = dev(synth.round_bf16(base), "bf16")
    xt.xt_accumulate(dstb, dev(src, "bf16")); sync()
    bb = synth.round_bf16(base)
    check(host(dstb), bb + src, "bf16", "bf16 += bf16", mag=np.abs(bb) + np.abs(src))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [5, 100003, 8192 * 768])
def test_sum(dtype, n):
    x = inputs((n,), 6, dtype)
    out = torch.zeros(1, dtype=torch.float32, device="cuda")
    xt.xt_sum_fwd(dev(x, dtype), out); sync()
    check_sum(host(out), [x.sum()], [np.abs(x).sum()], "f32", "sum")
    up = torch.tensor([1.75], device="cuda")
    dx = empty((n,), dtype)
    xt.xt_sum_bwd(up, dx); sync()
    assert np.all(host(dx) == 1.75)


# ----------------------------------------------------------------------------- norms


@pytest.mark.parametrize("dtype", DTYPES)
# (8192, 768): the stack's size, every block's dγ partial carried over several rows per warp
@pytest.mark.parametrize("rows,cols", ROWS_COLS + [(8192, 768)])
def test_rms_norm(dtype, rows, cols):
    x = inputs((rows, cols), 7, dtype)
    gamma = inputs((cols,), 8, dtype, std=0.1, mean=1.0)
    d = inputs((rows, cols), 9, dtype)
    eps = 1e-5
    y, ir = O.rms_norm_fwd(x, gamma, eps)
    X, G, Dd = dev(x, dtype), dev(gamma, dtype), dev(d, dtype)
    Y, IR = empty((rows, cols), dtype), empty((rows,), "f32")
    xt.xt_rms_norm_fwd(X, G, Y, IR, eps); sync()
    check(host(Y), y, dtype, "rms y")
    check(host(IR), ir, "f32", "rms inv_rms")
    IRo = dev(ir, "f32")
    dx, dg = O.rms_norm_bwd(d, x, gamma, np.float32(ir).astype(np.float64))
    DX, DG = empty((rows, cols), dtype), empty((cols,), "f32")
    xt.xt_rms_norm_bwd(Dd, X, G, IRo, DX, DG); sync()
    irr = np.float32(ir).astype(np.float64)
    # the row reduction Σ d·γ·x cancels: its rounding is relative to Σ|d·γ·x|, not to |Σ d·γ·x|
    mag_dx = np.abs(irr[:, None] * d * gamma) + np.abs(x * (irr ** 3 / cols * np.sum(np.abs(d * gamma * x), 1))[:, None])
    check(host(DX), dx, dtype, "rms dx", mag=mag_dx)
    check_sum(host(DG), dg, np.abs(d * x * ir[:, None]).sum(0), "f32", "rms dgamma")
    # accumulate paths: dx += , dγ +=
    DX2 = dev(np.ones((rows, cols)), dtype)
    DG2 = dev(np.ones(cols), "f32")
    xt.xt_rms_norm_bwd(Dd, X, G, IRo, DX2, DG2, acc_dx=1, acc_param=1); sync()
    check(host(DX2), 1 + dx, dtype, "rms dx acc", mag=1 + mag_dx)
    check_sum(host(DG2), 1 + dg, 1 + np.abs(d * x * ir[:, None]).sum(0), "f32", "rms dgamma acc")


@pytest.mark.parametrize("dtype", DTYPES)
# (1500, 2048): a bf16 row of 2048 runs with 128 threads of two vectors, two rows per block, and
# 1500 rows give each block two or three row pairs (the partials carried across rows);
# (8192, 768): the stack's size (304 blocks of eight row warps, three or four rows per warp)
@pytest.mark.parametrize("rows,cols", ROWS_COLS + [(1500, 2048), (8192, 768)])
def test_layernorm(dtype, rows, cols):
    x = inputs((rows, cols), 10, dtype, mean=0.3)
    gamma = inputs((cols,), 11, dtype, std=0.1, mean=1.0)
    beta = inputs((cols,), 12, dtype, std=0.1)
    d = inputs((rows, cols), 13, dtype)
    eps = 1e-5
    y, mu, rstd = O.layernorm_fwd(x, gamma, beta, eps)
    X = dev(x, dtype)
    Y, MU, RS = empty((rows, cols), dtype), empty((rows,), "f32"), empty((rows,), "f32")
    xt.xt_layernorm_fwd(X, dev(gamma, dtype), dev(beta, dtype), Y, MU, RS, eps); sync()
    xhat = (x - mu[:, None]) * rstd[:, None]
    # y is formed from x − μ, x̂γ and β: its error is relative to the largest of those terms, and
    # the centring x − μ carries the rounding of μ at the scale of |μ|·rstd·|γ|
    mag = np.abs(xhat * gamma) + np.abs(beta) + (np.abs(mu) * rstd)[:, None] * np.abs(gamma)
    check(host(Y), y, dtype, "ln y", mag=mag)
    assert np.max(np.abs(host(MU) - mu)) <= 1e-5 * np.max(np.abs(x))
    check(host(RS), rstd, "f32", "ln rstd")
    mu32, rs32 = np.float32(mu).astype(np.float64), np.float32(rstd).astype(np.float64)
    dx, dg, db = O.layernorm_bwd(d, x, gamma, mu32, rs32)
    DX, DG, DB = empty((rows, cols), dtype), empty((cols,), "f32"), empty((cols,), "f32")
    xt.xt_layernorm_bwd(dev(d, dtype), X, dev(gamma, dtype), dev(mu32), dev(rs32), DX, DG, DB); sync()
    # dx of LayerNorm cancels by construction (Σ dx = 0): floor relative to the row scale
    g = host(DX)
    scale = np.max(np.abs(rs32[:, None] * d * gamma), axis=1, keepdims=True)
    tol = (1e-5 if dtype == "f32" else 2.0 ** -8) * np.maximum(np.abs(dx), 1e-3 * scale) + 1e-6 * scale
    assert np.all(np.abs(g - dx) <= tol), f"ln dx max excess {np.max(np.abs(g - dx) / tol):.3f}"
    xh = (x - mu32[:, None]) * rs32[:, None]
    check_sum(host(DG), dg, np.abs(d * xh).sum(0), "f32", "ln dgamma")
    check_sum(host(DB), db, np.abs(d).sum(0), "f32", "ln dbeta")


def test_layernorm_bwd_stack_form():
    """LayerNorm backward as the 12-layer stack calls it at B 8 × S 1024, d 768: bf16 d, x and γ,
    the float32 residual gradient accumulated (dh += dx), and float32 dγ / dβ accumulated."""
    rows, cols = 8192, 768
    x = inputs((rows, cols), 14, "bf16", mean=0.3)
    gamma = inputs((cols,), 15, "bf16", std=0.1, mean=1.0)
    d = inputs((rows, cols), 16, "bf16")
    dh0 = inputs((rows, cols), 17, "f32")
    dg0, db0 = inputs((cols,), 18, "f32"), inputs((cols,), 19, "f32")
    _, mu, rstd = O.layernorm_fwd(x, gamma, np.zeros(cols), 1e-5)
    mu32, rs32 = np.float32(mu).astype(np.float64), np.float32(rstd).astype(np.float64)
    dx, dg, db = O.layernorm_bwd(d, x, gamma, mu32, rs32)
    DH, DG, DB = dev(dh0, "f32"), dev(dg0, "f32"), dev(db0, "f32")
    xt.xt_layernorm_bwd(dev(d, "bf16"), dev(x, "bf16"), dev(gamma, "bf16"), dev(mu32), dev(rs32), DH, DG, DB,
                        acc_dx=1, acc_param=1); sync()
    scale = np.max(np.abs(rs32[:, None] * d * gamma), axis=1, keepdims=True)
    tol = 1e-5 * (np.abs(dh0) + np.maximum(np.abs(dx), 1e-3 * scale)) + 1e-6 * scale
    g = host(DH)
    assert np.all(np.abs(g - (dh0 + dx)) <= tol), f"dh max excess {np.max(np.abs(g - dh0 - dx) / tol):.3f}"
    xh = (x - mu32[:, None]) * rs32[:, None]
    check_sum(host(DG), dg0 + dg, np.abs(dg0) + np.abs(d * xh).sum(0), "f32", "ln dgamma acc")
    check_sum(host(DB), db0 + db, np.abs(db0) + np.abs(d).sum(0), "f32", "ln dbeta acc")
    assert xt.device_errors() == 0


# ----------------------------------------------------------------------------- softmax


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rows,cols", [(37, 768), (5, 1000), (7, 33), (4, 8192), (64, 1024)])
def test_softmax(dtype, rows, cols):
    x = inputs((rows, cols), 14, dtype, std=3.0)
    d = inputs((rows, cols), 15, dtype)
    y = O.softmax_fwd(x)
    Y = empty((rows, cols), dtype)
    xt.xt_softmax_fwd(dev(x, dtype), Y); sync()
    check(host(Y), y, dtype, "softmax y")
    yin = synth.to_storage(y, dtype)
    dx = O.softmax_bwd(d, yin)
    DX = empty((rows, cols), dtype)
    xt.xt_softmax_bwd(dev(d, dtype), dev(yin, dtype), DX); sync()
    g = host(DX)
    scale = np.max(np.abs(yin * d), axis=1, keepdims=True)
    rel = 1e-5 if dtype == "f32" else 2.0 ** -8
    tol = rel * np.maximum(np.abs(dx), 1e-3 * scale) + 1e-6 * scale
    assert np.all(np.abs(g - dx) <= tol), f"softmax dx excess {np.max(np.abs(g - dx) / tol):.3f}"


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("S", [16, 200, 384])
@pytest.mark.parametrize("mode", [1, 2])
def test_softmax_causal(dtype, S, mode):
    BH = 3
    x = inputs((BH, S, S), 16, dtype, std=2.0)
    d = inputs((BH, S, S), 17, dtype)
    y = O.softmax_fwd(x, causal=True)
    X = dev(x, dtype)
    Y = empty((BH, S, S), dtype, fill=float("nan"))
    xt.xt_softmax_fwd(X, Y, causal=mode, q_len=S); sync()
    g = host(Y)
    s_idx = np.arange(S)[:, None]
    c_idx = np.arange(S)[None, :]
    ext = np.minimum((s_idx // 128 + 1) * 128, S) if mode == 2 else np.full((S, 1), S)
    written = np.broadcast_to(c_idx < ext, (BH, S, S))
    check(g[written], y[written], dtype, "causal softmax y")
    if mode == 2:
        assert np.all(np.isnan(g[~written])), "mode 2 wrote beyond the causal tile extent"
    yin = synth.to_storage(y, dtype)
    dx = O.softmax_bwd(d, yin)
    DX = empty((BH, S, S), dtype, fill=float("nan"))
    xt.xt_softmax_bwd(dev(d, dtype), dev(yin, dtype), DX, causal=mode, q_len=S); sync()
    gd = host(DX)
    assert np.all(gd[written & ~np.broadcast_to(c_idx <= s_idx, (BH, S, S))] == 0)
    scale = np.max(np.abs(yin * d), axis=-1, keepdims=True)
    rel = 1e-5 if dtype == "f32" else 2.0 ** -8
    tol = rel * np.maximum(np.abs(dx), 1e-3 * scale) + 1e-6 * scale
    assert np.all(np.abs(gd[written] - dx[written]) <= np.broadcast_to(tol, dx.shape)[written])


# ----------------------------------------------------------------------------- cross-entropy


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rows,V", [(37, 64), (16, 4096), (5, 1001), (3, 50304), (2, 128256)])
def test_cross_entropy(dtype, rows, V):
    x = inputs((rows, V), 18, dtype, std=2.0)
    t = synth.uniform_ids(rows, V, 19)
    loss, lse = O.cross_entropy_fwd(x, t)
    X, Tg = dev(x, dtype), torch.tensor(t, device="cuda")
    LSE, L = empty((rows,), "f32"), empty((1,), "f32")
    xt.xt_cross_entropy_fwd(X, Tg, LSE, L); sync()
    check(host(LSE), lse, "f32", "lse")
    assert abs(host(L)[0] - loss) <= 1e-5 * abs(loss)
    up = torch.tensor([1.3], device="cuda")
    lse32 = np.float32(lse).astype(np.float64)
    dx = O.cross_entropy_bwd(x, t, lse32, np.float32(1.3))
    for gdt in ("f32", dtype):
        DX = empty((rows, V), gdt)
        xt.xt_cross_entropy_bwd(X, Tg, dev(lse32), up, DX); sync()
        g = host(DX)
        scale = 1.3 / rows
        rel = 1e-5 if gdt == "f32" else 2.0 ** -8
        tol = rel * np.abs(dx) + 1e-6 * scale
        assert np.all(np.abs(g - dx) <= tol), f"ce dx ({gdt}) excess {np.max(np.abs(g - dx) / tol):.3f}"
    # in place, then accumulate into an fp32 buffer
    Xc = X.clone()
    xt.xt_cross_entropy_bwd(Xc, Tg, dev(lse32), up, Xc); sync()
    rel = 1e-5 if dtype == "f32" else 2.0 ** -8
    assert np.all(np.abs(host(Xc) - dx) <= rel * np.abs(dx) + 1e-6 * 1.3 / rows), "in-place ce bwd"
    DXa = dev(np.ones((rows, V)), "f32")
    xt.xt_cross_entropy_bwd(X, Tg, dev(lse32), up, DXa, acc=1); sync()
    assert np.max(np.abs(host(DXa) - 1 - dx)) <= 1e-5 * np.max(np.abs(dx)) + 1e-7


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rows,V", [(3, 64), (37, 1000), (7, 1001), (64, 50304), (5, 128256)])
def test_cross_entropy_fwd_bwd_fused(dtype, rows, V):
    """The one-pass forward + backward (the row held in shared memory) against the oracle, in
    place as the block runs it; rows that are not whole 16-byte vectors or exceed 200 KB
    (1001; float32 50304; 128256) take the two-kernel path."""
    x = inputs((rows, V), 21, dtype, std=2.0)
    t = synth.uniform_ids(rows, V, 22)
    loss, lse = O.cross_entropy_fwd(x, t)
    X, Tg = dev(x, dtype), torch.tensor(t, device="cuda")
    LSE, L = empty((rows,), "f32"), empty((1,), "f32")
    up = torch.tensor([1.3], device="cuda")
    xt.xt_cross_entropy_fwd_bwd(X, Tg, LSE, L, up, X); sync()
    assert xt.device_errors() == 0
    check(host(LSE), lse, "f32", "lse")
    assert abs(host(L)[0] - loss) <= 1e-5 * abs(loss)
    dx = O.cross_entropy_bwd(x, t, np.float32(host(LSE)).astype(np.float64), np.float32(1.3))
    rel = 1e-5 if dtype == "f32" else 2.0 ** -8
    assert np.all(np.abs(host(X) - dx) <= rel * np.abs(dx) + 1e-6 * 1.3 / rows), "fused ce dx"


def test_cross_entropy_bad_target_sets_flag():
    xt.clear_device_errors()
    x = dev(np.zeros((4, 64)))
    t = torch.tensor([0, 3, 64, 1], dtype=torch.int32, device="cuda")
    LSE, L = empty((4,), "f32"), empty((1,), "f32")
    xt.xt_cross_entropy_fwd(x, t, LSE, L)
    assert xt.device_errors() & xt.XT_DEVERR_INDEX
    xt.clear_device_errors()
    assert xt.device_errors() == 0


# ----------------------------------------------------------------------------- rope


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("B,S,H,hd", [(1, 16, 2, 16), (2, 100, 3, 64), (8, 1024, 2, 128), (1, 7, 1, 6)])
def test_rope(dtype, B, S, H, hd):
    d_model = H * hd
    ld = 3 * d_model   # q block inside a [T, 3d] qkv buffer
    buf = inputs((B * S, ld), 20, dtype)
    q = buf[:, :d_model].reshape(B, S, H, hd).transpose(0, 2, 1, 3)
    pos = np.arange(S)
    table = torch.empty(2 * S * (hd // 2), dtype=torch.float32, device="cuda")
    xt.xt_rope_table(table, S, hd, 10000.0)
    Buf = dev(buf, dtype)
    out = Buf.clone()
    xt.xt_rope_fwd(Buf, out, table, B, S, H, hd, ld); sync()
    want = O.rope_fwd(q, pos, 10000.0).transpose(0, 2, 1, 3).reshape(B * S, d_model)
    h = hd // 2
    th = O.rope_angles(pos, hd, 10000.0)
    qa = np.abs(q)
    mag = (np.concatenate([qa[..., :h] * np.abs(np.cos(th)) + qa[..., h:] * np.abs(np.sin(th))] * 2, axis=-1)
           .transpose(0, 2, 1, 3).reshape(B * S, d_model))
    g = host(out)
    check(g[:, :d_model], want, dtype, "rope fwd", mag=mag)
    assert np.array_equal(g[:, d_model:], host(Buf)[:, d_model:]), "rope touched other columns"
    # in place, backward
    xt.xt_rope_bwd(Buf, Buf, table, B, S, H, hd, ld); sync()
    wantb = O.rope_bwd(q, pos, 10000.0).transpose(0, 2, 1, 3).reshape(B * S, d_model)
    check(host(Buf)[:, :d_model], wantb, dtype, "rope bwd", mag=mag)


# ----------------------------------------------------------------------------- dropout


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("p", [0.0, 0.1, 0.5])
@pytest.mark.parametrize("n", [1, 1001, 8192 * 768])
def test_dropout_bit_exact(dtype, p, n):
    seed = synth.BASE_SEED_DROPOUT ^ 0xA77
    x = inputs((n,), 21, dtype)
    X = dev(x, dtype)
    Y = empty((n,), dtype)
    xt.xt_dropout_fwd(X, Y, p, seed); sync()
    want = OD.dropout_fwd(x, p, seed, dtype=dtype)
    g = Y.float().cpu().numpy()
    assert np.array_equal(g.view(np.uint32), want.astype(np.float32).view(np.uint32)), "dropout output not bit-exact"
    mask = torch.empty(n, dtype=torch.uint8, device="cuda")
    xt.xt_dropout_mask(mask, p, seed); sync()
    assert np.array_equal(mask.cpu().numpy().astype(bool), OD.keep_mask(n, p, seed))
    DX = empty((n,), dtype)
    xt.xt_dropout_bwd(X, DX, p, seed); sync()
    assert np.array_equal(DX.float().cpu().numpy().view(np.uint32), want.astype(np.float32).view(np.uint32))
    # eval is the identity
    xt.xt_dropout_fwd(X, Y, p, seed, training=0); sync()
    assert torch.equal(Y, X)


def test_dropout_add_and_errors():
    n = 70001
    h, a = inputs((n,), 22, "f32"), inputs((n,), 23, "f32")
    H, A = dev(h), dev(a)
    out = empty((n,), "f32")
    xt.xt_dropout_add_fwd(H, A, out, 0.1, 1234); sync()
    want = (np.float32(h) + OD.dropout_fwd(a, 0.1, 1234)).astype(np.float32)
    assert np.array_equal(out.cpu().numpy(), want)
    with pytest.raises(xt.XtError):
        xt.xt_dropout_fwd(H, out, 1.0, 1)
    with pytest.raises(xt.XtError):
        xt.xt_dropout_fwd(H, out, -0.1, 1)


# ----------------------------------------------------------------------------- embedding


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("B,S,d,V,pos", [(1, 16, 32, 64, False), (4, 256, 256, 4096, False),
                                          (8, 1024, 768, 50304, True), (3, 5, 12, 7, True)])
def test_embedding(dtype, B, S, d, V, pos):
    T = B * S
    E = inputs((V, d), 24, dtype, std=0.02)
    P = inputs((S, d), 25, dtype, std=0.02) if pos else None
    ids = synth.uniform_ids(T, V, 26)
    if T > 8:
        ids[: T // 4] = ids[0]  # many repeats of one id
    h = O.embedding_fwd(ids, E, P, S)
    Ids = torch.tensor(ids, device="cuda")
    Hh = empty((T, d), dtype)
    xt.xt_embedding_fwd(Ids, dev(E, dtype), dev(P, dtype) if pos else None, Hh, S); sync()
    check(host(Hh), h, dtype, "embedding fwd")
    dh = inputs((T, d), 27, dtype)
    dE, dP = O.embedding_bwd(ids, dh, V, S, with_pos=pos)
    DE = dev(np.full((V, d), 7.0), "f32")  # acc = 0 must clear untouched rows
    DP = empty((S, d), "f32") if pos else None
    xt.xt_embedding_bwd(Ids, dev(dh, dtype), DE, DP, S); sync()
    absE, _ = O.embedding_bwd(ids, np.abs(dh), V, S)
    check_sum(host(DE), dE, absE, "f32", "embedding dE")
    if pos:
        check_sum(host(DP), dP, np.abs(dh).reshape(-1, S, d).sum(0), "f32", "embedding dP")
    # accumulate adds onto the existing gradient
    xt.xt_embedding_bwd(Ids, dev(dh, dtype), DE, DP, S, acc=1); sync()
    check_sum(host(DE), 2 * dE, 2 * absE, "f32", "embedding dE acc")


def test_embedding_bad_id_sets_flag():
    xt.clear_device_errors()
    E = dev(np.zeros((8, 16)))
    Hh = empty((2, 16), "f32")
    xt.xt_embedding_fwd(torch.tensor([1, 9], dtype=torch.int32, device="cuda"), E, None, Hh, 2)
    assert xt.device_errors() & xt.XT_DEVERR_INDEX
    assert np.all(np.isnan(host(Hh)[1]))
    xt.clear_device_errors()


# ----------------------------------------------------------------------------- swiglu, add_bias


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rows,F", [(16, 64), (1024, 688), (33, 7)])
def test_swiglu(dtype, rows, F):
    gu = inputs((rows, 2 * F), 28, dtype, std=2.0)
    d = inputs((rows, F), 29, dtype)
    g, u = gu[:, :F], gu[:, F:]
    GU = dev(gu, dtype)
    Y = empty((rows, F), dtype)
    xt.xt_swiglu_fwd(GU[:, :F], GU[:, F:], Y); sync()
    check(host(Y), O.swiglu_fwd(g, u), dtype, "swiglu fwd")
    dg, du = O.swiglu_bwd(d, g, u)
    DGU = empty((rows, 2 * F), dtype)
    xt.xt_swiglu_bwd(dev(d, dtype), GU[:, :F], GU[:, F:], DGU[:, :F], DGU[:, F:]); sync()
    gd = host(DGU)
    sg = O.sigmoid(g)
    check(gd[:, :F], dg, dtype, "swiglu dg", mag=np.abs(d * u) * (sg + np.abs(g) * sg * (1 - sg)))
    check(gd[:, F:], du, dtype, "swiglu du")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rows,cols", [(37, 768), (8192, 2048), (5, 13), (1000, 520), (130, 1001)])
def test_add_bias(dtype, rows, cols):
    x = inputs((rows, cols), 30, dtype)
    b = inputs((cols,), 31, dtype, std=0.1)
    d = inputs((rows, cols), 32, dtype)
    Y = empty((rows, cols), dtype)
    xt.xt_add_bias_fwd(dev(x, dtype), dev(b, dtype), Y); sync()
    check(host(Y), O.add_bias_fwd(x, b), dtype, "add_bias fwd")
    DX, DB = empty((rows, cols), dtype), empty((cols,), "f32")
    xt.xt_add_bias_bwd(dev(d, dtype), DX, DB); sync()
    rdx, rdb = O.add_bias_bwd(d)
    check(host(DX), rdx, dtype, "add_bias dx")
    check_sum(host(DB), rdb, np.abs(d).sum(0), "f32", "add_bias dbias")
    # accumulate forms: dx += d into a buffer holding x, dbias += Σ into one holding b; dbias alone
    DXa, DBa = dev(x, dtype), dev(b, "f32")
    xt.xt_add_bias_bwd(dev(d, dtype), DXa, DBa, acc_dx=1, acc_dbias=1); sync()
    check(host(DXa), O.add_fwd(x, d), dtype, "add_bias dx accumulated")
    check_sum(host(DBa), rdb + b, np.abs(d).sum(0) + np.abs(b), "f32", "add_bias dbias accumulated")
    DB1 = empty((cols,), "f32")
    xt.xt_add_bias_bwd(dev(d, dtype), None, DB1); sync()
    assert np.array_equal(host(DB1), host(DB)), "dbias without dx differs"


@pytest.mark.parametrize("norm", ["rms", "ln"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("p,training", [(0.0, 1), (0.1, 1), (0.1, 0)])
@pytest.mark.parametrize("rows,cols", [(333, 768), (64, 97), (40, 2048)])
def test_dropout_add_norm_fused_equals_separate(norm, dtype, p, training, rows, cols):
    """[DO] § dropout 接在哪 (wiring): the residual add and the next pre-norm in one pass give the
    separate calls' results bit for bit (same masks, same arithmetic): sum, y and the statistics;
    and the norm backward fused with the preceding site's dropout backward gives the separate
    norm backward and xt_dropout_bwd_ex bit for bit (dx, dγ, dβ and the passed-on gradient)."""
    if dtype == "bf16" and cols % 8:
        cols += 8 - cols % 8
    seed = synth.BASE_SEED_DROPOUT + 7
    kind = xt.XT_NORM_RMS if norm == "rms" else xt.XT_NORM_LN
    h, a, dy = (dev(synth.normal((rows, cols), 90 + i, dtype=dtype), dtype) for i in range(3))
    gam = dev(synth.normal((cols,), 93, std=0.1, mean=1.0, dtype=dtype), dtype)
    bet = dev(synth.normal((cols,), 94, std=0.1, dtype=dtype), dtype)
    # forward: separate
    s1, y1 = empty((rows, cols), dtype), empty((rows, cols), dtype)
    st_a, st_b = empty((rows,)), empty((rows,))
    xt.xt_dropout_add_fwd(h, a, s1, p, seed, training)
    if norm == "rms":
        xt.xt_rms_norm_fwd(s1, gam, y1, st_a, 1e-5)
    else:
        xt.xt_layernorm_fwd(s1, gam, bet, y1, st_a, st_b, 1e-5)
    # forward: fused
    s2, y2 = empty((rows, cols), dtype), empty((rows, cols), dtype)
    st_c, st_d = empty((rows,)), empty((rows,))
    xt.xt_dropout_add_norm_fwd(h, a, s2, gam, bet, y2, st_c, st_d if norm == "ln" else None, p, seed, training, kind,
                               1e-5)
    sync()
    assert torch.equal(s1, s2) and torch.equal(y1, y2) and torch.equal(st_a, st_c)
    if norm == "ln":
        assert torch.equal(st_b, st_d)
    # backward: separate (dx accumulated into a float32 residual gradient, then the dropout backward)
    dh1 = dev(synth.normal((rows, cols), 95), "f32")
    dh2 = dh1.clone()
    dg1, dg2 = empty((cols,)), empty((cols,))
    db1, db2 = empty((cols,)), empty((cols,))
    g1, g2 = empty((rows, cols), dtype), empty((rows, cols), dtype)
    if norm == "rms":
        xt.xt_rms_norm_bwd(dy, s1, gam, st_a, dh1, dg1, acc_dx=1)
    else:
        xt.xt_layernorm_bwd(dy, s1, gam, st_a, st_b, dh1, dg1, db1, acc_dx=1)
    xt.xt_dropout_bwd_ex(dh1, g1, p, seed, training)
    xt.xt_norm_bwd_dropout(kind, dy, s1, gam, st_a, st_b if norm == "ln" else None, dh2, dg2,
                           db2 if norm == "ln" else None, g2, p, seed, training, acc_dx=1)
    sync()
    assert xt.device_errors() == 0
    assert torch.equal(dh1, dh2) and torch.equal(dg1, dg2) and torch.equal(g1, g2)
    if norm == "ln":
        assert torch.equal(db1, db2)
