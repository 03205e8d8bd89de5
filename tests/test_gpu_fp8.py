"""GPU parity of the FP8 E4M3 path against the oracle: per-tensor quantization bit for bit (the
codes are decided in the same float32 product x·scale on both sides), the dequantization factor
exactly, and the e4m3 GEMM against the float64 product of the same decoded codes (products of
e4m3 values are exact in float32, so only the float32 accumulation and the output rounding
remain: ≤ 1e-5 normalised for float32 C, ≤ 4e-3 for bf16 C)."""
import numpy as np
import pytest
import torch

import synth
from oracle import fp8 as F
from tests.gpu_util import norm_err

pytestmark = pytest.mark.gpu

xt = pytest.importorskip("transformer_fwd_bwd_gb300.xt")


def quant_gpu(x_dev):
    out = torch.empty(x_dev.numel(), dtype=torch.uint8, device="cuda")
    dq = torch.empty(1, dtype=torch.float32, device="cuda")
    xt.xt_quantize_fp8(x_dev, out, dq)
    torch.cuda.synchronize()
    return out, dq


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n,std", [(1, 1.0), (4097, 3.0), (100003, 1e-3), (65536, 1e4), (7, 0.0)])
def test_quantize_bit_exact(dtype, n, std):
    x = synth.normal((n,), 70 + n, std=std if std > 0 else 1.0, dtype=dtype)
    if std == 0:
        x = np.zeros(n, np.float32)
    xd = torch.tensor(np.asarray(x, np.float32), device="cuda")
    if dtype == "bf16":
        xd = xd.to(torch.bfloat16)
    codes, dq = quant_gpu(xd)
    want, scale = F.quantize(np.asarray(xd.float().cpu().numpy(), np.float32))
    assert np.array_equal(codes.cpu().numpy(), want.ravel())
    amax = np.float32(np.max(np.abs(xd.float().cpu().numpy()))) if n else np.float32(0)
    want_dq = np.float32(amax) / np.float32(448.0) if amax > 0 else np.float32(1.0)
    assert np.float32(dq.item()) == want_dq
    assert xt.device_errors() == 0


def codes_dev(codes, ld):
    M, K = codes.shape
    buf = torch.zeros((M, ld), dtype=torch.uint8, device="cuda")
    buf[:, :K] = torch.tensor(codes, device="cuda")
    return buf[:, :K]


@pytest.mark.parametrize("c", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (200, 136, 328), (1000, 776, 1000), (256, 3072, 768)])
def test_matmul_fp8_parity(c, M, N, K):
    rng = np.random.default_rng(M + N + K)
    A = F.quantize(rng.normal(size=(M, K)).astype(np.float32))[0]
    B = F.quantize(rng.normal(size=(N, K)).astype(np.float32))[0]
    ld = (K + 15) // 16 * 16 + 16   # padded rows: the kernel reads only K codes of each
    Ad, Bd = codes_dev(A, ld), codes_dev(B, ld)
    sa = torch.tensor([0.0123], dtype=torch.float32, device="cuda")
    sb = torch.tensor([0.75], dtype=torch.float32, device="cuda")
    Cd = torch.empty((M, N), dtype=torch.float32 if c == "f32" else torch.bfloat16, device="cuda")
    xt.xt_matmul_fp8_fwd(Ad, Bd, Cd, alpha=0.5, scale_a=sa, scale_b=sb)
    torch.cuda.synchronize()
    want = F.matmul_fp8(A, B, 0.5, float(np.float32(0.0123)), 0.75)
    assert norm_err(Cd.float().cpu().numpy(), want) <= (1e-5 if c == "f32" else 4e-3)
    assert xt.device_errors() == 0


def test_matmul_fp8_accumulate_and_full_size_rows():
    """8192 × 3072 × 768 (the MLP up projection's shape) with C += into float32, checked on
    sampled rows; scales NULL (1)."""
    M, N, K = 8192, 3072, 768
    rng = np.random.default_rng(3)
    A = F.quantize(rng.normal(size=(M, K)).astype(np.float32))[0]
    B = F.quantize(rng.normal(size=(N, K)).astype(np.float32))[0]
    C0 = rng.normal(size=(M, N)).astype(np.float32)
    Cd = torch.tensor(C0, device="cuda")
    xt.xt_matmul_fp8_fwd(torch.tensor(A, device="cuda"), torch.tensor(B, device="cuda"), Cd, alpha=0.25,
                         accumulate=1)
    torch.cuda.synchronize()
    rows = np.concatenate([rng.choice(M, 24, replace=False), [0, 127, 128, M - 1]])
    want = C0[rows] + F.matmul_fp8(A[rows], B, 0.25)
    got = Cd[torch.tensor(rows, device="cuda")].cpu().numpy()
    assert norm_err(got, want) <= 1e-5
    assert xt.device_errors() == 0


def test_fp8_end_to_end_close_to_unquantized():
    """Quantize activations and weights on the GPU, multiply in e4m3 with the dequant factors:
    within the format's resolution (3 mantissa bits) of the float64 product of the originals."""
    rng = np.random.default_rng(4)
    x = rng.normal(size=(512, 768)).astype(np.float32)
    w = (rng.normal(size=(1024, 768)) * 0.02).astype(np.float32)
    xq, dx = quant_gpu(torch.tensor(x, device="cuda"))
    wq, dw = quant_gpu(torch.tensor(w, device="cuda"))
    Cd = torch.empty((512, 1024), dtype=torch.float32, device="cuda")
    xt.xt_matmul_fp8_fwd(xq.view(512, 768), wq.view(1024, 768), Cd, scale_a=dx, scale_b=dw)
    torch.cuda.synchronize()
    assert norm_err(Cd.cpu().numpy(), x.astype(np.float64) @ w.astype(np.float64).T) <= 0.06


def test_matmul_fp8_rejects():
    A = torch.zeros((64, 40), dtype=torch.uint8, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(xt.XtError) as ei:   # 40-byte rows: not 16-byte multiples
        xt.xt_matmul_fp8_fwd(A, A, C[:, :64])
    assert ei.value.code == xt.XT_ERR_ALIGNMENT
