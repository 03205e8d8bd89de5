"""Bounded waits on the GPU (failure detection without a fault): with the wait limit set to
1 ns, the first wait of a tensor-core kernel that is not already satisfied runs out, the kernel
records XT_DEVERR_TIMEOUT in the device flag, stops issuing work, waits (with the default limit)
for its own copies and MMAs, releases its tensor memory and returns.  The call returns, the flag
reads back on the host, and after the flag is cleared and the limit restored the same call
gives the same result as before, bit for bit (and the GEMM the oracle's product)."""
import numpy as np
import pytest
import torch

import synth
from tests.gpu_util import dev, host, norm_err, sync

pytestmark = pytest.mark.gpu

xt = pytest.importorskip("transformer_fwd_bwd_gb300.xt")

DEFAULT_NS = 2_000_000_000


@pytest.fixture
def short_waits():
    xt.clear_device_errors()
    yield
    xt.set_wait_limit_ns(0)
    xt.gemm_set_pairing(0)
    xt.gemm_set_schedule(0)
    xt.clear_device_errors()


def test_wait_limit_setter():
    assert xt.wait_limit_ns() == DEFAULT_NS
    xt.set_wait_limit_ns(12345)
    assert xt.wait_limit_ns() == 12345
    xt.set_wait_limit_ns(0)
    assert xt.wait_limit_ns() == DEFAULT_NS


def test_gemm_wait_runs_out_then_recovers(short_waits):
    """Single-CTA GEMM, whole tiles (no stream-K flags in a workspace): the epilogue's first
    wait for an accumulator (256 k-blocks of MMAs) cannot be satisfied within 1 ns."""
    xt.gemm_set_pairing(1)
    xt.gemm_set_schedule(1)
    M, N, K = 1024, 1024, 16384
    A = synth.normal((M, K), 160, dtype="bf16")
    B = synth.normal((K, N), 161, dtype="bf16")
    Ad, Bd = dev(A, "bf16"), dev(B, "bf16")
    d = xt.matmul_desc(M, N, K)
    C0 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    xt.xt_matmul_fwd(d, Ad, Bd, C0); sync()
    assert xt.device_errors() == 0
    ref = host(C0)
    # K = 16384 float32 accumulation: the rounding of the running sums grows with K
    assert norm_err(ref, A @ B) <= 1e-4

    xt.set_wait_limit_ns(1)
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    xt.xt_matmul_fwd(d, Ad, Bd, C)   # enqueued normally: the give-up happens on the device
    sync()
    assert xt.device_errors() & xt.XT_DEVERR_TIMEOUT
    assert torch.cuda.is_available() and torch.cuda.synchronize() is None   # the context is usable

    xt.set_wait_limit_ns(0)
    xt.clear_device_errors()
    assert xt.device_errors() == 0
    xt.xt_matmul_fwd(d, Ad, Bd, C); sync()
    assert xt.device_errors() == 0
    assert np.array_equal(host(C), ref)


def test_attention_waits_run_out_then_recover(short_waits):
    """Fused attention forward and backward (causal, B2 H4 S1024 hd64): each kernel's first
    waits (tiles landing, scores computed) cannot be satisfied within 1 ns."""
    Bn, H, S, hd = 2, 4, 1024, 64
    d = H * hd
    qkv = dev(synth.normal((Bn * S, 3 * d), 162, dtype="bf16"), "bf16")
    dO = dev(synth.normal((Bn * S, d), 163, dtype="bf16"), "bf16")
    q, k, v = qkv[:, :d], qkv[:, d:2 * d], qkv[:, 2 * d:]
    nws = xt.ws_bytes("xt_attention_bwd_workspace_size", Bn, S, H)
    ws = torch.zeros(max(1, nws), dtype=torch.uint8, device="cuda")

    def run():
        o = torch.empty((Bn * S, d), dtype=torch.bfloat16, device="cuda")
        o_lo = torch.empty_like(o)
        lse = torch.empty((Bn, H, S), dtype=torch.float32, device="cuda")
        dqkv = torch.zeros_like(qkv)
        xt.xt_attention_fwd(q, k, v, o, lse, Bn, S, H, hd, 1, o_lo=o_lo)
        xt.xt_attention_bwd(q, k, v, o, dO, lse, dqkv[:, :d], dqkv[:, d:2 * d], dqkv[:, 2 * d:], Bn, S, H, hd, 1,
                            o_lo=o_lo, ws=ws)
        sync()
        return [host(t) for t in (o, lse, dqkv)]

    ref = run()
    assert xt.device_errors() == 0
    xt.set_wait_limit_ns(1)
    run()
    assert xt.device_errors() & xt.XT_DEVERR_TIMEOUT
    xt.set_wait_limit_ns(0)
    xt.clear_device_errors()
    again = run()
    assert xt.device_errors() == 0
    for a, b in zip(again, ref):
        assert np.array_equal(a, b)
