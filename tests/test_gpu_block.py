"""GPU parity of the native block stack (xt_block_fwd / xt_block_bwd) against the oracle:
the loss and every leaf gradient, normalised error ‖g − r‖/‖r‖ ≤ 2e-2 per leaf, for the three
block configurations (tiny fp32, 4×256 fp32 with dropout, 12-layer bf16 GPT stack) and small
variants; plus the dropout gates, determinism and += accumulation."""
import numpy as np
import pytest
import torch

import synth
from oracle import block as OB
from tests.gpu_util import norm_err

pytestmark = pytest.mark.gpu

xt = pytest.importorskip("transformer_fwd_bwd_gb300.xt")
from transformer_fwd_bwd_gb300.block import NativeBlock  # noqa: E402

SEED = synth.BASE_SEED_DROPOUT


def run_native(cfg, params, ids, tgt, training=True, base_seed=SEED, steps=1):
    nb = NativeBlock(cfg, training=training, base_seed=base_seed)
    nb.load(params)
    nb.zero_grads()
    I = torch.tensor(ids, device="cuda")
    Tg = torch.tensor(tgt, device="cuda")
    for _ in range(steps):
        loss = nb.step(I, Tg)
    torch.cuda.synchronize()
    assert xt.device_errors() == 0
    return float(loss.item()), nb.grads_named(), nb


def compare(cfg, training=True, base_seed=SEED, tol=2e-2, params=None, report=None):
    params = params if params is not None else synth.block_params(cfg)
    ids, tgt = synth.block_tokens(cfg)
    loss, grads, _ = run_native(cfg, params, ids, tgt, training, base_seed)
    rloss, rgrads = OB.forward_backward(cfg, params, ids, tgt, base_seed, training)
    errs = {k: norm_err(grads[k], rgrads[k]) for k in rgrads}
    worst = max(errs, key=errs.get)
    if report is not None:
        report.update(errs)
    assert abs(loss - rloss) <= 1e-3 * abs(rloss), f"loss {loss} vs oracle {rloss}"
    assert errs[worst] <= tol, f"{worst}: normalised grad error {errs[worst]:.3e}"
    return errs


def variant(name, **over):
    cfg = dict(synth.BLOCK_CONFIGS[name])
    cfg.update(over)
    return cfg


def test_block_tiny():
    """Tiny configuration: 1 block, fp32, RMSNorm + RoPE + SwiGLU, p = 0."""
    compare(synth.BLOCK_CONFIGS["tiny"])


def test_block_tiny_dropout():
    compare(variant("tiny", p=0.2), training=True)


def test_block_tiny_ln_gelu_pos_fp32():
    """The 12-layer stack's topology (LayerNorm, GELU, learned positions) at tiny size, fp32."""
    compare(variant("tiny", norm="ln", mlp="gelu", rope=False, learned_pos=True, n_layers=2),
            params=synth.block_params(variant("tiny", norm="ln", mlp="gelu", rope=False, learned_pos=True,
                                              n_layers=2), gain_jitter=0.1))


def test_block_small_bf16():
    cfg = variant("gpt12", B=2, S=256, d=128, H=2, hd=64, F=512, V=1000, n_layers=2)
    compare(cfg, params=synth.block_params(cfg, gain_jitter=0.1))


def test_block_small_bf16_composed():
    """The same stack through the composed attention (causal-tile GEMMs around the softmax)."""
    cfg = variant("gpt12", B=2, S=256, d=128, H=2, hd=64, F=512, V=1000, n_layers=2, attention="composed")
    compare(cfg, params=synth.block_params(cfg, gain_jitter=0.1))


def test_block_bf16_rope_swiglu_dropout_fused():
    """RMSNorm + RoPE + SwiGLU + residual dropout 0.1 in bf16 through the fused attention;
    bit-identical on a second run."""
    cfg = variant("block256", dtype="bf16", attention="fused")
    compare(cfg, training=True)
    params = synth.block_params(cfg)
    ids, tgt = synth.block_tokens(cfg)
    la, ga, _ = run_native(cfg, params, ids, tgt)
    lb, gb, _ = run_native(cfg, params, ids, tgt)
    assert la == lb
    for k in ga:
        assert np.array_equal(ga[k], gb[k]), k


def test_block_fused_attention_needs_bf16():
    with pytest.raises(xt.XtError):
        NativeBlock(variant("block256", attention="fused"))


def test_block_256():
    """Configuration 4×256, d 256, 4 heads, SwiGLU 688, vocab 4096, fp32, dropout 0.1."""
    compare(synth.BLOCK_CONFIGS["block256"], training=True)


def test_block_p0_bit_identity_and_eval():
    """[DO] gates: p = 0 in training is bit-identical to no dropout; eval is the identity."""
    cfg = synth.BLOCK_CONFIGS["block256"]
    params = synth.block_params(cfg)
    ids, tgt = synth.block_tokens(cfg)
    l0, g0, _ = run_native(dict(cfg, p=0.0), params, ids, tgt, training=True)
    l1, g1, _ = run_native(dict(cfg, p=0.1), params, ids, tgt, training=False)
    assert l0 == l1
    for k in g0:
        assert np.array_equal(g0[k], g1[k]), k
    l2, _, _ = run_native(dict(cfg, p=0.1), params, ids, tgt, training=True)
    assert l2 != l0


def test_block_deterministic_and_accumulates():
    cfg = synth.BLOCK_CONFIGS["block256"]
    params = synth.block_params(cfg)
    ids, tgt = synth.block_tokens(cfg)
    la, ga, _ = run_native(cfg, params, ids, tgt)
    lb, gb, _ = run_native(cfg, params, ids, tgt)
    assert la == lb
    for k in ga:
        assert np.array_equal(ga[k], gb[k]), k
    _, g2, _ = run_native(cfg, params, ids, tgt, steps=2)   # backward adds: two steps = 2×
    for k in ga:
        assert norm_err(g2[k], 2 * ga[k]) <= 1e-6, k


@pytest.mark.parametrize("cfg", [variant("gpt12", B=2, S=256, d=128, H=2, hd=64, F=512, V=1000, n_layers=3),
                                 variant("block256", p=0.1)], ids=["bf16-fused-3layers", "fp32-composed-dropout"])
def test_block_weight_gradient_stream_matches_one_stream(cfg):
    """The backward with its weight-gradient GEMMs on the second stream gives the one-stream
    backward's loss and every gradient bit for bit: the same kernels on the same inputs, so any
    missing ordering between the streams (a dW reading a buffer the main stream has already
    overwritten) would show as a difference."""
    params = synth.block_params(cfg, gain_jitter=0.1)
    ids, tgt = synth.block_tokens(cfg)
    xt.block_set_overlap(0)
    try:
        l0, g0, _ = run_native(cfg, params, ids, tgt, steps=2)
    finally:
        xt.block_set_overlap(1)
    l1, g1, _ = run_native(cfg, params, ids, tgt, steps=2)
    assert l0 == l1
    for k in g0:
        assert np.array_equal(g0[k], g1[k]), k


def test_block_gpt12_full():
    """12-layer GPT-style stack at full size (B 8, S 1024, d 768, 12 heads, GELU 3072, vocab
    50304, bf16) — the workload the benchmark times — against the float64 oracle."""
    errs = compare(synth.BLOCK_CONFIGS["gpt12"], training=True, report={})
    assert max(errs.values()) <= 2e-2


@pytest.mark.parametrize("cfg", [synth.BLOCK_CONFIGS["block256"], variant("block256", dtype="bf16")],
                         ids=["fp32-composed", "bf16-fused"])
def test_block_graph_replay_matches_eager(cfg):
    """One step (zero grads, forward, backward) captured into a CUDA graph and replayed gives the
    eager step's loss and gradients bit for bit (dropout included: the masks are counter-based);
    GEMM timing events enqueued during the capture are re-recorded by every replay."""
    params = synth.block_params(cfg)
    ids, tgt = synth.block_tokens(cfg)
    la, ga, _ = run_native(cfg, params, ids, tgt)

    nb = NativeBlock(cfg, training=True, base_seed=SEED)
    nb.load(params)
    I = torch.tensor(ids, device="cuda")
    Tg = torch.tensor(tgt, device="cuda")
    nb.step(I, Tg)   # warm-up outside the capture (kernel attributes, tensor maps)
    torch.cuda.synchronize()
    xt.profile_gemm(256)
    g = torch.cuda.CUDAGraph()
    n0 = xt.launch_count()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        s = torch.cuda.current_stream()
        nb.zero_grads(s)
        nb.forward(I, Tg, s)
        nb.backward(I, Tg, s)
    captured = xt.launch_count() - n0
    assert captured > 0
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert xt.device_errors() == 0
        flops, ms = xt.profile_gemm_read()
        assert len(ms) > 0 and np.all(np.asarray(ms) > 0) and np.all(np.asarray(flops) > 0)
        assert float(nb.loss.item()) == la
        gb = nb.grads_named()
        for k in ga:
            assert np.array_equal(ga[k], gb[k]), k
    del g
    xt.profile_gemm(0)


@pytest.mark.parametrize("cfg", [variant("block256", n_layers=2), variant("block256", dtype="bf16", n_layers=2),
                                 variant("gpt12", B=2, S=256, d=128, H=2, hd=64, F=512, V=1000, n_layers=3)],
                         ids=["fp32-composed-rope-swiglu-dropout", "bf16-fused", "bf16-ln-gelu-3layers"])
def test_block_recompute_bit_identical(cfg):
    """Activation recompute (keep each layer's input, redo the layer's forward in the backward;
    [DO] § RNG：counter-based … 与重计算兼容 requires the recomputed dropout masks to be the
    forward's): the workspace shrinks and the loss and every gradient are bit-identical to the
    run that keeps all activations (same kernels on the same inputs, masks from their counters)."""
    params = synth.block_params(cfg)
    ids, tgt = synth.block_tokens(cfg)
    l0, g0, nb0 = run_native(cfg, params, ids, tgt)
    l1, g1, nb1 = run_native(dict(cfg, recompute=1), params, ids, tgt)
    assert nb1.ws.numel() <= nb0.ws.numel() and (cfg["n_layers"] == 1 or nb1.ws.numel() < nb0.ws.numel())
    assert l0 == l1
    for k in g0:
        assert np.array_equal(g0[k], g1[k]), k
