"""Pins of the oracle's block stack: finite differences on every leaf (sampled entries),
the dropout gates at block level, and the fan-out closed form of the logits graph."""
import math

import numpy as np
import pytest

import synth
from oracle import block as OB
from oracle import dropout as D
from oracle import fd
from oracle import ops as O
from oracle import tape as t


def _tiny(**over):
    cfg = dict(synth.BLOCK_CONFIGS["tiny"])
    cfg.update(over)
    return cfg


@pytest.mark.parametrize("variant", ["rms_swiglu", "ln_gelu_pos"])
def test_block_fd_all_leaves(variant):
    if variant == "rms_swiglu":
        cfg = _tiny(p=0.2)
    else:
        cfg = _tiny(norm="ln", mlp="gelu", rope=False, learned_pos=True, n_layers=2, p=0.2)
    params = synth.block_params(cfg, gain_jitter=0.1)
    ids, tgt = synth.block_tokens(cfg)
    loss, grads = OB.forward_backward(cfg, params, ids, tgt, base_seed=0x5EED, training=True)
    r = np.random.default_rng(0)
    for name, g in grads.items():
        flat = params[name].reshape(-1)
        idx = r.choice(flat.size, size=min(12, flat.size), replace=False)

        def f(x, name=name):
            pp = dict(params)
            pp[name] = x
            return OB.loss_only(cfg, pp, ids, tgt, base_seed=0x5EED, training=True)
        num = fd.numeric_grad(f, params[name], eps=1e-4, idx=idx)   # round-off bound at 1e-6
        err = fd.max_rel_err(g.reshape(-1)[idx], num.reshape(-1)[idx], floor=1e-4)
        assert err < 1e-5, f"{name}: {err}"


def test_block_p0_equals_no_dropout_graph():
    """[DO] § 验证方法 gate 3: p = 0 (training) is bit-identical to the plain graph."""
    cfg = _tiny()
    params = synth.block_params(cfg)
    ids, tgt = synth.block_tokens(cfg)
    l0, g0 = OB.forward_backward(cfg, params, ids, tgt, 123, training=True)
    l1, g1 = OB.forward_backward(cfg, params, ids, tgt, 123, training=False)
    assert l0 == l1
    for k in g0:
        assert np.array_equal(g0[k], g1[k])


def test_block_eval_is_identity_of_dropout():
    cfg = _tiny(p=0.5)
    params = synth.block_params(cfg)
    ids, tgt = synth.block_tokens(cfg)
    le = OB.loss_only(cfg, params, ids, tgt, 9, training=False)
    l0 = OB.loss_only(_tiny(p=0.0), params, ids, tgt, 9, training=True)
    lt = OB.loss_only(cfg, params, ids, tgt, 9, training=True)
    assert le == l0 and lt != le


def test_block_initial_loss_near_log_vocab():
    """With N(0, 0.02) weights the logits are ≈ 0, so the loss is ≈ ln V."""
    cfg = _tiny()
    params = synth.block_params(cfg)
    ids, tgt = synth.block_tokens(cfg)
    assert abs(OB.loss_only(cfg, params, ids, tgt) - math.log(cfg["V"])) < 0.05


def test_fanout_logits_closed_form():
    """Large-vocab fan-out: L = CE(x) + Σ(0.5·x) + Σ(x∘x) ⇒ dx = (softmax − onehot)/R + 0.5 + 2x."""
    r = np.random.default_rng(5)
    R, V = 6, 13
    x0 = r.normal(0, 2, size=(R, V))
    tg = r.integers(0, V, size=R)
    x = t.leaf(x0)
    L = t.add(t.add(t.cross_entropy(x, tg), t.sum_all(t.scale(x, 0.5))), t.sum_all(t.mul(x, x)))
    t.backward(L)
    p = np.exp(x0 - x0.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    onehot = np.zeros_like(x0)
    onehot[np.arange(R), tg] = 1
    want = (p - onehot) / R + 0.5 + 2 * x0
    assert np.allclose(x.grad, want, rtol=1e-13, atol=1e-15)


def test_tied_embedding_gets_both_contributions():
    cfg = _tiny()
    params = synth.block_params(cfg)
    ids, tgt = synth.block_tokens(cfg)
    keep = {}
    loss, leaves = OB.model_loss(cfg, params, ids, tgt, keep=keep)
    t.backward(loss)
    # the logits matmul contribution alone: dE_logits = dlogitsᵀ @ hf
    _, lse = O.cross_entropy_fwd(keep["logits"].value, tgt)
    dlog = O.cross_entropy_bwd(keep["logits"].value, tgt, lse, 1.0)
    dE_logits = dlog.T @ keep["hf"].value
    dE_gather, _ = O.embedding_bwd(ids, keep["h0"].grad, cfg["V"])
    assert np.allclose(leaves["E"].grad, dE_logits + dE_gather, rtol=1e-12, atol=1e-15)


def test_dropout_sites_use_distinct_masks():
    cfg = _tiny(p=0.5)
    n = cfg["B"] * cfg["S"] * cfg["d"]
    a = D.keep_mask(n, 0.5, D.site_seed(0x5EED, 0, D.SITE_ATTN))
    f = D.keep_mask(n, 0.5, D.site_seed(0x5EED, 0, D.SITE_FFN))
    assert not np.array_equal(a, f)


# ----------------------------------------------------------------------------- structure pins
#
# The finite-difference pin above holds for any forward (the tape derives the backward from
# whatever graph is built), so the stack's structure is pinned separately: closed forms that
# follow when some weights are zero, written with the separately pinned ops and cumulative
# sums rather than with the stack's own code, and the causality / per-sequence invariants.

VARIANTS = ["rms_swiglu", "ln_gelu_pos"]


def _variant(name, **over):
    if name == "rms_swiglu":
        cfg = _tiny(B=2, S=6, n_layers=2)
    else:
        cfg = _tiny(B=2, S=6, norm="ln", mlp="gelu", rope=False, learned_pos=True, n_layers=2)
    cfg.update(over)
    return cfg


def _down(cfg):
    return "Wd" if cfg["mlp"] == "swiglu" else "W2"


def _norm(cfg, x, g, b):
    if cfg["norm"] == "rms":
        return O.rms_norm_fwd(x, g, cfg["eps"])[0]
    return O.layernorm_fwd(x, g, b, cfg["eps"])[0]


def _params(cfg, seed=3):
    """Block weights at N(0, 0.3) (large enough that every path moves the loss), gains jittered."""
    params = synth.block_params(cfg, gain_jitter=0.1)
    r = np.random.default_rng(seed)
    for k, v in params.items():
        if v.ndim == 2 and k not in ("E", "P"):
            params[k] = r.normal(0.0, 0.3, size=v.shape)
    return params


@pytest.mark.parametrize("variant", VARIANTS)
def test_block_zero_sublayers_is_residual_identity(variant):
    """Every W_O and MLP down projection zero: each sub-block adds exactly zero to the residual
    stream (its dropout, p = 0.3, acts on that zero), so the stack is embed → final norm → tied
    logits → mean cross-entropy, computed here from those ops alone."""
    cfg = _variant(variant, p=0.3)
    params = _params(cfg)
    for l in range(cfg["n_layers"]):
        params[f"l{l}.Wo"] = np.zeros_like(params[f"l{l}.Wo"])
        params[f"l{l}.{_down(cfg)}"] = np.zeros_like(params[f"l{l}.{_down(cfg)}"])
    ids, tgt = synth.block_tokens(cfg)
    h0 = O.embedding_fwd(ids, params["E"], params.get("P"), cfg["S"])
    hf = _norm(cfg, h0, params["gf"], params.get("bf"))
    want, _ = O.cross_entropy_fwd(hf @ params["E"].T, tgt)
    got = OB.loss_only(cfg, params, ids, tgt, base_seed=7, training=True)
    assert got == pytest.approx(want, rel=1e-12)


@pytest.mark.parametrize("variant", VARIANTS)
def test_block_uniform_attention_closed_form(variant):
    """W_Q = W_K = 0 makes every visible score 0, so causal attention is the plain mean of the
    values at positions 0..s (the softmax of a row of zeros is uniform over the visible keys);
    with the MLP's down projection zero as well, layer 0 outputs
    h0 + runningmean_s(norm1(h0) W_V) W_O per sequence, written here with cumulative sums."""
    cfg = _variant(variant, n_layers=1)
    params = _params(cfg)
    B, S, d = cfg["B"], cfg["S"], cfg["d"]
    params["l0.Wq"] = np.zeros((d, d))
    params["l0.Wk"] = np.zeros((d, d))
    params[f"l0.{_down(cfg)}"] = np.zeros_like(params[f"l0.{_down(cfg)}"])
    ids, tgt = synth.block_tokens(cfg)
    keep = {}
    OB.model_loss(cfg, params, ids, tgt, keep=keep)
    h0 = O.embedding_fwd(ids, params["E"], params.get("P"), S)
    v = (_norm(cfg, h0, params["l0.g1"], params.get("l0.b1")) @ params["l0.Wv"]).reshape(B, S, d)
    mean = np.cumsum(v, axis=1) / np.arange(1, S + 1)[None, :, None]
    want = h0 + mean.reshape(B * S, d) @ params["l0.Wo"]
    assert np.allclose(keep["h1"].value, want, rtol=1e-12, atol=1e-14)


def test_block_heads_are_separate():
    """Query / key weights nonzero only in head 0's columns: head 1 scores zero everywhere, so
    its output columns are the running mean of its own value columns, while head 0's are not.
    W_O = I and a zero MLP down projection expose the merged head outputs as h1 − h0."""
    cfg = _variant("ln_gelu_pos", n_layers=1)
    params = _params(cfg)
    d, hd, B, S = cfg["d"], cfg["hd"], cfg["B"], cfg["S"]
    for w in ("Wq", "Wk"):
        params[f"l0.{w}"][:, hd:] = 0.0
    params["l0.Wo"] = np.eye(d)
    params["l0.W2"] = np.zeros_like(params["l0.W2"])
    ids, tgt = synth.block_tokens(cfg)
    keep = {}
    OB.model_loss(cfg, params, ids, tgt, keep=keep)
    h0 = O.embedding_fwd(ids, params["E"], params["P"], S)
    o = (keep["h1"].value - h0).reshape(B, S, d)
    v = (_norm(cfg, h0, params["l0.g1"], params["l0.b1"]) @ params["l0.Wv"]).reshape(B, S, d)
    mean = np.cumsum(v, axis=1) / np.arange(1, S + 1)[None, :, None]
    assert np.allclose(o[..., hd:], mean[..., hd:], rtol=1e-10, atol=1e-12)
    assert not np.allclose(o[..., :hd], mean[..., :hd], rtol=1e-3, atol=1e-6)


@pytest.mark.parametrize("variant", VARIANTS)
def test_block_logits_causal_and_per_sequence(variant):
    """Changing the token at position j of sequence 0 leaves that sequence's logits before j
    and every logit of sequence 1 unchanged, and changes the logits from j on."""
    cfg = _variant(variant)
    params = _params(cfg)
    B, S, V = cfg["B"], cfg["S"], cfg["V"]
    ids, tgt = synth.block_tokens(cfg)
    j = 3
    ids2 = ids.copy()
    ids2[j] = (ids2[j] + 1) % V
    k0, k1 = {}, {}
    OB.model_loss(cfg, params, ids, tgt, keep=k0)
    OB.model_loss(cfg, params, ids2, tgt, keep=k1)
    L0, L1 = k0["logits"].value.reshape(B, S, V), k1["logits"].value.reshape(B, S, V)
    assert np.allclose(L1[0, :j], L0[0, :j], rtol=1e-13, atol=1e-15)
    assert np.allclose(L1[1], L0[1], rtol=1e-13, atol=1e-15)
    for s in range(j, S):
        assert not np.allclose(L1[0, s], L0[0, s], rtol=1e-6, atol=1e-9)
