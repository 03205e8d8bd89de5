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
