"""Pre-norm transformer stack forward + backward through the oracle tape (float64).

[BP] § Framåtgåendet: h = embed(ids); per layer h = h + attn(LN h), h = h + mlp(LN h);
logits = LN(h) @ embedᵀ (tied); loss = cross_entropy(logits, targets).
[DO] § dropout 接在哪（wiring）: h = h + dropout(attention(norm h)), h = h + dropout(mlp(norm h)),
site seeds base ⊕ layer ⊕ {0xA77, 0xF70}; dropout only when p > 0 and training.
[AE] § Attention 用组合: attention composed of matmul / scale / softmax / matmul.

Readings (pages silent): no biases in any linear layer (the per-block weight list in
[BP] § Var gradienter lever i minnet has none); attention is causal; RoPE (when used)
rotates Q and K per head with position = index within the sequence; the RMS variant
uses SwiGLU (silu(x W_g) ∘ x W_u) W_d, the LN variant exact GELU; learned positions
are added to the token embedding.
"""
from __future__ import annotations

import numpy as np

from . import dropout as D
from . import tape as t


def model_loss(cfg, params, ids, targets, base_seed=0, training=False, keep=None):
    """Builds the graph; returns (loss Var, leaves dict).  `keep` (optional dict) receives
    named intermediate Vars for inspection."""
    B, S, d, H, hd = cfg["B"], cfg["S"], cfg["d"], cfg["H"], cfg["hd"]
    eps, p = cfg["eps"], cfg["p"]
    leaves = {name: t.leaf(v, name) for name, v in params.items()}
    positions = np.arange(S)

    def norm(x, g, b):
        if cfg["norm"] == "rms":
            return t.rms_norm(x, leaves[g], eps)
        return t.layernorm(x, leaves[g], leaves[b], eps)

    h = t.embedding(ids, leaves["E"], leaves.get("P"), S)
    if keep is not None:
        keep["h0"] = h
    for l in range(cfg["n_layers"]):
        x = norm(h, f"l{l}.g1", f"l{l}.b1")
        q = t.split_heads(t.matmul(x, leaves[f"l{l}.Wq"]), B, S, H, hd)
        k = t.split_heads(t.matmul(x, leaves[f"l{l}.Wk"]), B, S, H, hd)
        v = t.split_heads(t.matmul(x, leaves[f"l{l}.Wv"]), B, S, H, hd)
        if cfg["rope"]:
            q = t.rope(q, positions, cfg["rope_base"])
            k = t.rope(k, positions, cfg["rope_base"])
        o = t.merge_heads(t.attention(q, k, v, causal=cfg["causal"]))
        a = t.matmul(o, leaves[f"l{l}.Wo"])
        a = t.dropout(a, p, D.site_seed(base_seed, l, D.SITE_ATTN), training)
        h = t.add(h, a)
        x = norm(h, f"l{l}.g2", f"l{l}.b2")
        if cfg["mlp"] == "swiglu":
            m = t.swiglu(t.matmul(x, leaves[f"l{l}.Wg"]), t.matmul(x, leaves[f"l{l}.Wu"]))
            f = t.matmul(m, leaves[f"l{l}.Wd"])
        else:
            m = t.gelu(t.matmul(x, leaves[f"l{l}.W1"]))
            f = t.matmul(m, leaves[f"l{l}.W2"])
        f = t.dropout(f, p, D.site_seed(base_seed, l, D.SITE_FFN), training)
        h = t.add(h, f)
        if keep is not None:
            keep[f"h{l + 1}"] = h
    hf = norm(h, "gf", "bf")
    logits = t.matmul(hf, t.transpose(leaves["E"]))
    if keep is not None:
        keep["hf"] = hf
        keep["logits"] = logits
    loss = t.cross_entropy(logits, targets)
    return loss, leaves


def forward_backward(cfg, params, ids, targets, base_seed=0, training=False, keep=None):
    """Returns (loss float, grads dict name → array)."""
    loss, leaves = model_loss(cfg, params, ids, targets, base_seed, training, keep)
    t.backward(loss)
    grads = {n: (v.grad if v.grad is not None else np.zeros_like(v.value)) for n, v in leaves.items()}
    return float(loss.value), grads


def loss_only(cfg, params, ids, targets, base_seed=0, training=False):
    loss, _ = model_loss(cfg, params, ids, targets, base_seed, training)
    return float(loss.value)
