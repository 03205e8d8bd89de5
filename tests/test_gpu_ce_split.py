"""Cross-entropy on rows split across a cluster of CTAs, and the fused fan-out loss, against the
oracle ([AE] op table row cross_entropy; § 梯度累加's fan-out, L = CE(x) + c_lin·Σx + c_sq·Σx∘x).

Rows wider than one CTA's shared memory (128256 bf16 logits: 250 KB; float32 rows of 400 KB to
1.6 MB) are held as 2, 4 or 8 chunks by the CTAs of a cluster, whose (max, Σ exp) pairs are
merged through distributed shared memory.  Bounds as for the other cross-entropy tests: lse
to the float32 row-op bound, the loss to 1e-5 relative, the gradient to 1e-5 of each element
(float32) or one bf16 rounding, plus 1e-6 of the gradient scale.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import ops as O
from tests.gpu_util import check, dev, empty, host, norm_err, sync

pytestmark = pytest.mark.gpu

xt = pytest.importorskip("transformer_fwd_bwd_gb300.xt")
T = pytest.importorskip("transformer_fwd_bwd_gb300.tape")


def inputs(shape, seed, dtype, std=2.0):
    return synth.normal(shape, seed, std=std, dtype=dtype)


def grad_tol(dx, gdt, scale):
    rel = 1e-5 if gdt == "f32" else 2.0 ** -8
    return rel * np.abs(dx) + 1e-6 * scale


# (rows, V): 128256 bf16 → 2 chunks; 128264 → 2 chunks of unequal width; 409600 bf16 → 4;
# float32 100008 → 2, 409600 → 8, 262144 → 8
SPLIT = [(5, 128256), (4, 128264), (3, 409600), (9, 100008), (2, 262144)]


@pytest.mark.parametrize("dtype,gdt", [("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32"), ("f32", "bf16")])
@pytest.mark.parametrize("rows,V", SPLIT)
def test_ce_split_rows(dtype, gdt, rows, V):
    x = inputs((rows, V), 31, dtype)
    t = synth.uniform_ids(rows, V, 32)
    loss, lse = O.cross_entropy_fwd(x, t)
    X, Tg = dev(x, dtype), torch.tensor(t, device="cuda")
    LSE, L = empty((rows,), "f32"), empty((1,), "f32")
    up = torch.tensor([1.3], device="cuda")
    DX = X if gdt == dtype else empty((rows, V), gdt)   # in place when the dtypes agree
    xt.xt_cross_entropy_fwd_bwd(X, Tg, LSE, L, up, DX); sync()
    assert xt.device_errors() == 0
    check(host(LSE), lse, "f32", "lse")
    assert abs(host(L)[0] - loss) <= 1e-5 * abs(loss)
    dx = O.cross_entropy_bwd(x, t, np.float32(host(LSE)).astype(np.float64), np.float32(1.3))
    err = np.abs(host(DX) - dx) / grad_tol(dx, gdt, 1.3 / rows)
    assert np.all(err <= 1.0), f"split ce dx excess {np.max(err):.3f}"


@pytest.mark.parametrize("cl,nb", [(2, 1), (4, 1), (4, 2), (8, 1), (8, 2)])
def test_ce_split_forced_configs(cl, nb):
    """Every (cluster size, chunk buffers) form on more rows than there are clusters, so each
    cluster walks several rows (the chunk copies of later rows, both buffer parities)."""
    rows, V = 320, 128256
    x = inputs((rows, V), 37, "bf16")
    t = synth.uniform_ids(rows, V, 38)
    X, Tg = dev(x, "bf16"), torch.tensor(t, device="cuda")
    LSE, L = empty((rows,), "f32"), empty((1,), "f32")
    G = empty((rows, V), "f32")
    one = torch.ones(1, device="cuda")
    xt.ce_set_split(cl, nb)
    try:
        xt.xt_cross_entropy_fwd_bwd(X, Tg, LSE, L, one, G); sync()
    finally:
        xt.ce_set_split(0, 0)
    assert xt.device_errors() == 0
    loss, lse = O.cross_entropy_fwd(x, t)
    check(host(LSE), lse, "f32", "lse")
    assert abs(host(L)[0] - loss) <= 1e-5 * abs(loss)
    rs = np.array([0, 1, 75, 76, 151, 152, 305, rows - 1])
    dx = O.cross_entropy_bwd(x[rs], t[rs], np.float32(host(LSE)[rs]).astype(np.float64), len(rs) / rows)
    err = np.abs(host(G)[rs] - dx) / grad_tol(dx, "f32", 1.0 / rows)
    assert np.all(err <= 1.0), f"forced split ce dx excess {np.max(err):.3f}"


def test_ce_split_bad_target_sets_flag():
    rows, V = 3, 128256
    xt.clear_device_errors()
    X = dev(np.zeros((rows, V)), "bf16")
    t = torch.tensor([0, V, 5], dtype=torch.int32, device="cuda")
    LSE, L = empty((rows,), "f32"), empty((1,), "f32")
    one = torch.ones(1, device="cuda")
    xt.xt_cross_entropy_fwd_bwd(X, t, LSE, L, one, X)
    assert xt.device_errors() & xt.XT_DEVERR_INDEX
    xt.clear_device_errors()


def fanout_ref(x, t, c_lin, c_sq, up):
    """The oracle's three consumers of x and their summed gradient, each from its own op."""
    ce, lse = O.cross_entropy_fwd(x, t)
    L = ce + c_lin * float(np.sum(x)) + c_sq * float(np.sum(x * x))
    ones = np.ones_like(x)
    g_ce = O.cross_entropy_bwd(x, t, lse, up)
    g_lin = O.scale_bwd(ones * up, c_lin)
    da, db = O.mul_bwd(ones * (up * c_sq), x, x)
    return L, ce, lse, g_ce, g_lin + da + db


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rows,V", [(6, 128256), (4, 1000), (3, 409600)])
@pytest.mark.parametrize("c_lin,c_sq", [(0.5, 1.0), (-0.25, 0.3)])
def test_ce_fanout(dtype, rows, V, c_lin, c_sq):
    x = inputs((rows, V), 33, dtype)
    t = synth.uniform_ids(rows, V, 34)
    L_ref, ce_ref, lse_ref, g_ce, g_rest = fanout_ref(x, t, c_lin, c_sq, 1.0)
    X, Tg = dev(x, dtype), torch.tensor(t, device="cuda")
    LSE, loss, sums = empty((rows,), "f32"), empty((1,), "f32"), empty((3,), "f32")
    G = empty((rows, V), "f32")
    xt.xt_cross_entropy_fanout_fwd_bwd(X, Tg, c_lin, c_sq, LSE, loss, sums, G); sync()
    assert xt.device_errors() == 0
    check(host(LSE), lse_ref, "f32", "lse")
    assert abs(host(loss)[0] - ce_ref) <= 1e-5 * abs(ce_ref)
    s = host(sums)
    assert abs(s[0] - np.sum(x)) <= 1e-5 * np.sum(np.abs(x))
    assert abs(s[1] - np.sum(x * x)) <= 1e-5 * np.sum(x * x)
    mag = abs(ce_ref) + abs(c_lin) * np.sum(np.abs(x)) + abs(c_sq) * np.sum(x * x)
    assert abs(s[2] - L_ref) <= 1e-5 * mag
    # the gradient: every element against the sum of the three contributions, to float32
    # rounding of the largest term (the cross-entropy part is ~1/(rows·V) per element)
    want = g_ce + g_rest
    term = np.abs(g_ce) + np.abs(c_lin) + np.abs(2 * c_sq * x)
    g = host(G)
    assert np.all(np.abs(g - want) <= 2e-7 * term + 1e-6 / rows), "fanout grad"
    # the cross-entropy part alone, where it is not swamped: the target entries
    ridx = np.arange(rows)
    resid = (g - g_rest)[ridx, t]
    assert np.all(np.abs(resid - g_ce[ridx, t]) <= 1e-6 * (1.0 + term[ridx, t]) * 8), "target entries"
    # upstream 1.7, accumulated into a buffer holding ones
    up = torch.tensor([1.7], device="cuda")
    Ga = dev(np.ones((rows, V)), "f32")
    xt.xt_cross_entropy_fanout_fwd_bwd(X, Tg, c_lin, c_sq, LSE, loss, sums, Ga, upstream=up, acc=1); sync()
    _, _, _, g_ce2, g_rest2 = fanout_ref(x, t, c_lin, c_sq, np.float32(1.7))
    want2 = 1.0 + g_ce2 + g_rest2
    assert np.all(np.abs(host(Ga) - want2) <= 2e-7 * (1.7 * term + 1.0) + 2e-6 / rows), "fanout grad, upstream + acc"


def test_ce_fanout_alignment_rejected():
    X = torch.zeros((2, 1001), dtype=torch.bfloat16, device="cuda")   # 2002-byte rows
    Tg = torch.zeros(2, dtype=torch.int32, device="cuda")
    LSE, loss, sums = empty((2,), "f32"), empty((1,), "f32"), empty((3,), "f32")
    G = empty((2, 1001), "f32")
    with pytest.raises(xt.XtError) as ei:
        xt.xt_cross_entropy_fanout_fwd_bwd(X, Tg, 0.5, 1.0, LSE, loss, sums, G)
    assert ei.value.code == xt.XT_ERR_ALIGNMENT


@pytest.mark.parametrize("root", [True, False])
def test_tape_fanout_node_matches_composed(root):
    """The fused node against the tape's composition of the three consumers on the same x:
    the same L and the same float32 gradient (to float32 summation order).  As the root its
    forward's gradient is pushed; under scale(·, 2) the backward runs the pass with the upstream."""
    rows, V = 16, 128256
    x = inputs((rows, V), 35, "bf16")
    tn = synth.uniform_ids(rows, V, 36)
    t = torch.tensor(tn, device="cuda")
    X = dev(x, "bf16")
    xc = T.leaf(X, grad_dtype=torch.float32)
    Lc = T.add(T.add(T.cross_entropy(xc, t), T.sum_all(T.scale(xc, 0.5))), T.sum_all(T.mul(xc, xc)))
    xf = T.leaf(X, grad_dtype=torch.float32)
    Lf = T.cross_entropy_fanout(xf, t, 0.5, 1.0)
    if not root:
        Lc, Lf = T.scale(Lc, 2.0), T.scale(Lf, 2.0)
    T.backward(Lc)
    T.backward(Lf)
    sync()
    assert xt.device_errors() == 0
    lc, lf = float(host(Lc.value)[0]), float(host(Lf.value)[0])
    # L against the oracle's exact value: the fused node sums the squares in float32; the
    # composed graph stores x∘x in bf16 before its sum (each square rounded to 8 bits), which
    # moves its L by ~1e-4 relative
    L_ref = fanout_ref(x, tn, 0.5, 1.0, 1.0)[0] * (1.0 if root else 2.0)
    assert math.isfinite(lf) and abs(lf - L_ref) <= 1e-5 * abs(L_ref), (lf, L_ref)
    assert abs(lc - L_ref) <= 2.0 ** -8 * abs(L_ref), (lc, L_ref)
    assert norm_err(host(xf.grad), host(xc.grad)) <= 1e-6
