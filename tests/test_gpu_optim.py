"""GPU parity of the optimizer step (xt_adamw_step) against the oracle's float64 restatement
([BP] § Ackumulation över mikrobatcher, § Parningsdisciplinen, § Optimiser-tillståndet):
microbatch scale, global-norm clipping, AdamW with decoupled weight decay, over several steps
and many tensors of ragged sizes.  Bounds from the float32 arithmetic: per step ≲ 1e-6 of lr
on the update and ≲ 2e-7 relative on θ, m, v; the bf16 shadow is bf16(θ) bit for bit."""
import numpy as np
import pytest
import torch

from oracle import optim as OP

pytestmark = pytest.mark.gpu

xt = pytest.importorskip("transformer_fwd_bwd_gb300.xt")

HP = dict(lr=2e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def make(sizes, seed, gscale=1.0):
    rng = np.random.default_rng(seed)
    p = [rng.normal(size=n).astype(np.float32) for n in sizes]
    g = [(rng.normal(size=n) * gscale).astype(np.float32) for n in sizes]
    return p, g


def dev(a):
    return torch.tensor(a, dtype=torch.float32, device="cuda")


def run(sizes, steps, max_norm, grad_scale, seed=0, shadow=None):
    p, _ = make(sizes, seed)
    P = [dev(x) for x in p]
    M = [torch.zeros_like(x) for x in P]
    V = [torch.zeros_like(x) for x in P]
    S = None if shadow is None else [torch.zeros(x.numel(), dtype=shadow, device="cuda") for x in P]
    rp, rm, rv = [x.astype(np.float64) for x in p], [np.zeros(n) for n in sizes], [np.zeros(n) for n in sizes]
    norm = torch.zeros(1, dtype=torch.float32, device="cuda")
    for t in range(1, steps + 1):
        _, g = make(sizes, seed + 100 * t, gscale=3.0)
        G = [dev(x) for x in g]
        cfg = xt.adamw_config(step=t, max_grad_norm=max_norm, grad_scale=grad_scale, **HP)
        xt.xt_adamw_step(cfg, P, G, M, V, shadows=S, norm_out=norm)
        torch.cuda.synchronize()
        rp, rm, rv, rnorm = OP.adamw_step(rp, g, rm, rv, t, **HP, max_norm=max_norm, grad_scale=grad_scale)
        assert abs(float(norm.item()) - rnorm) <= 1e-6 * rnorm
    assert xt.device_errors() == 0
    return P, M, V, S, rp, rm, rv


SIZES = [1, 3, 4095, 4096, 4097, 10000, 0, 777]


@pytest.mark.parametrize("max_norm,grad_scale", [(0.0, 1.0), (1.0, 0.5), (1e6, 0.25)],
                         ids=["no-clip", "clip-active", "clip-inactive"])
def test_adamw_parity(max_norm, grad_scale):
    steps = 4
    P, M, V, _, rp, rm, rv = run(SIZES, steps, max_norm, grad_scale)
    for i, n in enumerate(SIZES):
        if n == 0:
            continue
        p, m, v = (x.cpu().numpy().astype(np.float64) for x in (P[i], M[i], V[i]))
        assert np.max(np.abs(p - rp[i])) <= steps * (1e-6 * HP["lr"] + 2e-7 * np.max(np.abs(rp[i]))), i
        assert np.max(np.abs(m - rm[i])) <= steps * 2e-7 * np.max(np.abs(rm[i])) + 1e-30, i
        assert np.max(np.abs(v - rv[i])) <= steps * 2e-7 * np.max(np.abs(rv[i])) + 1e-30, i


def test_adamw_many_tensors_and_bf16_shadow():
    """More tensors than one launch's table (300 > 128) and a bf16 working copy: the copy is the
    round-to-nearest-even bf16 of the updated float32 master weights."""
    sizes = [int(s) for s in np.random.default_rng(5).integers(1, 3000, size=300)]
    P, M, V, S, rp, rm, rv = run(sizes, 2, 0.5, 1.0, seed=9, shadow=torch.bfloat16)
    for i in range(len(sizes)):
        assert torch.equal(S[i], P[i].to(torch.bfloat16)), i
        p = P[i].cpu().numpy().astype(np.float64)
        assert np.max(np.abs(p - rp[i])) <= 2 * (1e-6 * HP["lr"] + 2e-7 * np.max(np.abs(rp[i]))), i


def test_adamw_deterministic():
    a = run(SIZES, 3, 1.0, 0.5, seed=3)
    b = run(SIZES, 3, 1.0, 0.5, seed=3)
    for x, y in zip(a[0], b[0]):
        assert torch.equal(x, y)


def test_adamw_rejects():
    P = [torch.zeros(4, device="cuda")]
    with pytest.raises(xt.XtError):   # step must be ≥ 1
        xt.xt_adamw_step(xt.adamw_config(lr=1e-3, step=0), P, P, P, P)
    with pytest.raises(xt.XtError):   # β₁ outside [0, 1)
        xt.xt_adamw_step(xt.adamw_config(lr=1e-3, beta1=1.0), P, P, P, P)


from transformer_fwd_bwd_gb300.block import NativeBlock  # noqa: E402
import synth  # noqa: E402


def _variant(name, **over):
    cfg = dict(synth.BLOCK_CONFIGS[name])
    cfg.update(over)
    return cfg


@pytest.mark.parametrize("cfg", [synth.BLOCK_CONFIGS["block256"],
                                 _variant("gpt12", B=2, S=256, d=128, H=2, hd=64, F=512, V=1000, n_layers=2)],
                         ids=["fp32", "bf16-master-weights"])
def test_block_train_step_matches_oracle_adamw(cfg):
    """One training step of the native stack with two microbatches: the gradient buffers hold
    the sum of both backwards (checked against the two single-microbatch backwards), and the
    clipped AdamW update of the float32 master weights from those buffers matches the oracle;
    the bf16 working weights are bf16(master) bit for bit."""
    params = synth.block_params(cfg)
    nb = NativeBlock(cfg, training=True, base_seed=synth.BASE_SEED_DROPOUT)
    nb.load(params)
    nb.init_optimizer(lr=1e-3, max_grad_norm=0.5)
    mbs = []
    singles = []
    for k in range(2):
        ids, tgt = synth.block_tokens(cfg, seed=synth.SEED_TOKENS + 10 + k)
        mb = (torch.tensor(ids, device="cuda"), torch.tensor(tgt, device="cuda"))
        mbs.append(mb)
        nb.zero_grads()
        nb.step(*mb)
        singles.append({n: g.clone() for n, g in nb.g.items()})
    names = list(nb.p)
    master0 = {n: nb.master[n].clone() for n in names}
    nb.zero_grads()
    for mb in mbs:
        nb.step(*mb)
    torch.cuda.synchronize()
    for n in names:   # the buffers hold the sum (a tied or multiply-used weight adds in another order)
        want = (singles[0][n] + singles[1][n]).double()
        err = (nb.g[n].double() - want).norm() / max(float(want.norm()), 1e-30)
        assert float(err) <= 1e-6, n
    grads = {n: nb.g[n].cpu().numpy() for n in names}
    nb.optimizer_step(n_microbatches=2)
    torch.cuda.synchronize()
    assert xt.device_errors() == 0
    h = nb.hyper
    rp, _, _, rnorm = OP.adamw_step([master0[n].cpu().numpy().astype(np.float64) for n in names],
                                    [grads[n] for n in names], [np.zeros(nb.p[n].shape) for n in names],
                                    [np.zeros(nb.p[n].shape) for n in names], 1, h["lr"], h["beta1"], h["beta2"],
                                    h["eps"], h["weight_decay"], max_norm=h["max_grad_norm"], grad_scale=0.5)
    assert abs(float(nb.grad_norm.item()) - rnorm) <= 1e-6 * rnorm
    for n, r in zip(names, rp):
        got = nb.master[n].cpu().numpy().astype(np.float64)
        assert np.max(np.abs(got - r)) <= 1e-6 * h["lr"] + 2e-7 * np.max(np.abs(r)), n
        if nb.dt != torch.float32:
            assert torch.equal(nb.p[n], nb.master[n].to(nb.dt)), n


def test_block_training_loss_decreases():
    """A few microbatched AdamW steps on one fixed batch of the 4×256 stack: the loss falls and
    stays finite (the pages' small-training convergence gate, here with dropout 0.1)."""
    cfg = synth.BLOCK_CONFIGS["block256"]
    nb = NativeBlock(cfg, training=True, base_seed=synth.BASE_SEED_DROPOUT)
    nb.load(synth.block_params(cfg))
    nb.init_optimizer(lr=3e-3, max_grad_norm=1.0)
    ids, tgt = synth.block_tokens(cfg)
    I, T = torch.tensor(ids, device="cuda"), torch.tensor(tgt, device="cuda")
    first = None
    for _ in range(8):
        losses = nb.train_step([(I, T), (I, T)])
        val = float(losses[0].item())
        assert np.isfinite(val)
        first = val if first is None else first
    assert val < first - 0.1, (first, val)
    assert xt.device_errors() == 0
