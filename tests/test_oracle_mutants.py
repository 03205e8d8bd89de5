"""The pins must catch plausible mistakes: each case plants one mistake in the oracle
(on the CPU, through monkeypatch) and checks that a pin test then fails."""
import math

import numpy as np
import pytest

import oracle.dropout as D
import oracle.fp8 as F8
import oracle.ops as O
import oracle.optim as OP
from tests import test_oracle_block as TB
from tests import test_oracle_engine as TE
from tests import test_oracle_ops as TO
from tests import test_oracle_fp8 as TF8
from tests import test_oracle_optim as TOP


def _rms_bwd_dropped_term(d, x, gamma, ir):
    d, x = np.asarray(d, float), np.asarray(x, float)
    return ir[..., None] * d * gamma, np.sum((d * x * ir[..., None]).reshape(-1, x.shape[-1]), 0)


def _rms_bwd_wrong_power(d, x, gamma, ir):
    n = x.shape[-1]
    g = d * gamma
    s = np.sum(g * x, axis=-1)
    dx = ir[..., None] * g - x * (ir ** 2 / n * s)[..., None]
    return dx, np.sum((d * x * ir[..., None]).reshape(-1, n), axis=0)


def _softmax_bwd_sign(d, y):
    return y * (d + np.sum(d * y, axis=-1, keepdims=True))


def _rope_bwd_sign(d, positions, base):
    return O.rope_fwd(d, positions, base)


def _ln_bwd_no_mean(d, x, gamma, mu, rstd):
    xhat = (x - mu[..., None]) * rstd[..., None]
    g = d * gamma
    dx = rstd[..., None] * (g - xhat * np.mean(g * xhat, axis=-1, keepdims=True))
    n = x.shape[-1]
    return dx, np.sum((d * xhat).reshape(-1, n), 0), np.sum(d.reshape(-1, n), 0)


def _ce_bwd_no_rows(x, targets, lse, upstream):
    return O.cross_entropy_bwd.__wrapped__(x, targets, lse, upstream) * x.shape[0]


def _gelu_bwd_no_phi(d, x):
    from scipy.special import erf
    return d * 0.5 * (1 + erf(np.asarray(x) / math.sqrt(2)))


def _silu_bwd_wrong(d, x):
    s = O.sigmoid(x)
    return d * s * (1 - s)


def _matmul_bwd_transposed(d, A, B):
    return d @ B, np.swapaxes(A, -1, -2) @ d


def _embed_bwd_overwrite(ids, dh, V, S=None, with_pos=False):
    dE = np.zeros((V, dh.shape[1]))
    dE[np.asarray(ids)] = dh
    dP = dh.reshape(-1, S, dh.shape[1]).sum(0) if with_pos else None
    return dE, dP


def _splitmix_wrong_shift(state):
    z = np.asarray(state, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = z + D.GAMMA
        z = (z ^ (z >> np.uint64(30))) * D.MIX1
        z = (z ^ (z >> np.uint64(28))) * D.MIX2
    return z ^ (z >> np.uint64(31))


def _swiglu_bwd_swapped(d, g, u):
    dg, du = O.swiglu_bwd.__wrapped__(d, g, u)
    return du, dg


def _adamw_no_bias_correction(p, g, m, v, step, lr, beta1, beta2, eps, weight_decay):
    m = beta1 * np.asarray(m, float) + (1 - beta1) * g
    v = beta2 * np.asarray(v, float) + (1 - beta2) * g * g
    return p * (1 - lr * weight_decay) - lr * m / (np.sqrt(v) + eps), m, v


def _adamw_coupled_decay(p, g, m, v, step, lr, beta1, beta2, eps, weight_decay):
    # weight decay folded into the gradient (Adam with an L2 term) instead of decoupled
    return _adamw_coupled_decay.__wrapped__(p, np.asarray(g) + weight_decay * np.asarray(p), m, v, step, lr,
                                            beta1, beta2, eps, 0.0)


def _clip_always(norm, max_norm):
    return 1.0 if max_norm <= 0 else max_norm / (norm + 1e-6)


def _norm_unscaled(grads, scale=1.0):
    return math.sqrt(sum(float(np.sum(np.asarray(g, float) ** 2)) for g in grads))


def _fp8_ties_away(x):
    # nearest code with ties away from zero instead of to the even code
    x = np.asarray(x, float)
    out = _fp8_ties_away.__wrapped__(x)
    pos = F8.DECODE[:0x7F]
    for i, v in enumerate(x.ravel()):
        a = min(abs(v), F8.MAX)
        lo = int(np.searchsorted(pos, a, side="right")) - 1
        if lo < 0x7E and a - pos[lo] == pos[lo + 1] - a:
            out.ravel()[i] = (0x80 if v < 0 else 0) | (lo + 1)
    return out


def _fp8_no_saturation(x):
    out = _fp8_no_saturation.__wrapped__(x)
    out[np.abs(np.asarray(x, float)) > F8.MAX] = 0x7F
    return out


MUTANTS = [
    ("rms_norm_bwd", _rms_bwd_dropped_term, O, TO.test_rms_norm),
    ("rms_norm_bwd", _rms_bwd_wrong_power, O, TO.test_rms_norm),
    ("softmax_bwd", _softmax_bwd_sign, O, TO.test_softmax),
    ("rope_bwd", _rope_bwd_sign, O, TO.test_rope_identities),
    ("layernorm_bwd", _ln_bwd_no_mean, O, TO.test_layernorm),
    ("cross_entropy_bwd", _ce_bwd_no_rows, O, TO.test_cross_entropy),
    ("gelu_bwd", _gelu_bwd_no_phi, O, TO.test_gelu),
    ("silu_bwd", _silu_bwd_wrong, O, TO.test_silu),
    ("matmul_bwd", _matmul_bwd_transposed, O, TO.test_matmul_square_fd),
    ("embedding_bwd", _embed_bwd_overwrite, O, TO.test_embedding),
    ("splitmix64", _splitmix_wrong_shift, D, TE.test_splitmix64_published_sequence),
    ("swiglu_bwd", _swiglu_bwd_swapped, O, TO.test_swiglu_equals_composition),
    ("rms_norm_bwd", _rms_bwd_dropped_term, O, lambda: TB.test_block_fd_all_leaves("rms_swiglu")),
    ("layernorm_bwd", _ln_bwd_no_mean, O, lambda: TB.test_block_fd_all_leaves("ln_gelu_pos")),
    ("adamw_tensor", _adamw_no_bias_correction, OP, TOP.test_adamw_matches_torch_over_steps),
    ("adamw_tensor", _adamw_no_bias_correction, OP, TOP.test_first_step_closed_form),
    ("adamw_tensor", _adamw_coupled_decay, OP, TOP.test_adamw_matches_torch_over_steps),
    ("clip_coefficient", _clip_always, OP, lambda: TOP.test_clip_matches_torch(1e3)),
    ("global_grad_norm", _norm_unscaled, OP, lambda: TOP.test_microbatch_average_identity(2)),
    ("encode", _fp8_ties_away, F8, TF8.test_encode_matches_torch_in_range_and_on_ties),
    ("encode", _fp8_ties_away, F8, TF8.test_printed_constants_and_saturation),
    ("encode", _fp8_no_saturation, F8, TF8.test_printed_constants_and_saturation),
]


@pytest.mark.parametrize("i", range(len(MUTANTS)))
def test_pin_catches_mutant(i, monkeypatch):
    name, fn, mod, pin = MUTANTS[i]
    orig = getattr(mod, name)
    fn.__dict__.setdefault("__wrapped__", orig)   # lets a mutant call the true op
    monkeypatch.setattr(mod, name, fn)
    with pytest.raises(AssertionError):
        pin()
