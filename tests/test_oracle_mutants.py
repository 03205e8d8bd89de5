"""The pins must catch plausible mistakes: each case plants one mistake in the oracle
(on the CPU, through monkeypatch) and checks that a pin test then fails."""
import math

import numpy as np
import pytest

import oracle.dropout as D
import oracle.fp8 as F8
import oracle.ops as O
import oracle.optim as OP
import oracle.tape as T
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


def _gelu_tanh(x):
    # the tanh approximation instead of the erf definition
    x = np.asarray(x, float)
    return 0.5 * x * (1 + np.tanh(math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3)))


def _rms_eps_outside(x, gamma, eps):
    x = np.asarray(x, float)
    ir = 1.0 / (np.sqrt(np.mean(x * x, axis=-1)) + eps)
    return x * ir[..., None] * gamma, ir


def _ln_unbiased(x, gamma, beta, eps):
    x = np.asarray(x, float)
    mu = np.mean(x, axis=-1)
    xc = x - mu[..., None]
    rstd = 1.0 / np.sqrt(np.sum(xc * xc, axis=-1) / (x.shape[-1] - 1) + eps)
    return xc * rstd[..., None] * gamma + beta, mu, rstd


def _rope_half_frequency(positions, hd, base):
    i = np.arange(hd // 2, dtype=np.float64)
    return np.asarray(positions, float)[..., None] * base ** (-i / hd)


def _causal_diagonal_hidden(q_len, k_len):
    return np.arange(k_len)[None, :] < np.arange(q_len)[:, None]


def _ce_sum(x, targets):
    loss, lse = _ce_sum.__wrapped__(x, targets)
    return loss * np.asarray(x).shape[0], lse


def _embed_no_pos(ids, E, P=None, S=None):
    return _embed_no_pos.__wrapped__(ids, E)


def _attention_scale_hd(q, k, v, causal=True):
    q, k, v = (np.asarray(a, float) for a in (q, k, v))
    scores = np.einsum("bhsd,bhtd->bhst", q, k) / q.shape[-1]
    P = O.softmax_fwd(scores, causal=causal)
    return np.einsum("bhst,bhtd->bhsd", P, v), P


def _dropout_scale_inverse_p(p):
    return np.float32(1.0 / float(np.float32(p)))


def _keep_strict(n, p, seed):
    return D.uniforms(n, seed) > np.float32(p)


def _site_seed_added(base_seed, layer, site):
    return (int(base_seed) + int(layer) + int(site)) & 0xFFFFFFFFFFFFFFFF


# block structure mistakes, planted in the tape ops the stack is built from
def _residual_dropped(a, b):
    return b


def _post_norm(a, b):
    s = _post_norm.__wrapped__(a, b)
    return T.rms_norm(s, T.leaf(np.ones(s.value.shape[-1])), 1e-5)


def _attention_not_causal(q, k, v, causal=True):
    return _attention_not_causal.__wrapped__(q, k, v, causal=False)


def _heads_interleaved(x, B, S, H, hd):
    # columns read as [hd, H] instead of [H, hd]: every "head" mixes all heads' columns
    return T.Var(np.transpose(x.value.reshape(B, S, hd, H), (0, 3, 1, 2)), [x], lambda g, ps: None)


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
    ("gelu_fwd", _gelu_tanh, O, TO.test_gelu),
    ("rms_norm_fwd", _rms_eps_outside, O, TO.test_rms_norm),
    ("layernorm_fwd", _ln_unbiased, O, TO.test_layernorm),
    ("rope_angles", _rope_half_frequency, O, TO.test_rope_identities),
    ("causal_mask", _causal_diagonal_hidden, O, TO.test_softmax_causal),
    ("cross_entropy_fwd", _ce_sum, O, TO.test_cross_entropy),
    ("embedding_fwd", _embed_no_pos, O, TO.test_embedding),
    ("attention_fwd", _attention_scale_hd, O, TO.test_attention_composed),
    ("scale_f32", _dropout_scale_inverse_p, D, TE.test_dropout_expectation_and_identities),
    ("keep_mask", _keep_strict, D, TE.test_dropout_keep_boundary),
    ("site_seed", _site_seed_added, D, TE.test_site_seeds),
    ("add", _residual_dropped, T, lambda: TB.test_block_zero_sublayers_is_residual_identity("rms_swiglu")),
    ("add", _residual_dropped, T, lambda: TB.test_block_zero_sublayers_is_residual_identity("ln_gelu_pos")),
    ("add", _post_norm, T, lambda: TB.test_block_uniform_attention_closed_form("rms_swiglu")),
    ("add", _post_norm, T, lambda: TB.test_block_uniform_attention_closed_form("ln_gelu_pos")),
    ("attention", _attention_not_causal, T, lambda: TB.test_block_logits_causal_and_per_sequence("rms_swiglu")),
    ("attention", _attention_not_causal, T, lambda: TB.test_block_uniform_attention_closed_form("ln_gelu_pos")),
    ("split_heads", _heads_interleaved, T, TB.test_block_heads_are_separate),
]


@pytest.mark.parametrize("i", range(len(MUTANTS)))
def test_pin_catches_mutant(i, monkeypatch):
    name, fn, mod, pin = MUTANTS[i]
    orig = getattr(mod, name)
    fn.__dict__.setdefault("__wrapped__", orig)   # lets a mutant call the true op
    monkeypatch.setattr(mod, name, fn)
    with pytest.raises(AssertionError):
        pin()
