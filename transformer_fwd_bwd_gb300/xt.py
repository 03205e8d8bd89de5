"""ctypes binding of libxt (include/xt.h): the same entry points, taking torch tensors.

Argument marshalling only — every computation runs in libxt's CUDA kernels.  Tensors must
be CUDA tensors; sizes are taken from them where the C call needs them.  A non-zero status
raises XtError with libxt's message.  There is no fallback: without libxt.so importing the
library raises.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libxt.so")

XT_OK, XT_ERR_INVALID_ARG, XT_ERR_UNSUPPORTED, XT_ERR_ALIGNMENT, XT_ERR_CUDA, XT_ERR_TIMEOUT = range(6)
XT_F32, XT_BF16 = 0, 1
XT_DEVERR_INDEX, XT_DEVERR_TIMEOUT = 1, 2
XT_NORM_RMS, XT_NORM_LN = 0, 1
XT_MLP_SWIGLU, XT_MLP_GELU = 0, 1
XT_ATTN_AUTO, XT_ATTN_COMPOSED, XT_ATTN_FUSED = 0, 1, 2


class XtError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"libxt status {code}: {msg}")
        self.code = code


class MatmulDesc(C.Structure):
    _fields_ = [("M", C.c_int32), ("N", C.c_int32), ("K", C.c_int32),
                ("trans_a", C.c_int32), ("trans_b", C.c_int32),
                ("batch_outer", C.c_int32), ("batch_inner", C.c_int32),
                ("dtype_ab", C.c_int32), ("dtype_c", C.c_int32),
                ("accumulate", C.c_int32), ("causal", C.c_int32), ("alpha", C.c_float),
                ("lda", C.c_int64), ("ldb", C.c_int64), ("ldc", C.c_int64),
                ("stride_a_outer", C.c_int64), ("stride_a_inner", C.c_int64),
                ("stride_b_outer", C.c_int64), ("stride_b_inner", C.c_int64),
                ("stride_c_outer", C.c_int64), ("stride_c_inner", C.c_int64)]


class AdamWConfig(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float), ("eps", C.c_float),
                ("weight_decay", C.c_float), ("max_grad_norm", C.c_float), ("grad_scale", C.c_float),
                ("step", C.c_int32)]


class BlockConfig(C.Structure):
    _fields_ = [("B", C.c_int32), ("S", C.c_int32), ("d", C.c_int32), ("H", C.c_int32),
                ("hd", C.c_int32), ("F", C.c_int32), ("V", C.c_int32), ("n_layers", C.c_int32),
                ("norm", C.c_int32), ("mlp", C.c_int32), ("rope", C.c_int32),
                ("learned_pos", C.c_int32), ("causal", C.c_int32), ("training", C.c_int32),
                ("dtype", C.c_int32), ("grad_dtype", C.c_int32), ("eps", C.c_float),
                ("p", C.c_float), ("rope_base", C.c_double), ("base_seed", C.c_uint64),
                ("attention", C.c_int32), ("recompute", C.c_int32)]


_VP = C.c_void_p
_PP = C.POINTER(C.c_void_p)


class BlockParams(C.Structure):
    _fields_ = [("E", _VP), ("P", _VP), ("g1", _PP), ("b1", _PP), ("Wqkv", _PP), ("Wo", _PP),
                ("g2", _PP), ("b2", _PP), ("W_up", _PP), ("W_down", _PP), ("gf", _VP), ("bf", _VP),
                ("dE", _VP), ("dP", _VP), ("dg1", _PP), ("db1", _PP), ("dWqkv", _PP), ("dWo", _PP),
                ("dg2", _PP), ("db2", _PP), ("dW_up", _PP), ("dW_down", _PP), ("dgf", _VP), ("dbf", _VP)]


_I, _I64, _F, _D, _U64, _SZP = C.c_int, C.c_int64, C.c_float, C.c_double, C.c_uint64, C.POINTER(C.c_size_t)

# name → argtypes (restype is int for all but the two string getters)
_SIGS = {
    "xt_get_device_errors": [C.POINTER(C.c_uint32), _VP],
    "xt_clear_device_errors": [_VP],
    "xt_set_wait_limit_ns": [C.c_uint64],
    "xt_profile_gemm": [_I],
    "xt_profile_gemm_read": [C.POINTER(C.c_double), C.POINTER(C.c_float), C.POINTER(C.c_int), _I,
                             C.POINTER(C.c_int)],
    "xt_accumulate": [_VP, _I, _VP, _I, _I64, _VP],
    "xt_convert": [_VP, _I, _VP, _I, _I64, _VP],
    "xt_add_fwd": [_VP, _VP, _VP, _I64, _I, _VP],
    "xt_add_bwd": [_VP, _VP, _VP, _I64, _I, _I, _I, _VP],
    "xt_mul_fwd": [_VP, _VP, _VP, _I64, _I, _VP],
    "xt_mul_bwd": [_VP, _VP, _VP, _VP, _VP, _I64, _I, _I, _I, _VP],
    "xt_scale_fwd": [_VP, _VP, _I64, _F, _I, _VP],
    "xt_scale_bwd": [_VP, _VP, _I64, _F, _I, _I, _VP],
    "xt_sum_workspace_size": [_I64, _SZP],
    "xt_sum_fwd": [_VP, _I64, _I, _VP, _VP, _VP],
    "xt_sum_bwd": [_VP, _VP, _I64, _I, _I, _VP],
    "xt_colsum_workspace_size": [_I64, _I64, _SZP],
    "xt_add_bias_fwd": [_VP, _VP, _VP, _I64, _I64, _I, _VP],
    "xt_add_bias_bwd": [_VP, _VP, _VP, _I64, _I64, _I, _I, _VP, _I, _I, _VP],
    "xt_silu_fwd": [_VP, _VP, _I64, _I, _VP],
    "xt_silu_bwd": [_VP, _VP, _VP, _I64, _I, _I, _VP],
    "xt_swiglu_fwd": [_VP, _VP, _I64, _VP, _I64, _I64, _I64, _I, _VP],
    "xt_swiglu_bwd": [_VP, _I64, _VP, _VP, _I64, _VP, _VP, _I64, _I64, _I64, _I, _I, _VP],
    "xt_gelu_fwd": [_VP, _VP, _I64, _I, _VP],
    "xt_gelu_bwd": [_VP, _VP, _VP, _I64, _I, _I, _VP],
    "xt_norm_bwd_workspace_size": [_I64, _I64, _SZP],
    "xt_rms_norm_fwd": [_VP, _VP, _VP, _VP, _I64, _I64, _F, _I, _VP],
    "xt_rms_norm_bwd": [_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I, _I, _I, _VP, _I, _I, _VP],
    "xt_rms_norm_bwd_noalloc": [_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I, _I, _I, _I, _I, _VP],
    "xt_layernorm_fwd": [_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _F, _I, _VP],
    "xt_layernorm_bwd": [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I, _I, _I, _VP, _I, _I, _VP],
    "xt_rope_table": [_VP, _I, _I, _D, _I, _VP],
    "xt_rope_fwd": [_VP, _VP, _VP, _I, _I, _I, _I, _I64, _I, _VP],
    "xt_rope_bwd": [_VP, _VP, _VP, _I, _I, _I, _I, _I64, _I, _I, _VP],
    "xt_softmax_fwd": [_VP, _VP, _I64, _I64, _I, _I64, _I, _VP],
    "xt_dropout_add_norm_fwd": [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _F, _U64, _I, _I, _F, _I, _VP],
    "xt_norm_bwd_dropout": [_I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I, _I, _I, _VP, _I, _I, _F,
                            _U64, _I, _VP],
    "xt_softmax_bwd": [_VP, _VP, _VP, _I64, _I64, _I, _I64, _I, _I, _VP],
    "xt_attention_fwd": [_VP, _VP, _VP, _I64, _VP, _VP, _I64, _VP, _I, _I, _I, _I, _I, _I, _VP],
    "xt_attention_bwd_workspace_size": [_I, _I, _I, _SZP],
    "xt_attention_bwd": [_VP, _VP, _VP, _I64, _VP, _VP, _VP, _I64, _VP, _VP, _VP, _VP, _I64, _VP, C.c_size_t,
                         _I, _I, _I, _I, _I, _I, _VP],
    "xt_cross_entropy_workspace_size": [_I64, _SZP],
    "xt_cross_entropy_fwd": [_VP, _VP, _VP, _VP, _I64, _I64, _I, _VP, _VP],
    "xt_cross_entropy_fwd_bwd": [_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I, _I, _VP, _VP],
    "xt_cross_entropy_bwd": [_VP, _VP, _VP, _VP, _VP, _I64, _I64, _I, _I, _I, _VP],
    "xt_cross_entropy_fanout_workspace_size": [_I64, _SZP],
    "xt_ce_set_split": [_I, _I],
    "xt_cross_entropy_fanout_fwd_bwd": [_VP, _VP, _F, _F, _VP, _VP, _VP, _VP, _VP, _I, _I64, _I64, _I, _VP,
                                        C.c_size_t, _VP],
    "xt_dropout_fwd": [_VP, _VP, _I64, _F, _U64, _I, _I, _VP],
    "xt_dropout_bwd": [_VP, _VP, _I64, _F, _U64, _I, _I, _I, _VP],
    "xt_dropout_bwd_ex": [_VP, _I, _VP, _I, _I64, _F, _U64, _I, _I, _VP],
    "xt_dropout_mask": [_VP, _I64, _F, _U64, _VP],
    "xt_dropout_add_fwd": [_VP, _VP, _VP, _I64, _F, _U64, _I, _I, _VP],
    "xt_embedding_workspace_size": [_I64, _SZP],
    "xt_embedding_fwd": [_VP, _VP, _VP, _VP, _I64, _I, _I64, _I64, _I, _VP],
    "xt_embedding_bwd": [_VP, _VP, _VP, _VP, _I64, _I, _I64, _I64, _I, _I, _VP, _I, _VP],
    "xt_matmul_workspace_size": [C.POINTER(MatmulDesc), _SZP],
    "xt_gemm_set_schedule": [_I],
    "xt_gemm_set_pairing": [_I],
    "xt_block_set_overlap": [_I],
    "xt_gemm_set_tile": [_I],
    "xt_quantize_fp8_workspace_size": [_I64, _SZP],
    "xt_quantize_fp8": [_VP, _I64, _I, _VP, _VP, _VP, C.c_size_t, _VP],
    "xt_matmul_fp8_fwd": [_I64, _I64, _I64, _VP, _I64, _VP, _I64, _VP, _I64, _I, _F, _VP, _VP, _I, _VP],
    "xt_adamw_workspace_size": [_I, C.POINTER(C.c_int64), _SZP],
    "xt_adamw_step": [C.POINTER(AdamWConfig), _I, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p),
                      C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), _I,
                      C.POINTER(C.c_int64), _VP, _VP, C.c_size_t, _VP],
    "xt_matmul_fwd": [C.POINTER(MatmulDesc), _VP, _VP, _VP, _VP, C.c_size_t, _VP],
    "xt_matmul_gelu_fwd": [C.POINTER(MatmulDesc), _VP, _VP, _VP, _VP, _VP, C.c_size_t, _VP],
    "xt_matmul_gelu_bwd": [C.POINTER(MatmulDesc), _VP, _VP, _VP, _VP, _VP, C.c_size_t, _VP],
    "xt_matmul_bwd_workspace_size": [C.POINTER(MatmulDesc), _SZP],
    "xt_matmul_bwd": [C.POINTER(MatmulDesc), _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP, C.c_size_t, _VP],
    "xt_block_workspace_size": [C.POINTER(BlockConfig), _SZP],
    "xt_block_fwd": [C.POINTER(BlockConfig), C.POINTER(BlockParams), _VP, _VP, _VP, _VP, _VP],
    "xt_block_bwd": [C.POINTER(BlockConfig), C.POINTER(BlockParams), _VP, _VP, _VP, _VP],
    "xt_block_zero_grads": [C.POINTER(BlockConfig), C.POINTER(BlockParams), _VP],
}

_lib = None


def lib():
    """Loads libxt.so (built in-tree by __graft_entry__.build()); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() first")
        L = C.CDLL(LIB_PATH)
        L.xt_last_error.restype = C.c_char_p
        L.xt_last_error.argtypes = []
        L.xt_version.restype = C.c_char_p
        L.xt_version.argtypes = []
        L.xt_launch_count.restype = C.c_uint64
        L.xt_launch_count.argtypes = []
        L.xt_get_wait_limit_ns.restype = C.c_uint64
        L.xt_get_wait_limit_ns.argtypes = []
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = C.c_int
        _lib = L
    return _lib


def exported_symbols():
    return ["xt_last_error", "xt_version", "xt_launch_count", "xt_get_wait_limit_ns", *_SIGS.keys()]


def launch_count() -> int:
    return int(lib().xt_launch_count())


def set_wait_limit_ns(ns: int):
    """Limit of the tensor-core kernels' bounded waits on work (0: the default, 2 s)."""
    call("xt_set_wait_limit_ns", int(ns))


def wait_limit_ns() -> int:
    return int(lib().xt_get_wait_limit_ns())


def profile_gemm(capacity: int):
    call("xt_profile_gemm", int(capacity))


def profile_gemm_read(max_records: int = 1 << 16, shapes: bool = False):
    """Returns (flops, ms) numpy arrays of the GEMM launches recorded since profile_gemm(),
    plus an [n, 8] int array (M, N, K, batches, BN, A MN-major, B MN-major, causal) if shapes."""
    import numpy as np
    fl = (C.c_double * max_records)()
    ms = (C.c_float * max_records)()
    sh = (C.c_int * (8 * max_records))()
    n = C.c_int(0)
    call("xt_profile_gemm_read", fl, ms, sh, max_records, C.byref(n))
    k = min(n.value, max_records)
    out = (np.array(fl[:k]), np.array(ms[:k], dtype=np.float64))
    if shapes:
        out = out + (np.array(sh[:8 * k], dtype=np.int64).reshape(k, 8),)
    return out


def _check(code):
    if code != XT_OK:
        raise XtError(code, lib().xt_last_error().decode(errors="replace"))


def call(name, *args):
    """Calls a libxt entry point with already-marshalled arguments; raises on failure."""
    _check(getattr(lib(), name)(*args))


# ------------------------------------------------------------------------------ marshalling

def dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return XT_F32
    if t.dtype == torch.bfloat16:
        return XT_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def ptr(t, contiguous=True):
    """Device address of `t`.  Entry points that take their sizes from a tensor read it as
    dense row-major, so such tensors must be contiguous; strided views (matmul operands,
    swiglu column blocks) pass contiguous=False and describe their layout explicitly."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("libxt takes CUDA tensors")
    if contiguous and not t.is_contiguous():
        raise ValueError("libxt reads this tensor as dense row-major: pass a contiguous tensor")
    return t.data_ptr()


def stream(s=None):
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    return s.cuda_stream if hasattr(s, "cuda_stream") else s


def ws_bytes(name, *args) -> int:
    out = C.c_size_t(0)
    call(name, *args, C.byref(out))
    return int(out.value)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zero-filled scratch (the matmul workspace's flag words must start at zero)."""
    return torch.zeros(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def gemm_set_schedule(mode: int):
    """0 model's choice, 1 whole tiles, 2 K split, 3 stream-K over every SM, 4 stream-K in
    lockstep K slices (2-4 where allowed)."""
    call("xt_gemm_set_schedule", int(mode))


def gemm_set_pairing(mode: int):
    """0 model's choice, 1 never the paired-CTA kernel, 2 the paired kernel wherever allowed, 3 its
    multicast form (two pairs of a cluster sharing B) wherever allowed."""
    call("xt_gemm_set_pairing", int(mode))


def block_set_overlap(on: int):
    """1 (default): the block backward's weight-gradient GEMMs on a second stream; 0: one stream."""
    call("xt_block_set_overlap", int(on))


def ce_set_split(cl: int, nb: int):
    """Cross-entropy row split: clusters of cl CTAs with nb chunk buffers, (0, 0) automatic."""
    call("xt_ce_set_split", int(cl), int(nb))


def gemm_set_tile(bn: int):
    """0 model's choice, else the GEMM tile width BN (64, 128, 192, 256) wherever allowed."""
    call("xt_gemm_set_tile", int(bn))


def device_errors(s=None) -> int:
    out = C.c_uint32(0)
    code = lib().xt_get_device_errors(C.byref(out), stream(s))
    if code not in (XT_OK, XT_ERR_TIMEOUT):
        _check(code)
    return int(out.value)


def clear_device_errors(s=None):
    call("xt_clear_device_errors", stream(s))


def version() -> str:
    return lib().xt_version().decode()


# ------------------------------------------------------------------------------ op wrappers
# Same names as the C entry points; tensors in, results written into caller tensors.

def xt_accumulate(dst, src, s=None):
    call("xt_accumulate", ptr(dst), dt(dst), ptr(src), dt(src), src.numel(), stream(s))


def xt_convert(dst, src, s=None):
    call("xt_convert", ptr(dst), dt(dst), ptr(src), dt(src), src.numel(), stream(s))


def xt_add_fwd(a, b, y, s=None):
    call("xt_add_fwd", ptr(a), ptr(b), ptr(y), a.numel(), dt(a), stream(s))


def xt_add_bwd(d, da, db, acc_a=0, acc_b=0, s=None):
    call("xt_add_bwd", ptr(d), ptr(da), ptr(db), d.numel(), dt(d), acc_a, acc_b, stream(s))


def xt_mul_fwd(a, b, y, s=None):
    call("xt_mul_fwd", ptr(a), ptr(b), ptr(y), a.numel(), dt(a), stream(s))


def xt_mul_bwd(d, a, b, da, db, acc_a=0, acc_b=0, s=None):
    call("xt_mul_bwd", ptr(d), ptr(a), ptr(b), ptr(da), ptr(db), d.numel(), dt(d), acc_a, acc_b, stream(s))


def xt_scale_fwd(x, y, alpha, s=None):
    call("xt_scale_fwd", ptr(x), ptr(y), x.numel(), float(alpha), dt(x), stream(s))


def xt_scale_bwd(d, dx, alpha, acc=0, s=None):
    call("xt_scale_bwd", ptr(d), ptr(dx), d.numel(), float(alpha), dt(d), acc, stream(s))


def xt_sum_fwd(x, out, ws=None, s=None):
    if ws is None:
        ws = workspace(ws_bytes("xt_sum_workspace_size", x.numel()), x.device)
    call("xt_sum_fwd", ptr(x), x.numel(), dt(x), ptr(out), ptr(ws), stream(s))


def xt_sum_bwd(upstream, dx, acc=0, s=None):
    call("xt_sum_bwd", ptr(upstream), ptr(dx), dx.numel(), dt(dx), acc, stream(s))


def xt_add_bias_fwd(x, bias, y, s=None):
    rows, cols = x.shape
    call("xt_add_bias_fwd", ptr(x), ptr(bias), ptr(y), rows, cols, dt(x), stream(s))


def xt_add_bias_bwd(d, dx, dbias, acc_dx=0, acc_dbias=0, ws=None, s=None):
    rows, cols = d.shape
    if ws is None:
        ws = workspace(ws_bytes("xt_colsum_workspace_size", rows, cols), d.device)
    call("xt_add_bias_bwd", ptr(d), ptr(dx), ptr(dbias), rows, cols, dt(d), dt(dbias), ptr(ws), acc_dx,
         acc_dbias, stream(s))


def xt_silu_fwd(x, y, s=None):
    call("xt_silu_fwd", ptr(x), ptr(y), x.numel(), dt(x), stream(s))


def xt_silu_bwd(d, x, dx, acc=0, s=None):
    call("xt_silu_bwd", ptr(d), ptr(x), ptr(dx), d.numel(), dt(d), acc, stream(s))


def xt_gelu_fwd(x, y, s=None):
    call("xt_gelu_fwd", ptr(x), ptr(y), x.numel(), dt(x), stream(s))


def xt_gelu_bwd(d, x, dx, acc=0, s=None):
    call("xt_gelu_bwd", ptr(d), ptr(x), ptr(dx), d.numel(), dt(d), acc, stream(s))


def xt_swiglu_fwd(g, u, y, s=None):
    rows, cols = g.shape
    for t in (g, u, y):
        assert t.stride(1) == 1, "swiglu operands need unit column stride"
    call("xt_swiglu_fwd", ptr(g, False), ptr(u, False), g.stride(0), ptr(y, False), y.stride(0), rows, cols, dt(g),
         stream(s))


def xt_swiglu_bwd(d, g, u, dg, du, acc=0, s=None):
    rows, cols = g.shape
    assert u.stride(0) == g.stride(0) and du.stride(0) == dg.stride(0)
    for t in (d, g, u, dg, du):
        assert t.stride(1) == 1, "swiglu operands need unit column stride"
    call("xt_swiglu_bwd", ptr(d, False), d.stride(0), ptr(g, False), ptr(u, False), g.stride(0), ptr(dg, False),
         ptr(du, False), dg.stride(0), rows, cols, dt(g), acc, stream(s))


def xt_rms_norm_fwd(x, gamma, y, inv_rms, eps, s=None):
    rows, cols = x.shape
    call("xt_rms_norm_fwd", ptr(x), ptr(gamma), ptr(y), ptr(inv_rms), rows, cols, float(eps), dt(x), stream(s))


def xt_rms_norm_bwd(d, x, gamma, inv_rms, dx, dgamma, acc_dx=0, acc_param=0, ws=None, s=None):
    rows, cols = x.shape
    if ws is None:
        ws = workspace(ws_bytes("xt_norm_bwd_workspace_size", rows, cols), x.device)
    call("xt_rms_norm_bwd", ptr(d), ptr(x), ptr(gamma), ptr(inv_rms), ptr(dx), ptr(dgamma), rows, cols, dt(x),
         dt(dx) if dx is not None else dt(x), dt(dgamma) if dgamma is not None else dt(x), ptr(ws), acc_dx,
         acc_param, stream(s))


def xt_rms_norm_bwd_noalloc(d, x, gamma, inv_rms, dx, dgamma, acc_dx=0, acc_param=0, s=None):
    """Same result as xt_rms_norm_bwd without a workspace argument (scratch is fixed in libxt)."""
    rows, cols = x.shape
    call("xt_rms_norm_bwd_noalloc", ptr(d), ptr(x), ptr(gamma), ptr(inv_rms), ptr(dx), ptr(dgamma), rows, cols,
         dt(x), dt(dx) if dx is not None else dt(x), dt(dgamma) if dgamma is not None else dt(x), acc_dx, acc_param,
         stream(s))


def xt_layernorm_fwd(x, gamma, beta, y, mean, rstd, eps, s=None):
    rows, cols = x.shape
    call("xt_layernorm_fwd", ptr(x), ptr(gamma), ptr(beta), ptr(y), ptr(mean), ptr(rstd), rows, cols, float(eps),
         dt(x), stream(s))


def xt_layernorm_bwd(d, x, gamma, mean, rstd, dx, dgamma, dbeta, acc_dx=0, acc_param=0, ws=None, s=None):
    rows, cols = x.shape
    if ws is None:
        ws = workspace(ws_bytes("xt_norm_bwd_workspace_size", rows, cols), x.device)
    pdt = dt(dgamma) if dgamma is not None else (dt(dbeta) if dbeta is not None else dt(x))
    call("xt_layernorm_bwd", ptr(d), ptr(x), ptr(gamma), ptr(mean), ptr(rstd), ptr(dx), ptr(dgamma), ptr(dbeta),
         rows, cols, dt(x), dt(dx) if dx is not None else dt(x), pdt, ptr(ws), acc_dx, acc_param, stream(s))


def xt_dropout_add_norm_fwd(h, a, sum_out, gamma, beta, y, stat0, stat1, p, seed, training, norm, eps, s=None):
    rows, cols = h.shape
    call("xt_dropout_add_norm_fwd", ptr(h), ptr(a), ptr(sum_out), ptr(gamma), ptr(beta), ptr(y), ptr(stat0),
         ptr(stat1), rows, cols, float(p), int(seed) & (2**64 - 1), int(training), norm, float(eps), dt(h), stream(s))


def xt_norm_bwd_dropout(norm, d, x, gamma, stat0, stat1, dx, dgamma, dbeta, g, p, seed, training, acc_dx=0,
                        acc_param=0, ws=None, s=None):
    rows, cols = x.shape
    if ws is None:
        ws = workspace(ws_bytes("xt_norm_bwd_workspace_size", rows, cols), x.device)
    pdt = dt(dgamma) if dgamma is not None else (dt(dbeta) if dbeta is not None else dt(x))
    call("xt_norm_bwd_dropout", norm, ptr(d), ptr(x), ptr(gamma), ptr(stat0), ptr(stat1), ptr(dx), ptr(dgamma),
         ptr(dbeta), ptr(g), rows, cols, dt(x), dt(dx), pdt, ptr(ws), acc_dx, acc_param, float(p),
         int(seed) & (2**64 - 1), int(training), stream(s))


def xt_rope_table(table, S, hd, base, pos_offset=0, s=None):
    call("xt_rope_table", ptr(table), S, hd, float(base), pos_offset, stream(s))


def xt_rope_fwd(x, y, table, B, S, H, hd, ld, s=None):
    call("xt_rope_fwd", ptr(x, False), ptr(y, False), ptr(table), B, S, H, hd, ld, dt(x), stream(s))


def xt_rope_bwd(d, dx, table, B, S, H, hd, ld, acc=0, s=None):
    call("xt_rope_bwd", ptr(d, False), ptr(dx, False), ptr(table), B, S, H, hd, ld, dt(d), acc, stream(s))


def xt_softmax_fwd(x, y, causal=0, q_len=0, s=None):
    cols = x.shape[-1]
    rows = x.numel() // cols
    call("xt_softmax_fwd", ptr(x), ptr(y), rows, cols, causal, q_len, dt(x), stream(s))


def xt_attention_fwd(q, k, v, o, lse, B, S, H, hd, causal=1, o_lo=None, s=None):
    """q, k, v: [B·S, ld] views (head h at columns h·hd); o (and the optional rounding residual
    o_lo, same layout): [B·S, ld_o] bf16; lse: float32 [B, H, S]."""
    if o_lo is not None and o_lo.stride(0) != o.stride(0):
        raise ValueError("o_lo must have o's row stride")
    call("xt_attention_fwd", ptr(q, False), ptr(k, False), ptr(v, False), q.stride(0), ptr(o, False),
         ptr(o_lo, False), o.stride(0), ptr(lse), B, S, H, hd, causal, dt(q), stream(s))


def xt_attention_bwd(q, k, v, o, d_o, lse, dq, dk, dv, B, S, H, hd, causal=1, o_lo=None, ws=None, s=None):
    if d_o.stride(0) != o.stride(0) or (o_lo is not None and o_lo.stride(0) != o.stride(0)):
        raise ValueError("o, o_lo and d_o must share a row stride")
    n = C.c_size_t(0)
    call("xt_attention_bwd_workspace_size", B, S, H, C.byref(n))
    if ws is None:
        ws = torch.empty(max(1, n.value), dtype=torch.uint8, device=q.device)
    call("xt_attention_bwd", ptr(q, False), ptr(k, False), ptr(v, False), q.stride(0), ptr(o, False),
         ptr(o_lo, False), ptr(d_o, False), o.stride(0), ptr(lse), ptr(dq, False), ptr(dk, False), ptr(dv, False),
         dq.stride(0), ptr(ws), ws.numel(), B, S, H, hd, causal, dt(q), stream(s))


def xt_softmax_bwd(d, y, dx, causal=0, q_len=0, acc=0, s=None):
    cols = y.shape[-1]
    rows = y.numel() // cols
    call("xt_softmax_bwd", ptr(d), ptr(y), ptr(dx), rows, cols, causal, q_len, dt(y), acc, stream(s))


def xt_cross_entropy_fwd(logits, targets, lse, loss, ws=None, s=None):
    rows, V = logits.shape
    if ws is None:
        ws = workspace(ws_bytes("xt_cross_entropy_workspace_size", rows), logits.device)
    call("xt_cross_entropy_fwd", ptr(logits), ptr(targets), ptr(lse), ptr(loss), rows, V, dt(logits), ptr(ws),
         stream(s))


def xt_cross_entropy_fwd_bwd(logits, targets, lse, loss, upstream, dlogits, ws=None, s=None):
    """Forward and backward in one pass (dlogits may be logits)."""
    rows, V = logits.shape
    if ws is None:
        ws = workspace(ws_bytes("xt_cross_entropy_workspace_size", rows), logits.device)
    call("xt_cross_entropy_fwd_bwd", ptr(logits), ptr(targets), ptr(lse), ptr(loss), ptr(upstream), ptr(dlogits),
         rows, V, dt(logits), dt(dlogits), ptr(ws), stream(s))


def xt_cross_entropy_fanout_fwd_bwd(logits, targets, c_lin, c_sq, lse, loss, sums, grad, upstream=None, acc=0,
                                    ws=None, s=None):
    """L = CE(x) + c_lin·Σx + c_sq·Σx∘x forward and backward in one pass; grad (+)= u·dL/dx (float32),
    u the device scalar `upstream` (None: 1)."""
    rows, V = logits.shape
    if ws is None:
        ws = workspace(ws_bytes("xt_cross_entropy_fanout_workspace_size", rows), logits.device)
    call("xt_cross_entropy_fanout_fwd_bwd", ptr(logits), ptr(targets), float(c_lin), float(c_sq), ptr(upstream),
         ptr(lse), ptr(loss), ptr(sums), ptr(grad), int(acc), rows, V, dt(logits), ptr(ws), ws.numel(), stream(s))


def xt_cross_entropy_bwd(logits, targets, lse, upstream, dlogits, acc=0, s=None):
    rows, V = logits.shape
    call("xt_cross_entropy_bwd", ptr(logits), ptr(targets), ptr(lse), ptr(upstream), ptr(dlogits), rows, V,
         dt(logits), dt(dlogits), acc, stream(s))


def xt_dropout_fwd(x, y, p, seed, training=1, s=None):
    call("xt_dropout_fwd", ptr(x), ptr(y), x.numel(), float(p), int(seed) & (2**64 - 1), int(training), dt(x),
         stream(s))


def xt_dropout_bwd(d, dx, p, seed, training=1, acc=0, s=None):
    call("xt_dropout_bwd", ptr(d), ptr(dx), d.numel(), float(p), int(seed) & (2**64 - 1), int(training), dt(d),
         acc, stream(s))


def xt_dropout_bwd_ex(d, dx, p, seed, training=1, acc=0, s=None):
    call("xt_dropout_bwd_ex", ptr(d), dt(d), ptr(dx), dt(dx), d.numel(), float(p), int(seed) & (2**64 - 1),
         int(training), acc, stream(s))


def xt_dropout_mask(mask, p, seed, s=None):
    call("xt_dropout_mask", ptr(mask), mask.numel(), float(p), int(seed) & (2**64 - 1), stream(s))


def xt_dropout_add_fwd(h, a, out, p, seed, training=1, s=None):
    call("xt_dropout_add_fwd", ptr(h), ptr(a), ptr(out), h.numel(), float(p), int(seed) & (2**64 - 1),
         int(training), dt(h), stream(s))


def xt_embedding_fwd(ids, E, P, h, S, s=None):
    V, d = E.shape
    call("xt_embedding_fwd", ptr(ids), ptr(E), ptr(P), ptr(h), ids.numel(), S, d, V, dt(E), stream(s))


def xt_embedding_bwd(ids, dh, dE, dP, S, acc=0, ws=None, s=None):
    V, d = dE.shape
    T = ids.numel()
    if ws is None:
        ws = workspace(ws_bytes("xt_embedding_workspace_size", T), dh.device)
    call("xt_embedding_bwd", ptr(ids), ptr(dh), ptr(dE), ptr(dP), T, S, d, V, dt(dh), dt(dE), ptr(ws), acc,
         stream(s))


def matmul_desc(M, N, K, *, trans_a=0, trans_b=0, lda=None, ldb=None, ldc=None, batch_outer=1, batch_inner=1,
                dtype_ab=XT_BF16, dtype_c=XT_F32, accumulate=0, causal=0, alpha=1.0, strides=(0, 0, 0, 0, 0, 0)):
    d = MatmulDesc()
    d.M, d.N, d.K = M, N, K
    d.trans_a, d.trans_b = trans_a, trans_b
    d.lda = lda if lda is not None else (M if trans_a else K)
    d.ldb = ldb if ldb is not None else (K if trans_b else N)
    d.ldc = ldc if ldc is not None else N
    d.batch_outer, d.batch_inner = batch_outer, batch_inner
    d.dtype_ab, d.dtype_c = dtype_ab, dtype_c
    d.accumulate, d.causal, d.alpha = accumulate, causal, alpha
    (d.stride_a_outer, d.stride_a_inner, d.stride_b_outer, d.stride_b_inner,
     d.stride_c_outer, d.stride_c_inner) = strides
    return d


def adamw_config(lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0, max_grad_norm=0.0, grad_scale=1.0, step=1):
    return AdamWConfig(lr, beta1, beta2, eps, weight_decay, max_grad_norm, grad_scale, step)


def adamw_workspace(numels, device="cuda"):
    arr = (C.c_int64 * max(1, len(numels)))(*numels)
    return workspace(ws_bytes("xt_adamw_workspace_size", len(numels), arr), device)


def xt_adamw_step(cfg, params, grads, m, v, shadows=None, norm_out=None, ws=None, s=None):
    """One AdamW step over lists of float32 tensors (params, grads, m, v updated in place
    except grads); shadows: None or a list (entries may be None) of bf16 / float32 tensors that
    receive the updated weights; norm_out: a float32 device tensor of one element or None."""
    n = len(params)
    if not (len(grads) == len(m) == len(v) == n):
        raise ValueError("params, grads, m, v must have the same length")
    for t in list(params) + list(grads) + list(m) + list(v):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("params, grads, m, v must be contiguous float32")
    numel = [t.numel() for t in params]
    for lst in (grads, m, v):
        if [t.numel() for t in lst] != numel:
            raise ValueError("tensor sizes differ")
    P = (C.c_void_p * n)(*[t.data_ptr() for t in params])
    G = (C.c_void_p * n)(*[t.data_ptr() for t in grads])
    M = (C.c_void_p * n)(*[t.data_ptr() for t in m])
    V = (C.c_void_p * n)(*[t.data_ptr() for t in v])
    SH, sdt = None, XT_F32
    if shadows is not None:
        dts = {t.dtype for t in shadows if t is not None}
        if len(dts) > 1:
            raise ValueError("shadows must share one dtype")
        sdt = XT_BF16 if dts == {torch.bfloat16} else XT_F32
        for t, p in zip(shadows, params):
            if t is not None and (t.numel() != p.numel() or not t.is_contiguous()):
                raise ValueError("shadow shapes must match params")
        SH = (C.c_void_p * n)(*[(t.data_ptr() if t is not None else None) for t in shadows])
    N = (C.c_int64 * n)(*numel)
    if ws is None and (cfg.max_grad_norm > 0 or norm_out is not None):
        ws = adamw_workspace(numel, params[0].device)
    call("xt_adamw_step", C.byref(cfg), n, P, G, M, V, SH, sdt, N, ptr(norm_out), ptr(ws),
         ws.numel() if ws is not None else 0, stream(s))


def xt_quantize_fp8(x, out, dequant, ws=None, s=None):
    """Per-tensor e4m3 quantization of x (float32 / bf16) into out (uint8, x's element count);
    dequant: a float32 device tensor of one element receiving max|x| / 448."""
    if out.dtype != torch.uint8 or out.numel() != x.numel():
        raise ValueError("out must be uint8 with x's element count")
    n = x.numel()
    if ws is None:
        ws = workspace(ws_bytes("xt_quantize_fp8_workspace_size", n), x.device)
    call("xt_quantize_fp8", ptr(x), n, dt(x), ptr(out), ptr(dequant), ptr(ws), ws.numel(), stream(s))


def xt_matmul_fp8_fwd(A, B, Cm, alpha=1.0, scale_a=None, scale_b=None, accumulate=0, s=None):
    """C [M, N] (+)= alpha·sa·sb·A Bᵀ with A [M, K] and B [N, K] uint8 e4m3 codes (row strides
    from the tensors), C float32 or bf16; scale_a / scale_b: float32 device tensors of one
    element or None."""
    if A.dtype != torch.uint8 or B.dtype != torch.uint8:
        raise ValueError("A and B must be uint8 e4m3 codes")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K or tuple(Cm.shape) != (M, N):
        raise ValueError("shape mismatch")
    call("xt_matmul_fp8_fwd", M, N, K, ptr(A, False), A.stride(0), ptr(B, False), B.stride(0), ptr(Cm, False),
         Cm.stride(0), dt(Cm), float(alpha), ptr(scale_a), ptr(scale_b), int(accumulate), stream(s))


def matmul_workspace(desc, device="cuda"):
    """A zero-filled workspace of the size xt_matmul_workspace_size reports (None if 0)."""
    n = ws_bytes("xt_matmul_workspace_size", C.byref(desc))
    return workspace(n, device) if n else None


def xt_matmul_fwd(desc, A, B, Cm, ws=None, s=None):
    n = ws_bytes("xt_matmul_workspace_size", C.byref(desc))
    if n and ws is None:
        ws = workspace(n, Cm.device)
    call("xt_matmul_fwd", C.byref(desc), ptr(A, False), ptr(B, False), ptr(Cm, False), ptr(ws),
         ws.numel() if ws is not None else 0, stream(s))


def xt_matmul_gelu_fwd(desc, A, B, Cm, Y, ws=None, s=None):
    """Cm = alpha·op(A)@op(B) (bf16) and Y = gelu(Cm), from one GEMM."""
    n = ws_bytes("xt_matmul_workspace_size", C.byref(desc))
    if n and ws is None:
        ws = workspace(n, Cm.device)
    call("xt_matmul_gelu_fwd", C.byref(desc), ptr(A, False), ptr(B, False), ptr(Cm, False), ptr(Y, False), ptr(ws),
         ws.numel() if ws is not None else 0, stream(s))


def xt_matmul_gelu_bwd(desc, A, B, X, Cm, ws=None, s=None):
    """Cm = (alpha·op(A)@op(B)) ∘ gelu'(X), X the saved pre-activation (Cm's layout)."""
    n = ws_bytes("xt_matmul_workspace_size", C.byref(desc))
    if n and ws is None:
        ws = workspace(n, Cm.device)
    call("xt_matmul_gelu_bwd", C.byref(desc), ptr(A, False), ptr(B, False), ptr(X, False), ptr(Cm, False), ptr(ws),
         ws.numel() if ws is not None else 0, stream(s))


def xt_matmul_bwd(desc, A, B, dC, dA, dB, acc_a=0, acc_b=0, ws=None, s=None):
    n = ws_bytes("xt_matmul_bwd_workspace_size", C.byref(desc))
    if n and ws is None:
        ws = workspace(n, dC.device)
    call("xt_matmul_bwd", C.byref(desc), ptr(A, False), ptr(B, False), ptr(dC, False), ptr(dA, False),
         ptr(dB, False),
         dt(dA) if dA is not None else XT_F32, dt(dB) if dB is not None else XT_F32, acc_a, acc_b, ptr(ws),
         ws.numel() if ws is not None else 0, stream(s))
