"""The C ABI without a GPU: the library builds, loads, exports every entry point that
include/xt.h declares, the binding declares them all, and host-side validation rejects bad
arguments before anything touches the device."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "xt.h")


def header_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*|uint64_t)\s+(xt_\w+)\s*\(", src, re.M)))


@pytest.fixture(scope="module")
def xt():
    from transformer_fwd_bwd_gb300 import build
    build.build()
    from transformer_fwd_bwd_gb300 import xt as m
    m.lib()
    return m


def test_header_parses():
    fns = header_functions()
    assert "xt_matmul_fwd" in fns and "xt_rms_norm_bwd" in fns and len(fns) > 40


def test_exports_every_declared_symbol(xt):
    L = xt.lib()
    missing = [f for f in header_functions() if not hasattr(L, f)]
    assert not missing, f"not exported: {missing}"


def test_binding_declares_every_symbol(xt):
    declared = set(xt.exported_symbols())
    missing = [f for f in header_functions() if f not in declared]
    assert not missing, f"binding lacks: {missing}"


def test_host_validation(xt):
    L = xt.lib()
    assert L.xt_matmul_fwd(None, None, None, None, None, 0, None) == xt.XT_ERR_INVALID_ARG
    assert b"desc is NULL" in L.xt_last_error()
    assert L.xt_dropout_fwd(None, None, 10, C.c_float(1.5), 1, 1, 0, None) == xt.XT_ERR_INVALID_ARG
    assert L.xt_rope_table(None, 4, 7, C.c_double(1e4), 0, None) == xt.XT_ERR_INVALID_ARG
    assert L.xt_softmax_fwd(None, None, 4, 8, 5, 0, 0, None) == xt.XT_ERR_INVALID_ARG
    assert L.xt_rms_norm_fwd(None, None, None, None, -1, 8, C.c_float(1e-5), 0, None) == xt.XT_ERR_INVALID_ARG
    assert L.xt_accumulate(None, 7, None, 0, 4, None) == xt.XT_ERR_INVALID_ARG
    sz = C.c_size_t(0)
    d = xt.matmul_desc(64, 64, 60, lda=60, ldb=64)
    assert L.xt_matmul_fwd(C.byref(d), 16, 16, 16, None, 0, None) == xt.XT_ERR_ALIGNMENT
    d = xt.matmul_desc(64, 64, 64, lda=8)
    assert L.xt_matmul_fwd(C.byref(d), 16, 16, 16, None, 0, None) == xt.XT_ERR_INVALID_ARG
    # every matmul workspace starts with 4096 bytes of stream-K flag words; fp32 operands read
    # MN-major add tf32 staging scratch; a short-K bf16 problem (no split, no stream-K) nothing
    d = xt.matmul_desc(256, 128, 64, trans_a=1, dtype_ab=xt.XT_F32)
    assert L.xt_matmul_workspace_size(C.byref(d), C.byref(sz)) == 0
    assert sz.value >= 4096 + 256 * 64 * 4 + 128 * 64 * 4
    d = xt.matmul_desc(256, 128, 64, trans_a=1, dtype_ab=xt.XT_BF16)
    assert L.xt_matmul_workspace_size(C.byref(d), C.byref(sz)) == 0 and sz.value == 4096
    d = xt.matmul_desc(0, 128, 64)
    assert L.xt_matmul_workspace_size(C.byref(d), C.byref(sz)) == 0 and sz.value == 0
    assert L.xt_gemm_set_schedule(5) == xt.XT_ERR_INVALID_ARG and L.xt_gemm_set_schedule(0) == 0
    assert L.xt_embedding_workspace_size(1000, C.byref(sz)) == 0 and sz.value == 16
    assert L.xt_sum_workspace_size(-1, C.byref(sz)) == xt.XT_ERR_INVALID_ARG
    assert xt.version().startswith("xt")


def test_block_recompute_workspace_and_validation(xt):
    """The recompute option keeps one layer's activations instead of every layer's: the block
    workspace shrinks by about (n_layers − 1) layers' worth; modes other than 0/1 are rejected."""
    import synth
    from transformer_fwd_bwd_gb300.block import config_struct
    L = xt.lib()
    cfg = dict(synth.BLOCK_CONFIGS["gpt12"])
    sizes = {}
    for rc in (0, 1):
        c = config_struct(dict(cfg, recompute=rc))
        n = C.c_size_t(0)
        assert L.xt_block_workspace_size(C.byref(c), C.byref(n)) == 0
        sizes[rc] = n.value
    assert sizes[1] < sizes[0] * 0.7, sizes
    c = config_struct(dict(cfg, recompute=2))
    n = C.c_size_t(0)
    assert L.xt_block_workspace_size(C.byref(c), C.byref(n)) == xt.XT_ERR_INVALID_ARG
