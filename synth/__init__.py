"""Seeded synthetic inputs shared by the CPU oracle tests and the CUDA path.

This module holds NO arithmetic of the method: it only draws random numbers,
rounds them to the storage type of a run, and describes workload shapes.  Both
sides (oracle tests, GPU tests, bench) call it so that they see the same inputs;
neither side's results ever flow back into it.

Seeds (fixed): 1234 weights, 1235 token ids / targets, 1236 op-sweep data,
0x5EED dropout base seed.
"""
from __future__ import annotations

import numpy as np

SEED_WEIGHTS = 1234
SEED_TOKENS = 1235
SEED_SWEEP = 1236
BASE_SEED_DROPOUT = 0x5EED


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def round_bf16(a) -> np.ndarray:
    """Round float values to the nearest bfloat16 (ties to even), returned as float64.

    Storage conversion only: bfloat16 keeps the top 16 bits of an IEEE float32.
    """
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    nan = np.isnan(f)
    r = np.where(nan, np.uint64(0x7FC0), r)
    out = (r << np.uint64(16)).astype(np.uint32).view(np.float32)
    return out.astype(np.float64)


def bf16_bits(a) -> np.ndarray:
    """uint16 bit patterns of `a` rounded to bfloat16 (for uploading bf16 tensors)."""
    f = np.ascontiguousarray(round_bf16(a).astype(np.float32))
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def from_bf16_bits(bits) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16)).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def to_storage(a, dtype: str) -> np.ndarray:
    """Round to the storage type ('f32' or 'bf16'); the result is float64 holding exact values."""
    if dtype == "f32":
        return np.ascontiguousarray(np.asarray(a, dtype=np.float32), dtype=np.float64)
    if dtype == "bf16":
        return round_bf16(a)
    raise ValueError(dtype)


def normal(shape, seed: int, std: float = 1.0, mean: float = 0.0, dtype: str = "f32") -> np.ndarray:
    g = rng(seed)
    return to_storage(g.normal(mean, std, size=shape), dtype)


def normal_bf16_bits(shape, seed: int, std: float = 1.0, chunk_rows: int = 512) -> np.ndarray:
    """N(0, std) draws (float32) rounded to bfloat16, returned as uint16 bit patterns; drawn
    in row chunks so host memory stays bounded for multi-GB tensors."""
    g = rng(seed)
    out = np.empty(shape, dtype=np.uint16)
    for r0 in range(0, shape[0], chunk_rows):
        n = min(chunk_rows, shape[0] - r0)
        blk = g.standard_normal((n,) + tuple(shape[1:]), dtype=np.float32) * np.float32(std)
        out[r0:r0 + n] = bf16_bits(blk)
    return out


def uniform_ids(n: int, vocab: int, seed: int) -> np.ndarray:
    return rng(seed).integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


# --------------------------------------------------------------------------------------
# Workload shapes (the five configurations the hot path is exercised on)
# --------------------------------------------------------------------------------------

BLOCK_CONFIGS = {
    # One pre-norm block, fp32, RMSNorm + RoPE + SwiGLU, tied logits, causal, p = 0.
    "tiny": dict(B=1, S=16, d=32, H=2, hd=16, F=64, V=64, n_layers=1, norm="rms", mlp="swiglu",
                 rope=True, rope_base=10000.0, learned_pos=False, eps=1e-5, causal=True,
                 p=0.0, dtype="f32"),
    # Same topology, larger, residual dropout p = 0.1 at both sites.
    "block256": dict(B=4, S=256, d=256, H=4, hd=64, F=688, V=4096, n_layers=1, norm="rms",
                     mlp="swiglu", rope=True, rope_base=10000.0, learned_pos=False, eps=1e-5,
                     causal=True, p=0.1, dtype="f32"),
    # 12-layer GPT-style stack: LayerNorm, exact GELU MLP, learned positions, tied output, bf16.
    "gpt12": dict(B=8, S=1024, d=768, H=12, hd=64, F=3072, V=50304, n_layers=12, norm="ln",
                  mlp="gelu", rope=False, rope_base=10000.0, learned_pos=True, eps=1e-5,
                  causal=True, p=0.0, dtype="bf16"),
}

SWEEP_ROWS = 8192
SWEEP_COLS = (768, 2048, 4096, 8192)
SWEEP_ROPE_HD = 128
SWEEP_ROPE_SEQ = 1024
SWEEP_DROPOUT_P = (0.0, 0.1, 0.5)

BIGVOCAB = dict(rows=8192, V=128256, std=2.0, dtype="bf16")


def block_param_shapes(cfg: dict) -> dict:
    """Leaf parameter shapes of a block stack; weights are [in, out] (y = x @ W)."""
    d, F, V = cfg["d"], cfg["F"], cfg["V"]
    shapes = {"E": (V, d)}
    if cfg["learned_pos"]:
        shapes["P"] = (cfg["S"], d)
    for l in range(cfg["n_layers"]):
        shapes[f"l{l}.g1"] = (d,)
        if cfg["norm"] == "ln":
            shapes[f"l{l}.b1"] = (d,)
        shapes[f"l{l}.Wq"] = (d, d)
        shapes[f"l{l}.Wk"] = (d, d)
        shapes[f"l{l}.Wv"] = (d, d)
        shapes[f"l{l}.Wo"] = (d, d)
        shapes[f"l{l}.g2"] = (d,)
        if cfg["norm"] == "ln":
            shapes[f"l{l}.b2"] = (d,)
        if cfg["mlp"] == "swiglu":
            shapes[f"l{l}.Wg"] = (d, F)
            shapes[f"l{l}.Wu"] = (d, F)
            shapes[f"l{l}.Wd"] = (F, d)
        else:
            shapes[f"l{l}.W1"] = (d, F)
            shapes[f"l{l}.W2"] = (F, d)
    shapes["gf"] = (d,)
    if cfg["norm"] == "ln":
        shapes["bf"] = (d,)
    return shapes


def block_params(cfg: dict, seed: int = SEED_WEIGHTS, gain_jitter: float = 0.0) -> dict:
    """Weights ~ N(0, 0.02); norm gains 1 (+ optional N(0, jitter)); betas 0 (+ jitter).

    Returned values are rounded to the run's storage type and held as float64.
    """
    g = rng(seed)
    out = {}
    for name, shape in block_param_shapes(cfg).items():
        leaf = name.split(".")[-1]
        if leaf.startswith("g") and len(shape) == 1:
            v = np.ones(shape) + (g.normal(0.0, gain_jitter, size=shape) if gain_jitter else 0.0)
        elif leaf.startswith("b") and len(shape) == 1:
            v = np.zeros(shape) + (g.normal(0.0, gain_jitter, size=shape) if gain_jitter else 0.0)
        else:
            v = g.normal(0.0, 0.02, size=shape)
        out[name] = to_storage(v, cfg["dtype"])
    return out


def block_tokens(cfg: dict, seed: int = SEED_TOKENS):
    T = cfg["B"] * cfg["S"]
    g = rng(seed)
    ids = g.integers(0, cfg["V"], size=T, dtype=np.int64).astype(np.int32)
    tgt = g.integers(0, cfg["V"], size=T, dtype=np.int64).astype(np.int32)
    return ids, tgt
