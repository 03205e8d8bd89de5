"""Native block stack from Python: parameter / gradient storage and the xt_block_* calls.

Device buffers are torch tensors (memory and streams only); every step of the forward and
backward runs in libxt through xt_block_fwd / xt_block_bwd.  Weights follow the native
layout: W_qkv = [W_Q | W_K | W_V] ([d, 3d]) and, for SwiGLU, W_up = [W_g | W_u] ([d, 2F]).
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import xt

_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}


def config_struct(cfg: dict, training: bool = True, base_seed: int = 0, grad_dtype: str = "f32") -> xt.BlockConfig:
    c = xt.BlockConfig()
    c.B, c.S, c.d, c.H, c.hd = cfg["B"], cfg["S"], cfg["d"], cfg["H"], cfg["hd"]
    c.F, c.V, c.n_layers = cfg["F"], cfg["V"], cfg["n_layers"]
    c.norm = xt.XT_NORM_RMS if cfg["norm"] == "rms" else xt.XT_NORM_LN
    c.mlp = xt.XT_MLP_SWIGLU if cfg["mlp"] == "swiglu" else xt.XT_MLP_GELU
    c.rope = int(cfg["rope"])
    c.learned_pos = int(cfg["learned_pos"])
    c.causal = 1
    c.training = int(training)
    c.dtype = xt.XT_F32 if cfg["dtype"] == "f32" else xt.XT_BF16
    c.grad_dtype = xt.XT_F32 if grad_dtype == "f32" else xt.XT_BF16
    c.eps = cfg["eps"]
    c.p = cfg["p"]
    c.rope_base = cfg["rope_base"]
    c.base_seed = base_seed & (2**64 - 1)
    c.attention = {"auto": xt.XT_ATTN_AUTO, "composed": xt.XT_ATTN_COMPOSED,
                   "fused": xt.XT_ATTN_FUSED}[cfg.get("attention", "auto")]
    c.recompute = int(cfg.get("recompute", 0))
    return c


class NativeBlock:
    """Owns the parameters, gradients and workspace of one block stack on one device."""

    def __init__(self, cfg: dict, device="cuda", training=True, base_seed=0, grad_dtype="f32"):
        self.cfg = dict(cfg)
        self.device = torch.device(device)
        self.dt = _TORCH[cfg["dtype"]]
        self.gdt = _TORCH[grad_dtype]
        self.c = config_struct(cfg, training, base_seed, grad_dtype)
        L, d, F, V, S = cfg["n_layers"], cfg["d"], cfg["F"], cfg["V"], cfg["S"]
        up = 2 * F if cfg["mlp"] == "swiglu" else F
        ln = cfg["norm"] == "ln"
        z = lambda *shape, dt=self.dt: torch.zeros(shape, dtype=dt, device=self.device)  # noqa: E731
        self.p = {"E": z(V, d), "gf": z(d)}
        if cfg["learned_pos"]:
            self.p["P"] = z(S, d)
        if ln:
            self.p["bf"] = z(d)
        for l in range(L):
            self.p[f"l{l}.g1"] = z(d)
            self.p[f"l{l}.g2"] = z(d)
            if ln:
                self.p[f"l{l}.b1"] = z(d)
                self.p[f"l{l}.b2"] = z(d)
            self.p[f"l{l}.Wqkv"] = z(d, 3 * d)
            self.p[f"l{l}.Wo"] = z(d, d)
            self.p[f"l{l}.Wup"] = z(d, up)
            self.p[f"l{l}.Wdown"] = z(F, d)
        self.g = {k: torch.zeros(v.shape, dtype=self.gdt, device=self.device) for k, v in self.p.items()}
        self._arrays = []
        self.params = self._params_struct()
        nbytes = C.c_size_t(0)
        xt.call("xt_block_workspace_size", C.byref(self.c), C.byref(nbytes))
        # zero-filled: the matmul scratch inside it starts with stream-K flag words
        self.ws = torch.zeros(int(nbytes.value), dtype=torch.uint8, device=self.device)
        self.loss = torch.zeros(1, dtype=torch.float32, device=self.device)

    # -------------------------------------------------------------------------- structs

    def _ptr_array(self, tensors):
        arr = (C.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])
        self._arrays.append(arr)
        return C.cast(arr, C.POINTER(C.c_void_p))

    def _params_struct(self) -> xt.BlockParams:
        L = self.cfg["n_layers"]
        ln = self.cfg["norm"] == "ln"
        p, g = self.p, self.g
        s = xt.BlockParams()
        per = lambda d_, k: self._ptr_array([d_[f"l{l}.{k}"] for l in range(L)])  # noqa: E731
        s.E, s.dE = p["E"].data_ptr(), g["E"].data_ptr()
        if "P" in p:
            s.P, s.dP = p["P"].data_ptr(), g["P"].data_ptr()
        s.gf, s.dgf = p["gf"].data_ptr(), g["gf"].data_ptr()
        if ln:
            s.bf, s.dbf = p["bf"].data_ptr(), g["bf"].data_ptr()
            s.b1, s.db1, s.b2, s.db2 = per(p, "b1"), per(g, "b1"), per(p, "b2"), per(g, "b2")
        s.g1, s.dg1, s.g2, s.dg2 = per(p, "g1"), per(g, "g1"), per(p, "g2"), per(g, "g2")
        s.Wqkv, s.dWqkv = per(p, "Wqkv"), per(g, "Wqkv")
        s.Wo, s.dWo = per(p, "Wo"), per(g, "Wo")
        s.W_up, s.dW_up = per(p, "Wup"), per(g, "Wup")
        s.W_down, s.dW_down = per(p, "Wdown"), per(g, "Wdown")
        return s

    # -------------------------------------------------------------------------- parameters

    def load(self, params: dict):
        """Copies parameters given in the per-matrix naming (Wq, Wk, Wv, Wo, Wg, Wu, Wd / W1, W2,
        g1, b1, g2, b2, E, P, gf, bf) into the native layout."""
        def put(name, arr):
            self.p[name].copy_(torch.tensor(np.asarray(arr, np.float32)).to(self.dt))
        for name in ("E", "P", "gf", "bf"):
            if name in params and name in self.p:
                put(name, params[name])
        for l in range(self.cfg["n_layers"]):
            k = lambda n: params[f"l{l}.{n}"]  # noqa: E731
            for n in ("g1", "g2", "b1", "b2"):
                if f"l{l}.{n}" in self.p:
                    put(f"l{l}.{n}", k(n))
            put(f"l{l}.Wqkv", np.concatenate([k("Wq"), k("Wk"), k("Wv")], axis=1))
            put(f"l{l}.Wo", k("Wo"))
            if self.cfg["mlp"] == "swiglu":
                put(f"l{l}.Wup", np.concatenate([k("Wg"), k("Wu")], axis=1))
                put(f"l{l}.Wdown", k("Wd"))
            else:
                put(f"l{l}.Wup", k("W1"))
                put(f"l{l}.Wdown", k("W2"))

    def grads_named(self) -> dict:
        """Gradients on the host (float64) in the per-matrix naming of `load`."""
        d, F = self.cfg["d"], self.cfg["F"]
        h = {k: v.float().cpu().numpy().astype(np.float64) for k, v in self.g.items()}
        out = {}
        for name in ("E", "P", "gf", "bf"):
            if name in h:
                out[name] = h[name]
        for l in range(self.cfg["n_layers"]):
            for n in ("g1", "g2", "b1", "b2"):
                if f"l{l}.{n}" in h:
                    out[f"l{l}.{n}"] = h[f"l{l}.{n}"]
            qkv = h[f"l{l}.Wqkv"]
            out[f"l{l}.Wq"], out[f"l{l}.Wk"], out[f"l{l}.Wv"] = qkv[:, :d], qkv[:, d:2 * d], qkv[:, 2 * d:]
            out[f"l{l}.Wo"] = h[f"l{l}.Wo"]
            if self.cfg["mlp"] == "swiglu":
                out[f"l{l}.Wg"], out[f"l{l}.Wu"] = h[f"l{l}.Wup"][:, :F], h[f"l{l}.Wup"][:, F:]
                out[f"l{l}.Wd"] = h[f"l{l}.Wdown"]
            else:
                out[f"l{l}.W1"], out[f"l{l}.W2"] = h[f"l{l}.Wup"], h[f"l{l}.Wdown"]
        return out

    # -------------------------------------------------------------------------- steps

    def zero_grads(self, stream=None):
        xt.call("xt_block_zero_grads", C.byref(self.c), C.byref(self.params), xt.stream(stream))

    def forward(self, ids: torch.Tensor, targets: torch.Tensor, stream=None):
        xt.call("xt_block_fwd", C.byref(self.c), C.byref(self.params), ids.data_ptr(), targets.data_ptr(),
                self.loss.data_ptr(), self.ws.data_ptr(), xt.stream(stream))
        return self.loss

    def backward(self, ids: torch.Tensor, targets: torch.Tensor, stream=None):
        xt.call("xt_block_bwd", C.byref(self.c), C.byref(self.params), ids.data_ptr(), targets.data_ptr(),
                self.ws.data_ptr(), xt.stream(stream))

    def step(self, ids, targets, stream=None):
        """One forward + backward (gradients accumulate into the grad buffers)."""
        self.forward(ids, targets, stream)
        self.backward(ids, targets, stream)
        return self.loss

    # -------------------------------------------------------------------------- optimizer

    def init_optimizer(self, lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, max_grad_norm=1.0):
        """AdamW state ([BP] § Optimiser-tillståndet): float32 master weights (the parameters
        themselves when they are float32; for bf16 parameters a float32 copy, the bf16 tensors
        then being the working copy every step rewrites), first and second moments at zero."""
        if self.gdt != torch.float32:
            raise ValueError("the optimizer reads float32 gradients (grad_dtype='f32')")
        self.hyper = dict(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay,
                          max_grad_norm=max_grad_norm)
        self._names = list(self.p)
        self.master = {k: (v if v.dtype == torch.float32 else v.float().contiguous()) for k, v in self.p.items()}
        self.m = {k: torch.zeros(v.shape, dtype=torch.float32, device=self.device) for k, v in self.p.items()}
        self.v = {k: torch.zeros(v.shape, dtype=torch.float32, device=self.device) for k, v in self.p.items()}
        self.opt_step = 0
        self.grad_norm = torch.zeros(1, dtype=torch.float32, device=self.device)
        self._opt_ws = xt.adamw_workspace([self.p[k].numel() for k in self._names], self.device)

    def optimizer_step(self, n_microbatches=1, stream=None):
        """Clipped AdamW over every parameter with the gradients scaled by 1 / n_microbatches
        (the buffers hold the sum over the microbatches); the gradient norm before clipping
        lands in self.grad_norm."""
        self.opt_step += 1
        h = self.hyper
        cfg = xt.adamw_config(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], h["max_grad_norm"],
                              1.0 / n_microbatches, self.opt_step)
        names = self._names
        shadows = None
        if self.dt != torch.float32:
            shadows = [self.p[k] for k in names]
        xt.xt_adamw_step(cfg, [self.master[k] for k in names], [self.g[k] for k in names],
                         [self.m[k] for k in names], [self.v[k] for k in names], shadows=shadows,
                         norm_out=self.grad_norm, ws=self._opt_ws, s=stream)

    def train_step(self, microbatches, stream=None):
        """[BP] § Ackumulation över mikrobatcher: zero the gradients, forward + backward every
        microbatch (each backward adds into the buffers), one optimizer step on the average.
        Returns the microbatch losses (device tensors)."""
        self.zero_grads(stream)
        losses = []
        for ids, targets in microbatches:
            self.forward(ids, targets, stream)
            losses.append(self.loss.clone())
            self.backward(ids, targets, stream)
        self.optimizer_step(len(microbatches), stream)
        return losses
