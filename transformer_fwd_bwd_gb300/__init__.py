"""GB300-native forward / analytic-backward kernels of a pre-norm transformer block.

`xt` is the ctypes binding of libxt.so (include/xt.h); `tape` is the reverse-mode tape
that drives the per-op kernels; `block` runs the native whole-stack path.
"""
