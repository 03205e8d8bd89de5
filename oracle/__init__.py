"""CPU oracle for the pre-norm transformer block forward/backward hot path.

TEST INFRASTRUCTURE ONLY.  Plain, slow, obviously-correct NumPy code in float64
(dropout masks in exact uint64 integer arithmetic).  Only the tests, the smoke
check and the CPU-baseline leg of the benchmark may import it; the product path
(the CUDA library and its Python binding) never does, and this package imports
nothing from the product path.

Sources (cited by page title and section throughout):
  [AE] xtrain "Phase: Autograd Engine + Op Backward — Design Document"
       (docs/03-autograd-engine.md): tape design, per-op backward table,
       RMSNorm / RoPE / softmax / cross-entropy derivations, composed attention,
       validation method.
  [BP] unhomeschool "Träna en språkmodell: Backprop i anpassad CUDA":
       forward pass of the GPT-style stack, forward/backward kernel pairs,
       saved tensors, per-weight gradient buffers, += accumulation.
  [DO] xtrain "Phase T18: Dropout (device RNG + mask) — Design Document"
       (docs/17-dropout.md): counter-based RNG, per-site seeds, train/eval,
       residual-path wiring, validation gates.
  [AD] "从零构建自动微分引擎：对偶数、计算图与反向传播的 Rust 深度实战":
       dual numbers, computation-graph reverse mode, HyperDual.

Parity status: every function here is pinned by a `-m "not gpu"` test against
something other than itself (finite differences, closed forms, printed values,
library routines on special cases, a second engine).  No function is unpinned.
"""
