// Entry points shared between translation units of libxt (not part of the C ABI).
#pragma once

#include "common.cuh"

namespace xt {
// C (+)= alpha·op(A)@op(B) with tf32 staging scratch `ws` (see xt_matmul_workspace_size).
int matmul(const xt_matmul_desc& d, const void* A, const void* B, void* C, void* ws, size_t ws_bytes,
           cudaStream_t s);
size_t matmul_workspace(const xt_matmul_desc& d);

// Cross-entropy over rows split across a cluster of CTAs (ce_split.cu): the cluster size whose
// per-CTA chunk of a row fits shared memory (0: none; *nb: chunk buffers), and one forward +
// backward pass
// (dlogits (+)= upstream·((softmax − onehot)/rows + c_lin + 2·c_sq·x); with sums != null,
// sums[0] = Σx, sums[1] = Σx² over all elements and sums[2] = loss + c_lin·Σx + c_sq·Σx²).
// ws holds rows × (1 + 2·cluster) floats.
int ce_split_cluster(int64_t V, int dt, int* nb = nullptr);
int ce_split_run(const void* logits, const int32_t* targets, float* lse, float* loss, float* sums,
                 const float* upstream, void* dlogits, int64_t rows, int64_t V, int dt, int dt_grad, int acc,
                 float c_lin, float c_sq, void* ws, cudaStream_t s);

}  // namespace xt
