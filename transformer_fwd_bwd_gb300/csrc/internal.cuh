// Entry points shared between translation units of libxt (not part of the C ABI).
#pragma once

#include "common.cuh"

namespace xt {
// C (+)= alpha·op(A)@op(B) with tf32 staging scratch `ws` (see xt_matmul_workspace_size).
int matmul(const xt_matmul_desc& d, const void* A, const void* B, void* C, void* ws, size_t ws_bytes,
           cudaStream_t s);
size_t matmul_workspace(const xt_matmul_desc& d);

}  // namespace xt
