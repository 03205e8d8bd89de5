// FP8 E4M3 path ([BP] § Vad generiska ramverk kostar, item 4: an FP8 E4M3 tensor-core path in
// the mixed-precision pipeline): per-tensor quantization to e4m3 and the GEMM on e4m3
// operands (tcgen05 kind::f8f6f4, K-major A [M, K] and B [N, K], float32 accumulation), whose
// epilogue multiplies by the operands' dequantization factors read from device memory.
#include <cuda_fp8.h>

#include "gemm.cuh"
#include "internal.cuh"

namespace xt {
namespace gemm {

int launch_fp8(int bn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tc2,
               const Params& p, int grid, cudaStream_t s) {
  switch (bn) {
    case 128: return launch_one<kFp8, 128, false, false>(ta, tb, tc, tc2, p, grid, s);
    case 256: return launch_one<kFp8, 256, false, false>(ta, tb, tc, tc2, p, grid, s);
    default: return fail(XT_ERR_UNSUPPORTED, "gemm fp8: tile width %d", bn);
  }
}

}  // namespace gemm

namespace {

constexpr int kQThreads = 256;
constexpr float kE4M3Max = 448.f;

// Per-block max |x| of a grid-stride share (max is exact, so any order gives the same value).
template <typename T>
__global__ void __launch_bounds__(kQThreads) amax_partials(const T* __restrict__ x, int64_t n, float* __restrict__ part) {
  pdl_begin();
  __shared__ float sh[kQThreads];
  float m = 0.f;
  for (int64_t i = int64_t(blockIdx.x) * kQThreads + threadIdx.x; i < n; i += int64_t(gridDim.x) * kQThreads)
    m = fmaxf(m, fabsf(to_f(x[i])));
  sh[threadIdx.x] = m;
  __syncthreads();
  for (int w = kQThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) sh[threadIdx.x] = fmaxf(sh[threadIdx.x], sh[threadIdx.x + w]);
    __syncthreads();
  }
  if (threadIdx.x == 0) part[blockIdx.x] = sh[0];
}

// amax from the partials (every block forms the same value), scale = 448 / amax, codes =
// e4m3(x·scale) rounded to nearest even and saturated; block 0 writes the dequantization
// factor amax / 448 (1 when amax = 0).
template <typename T>
__global__ void __launch_bounds__(kQThreads) quantize_e4m3(const T* __restrict__ x, int64_t n,
                                                           const float* __restrict__ part, int nparts,
                                                           uint8_t* __restrict__ out, float* __restrict__ dequant) {
  pdl_begin();
  __shared__ float sh[kQThreads];
  float m = 0.f;
  for (int i = threadIdx.x; i < nparts; i += kQThreads) m = fmaxf(m, part[i]);
  sh[threadIdx.x] = m;
  __syncthreads();
  for (int w = kQThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) sh[threadIdx.x] = fmaxf(sh[threadIdx.x], sh[threadIdx.x + w]);
    __syncthreads();
  }
  const float amax = sh[0];
  const float scale = amax > 0.f ? kE4M3Max / amax : 1.f;
  if (blockIdx.x == 0 && threadIdx.x == 0) *dequant = amax > 0.f ? amax / kE4M3Max : 1.f;
  for (int64_t i = int64_t(blockIdx.x) * kQThreads + threadIdx.x; i < n; i += int64_t(gridDim.x) * kQThreads)
    out[i] = __nv_cvt_float_to_fp8(to_f(x[i]) * scale, __NV_SATFINITE, __NV_E4M3);
}

int quant_blocks(int64_t n) {
  const int64_t b = ceil_div(n, kQThreads * 8);
  const int64_t cap = int64_t(num_sms()) * 8;
  return int(b < 1 ? 1 : b > cap ? cap : b);
}

}  // namespace
}  // namespace xt

using namespace xt;

extern "C" {

int xt_quantize_fp8_workspace_size(int64_t n, size_t* bytes) {
  XT_REQUIRE(n >= 0 && bytes, "xt_quantize_fp8_workspace_size: bad arguments");
  *bytes = (size_t(quant_blocks(n)) * 4 + 255) & ~size_t(255);
  return XT_OK;
}

int xt_quantize_fp8(const void* x, int64_t n, int dt, uint8_t* out, float* dequant, void* ws, size_t ws_bytes,
                    void* stream) {
  XT_REQUIRE(n >= 0, "xt_quantize_fp8: n < 0");
  XT_REQUIRE(valid_dtype(dt), "xt_quantize_fp8: bad dtype");
  XT_REQUIRE(dequant != nullptr, "xt_quantize_fp8: dequant is NULL");
  XT_REQUIRE(n == 0 || (x && out), "xt_quantize_fp8: NULL pointer");
  size_t need = 0;
  XT_TRY(xt_quantize_fp8_workspace_size(n, &need));
  XT_REQUIRE(ws && ws_bytes >= need, "xt_quantize_fp8: workspace too small (%zu < %zu)", ws_bytes, need);
  cudaStream_t s = as_stream(stream);
  const int nb = quant_blocks(n);
  float* part = static_cast<float*>(ws);
  if (dt == XT_BF16) {
    launch(amax_partials<bf16>, nb, kQThreads, 0, s, static_cast<const bf16*>(x), n, part);
    XT_TRY(check_launch("xt_quantize_fp8 (amax)"));
    launch(quantize_e4m3<bf16>, nb, kQThreads, 0, s, static_cast<const bf16*>(x), n,
           static_cast<const float*>(part), nb, out, dequant);
  } else {
    launch(amax_partials<float>, nb, kQThreads, 0, s, static_cast<const float*>(x), n, part);
    XT_TRY(check_launch("xt_quantize_fp8 (amax)"));
    launch(quantize_e4m3<float>, nb, kQThreads, 0, s, static_cast<const float*>(x), n,
           static_cast<const float*>(part), nb, out, dequant);
  }
  return check_launch("xt_quantize_fp8");
}

int xt_matmul_fp8_fwd(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda, const uint8_t* B, int64_t ldb,
                      void* C, int64_t ldc, int dt_c, float alpha, const float* scale_a, const float* scale_b,
                      int accumulate, void* stream) {
  XT_REQUIRE(M >= 0 && N >= 0 && K >= 0, "xt_matmul_fp8_fwd: negative size");
  XT_REQUIRE(valid_dtype(dt_c), "xt_matmul_fp8_fwd: bad output dtype");
  XT_REQUIRE(accumulate == 0 || accumulate == 1, "xt_matmul_fp8_fwd: accumulate must be 0 or 1");
  if (M == 0 || N == 0) return XT_OK;
  XT_REQUIRE(K > 0, "xt_matmul_fp8_fwd: K must be positive");
  XT_REQUIRE(A && B && C, "xt_matmul_fp8_fwd: NULL pointer");
  XT_REQUIRE(lda >= K && ldb >= K && ldc >= N, "xt_matmul_fp8_fwd: leading dimension too small");
  XT_REQUIRE(M < (int64_t(1) << 31) && N < (int64_t(1) << 31) && K < (int64_t(1) << 31),
             "xt_matmul_fp8_fwd: size above 2^31");
  const int64_t ec = int64_t(dtype_size(dt_c));
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || lda % 16 || ldb % 16 || (ldc * ec) % 16)
    return fail(XT_ERR_ALIGNMENT, "xt_matmul_fp8_fwd: A, B, C and the row strides must be 16-byte aligned");
  gemm::Problem pb{};
  pb.tf32 = false;
  pb.fp8 = true;
  pb.scale_a = scale_a;
  pb.scale_b = scale_b;
  pb.M = M;
  pb.N = N;
  pb.K = K;
  pb.batch_inner = pb.batch_outer = 1;
  pb.A = gemm::Operand{A, false, M, K, lda, 0, 0, 1, 1};
  pb.B = gemm::Operand{B, false, N, K, ldb, 0, 0, 1, 1};
  pb.C = C;
  pb.ldc = ldc;
  pb.c_bf16 = dt_c == XT_BF16;
  pb.alpha = alpha;
  pb.accumulate = accumulate;
  pb.causal = 0;
  pb.split_ws = nullptr;
  pb.split_ws_bytes = 0;
  pb.sk_flags = nullptr;
  return gemm::run(pb, as_stream(stream));
}

}  // extern "C"
