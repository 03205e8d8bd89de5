// Shared helpers of libxt: status reporting, dtype conversion, 16-byte vector access,
// warp / row-group reductions, device facts.
#pragma once

#include <cmath>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <utility>
#include <cstdio>

#include "../../include/xt.h"

namespace xt {

// ------------------------------------------------------------------------------ host status

// Records the message for xt_last_error() and returns `code`.
int fail(int code, const char* fmt, ...);
// Maps the last CUDA launch error (if any) to XT_ERR_CUDA.
int check_launch(const char* what);
// Device address of the error flag word on the current device.
uint32_t* errflag();
// Multiprocessor count of the current device (cached per device).
int num_sms();
// Limit of the kernels' bounded waits on work, in ns (xt_set_wait_limit_ns; default 2 s).
uint64_t wait_limit_ns();
// GEMM timing hooks (active only between xt_profile_gemm(capacity > 0) and (0)): a record per
// GEMM launch and its timestamp region, kProfSlots pairs of words: [0, kProfGemmSlots) for
// the GEMM kernel's CTAs, the rest for a K split's reduce kernel.  Each CTA writes
// (start, end) %globaltimer words at 2·cta.
constexpr int kProfGemmSlots = 256;
constexpr int kProfSlots = 2048;
bool gemm_profile_begin(double flops, const int* shape, unsigned long long** ts, void** token);
void gemm_profile_grids(void* token, int grid, int rgrid);

#define XT_REQUIRE(cond, ...)                                      \
  do {                                                             \
    if (!(cond)) return ::xt::fail(XT_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)

#define XT_TRY(expr)              \
  do {                            \
    int _st = (expr);             \
    if (_st != XT_OK) return _st; \
  } while (0)

// Launches `kernel` on `s` with programmatic stream serialization allowed (see pdl_begin).
template <typename... KArgs, typename... Args>
inline void launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// As launch(), as clusters of `cluster_x` CTAs along x (gridDim.x a multiple of it).
template <typename... KArgs, typename... Args>
inline void launch_clustered(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             int cluster_x, Args&&... args) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = unsigned(cluster_x);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

inline bool valid_dtype(int dt) { return dt == XT_F32 || dt == XT_BF16; }
inline size_t dtype_size(int dt) { return dt == XT_BF16 ? 2 : 4; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------------------------------ device: dtype

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

// 16-byte vector of T: VW = 4 floats or 8 bf16.
template <typename T> struct Vec;
template <> struct Vec<float> {
  static constexpr int W = 4;
  __device__ __forceinline__ static void load(const float* p, float (&v)[4]) {
    float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  __device__ __forceinline__ static void load_nc(const float* p, float (&v)[4]) {
    float4 q = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  __device__ __forceinline__ static void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <> struct Vec<bf16> {
  static constexpr int W = 8;
  __device__ __forceinline__ static void unpack(const uint4& q, float (&v)[8]) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ __forceinline__ static void load(const bf16* p, float (&v)[8]) {
    unpack(*reinterpret_cast<const uint4*>(p), v);
  }
  __device__ __forceinline__ static void load_nc(const bf16* p, float (&v)[8]) {
    unpack(__ldg(reinterpret_cast<const uint4*>(p)), v);
  }
  __device__ __forceinline__ static void store(bf16* p, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// 8 elements at a time for any storage type (fp32: two 16-byte loads, bf16: one).
template <typename T> struct V8;
template <> struct V8<float> {
  __device__ __forceinline__ static void load(const float* p, float (&v)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  __device__ __forceinline__ static void store(float* p, const float (&v)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
};
template <> struct V8<bf16> {
  __device__ __forceinline__ static void load(const bf16* p, float (&v)[8]) { Vec<bf16>::load(p, v); }
  __device__ __forceinline__ static void store(bf16* p, const float (&v)[8]) { Vec<bf16>::store(p, v); }
};

// Generic access with a vector width VW of 1 (scalar path for ragged or misaligned data),
// 4 (fp32, one 16-byte access) or 8 (any type; 16-byte aligned).
template <typename T, int VW> struct Acc {
  __device__ __forceinline__ static void load(const T* p, float (&v)[VW]) {
    if constexpr (VW == 1) v[0] = to_f(p[0]);
    else if constexpr (VW == 8) V8<T>::load(p, v);
    else Vec<T>::load(p, v);
  }
  __device__ __forceinline__ static void store(T* p, const float (&v)[VW]) {
    if constexpr (VW == 1) p[0] = from_f<T>(v[0]);
    else if constexpr (VW == 8) V8<T>::store(p, v);
    else Vec<T>::store(p, v);
  }
};

// ------------------------------------------------------------------------------ reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Reduction over a row group of `tpr` consecutive threads (tpr a power of two, 32..1024;
// groups are warp aligned).  `red` is shared scratch of blockDim/32 floats.  Every thread
// of the group gets the result.  All threads of the block must call it together.
template <bool MAX>
__device__ __forceinline__ float group_reduce(float v, int tpr, float* red) {
  v = MAX ? warp_max(v) : warp_sum(v);
  if (tpr <= 32) return v;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpg = tpr >> 5;                 // warps per group
  const int g0 = (warp / wpg) * wpg;        // first warp of this group
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[g0];
  for (int w = 1; w < wpg; ++w) r = MAX ? fmaxf(r, red[g0 + w]) : r + red[g0 + w];
  return r;
}

// Online-softmax pair (running max m, running Σ exp(x − m)).
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float mm = fmaxf(m, m2);
  if (mm == -INFINITY) { m = mm; s = 0.f; return; }
  s = s * expf(m - mm) + s2 * expf(m2 - mm);
  m = mm;
}

// [DO] § RNG：counter-based.  splitmix64 (Steele, Lea & Flood) from state `key`; the keep
// decision uses the top 24 bits only.  The final `z ^ (z >> 31)` step of the mixer leaves
// bits 63..40 unchanged (z >> 31 has its top 31 bits clear), so it is omitted.
__device__ __forceinline__ bool dropout_keep(uint64_t seed, uint64_t i, float p) {
  uint64_t z = seed ^ (i * 0x9E3779B97F4A7C15ull);
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  const float u = static_cast<float>(static_cast<uint32_t>(z >> 40)) * 0x1.0p-24f;
  return u >= p;
}

// The same decision as an integer test: with k = z >> 40 (an integer below 2²⁴, so k·2⁻²⁴ and
// p·2²⁴ are exact in float), k·2⁻²⁴ ≥ p ⟺ k ≥ ⌈p·2²⁴⌉ ⟺ z ≥ ⌈p·2²⁴⌉·2⁴⁰ — the threshold
// dropout_threshold(p).  Eight consecutive counters i0 .. i0 + 7 share one multiply: the
// counter's i·γ is i0·γ + j·γ (mod 2⁶⁴).
inline uint64_t dropout_threshold(float p) {
  return static_cast<uint64_t>(std::ceil(static_cast<double>(p) * 16777216.0)) << 40;
}
// Only the high word of the last product is formed (the threshold's low 40 bits are zero, so
// z ≥ thr ⟺ z >> 32 ≥ thr >> 32): hi32(y·C) = umulhi(y_lo, C_lo) + y_lo·C_hi + y_hi·C_lo (mod 2³²).
__device__ __forceinline__ uint32_t dropout_keep8(uint64_t seed, uint64_t i0, uint64_t thr) {
  constexpr uint64_t kG = 0x9E3779B97F4A7C15ull;
  constexpr uint32_t kC2lo = 0x133111EBu, kC2hi = 0x94D049BBu;
  const uint32_t thr_hi = uint32_t(thr >> 32);
  const uint64_t base = i0 * kG;
  uint32_t bits = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint64_t z = (seed ^ (base + uint64_t(j) * kG)) + kG;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    const uint64_t y = z ^ (z >> 27);
    const uint32_t ylo = uint32_t(y), yhi = uint32_t(y >> 32);
    const uint32_t hi = __umulhi(ylo, kC2lo) + ylo * kC2hi + yhi * kC2lo;
    bits |= (hi >= thr_hi ? 1u : 0u) << j;
  }
  return bits;
}

// Φ(x) = ½·erfc(−x/√2) (no cancellation for x ≪ 0, unlike ½(1 + erf(x/√2))), with erfc from the
// Chebyshev-fitted form of Press, Teukolsky, Vetterling & Flannery, Numerical Recipes (§6.2,
// erfcc): for z ≥ 0, erfc(z) = t·exp(−z² + P(t)), t = 1/(1 + z/2), P a degree-9 polynomial in t;
// fractional error below 1.2e-7 for every z, and erfc(−z) = 2 − erfc(z).  One reciprocal, one
// exponential and nine FMAs.  The backward also needs φ(x) = exp(−x²/2)/√(2π) = exp(−z²)/√(2π),
// so both come out of one evaluation.
struct Gauss {
  float cdf, pdf;
};
// t and P(t) of the erfc form for z = |x|/√2.
__device__ __forceinline__ float erfc_poly(float z, float& t) {
  t = __fdividef(1.f, fmaf(0.5f, z, 1.f));
  float q = 0.17087277f;
  q = fmaf(q, t, -0.82215223f);
  q = fmaf(q, t, 1.48851587f);
  q = fmaf(q, t, -1.13520398f);
  q = fmaf(q, t, 0.27886807f);
  q = fmaf(q, t, -0.18628806f);
  q = fmaf(q, t, 0.09678418f);
  q = fmaf(q, t, 0.37409196f);
  q = fmaf(q, t, 1.00002368f);
  return fmaf(q, t, -1.26551223f);
}
// Two fp32 lanes in one 64-bit register for the paired FP32 instructions of sm_100+ (PTX
// fma.rn.f32x2): each lane is rounded as the scalar fma.rn.f32 rounds it, so a pair of Horner
// chains evaluated this way is bit-identical to two scalar chains, in half the issue slots.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// erfc_poly for two arguments at once (the same operations, the Horner steps paired).
__device__ __forceinline__ void erfc_poly2(float z0, float z1, float& t0, float& t1, float& q0, float& q1) {
  t0 = __fdividef(1.f, fmaf(0.5f, z0, 1.f));
  t1 = __fdividef(1.f, fmaf(0.5f, z1, 1.f));
  const uint64_t t = f32x2_pack(t0, t1);
  constexpr float c[9] = {-0.82215223f, 1.48851587f, -1.13520398f, 0.27886807f, -0.18628806f,
                          0.09678418f,  0.37409196f, 1.00002368f,  -1.26551223f};
  uint64_t q = f32x2_pack(0.17087277f, 0.17087277f);
#pragma unroll
  for (int k = 0; k < 9; ++k) q = f32x2_fma(q, t, f32x2_pack(c[k], c[k]));
  f32x2_unpack(q, q0, q1);
}
// Φ alone: one reciprocal and one exponential.
__device__ __forceinline__ float gelu_cdf(float x) {
  const float z = fabsf(x) * 0.70710678118654752f;
  float t;
  const float q = erfc_poly(z, t);
  const float half_erfc = 0.5f * t * __expf(fmaf(-z, z, q));  // ½·erfc(|x|/√2) = Φ(−|x|)
  return x <= 0.f ? half_erfc : 1.f - half_erfc;
}
// Φ and φ: φ needs exp(−x²/2) on its own, so one more exponential.
__device__ __forceinline__ Gauss gauss(float x) {
  const float z = fabsf(x) * 0.70710678118654752f;
  float t;
  const float q = erfc_poly(z, t);
  const float e = __expf(-z * z);                    // exp(−x²/2)
  const float half_erfc = 0.5f * t * e * __expf(q);  // ½·erfc(|x|/√2) = Φ(−|x|)
  return Gauss{x <= 0.f ? half_erfc : 1.f - half_erfc, 0.39894228040143268f * e};
}
// gelu(x) = x·Φ(x) (MODE 0) or d·gelu′(x) = d·(Φ(x) + x·φ(x)) (MODE 1) for a pair, with the
// expressions of gelu_cdf / gauss around the paired polynomial.
template <int MODE>
__device__ __forceinline__ void gelu_pair(float x0, float x1, float d0, float d1, float& r0, float& r1) {
  const float z0 = fabsf(x0) * 0.70710678118654752f, z1 = fabsf(x1) * 0.70710678118654752f;
  float t0, t1, q0, q1;
  erfc_poly2(z0, z1, t0, t1, q0, q1);
  if constexpr (MODE == 0) {
    const float h0 = 0.5f * t0 * __expf(fmaf(-z0, z0, q0));
    const float h1 = 0.5f * t1 * __expf(fmaf(-z1, z1, q1));
    r0 = x0 * (x0 <= 0.f ? h0 : 1.f - h0);
    r1 = x1 * (x1 <= 0.f ? h1 : 1.f - h1);
  } else {
    const float e0 = __expf(-z0 * z0), e1 = __expf(-z1 * z1);
    const float h0 = 0.5f * t0 * e0 * __expf(q0), h1 = 0.5f * t1 * e1 * __expf(q1);
    const float c0 = x0 <= 0.f ? h0 : 1.f - h0, c1 = x1 <= 0.f ? h1 : 1.f - h1;
    r0 = d0 * fmaf(x0, 0.39894228040143268f * e0, c0);
    r1 = d1 * fmaf(x1, 0.39894228040143268f * e1, c1);
  }
}


// N GELU evaluations at once, phase by phase (every phase is N independent operations, so a
// single warp keeps its pipes busy instead of waiting on one dependent chain per element).
// MODE 0: out = x·Φ(x); MODE 1: out = Φ(x) + x·φ(x) (the derivative).
template <int N, int MODE>
__device__ __forceinline__ void gelu_batch(const float (&x)[N], float (&out)[N]) {
  float z[N], t[N], q[N];
#pragma unroll
  for (int i = 0; i < N; ++i) z[i] = fabsf(x[i]) * 0.70710678118654752f;
#pragma unroll
  for (int i = 0; i < N; ++i) t[i] = __fdividef(1.f, fmaf(0.5f, z[i], 1.f));
#pragma unroll
  for (int i = 0; i < N; ++i) q[i] = fmaf(0.17087277f, t[i], -0.82215223f);
  constexpr float c[8] = {1.48851587f, -1.13520398f, 0.27886807f, -0.18628806f,
                          0.09678418f, 0.37409196f,  1.00002368f, -1.26551223f};
#pragma unroll
  for (int k = 0; k < 8; ++k)
#pragma unroll
    for (int i = 0; i < N; ++i) q[i] = fmaf(q[i], t[i], c[k]);
  if constexpr (MODE == 0) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float he = 0.5f * t[i] * __expf(fmaf(-z[i], z[i], q[i]));
      out[i] = x[i] * (x[i] <= 0.f ? he : 1.f - he);
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float e = __expf(-z[i] * z[i]);
      const float he = 0.5f * t[i] * e * __expf(q[i]);
      const float cdf = x[i] <= 0.f ? he : 1.f - he;
      out[i] = fmaf(x[i], 0.39894228040143268f * e, cdf);
    }
  }
}

// Programmatic dependent launch.  Every kernel is launched with programmatic stream
// serialization (launch() below), so it can be resident while its predecessor on the stream
// drains; pdl_begin() is each kernel's first statement: it waits until the predecessor has
// completed and its writes are visible (immediate when there is none), then lets the successor
// be scheduled.  Nothing a kernel does precedes the wait.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Split form of pdl_begin() for kernels whose set-up touches nothing a predecessor writes:
// the set-up runs before pdl_wait(), overlapping the predecessor's drain when the CTA is
// already resident.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void flag_error(uint32_t* flag, uint32_t bit) {
  if (flag) atomicOr(flag, bit);
}

}  // namespace xt
