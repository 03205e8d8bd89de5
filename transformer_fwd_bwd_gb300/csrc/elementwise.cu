// Elementwise ops: accumulate, add, mul, scale, sum, silu, gelu, swiglu, dropout, add_bias.
// All are HBM-bound streaming kernels: 8 elements per thread per step (fp32: two 16-byte
// accesses, bf16: one), grid-stride loops over a grid of a few waves, a scalar tail.
#include <math_constants.h>

#include "common.cuh"

namespace xt {

enum EwOp {
  EW_ACC,         // o0 += a
  EW_ADD,         // o0 = a + b
  EW_COPY2,       // o0 = a, o1 = a              (add backward)
  EW_MUL,         // o0 = a * b
  EW_MUL_BWD,     // o0 = a * c, o1 = a * b      (a = d, b = x, c = y)
  EW_SCALE,       // o0 = alpha * a
  EW_SILU,        // o0 = silu(a)
  EW_SILU_BWD,    // o0 = a * silu'(b)           (a = d, b = x)
  EW_GELU,        // o0 = gelu(a)
  EW_GELU_BWD,    // o0 = a * gelu'(b)
  EW_DROPOUT,     // o0 = keep ? a * scale : 0
  EW_DROPOUT_ADD, // o0 = a + (keep ? b * scale : 0)
  EW_FILL,        // o0 = *scalar
};

struct EwArgs {
  const void* a;
  const void* b;
  const void* c;
  void* o0;
  void* o1;
  int64_t n;
  float alpha;
  float p;
  float dscale;
  uint64_t seed;
  uint64_t thr;  // dropout_threshold(p)
  int acc0, acc1;
  const float* scalar;
};

// σ(x) = 1/(1 + e^(−x)) with the hardware exponential (ex2.approx of −x·log2 e: relative error
// ≲ |x|·2⁻²⁴ from rounding the argument, ≈ 5e-6 at the edge of the fp32 range) and the
// correctly rounded reciprocal, inside the fp32 ops' 1e-5 bound.
__device__ __forceinline__ float sigmoidf_(float x) { return __frcp_rn(1.f + __expf(-x)); }

template <EwOp OP>
__device__ __forceinline__ void ew_apply(float a, float b, float c, uint64_t i, const EwArgs& g,
                                         float& r0, float& r1) {
  if constexpr (OP == EW_ACC) {
    r0 = a;
  } else if constexpr (OP == EW_ADD) {
    r0 = a + b;
  } else if constexpr (OP == EW_COPY2) {
    r0 = a; r1 = a;
  } else if constexpr (OP == EW_MUL) {
    r0 = a * b;
  } else if constexpr (OP == EW_MUL_BWD) {
    r0 = a * c; r1 = a * b;
  } else if constexpr (OP == EW_SCALE) {
    r0 = a * g.alpha;
  } else if constexpr (OP == EW_SILU) {
    r0 = a * sigmoidf_(a);
  } else if constexpr (OP == EW_SILU_BWD) {
    const float s = sigmoidf_(b);
    r0 = a * (s + b * s * (1.f - s));
  } else if constexpr (OP == EW_GELU) {
    r0 = a * gelu_cdf(a);
  } else if constexpr (OP == EW_GELU_BWD) {
    const Gauss g = gauss(b);
    r0 = a * fmaf(b, g.pdf, g.cdf);
  } else if constexpr (OP == EW_DROPOUT) {
    r0 = dropout_keep(g.seed, i, g.p) ? a * g.dscale : 0.f;
  } else if constexpr (OP == EW_DROPOUT_ADD) {
    r0 = a + (dropout_keep(g.seed, i, g.p) ? b * g.dscale : 0.f);
  } else if constexpr (OP == EW_FILL) {
    r0 = *g.scalar;
  }
}

template <EwOp OP> struct EwIO {
  static constexpr bool B = OP == EW_ADD || OP == EW_MUL || OP == EW_MUL_BWD || OP == EW_SILU_BWD ||
                            OP == EW_GELU_BWD || OP == EW_DROPOUT_ADD;
  static constexpr bool C = OP == EW_MUL_BWD;
  static constexpr bool A = OP != EW_FILL;
  static constexpr bool TWO_OUT = OP == EW_COPY2 || OP == EW_MUL_BWD;
};

// Eight elements as loaded: one 16-byte word of bf16, two of fp32; unpacked per element.
template <typename T> struct Raw8;
template <> struct Raw8<bf16> {
  uint4 q;
  __device__ __forceinline__ void load(const bf16* p) { q = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ float get(int j) const {
    const uint32_t w = j < 2 ? q.x : j < 4 ? q.y : j < 6 ? q.z : q.w;
    return __uint_as_float((j & 1) ? (w & 0xffff0000u) : (w << 16));
  }
};
template <> struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = reinterpret_cast<const float4*>(p)[0];
    b = reinterpret_cast<const float4*>(p)[1];
  }
  __device__ __forceinline__ float get(int j) const {
    const float4& f = j < 4 ? a : b;
    const int k = j & 3;
    return k == 0 ? f.x : k == 1 ? f.y : k == 2 ? f.z : f.w;
  }
};

template <EwOp OP, typename TI, typename TO, bool VEC>
__global__ void __launch_bounds__(256, 4) ew_kernel(EwArgs g) {
  pdl_begin();
  using IO = EwIO<OP>;
  const TI* a = static_cast<const TI*>(g.a);
  const TI* b = static_cast<const TI*>(g.b);
  const TI* c = static_cast<const TI*>(g.c);
  TO* o0 = static_cast<TO*>(g.o0);
  TO* o1 = static_cast<TO*>(g.o1);
  const bool acc0 = OP == EW_ACC || g.acc0;
  const bool acc1 = g.acc1;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if constexpr (VEC) {
    const int64_t nv = g.n / 8;
    // The plain streaming ops take U vectors per thread per step, all loads issued before any is
    // used, so an SM keeps U times the bytes in flight; GELU (bound by its erfc arithmetic) and
    // fp32 dropout keep one, as their registers set their occupancy; bf16 dropout two.
    constexpr int U = (OP == EW_GELU || OP == EW_GELU_BWD) ? 1
                      : (OP == EW_DROPOUT || OP == EW_DROPOUT_ADD) ? (sizeof(TI) == 2 ? 2 : 1)
                      : OP == EW_MUL_BWD ? (sizeof(TI) == 2 ? 2 : 1) : 16 / int(sizeof(TI)) / 2;
    if constexpr (U > 1) {
      for (int64_t v0 = t; v0 < nv; v0 += U * stride) {
        // raw 16-byte words: the loads of all U vectors are in flight before any is unpacked
        Raw8<TI> ra[U], rb[U], rc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t v = v0 + int64_t(u) * stride;
          if (v < nv) {
            if constexpr (IO::A) ra[u].load(a + v * 8);
            if constexpr (IO::B) rb[u].load(b + v * 8);
            if constexpr (IO::C) rc[u].load(c + v * 8);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t v = v0 + int64_t(u) * stride;
          if (v >= nv) break;
          const int64_t i0 = v * 8;
          float r0[8], r1[8];
          if constexpr (OP == EW_DROPOUT || OP == EW_DROPOUT_ADD) {
            const uint32_t keep = dropout_keep8(g.seed, uint64_t(i0), g.thr);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if constexpr (OP == EW_DROPOUT) r0[j] = ((keep >> j) & 1u) ? ra[u].get(j) * g.dscale : 0.f;
              else r0[j] = ra[u].get(j) + (((keep >> j) & 1u) ? rb[u].get(j) * g.dscale : 0.f);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              ew_apply<OP>(IO::A ? ra[u].get(j) : 0.f, IO::B ? rb[u].get(j) : 0.f, IO::C ? rc[u].get(j) : 0.f,
                           uint64_t(i0 + j), g, r0[j], r1[j]);
          }
          if (o0) {
            if (acc0) {
              float old[8];
              V8<TO>::load(o0 + i0, old);
#pragma unroll
              for (int j = 0; j < 8; ++j) r0[j] += old[j];
            }
            V8<TO>::store(o0 + i0, r0);
          }
          if constexpr (IO::TWO_OUT) {
            if (o1) {
              if (acc1) {
                float old[8];
                V8<TO>::load(o1 + i0, old);
#pragma unroll
                for (int j = 0; j < 8; ++j) r1[j] += old[j];
              }
              V8<TO>::store(o1 + i0, r1);
            }
          }
        }
      }
    } else
    for (int64_t v = t; v < nv; v += stride) {
      const int64_t i0 = v * 8;
      float va[8] = {}, vb[8] = {}, vc[8] = {}, r0[8], r1[8];
      if constexpr (IO::A) V8<TI>::load(a + i0, va);
      if constexpr (IO::B) V8<TI>::load(b + i0, vb);
      if constexpr (IO::C) V8<TI>::load(c + i0, vc);
      if constexpr (OP == EW_GELU) {
#pragma unroll
        for (int j = 0; j < 8; j += 2) gelu_pair<0>(va[j], va[j + 1], 0.f, 0.f, r0[j], r0[j + 1]);
      } else if constexpr (OP == EW_DROPOUT || OP == EW_DROPOUT_ADD) {
        const uint32_t keep = dropout_keep8(g.seed, uint64_t(i0), g.thr);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if constexpr (OP == EW_DROPOUT) r0[j] = ((keep >> j) & 1u) ? va[j] * g.dscale : 0.f;
          else r0[j] = va[j] + (((keep >> j) & 1u) ? vb[j] * g.dscale : 0.f);
        }
      } else if constexpr (OP == EW_GELU_BWD) {
#pragma unroll
        for (int j = 0; j < 8; j += 2) gelu_pair<1>(vb[j], vb[j + 1], va[j], va[j + 1], r0[j], r0[j + 1]);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) ew_apply<OP>(va[j], vb[j], vc[j], uint64_t(i0 + j), g, r0[j], r1[j]);
      }
      if (o0) {
        if (acc0) {
          float old[8];
          V8<TO>::load(o0 + i0, old);
#pragma unroll
          for (int j = 0; j < 8; ++j) r0[j] += old[j];
        }
        V8<TO>::store(o0 + i0, r0);
      }
      if constexpr (IO::TWO_OUT) {
        if (o1) {
          if (acc1) {
            float old[8];
            V8<TO>::load(o1 + i0, old);
#pragma unroll
            for (int j = 0; j < 8; ++j) r1[j] += old[j];
          }
          V8<TO>::store(o1 + i0, r1);
        }
      }
    }
    t += (g.n / 8) * 8;  // scalar tail starts after the vectors
    for (int64_t i = t; i < g.n; i += stride) {
      float r0 = 0.f, r1 = 0.f;
      ew_apply<OP>(IO::A ? to_f(a[i]) : 0.f, IO::B ? to_f(b[i]) : 0.f, IO::C ? to_f(c[i]) : 0.f,
                   uint64_t(i), g, r0, r1);
      if (o0) o0[i] = from_f<TO>(acc0 ? r0 + to_f(o0[i]) : r0);
      if (IO::TWO_OUT && o1) o1[i] = from_f<TO>(acc1 ? r1 + to_f(o1[i]) : r1);
    }
  } else {
    for (int64_t i = t; i < g.n; i += stride) {
      float r0 = 0.f, r1 = 0.f;
      ew_apply<OP>(IO::A ? to_f(a[i]) : 0.f, IO::B ? to_f(b[i]) : 0.f, IO::C ? to_f(c[i]) : 0.f,
                   uint64_t(i), g, r0, r1);
      if (o0) o0[i] = from_f<TO>(acc0 ? r0 + to_f(o0[i]) : r0);
      if (IO::TWO_OUT && o1) o1[i] = from_f<TO>(acc1 ? r1 + to_f(o1[i]) : r1);
    }
  }
}

static int grid_for(int64_t work_items) {
  const int64_t want = ceil_div(work_items, 256);
  const int64_t cap = int64_t(num_sms()) * 8;
  return int(want < 1 ? 1 : (want > cap ? cap : want));
}

template <EwOp OP, typename TI, typename TO>
static int ew_run(const EwArgs& g, cudaStream_t s, const char* name) {
  if (g.n <= 0) return XT_OK;
  const bool vec = aligned16(g.a) && aligned16(g.b) && aligned16(g.c) && aligned16(g.o0) &&
                   aligned16(g.o1);
  if (vec)
    launch(ew_kernel<OP, TI, TO, true>, grid_for(g.n / 8 + 1), 256, 0, s, g);
  else
    launch(ew_kernel<OP, TI, TO, false>, grid_for(g.n), 256, 0, s, g);
  return check_launch(name);
}

template <EwOp OP>
static int ew_dispatch(int dt_in, int dt_out, const EwArgs& g, void* stream, const char* name) {
  cudaStream_t s = as_stream(stream);
  if (dt_in == XT_F32 && dt_out == XT_F32) return ew_run<OP, float, float>(g, s, name);
  if (dt_in == XT_BF16 && dt_out == XT_BF16) return ew_run<OP, bf16, bf16>(g, s, name);
  if (dt_in == XT_BF16 && dt_out == XT_F32) return ew_run<OP, bf16, float>(g, s, name);
  if (dt_in == XT_F32 && dt_out == XT_BF16) return ew_run<OP, float, bf16>(g, s, name);
  return fail(XT_ERR_INVALID_ARG, "%s: bad dtype", name);
}

static EwArgs ew_args(const void* a, const void* b, const void* c, void* o0, void* o1, int64_t n) {
  EwArgs g{};
  g.a = a; g.b = b; g.c = c; g.o0 = o0; g.o1 = o1; g.n = n;
  return g;
}

// ------------------------------------------------------------------------------ sum

constexpr int kSumThreads = 256;
constexpr int kSumMaxBlocks = 1024;

static int sum_blocks(int64_t n) {
  int64_t b = ceil_div(n, int64_t(kSumThreads) * 16);
  return int(b < 1 ? 1 : (b > kSumMaxBlocks ? kSumMaxBlocks : b));
}

template <typename T>
__global__ void __launch_bounds__(kSumThreads) sum_stage1(const T* x, int64_t n, float* part) {
  pdl_begin();
  __shared__ float red[kSumThreads / 32];
  float acc = 0.f;
  for (int64_t i = int64_t(blockIdx.x) * kSumThreads + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * kSumThreads)
    acc += to_f(x[i]);
  acc = warp_sum(acc);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < kSumThreads / 32; ++w) s += red[w];
    part[blockIdx.x] = s;
  }
}

__global__ void sum_stage2(const float* part, int nb, float* out) {
  pdl_begin();
  __shared__ float red[32];
  float acc = 0.f;
  for (int i = threadIdx.x; i < nb; i += blockDim.x) acc += part[i];
  acc = warp_sum(acc);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < int(blockDim.x / 32); ++w) s += red[w];
    *out = s;
  }
}

// ------------------------------------------------------------------------------ 2-D ops

// swiglu forward: y = silu(g) ∘ u over a [rows, cols] block with row strides.
template <typename T, bool VEC>
__global__ void __launch_bounds__(256) swiglu_fwd_kernel(const T* g, const T* u, int64_t ld_in, T* y,
                                                         int64_t ld_out, int64_t rows, int64_t cols) {
  pdl_begin();
  const int64_t W = VEC ? 8 : 1;
  const int64_t per_row = cols / W;
  const int64_t total = rows * per_row;
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < total;
       v += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = v / per_row, c = (v - r * per_row) * W;
    if constexpr (VEC) {
      float vg[8], vu[8], o[8];
      V8<T>::load(g + r * ld_in + c, vg);
      V8<T>::load(u + r * ld_in + c, vu);
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j] = vg[j] * sigmoidf_(vg[j]) * vu[j];
      V8<T>::store(y + r * ld_out + c, o);
    } else {
      const float a = to_f(g[r * ld_in + c]);
      y[r * ld_out + c] = from_f<T>(a * sigmoidf_(a) * to_f(u[r * ld_in + c]));
    }
  }
}

// swiglu backward by composition ([AE] op table row swiglu): with a = silu(g),
// du = d∘a, dg = (d∘u)∘silu'(g).
template <typename T, bool VEC>
__global__ void __launch_bounds__(256) swiglu_bwd_kernel(const T* d, int64_t ld_d, const T* g, const T* u,
                                                         int64_t ld_in, T* dg, T* du, int64_t ld_grad,
                                                         int64_t rows, int64_t cols, int acc) {
  pdl_begin();
  const int64_t W = VEC ? 8 : 1;
  const int64_t per_row = cols / W;
  const int64_t total = rows * per_row;
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < total;
       v += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = v / per_row, c = (v - r * per_row) * W;
    float vd[8], vg[8], vu[8], og[8], ou[8];
    if constexpr (VEC) {
      V8<T>::load(d + r * ld_d + c, vd);
      V8<T>::load(g + r * ld_in + c, vg);
      V8<T>::load(u + r * ld_in + c, vu);
    } else {
      vd[0] = to_f(d[r * ld_d + c]); vg[0] = to_f(g[r * ld_in + c]); vu[0] = to_f(u[r * ld_in + c]);
    }
#pragma unroll
    for (int j = 0; j < (VEC ? 8 : 1); ++j) {
      const float s = sigmoidf_(vg[j]);
      const float a = vg[j] * s;
      ou[j] = vd[j] * a;
      og[j] = (vd[j] * vu[j]) * (s + vg[j] * s * (1.f - s));
    }
    T* pg = dg + r * ld_grad + c;
    T* pu = du + r * ld_grad + c;
    if constexpr (VEC) {
      if (acc) {
        float o1[8], o2[8];
        V8<T>::load(pg, o1);
        V8<T>::load(pu, o2);
#pragma unroll
        for (int j = 0; j < 8; ++j) { og[j] += o1[j]; ou[j] += o2[j]; }
      }
      V8<T>::store(pg, og);
      V8<T>::store(pu, ou);
    } else {
      if (acc) { og[0] += to_f(*pg); ou[0] += to_f(*pu); }
      *pg = from_f<T>(og[0]);
      *pu = from_f<T>(ou[0]);
    }
  }
}

// add_bias forward: y[r, c] = x[r, c] + bias[c].
template <typename T, bool VEC>
__global__ void __launch_bounds__(256) add_bias_kernel(const T* x, const T* bias, T* y, int64_t rows,
                                                       int64_t cols) {
  pdl_begin();
  const int64_t W = VEC ? 8 : 1;
  const int64_t per_row = cols / W;
  const int64_t total = rows * per_row;
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < total;
       v += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = v / per_row, c = (v - r * per_row) * W;
    if constexpr (VEC) {
      float vx[8], vb[8];
      V8<T>::load(x + r * cols + c, vx);
      V8<T>::load(bias + c, vb);
#pragma unroll
      for (int j = 0; j < 8; ++j) vx[j] += vb[j];
      V8<T>::store(y + r * cols + c, vx);
    } else {
      y[r * cols + c] = from_f<T>(to_f(x[r * cols + c]) + to_f(bias[c]));
    }
  }
}

}  // namespace xt

// ==================================================================================== C ABI
using namespace xt;

#define XT_CHECK_N(n) XT_REQUIRE((n) >= 0, "negative size")
#define XT_CHECK_DT(dt) XT_REQUIRE(valid_dtype(dt), "bad dtype %d", int(dt))

extern "C" {

int xt_accumulate(void* dst, int dt_dst, const void* src, int dt_src, int64_t n, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt_dst);
  XT_CHECK_DT(dt_src);
  XT_REQUIRE(n == 0 || (dst && src), "xt_accumulate: NULL pointer");
  return ew_dispatch<EW_ACC>(dt_src, dt_dst, ew_args(src, nullptr, nullptr, dst, nullptr, n), stream,
                             "xt_accumulate");
}

int xt_convert(void* dst, int dt_dst, const void* src, int dt_src, int64_t n, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt_dst);
  XT_CHECK_DT(dt_src);
  XT_REQUIRE(n == 0 || (dst && src), "xt_convert: NULL pointer");
  EwArgs g = ew_args(src, nullptr, nullptr, dst, nullptr, n);
  g.alpha = 1.f;
  return ew_dispatch<EW_SCALE>(dt_src, dt_dst, g, stream, "xt_convert");
}

int xt_add_fwd(const void* a, const void* b, void* y, int64_t n, int dt, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt);
  XT_REQUIRE(n == 0 || (a && b && y), "xt_add_fwd: NULL pointer");
  return ew_dispatch<EW_ADD>(dt, dt, ew_args(a, b, nullptr, y, nullptr, n), stream, "xt_add_fwd");
}

int xt_add_bwd(const void* d, void* da, void* db, int64_t n, int dt, int acc_a, int acc_b,
               void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt);
  XT_REQUIRE(n == 0 || d, "xt_add_bwd: d is NULL");
  EwArgs g = ew_args(d, nullptr, nullptr, da, db, n);
  g.acc0 = acc_a; g.acc1 = acc_b;
  return ew_dispatch<EW_COPY2>(dt, dt, g, stream, "xt_add_bwd");
}

int xt_mul_fwd(const void* a, const void* b, void* y, int64_t n, int dt, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt);
  XT_REQUIRE(n == 0 || (a && b && y), "xt_mul_fwd: NULL pointer");
  return ew_dispatch<EW_MUL>(dt, dt, ew_args(a, b, nullptr, y, nullptr, n), stream, "xt_mul_fwd");
}

int xt_mul_bwd(const void* d, const void* a, const void* b, void* da, void* db, int64_t n, int dt,
               int acc_a, int acc_b, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt);
  XT_REQUIRE(n == 0 || (d && a && b), "xt_mul_bwd: NULL input");
  // o0 = d∘b is the grad of a, o1 = d∘a the grad of b
  EwArgs g = ew_args(d, a, b, da, db, n);
  g.acc0 = acc_a; g.acc1 = acc_b;
  return ew_dispatch<EW_MUL_BWD>(dt, dt, g, stream, "xt_mul_bwd");
}

int xt_scale_fwd(const void* x, void* y, int64_t n, float alpha, int dt, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt);
  XT_REQUIRE(n == 0 || (x && y), "xt_scale_fwd: NULL pointer");
  EwArgs g = ew_args(x, nullptr, nullptr, y, nullptr, n);
  g.alpha = alpha;
  return ew_dispatch<EW_SCALE>(dt, dt, g, stream, "xt_scale_fwd");
}

int xt_scale_bwd(const void* d, void* dx, int64_t n, float alpha, int dt, int acc, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt);
  XT_REQUIRE(n == 0 || (d && dx), "xt_scale_bwd: NULL pointer");
  EwArgs g = ew_args(d, nullptr, nullptr, dx, nullptr, n);
  g.alpha = alpha; g.acc0 = acc;
  return ew_dispatch<EW_SCALE>(dt, dt, g, stream, "xt_scale_bwd");
}

int xt_sum_workspace_size(int64_t n, size_t* bytes) {
  XT_CHECK_N(n);
  XT_REQUIRE(bytes, "xt_sum_workspace_size: bytes is NULL");
  *bytes = size_t(sum_blocks(n)) * sizeof(float);
  return XT_OK;
}

int xt_sum_fwd(const void* x, int64_t n, int dt, float* out, void* ws, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt);
  XT_REQUIRE(out && ws && (n == 0 || x), "xt_sum_fwd: NULL pointer");
  cudaStream_t s = as_stream(stream);
  const int nb = sum_blocks(n);
  float* part = static_cast<float*>(ws);
  if (dt == XT_F32)
    launch(sum_stage1<float>, nb, kSumThreads, 0, s, static_cast<const float*>(x), n, part);
  else
    launch(sum_stage1<bf16>, nb, kSumThreads, 0, s, static_cast<const bf16*>(x), n, part);
  XT_TRY(check_launch("xt_sum_fwd"));
  launch(sum_stage2, 1, 1024, 0, s, part, nb, out);
  return check_launch("xt_sum_fwd");
}

int xt_sum_bwd(const float* upstream, void* dx, int64_t n, int dt, int acc, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt);
  XT_REQUIRE(n == 0 || (upstream && dx), "xt_sum_bwd: NULL pointer");
  EwArgs g = ew_args(nullptr, nullptr, nullptr, dx, nullptr, n);
  g.scalar = upstream; g.acc0 = acc;
  return ew_dispatch<EW_FILL>(dt, dt, g, stream, "xt_sum_bwd");
}

int xt_silu_fwd(const void* x, void* y, int64_t n, int dt, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt);
  XT_REQUIRE(n == 0 || (x && y), "xt_silu_fwd: NULL pointer");
  return ew_dispatch<EW_SILU>(dt, dt, ew_args(x, nullptr, nullptr, y, nullptr, n), stream, "xt_silu_fwd");
}

int xt_silu_bwd(const void* d, const void* x, void* dx, int64_t n, int dt, int acc, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt);
  XT_REQUIRE(n == 0 || (d && x && dx), "xt_silu_bwd: NULL pointer");
  EwArgs g = ew_args(d, x, nullptr, dx, nullptr, n);
  g.acc0 = acc;
  return ew_dispatch<EW_SILU_BWD>(dt, dt, g, stream, "xt_silu_bwd");
}

int xt_gelu_fwd(const void* x, void* y, int64_t n, int dt, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt);
  XT_REQUIRE(n == 0 || (x && y), "xt_gelu_fwd: NULL pointer");
  return ew_dispatch<EW_GELU>(dt, dt, ew_args(x, nullptr, nullptr, y, nullptr, n), stream, "xt_gelu_fwd");
}

int xt_gelu_bwd(const void* d, const void* x, void* dx, int64_t n, int dt, int acc, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt);
  XT_REQUIRE(n == 0 || (d && x && dx), "xt_gelu_bwd: NULL pointer");
  EwArgs g = ew_args(d, x, nullptr, dx, nullptr, n);
  g.acc0 = acc;
  return ew_dispatch<EW_GELU_BWD>(dt, dt, g, stream, "xt_gelu_bwd");
}

static int check_dropout(float p) {
  if (!(p >= 0.f && p < 1.f)) return fail(XT_ERR_INVALID_ARG, "dropout: p must be in [0, 1), got %g", double(p));
  return XT_OK;
}

static float dropout_scale(float p) { return static_cast<float>(1.0 / (1.0 - static_cast<double>(p))); }

int xt_dropout_fwd(const void* x, void* y, int64_t n, float p, uint64_t seed, int training, int dt,
                   void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt);
  XT_TRY(check_dropout(p));
  XT_REQUIRE(n == 0 || (x && y), "xt_dropout_fwd: NULL pointer");
  if (p == 0.f || !training) {  // exact identity ([DO] § train / eval 开关)
    if (x == y || n == 0) return XT_OK;
    if (cudaMemcpyAsync(y, x, size_t(n) * dtype_size(dt), cudaMemcpyDeviceToDevice, as_stream(stream)) != cudaSuccess)
      return check_launch("xt_dropout_fwd copy");
    return XT_OK;
  }
  EwArgs g = ew_args(x, nullptr, nullptr, y, nullptr, n);
  g.p = p; g.dscale = dropout_scale(p); g.seed = seed; g.thr = dropout_threshold(p);
  return ew_dispatch<EW_DROPOUT>(dt, dt, g, stream, "xt_dropout_fwd");
}

int xt_dropout_bwd(const void* d, void* dx, int64_t n, float p, uint64_t seed, int training, int dt,
                   int acc, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt);
  XT_TRY(check_dropout(p));
  XT_REQUIRE(n == 0 || (d && dx), "xt_dropout_bwd: NULL pointer");
  EwArgs g = ew_args(d, nullptr, nullptr, dx, nullptr, n);
  g.acc0 = acc;
  if (p == 0.f || !training) {
    if (!acc && d == dx) return XT_OK;
    g.alpha = 1.f;
    return ew_dispatch<EW_SCALE>(dt, dt, g, stream, "xt_dropout_bwd");
  }
  g.p = p; g.dscale = dropout_scale(p); g.seed = seed; g.thr = dropout_threshold(p);
  return ew_dispatch<EW_DROPOUT>(dt, dt, g, stream, "xt_dropout_bwd");
}

int xt_dropout_bwd_ex(const void* d, int dt_d, void* dx, int dt_dx, int64_t n, float p, uint64_t seed,
                      int training, int acc, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt_d);
  XT_CHECK_DT(dt_dx);
  XT_TRY(check_dropout(p));
  XT_REQUIRE(n == 0 || (d && dx), "xt_dropout_bwd_ex: NULL pointer");
  EwArgs g = ew_args(d, nullptr, nullptr, dx, nullptr, n);
  g.acc0 = acc;
  if (p == 0.f || !training) {
    g.alpha = 1.f;
    return ew_dispatch<EW_SCALE>(dt_d, dt_dx, g, stream, "xt_dropout_bwd_ex");
  }
  g.p = p; g.dscale = dropout_scale(p); g.seed = seed; g.thr = dropout_threshold(p);
  return ew_dispatch<EW_DROPOUT>(dt_d, dt_dx, g, stream, "xt_dropout_bwd_ex");
}

int xt_dropout_add_fwd(const void* h, const void* a, void* out, int64_t n, float p, uint64_t seed,
                       int training, int dt, void* stream) {
  XT_CHECK_N(n);
  XT_CHECK_DT(dt);
  XT_TRY(check_dropout(p));
  XT_REQUIRE(n == 0 || (h && a && out), "xt_dropout_add_fwd: NULL pointer");
  EwArgs g = ew_args(h, a, nullptr, out, nullptr, n);
  if (p == 0.f || !training) return ew_dispatch<EW_ADD>(dt, dt, g, stream, "xt_dropout_add_fwd");
  g.p = p; g.dscale = dropout_scale(p); g.seed = seed; g.thr = dropout_threshold(p);
  return ew_dispatch<EW_DROPOUT_ADD>(dt, dt, g, stream, "xt_dropout_add_fwd");
}

}  // extern "C"

namespace xt {
__global__ void dropout_mask_kernel(uint8_t* mask, int64_t n, float p, uint64_t seed) {
  pdl_begin();
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x)
    mask[i] = dropout_keep(seed, uint64_t(i), p) ? 1 : 0;
}
}  // namespace xt

extern "C" {

int xt_dropout_mask(uint8_t* mask, int64_t n, float p, uint64_t seed, void* stream) {
  XT_CHECK_N(n);
  XT_TRY(check_dropout(p));
  XT_REQUIRE(n == 0 || mask, "xt_dropout_mask: NULL pointer");
  if (n == 0) return XT_OK;
  launch(dropout_mask_kernel, grid_for(n), 256, 0, as_stream(stream), mask, n, p, seed);
  return check_launch("xt_dropout_mask");
}

int xt_swiglu_fwd(const void* g, const void* u, int64_t ld_in, void* y, int64_t ld_out, int64_t rows,
                  int64_t cols, int dt, void* stream) {
  XT_REQUIRE(rows >= 0 && cols >= 0 && ld_in >= cols && ld_out >= cols, "xt_swiglu_fwd: bad sizes");
  XT_CHECK_DT(dt);
  XT_REQUIRE(rows * cols == 0 || (g && u && y), "xt_swiglu_fwd: NULL pointer");
  if (rows * cols == 0) return XT_OK;
  cudaStream_t s = as_stream(stream);
  const size_t e = dtype_size(dt);
  const bool vec = cols % 8 == 0 && (ld_in * e) % 16 == 0 && (ld_out * e) % 16 == 0 && aligned16(g) &&
                   aligned16(u) && aligned16(y);
  const int grid = grid_for(rows * cols / (vec ? 8 : 1));
  if (dt == XT_F32) {
    auto G = static_cast<const float*>(g); auto U = static_cast<const float*>(u); auto Y = static_cast<float*>(y);
    if (vec) launch(swiglu_fwd_kernel<float, true>, grid, 256, 0, s, G, U, ld_in, Y, ld_out, rows, cols);
    else launch(swiglu_fwd_kernel<float, false>, grid, 256, 0, s, G, U, ld_in, Y, ld_out, rows, cols);
  } else {
    auto G = static_cast<const bf16*>(g); auto U = static_cast<const bf16*>(u); auto Y = static_cast<bf16*>(y);
    if (vec) launch(swiglu_fwd_kernel<bf16, true>, grid, 256, 0, s, G, U, ld_in, Y, ld_out, rows, cols);
    else launch(swiglu_fwd_kernel<bf16, false>, grid, 256, 0, s, G, U, ld_in, Y, ld_out, rows, cols);
  }
  return check_launch("xt_swiglu_fwd");
}

int xt_swiglu_bwd(const void* d, int64_t ld_d, const void* g, const void* u, int64_t ld_in, void* dg,
                  void* du, int64_t ld_grad, int64_t rows, int64_t cols, int dt, int acc, void* stream) {
  XT_REQUIRE(rows >= 0 && cols >= 0 && ld_d >= cols && ld_in >= cols && ld_grad >= cols,
             "xt_swiglu_bwd: bad sizes");
  XT_CHECK_DT(dt);
  XT_REQUIRE(rows * cols == 0 || (d && g && u && dg && du), "xt_swiglu_bwd: NULL pointer");
  if (rows * cols == 0) return XT_OK;
  cudaStream_t s = as_stream(stream);
  const size_t e = dtype_size(dt);
  const bool vec = cols % 8 == 0 && (ld_in * e) % 16 == 0 && (ld_d * e) % 16 == 0 &&
                   (ld_grad * e) % 16 == 0 && aligned16(d) && aligned16(g) && aligned16(u) &&
                   aligned16(dg) && aligned16(du);
  const int grid = grid_for(rows * cols / (vec ? 8 : 1));
  if (dt == XT_F32) {
    auto D = static_cast<const float*>(d); auto G = static_cast<const float*>(g);
    auto U = static_cast<const float*>(u);
    auto DG = static_cast<float*>(dg); auto DU = static_cast<float*>(du);
    if (vec) launch(swiglu_bwd_kernel<float, true>, grid, 256, 0, s, D, ld_d, G, U, ld_in, DG, DU, ld_grad, rows, cols, acc);
    else launch(swiglu_bwd_kernel<float, false>, grid, 256, 0, s, D, ld_d, G, U, ld_in, DG, DU, ld_grad, rows, cols, acc);
  } else {
    auto D = static_cast<const bf16*>(d); auto G = static_cast<const bf16*>(g);
    auto U = static_cast<const bf16*>(u);
    auto DG = static_cast<bf16*>(dg); auto DU = static_cast<bf16*>(du);
    if (vec) launch(swiglu_bwd_kernel<bf16, true>, grid, 256, 0, s, D, ld_d, G, U, ld_in, DG, DU, ld_grad, rows, cols, acc);
    else launch(swiglu_bwd_kernel<bf16, false>, grid, 256, 0, s, D, ld_d, G, U, ld_in, DG, DU, ld_grad, rows, cols, acc);
  }
  return check_launch("xt_swiglu_bwd");
}

int xt_add_bias_fwd(const void* x, const void* bias, void* y, int64_t rows, int64_t cols, int dt,
                    void* stream) {
  XT_REQUIRE(rows >= 0 && cols >= 0, "xt_add_bias_fwd: bad sizes");
  XT_CHECK_DT(dt);
  XT_REQUIRE(rows * cols == 0 || (x && bias && y), "xt_add_bias_fwd: NULL pointer");
  if (rows * cols == 0) return XT_OK;
  cudaStream_t s = as_stream(stream);
  const bool vec = cols % 8 == 0 && aligned16(x) && aligned16(bias) && aligned16(y);
  const int grid = grid_for(rows * cols / (vec ? 8 : 1));
  if (dt == XT_F32) {
    auto X = static_cast<const float*>(x); auto Bb = static_cast<const float*>(bias); auto Y = static_cast<float*>(y);
    if (vec) launch(add_bias_kernel<float, true>, grid, 256, 0, s, X, Bb, Y, rows, cols);
    else launch(add_bias_kernel<float, false>, grid, 256, 0, s, X, Bb, Y, rows, cols);
  } else {
    auto X = static_cast<const bf16*>(x); auto Bb = static_cast<const bf16*>(bias); auto Y = static_cast<bf16*>(y);
    if (vec) launch(add_bias_kernel<bf16, true>, grid, 256, 0, s, X, Bb, Y, rows, cols);
    else launch(add_bias_kernel<bf16, false>, grid, 256, 0, s, X, Bb, Y, rows, cols);
  }
  return check_launch("xt_add_bias_fwd");
}

}  // extern "C"
