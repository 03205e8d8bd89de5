// Row-wise ops: RMSNorm, LayerNorm, softmax, cross-entropy; RoPE; embedding; column sums.
//
// Row-resident kernels keep a thread's share of one row in registers as packed 16-byte
// vectors (4 registers per vector for both fp32 and bf16): a row of `cols` elements is split
// over a row group of `tpr` threads (power of two, 32..1024), each holding up to NV = 4
// vectors, so one global read feeds the reductions and the outputs.  Several row groups
// share a block when rows are short.  Column reductions (dγ, dβ, dbias) are deterministic:
// per-block partial rows in the workspace, then one ordered pass.
#include <mutex>

#include "common.cuh"
#include "internal.cuh"

namespace xt {

constexpr int NV = 4;  // vectors per thread in row-resident kernels
constexpr float kLog2e = 1.4426950408889634f;

// 2^x with the hardware approximation (ex2.approx.ftz: relative error ~2⁻²², −inf → +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed storage of one vector (VW elements) of T.
template <typename T, int VW> struct Raw;
template <typename T> struct Raw<T, 1> {
  float v;
  __device__ __forceinline__ void load(const T* p) { v = to_f(*p); }
  __device__ __forceinline__ float get(int) const { return v; }
  __device__ __forceinline__ void zero() { v = 0.f; }
  __device__ __forceinline__ void keep_first(int n) { if (n < 1) v = 0.f; }
};
template <> struct Raw<float, 4> {
  float4 q;
  __device__ __forceinline__ void load(const float* p) { q = *reinterpret_cast<const float4*>(p); }
  __device__ __forceinline__ float get(int e) const {
    return e == 0 ? q.x : e == 1 ? q.y : e == 2 ? q.z : q.w;
  }
  __device__ __forceinline__ void zero() { q = make_float4(0.f, 0.f, 0.f, 0.f); }
  // zero elements n.. (n in 0..VW)
  __device__ __forceinline__ void keep_first(int n) {
    if (n < 4) q.w = 0.f;
    if (n < 3) q.z = 0.f;
    if (n < 2) q.y = 0.f;
    if (n < 1) q.x = 0.f;
  }
};
template <> struct Raw<bf16, 8> {
  uint4 q;
  __device__ __forceinline__ void load(const bf16* p) { q = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ float get(int e) const {
    const uint32_t w = e < 2 ? q.x : e < 4 ? q.y : e < 6 ? q.z : q.w;
    return (e & 1) ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
  }
  __device__ __forceinline__ void zero() { q = make_uint4(0, 0, 0, 0); }
  // zero elements n.. (n in 0..VW); element e is the low half of word e/2 when e is even
  __device__ __forceinline__ void keep_first(int n) {
    q.x &= word_keep(n, 0);
    q.y &= word_keep(n, 1);
    q.z &= word_keep(n, 2);
    q.w &= word_keep(n, 3);
  }
  static __device__ __forceinline__ uint32_t word_keep(int n, int i) {
    return n >= 2 * i + 2 ? 0xFFFFFFFFu : n == 2 * i + 1 ? 0x0000FFFFu : 0u;
  }
};

template <typename T, int VW>
__device__ __forceinline__ void store_vec(T* p, const float (&v)[VW]) {
  Acc<T, VW>::store(p, v);
}
template <typename T, int VW>
__device__ __forceinline__ void load_vec(const T* p, float (&v)[VW]) {
  Acc<T, VW>::load(p, v);
}

struct RowPlan {
  int vw, tpr, threads, rpb;
  bool ok;
};

static int next_pow2(int64_t v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

// Plans a row-resident launch: vector width, threads per row, block size, rows per block; nv is
// the most vectors a thread holds (≤ NV).
static RowPlan plan_rows(int64_t cols, int vw, int max_tpr = 1024, int nv = NV) {
  RowPlan pl{};
  pl.vw = vw;
  const int64_t nvec = ceil_div(cols, vw);
  if (nvec > int64_t(nv) * max_tpr) { pl.ok = false; return pl; }
  int tpr = next_pow2(ceil_div(nvec, nv));
  if (tpr < 32) tpr = 32;
  pl.tpr = tpr;
  pl.threads = tpr < 256 ? 256 : tpr;
  pl.rpb = pl.threads / tpr;
  pl.ok = true;
  return pl;
}

static bool rows_vec_ok(int64_t cols, int dt, std::initializer_list<const void*> ptrs) {
  const int vw = dt == XT_BF16 ? 8 : 4;
  if (cols % vw) return false;
  for (const void* p : ptrs)
    if (!aligned16(p)) return false;
  return true;
}

static int row_grid(int64_t rows, int rpb, int cap_per_sm = 32) {
  int64_t g = ceil_div(rows, rpb);
  const int64_t cap = int64_t(num_sms()) * cap_per_sm;
  if (g > cap) g = cap;
  return int(g < 1 ? 1 : g);
}

// Fixed number of blocks of the column-reducing backward kernels (one partial row each).
static int bwd_blocks(int64_t rows, int rpb) {
  int64_t g = ceil_div(rows, rpb);
  const int64_t cap = int64_t(num_sms()) * 4;
  if (g > cap) g = cap;
  return int(g < 1 ? 1 : g);
}

__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Rows of 4 KB or more: a row group asks L2 for the row it takes next (its vectors of row rn)
// while it still waits on this row's loads, so that row's loads are L2 hits.  With one or two
// row groups per SM, a row's DRAM latency is otherwise paid once per row, unhidden.
template <typename T, int VW>
__device__ __forceinline__ void prefetch_next_row(const T* base, int64_t rn, int64_t rows, int64_t cols, int l,
                                                  int tpr) {
  if (rn >= rows || cols * int64_t(sizeof(T)) < 4096) return;
  const int64_t nvec = cols / VW;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int64_t j = l + int64_t(k) * tpr;
    if (j < nvec) prefetch_l2(base + rn * cols + j * VW);
  }
}

// ============================================================================== RMSNorm

template <typename T, int VW>
__global__ void __launch_bounds__(1024) rms_fwd_kernel(const T* __restrict__ x, const T* __restrict__ gamma,
                                                      T* __restrict__ y, float* __restrict__ inv_rms,
                                                      int64_t rows, int64_t cols, float eps, int tpr) {
  pdl_begin();
  __shared__ float red[32];
  const int rpb = blockDim.x / tpr, l = threadIdx.x % tpr;
  const int64_t nvec = cols / VW;
  for (int64_t r0 = int64_t(blockIdx.x) * rpb; r0 < rows; r0 += int64_t(gridDim.x) * rpb) {
    const int64_t r = r0 + threadIdx.x / tpr;
    const bool act = r < rows;
    Raw<T, VW> v[NV];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t j = l + int64_t(k) * tpr;
      if (act && j < nvec) v[k].load(x + r * cols + j * VW); else v[k].zero();
    }
    prefetch_next_row<T, VW>(x, r + int64_t(gridDim.x) * rpb, rows, cols, l, tpr);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
#pragma unroll
      for (int e = 0; e < VW; ++e) ss += v[k].get(e) * v[k].get(e);
    }
    ss = group_reduce<false>(ss, tpr, red);
    const float ir = 1.f / sqrtf(ss / float(cols) + eps);
    if (act && l == 0) inv_rms[r] = ir;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t j = l + int64_t(k) * tpr;
      if (act && j < nvec) {
        float gm[VW], o[VW];
        load_vec<T, VW>(gamma + j * VW, gm);
#pragma unroll
        for (int e = 0; e < VW; ++e) o[e] = v[k].get(e) * ir * gm[e];
        store_vec<T, VW>(y + r * cols + j * VW, o);
      }
    }
  }
}

// Column partials of the backward kernels live in shared memory, one slice of `cols` floats
// per row group; each (group, column) is owned by exactly one thread, so no atomics are
// needed and the order of additions is fixed.  slice_add adds one vector's contribution.
template <int VW>
__device__ __forceinline__ void slice_add(float* p, const float (&v)[VW]) {
  if constexpr (VW % 4 == 0) {
#pragma unroll
    for (int e = 0; e < VW; e += 4) {
      float4 q = *reinterpret_cast<float4*>(p + e);
      q.x += v[e]; q.y += v[e + 1]; q.z += v[e + 2]; q.w += v[e + 3];
      *reinterpret_cast<float4*>(p + e) = q;
    }
  } else {
#pragma unroll
    for (int e = 0; e < VW; ++e) p[e] += v[e];
  }
}

// Zeroes this thread's columns of its group's slice.
template <int VW>
__device__ __forceinline__ void slice_zero(float* slice, int l, int tpr, int64_t nvec) {
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int64_t j = l + int64_t(k) * tpr;
    if (j < nvec)
#pragma unroll
      for (int e = 0; e < VW; ++e) slice[j * VW + e] = 0.f;
  }
}

// part[blockIdx.x][c] = Σ over the block's row groups (in group order) of slice[g][c].
__device__ __forceinline__ void slices_fold(const float* slices, int rpb, float* part, int64_t cols) {
  __syncthreads();
  for (int64_t c = threadIdx.x; c < cols; c += blockDim.x) {
    float a = 0.f;
    for (int g = 0; g < rpb; ++g) a += slices[int64_t(g) * cols + c];
    part[int64_t(blockIdx.x) * cols + c] = a;
  }
}

// Optional second output of the norm backward kernels: the gradient the preceding residual
// dropout passes on, g = keep(seed, i) ? dh·dscale : 0 (dh itself when drop is 0), written in
// the activation dtype from the final residual gradient dh the kernel stores (i the flat index).
struct GradOut {
  void* g;
  float p, dscale;
  uint64_t seed;
  int drop;
};
template <typename T, int VW>
__device__ __forceinline__ void grad_out_store(const GradOut& go, int64_t off, const float (&dh)[VW]) {
  float v[VW];
#pragma unroll
  for (int e = 0; e < VW; ++e)
    v[e] = go.drop ? (dropout_keep(go.seed, uint64_t(off + e), go.p) ? dh[e] * go.dscale : 0.f) : dh[e];
  store_vec<T, VW>(static_cast<T*>(go.g) + off, v);
}

template <typename T, typename TD, int VW, int MAXT>
__global__ void __launch_bounds__(MAXT, MAXT <= 256 ? 2 : 1) rms_bwd_kernel(const T* __restrict__ d, const T* __restrict__ x,
                                                      const T* __restrict__ gamma, const float* __restrict__ inv_rms,
                                                      TD* dx, float* __restrict__ part, int64_t rows, int64_t cols,
                                                      int tpr, int acc_dx, GradOut go) {
  pdl_begin();
  extern __shared__ float smem[];
  float* red = smem;  // 32
  const int rpb = blockDim.x / tpr, l = threadIdx.x % tpr;
  float* pg = smem + 32 + int64_t(threadIdx.x / tpr) * cols;  // this row group's dγ slice
  const int64_t nvec = cols / VW;
  Raw<T, VW> gm[NV];  // this thread's columns of γ, the same for every row
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int64_t j = l + int64_t(k) * tpr;
    if (j < nvec) gm[k].load(gamma + j * VW); else gm[k].zero();
  }
  if (part) slice_zero<VW>(pg, l, tpr, nvec);
  for (int64_t r0 = int64_t(blockIdx.x) * rpb; r0 < rows; r0 += int64_t(gridDim.x) * rpb) {
    const int64_t r = r0 + threadIdx.x / tpr;
    const bool act = r < rows;
    Raw<T, VW> vd[NV], vx[NV];
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t j = l + int64_t(k) * tpr;
      if (act && j < nvec) {
        vd[k].load(d + r * cols + j * VW);
        vx[k].load(x + r * cols + j * VW);
      } else {
        vd[k].zero(); vx[k].zero();
      }
    }
    prefetch_next_row<T, VW>(d, r + int64_t(gridDim.x) * rpb, rows, cols, l, tpr);
    prefetch_next_row<T, VW>(x, r + int64_t(gridDim.x) * rpb, rows, cols, l, tpr);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
#pragma unroll
      for (int e = 0; e < VW; ++e) s += vd[k].get(e) * gm[k].get(e) * vx[k].get(e);
    }
    s = group_reduce<false>(s, tpr, red);
    const float ir = act ? inv_rms[r] : 0.f;
    const float c2 = ir * ir * ir / float(cols) * s;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t j = l + int64_t(k) * tpr;
      if (act && j < nvec) {
        float o[VW], pgv[VW];
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          const float xv = vx[k].get(e), dv = vd[k].get(e);
          o[e] = ir * dv * gm[k].get(e) - xv * c2;
          pgv[e] = dv * xv * ir;
        }
        if (part) slice_add<VW>(pg + j * VW, pgv);
        if (dx) {
          TD* p = dx + r * cols + j * VW;
          if (acc_dx) {
            float old[VW];
            load_vec<TD, VW>(p, old);
#pragma unroll
            for (int e = 0; e < VW; ++e) o[e] += old[e];
          }
          store_vec<TD, VW>(p, o);
          if (go.g) grad_out_store<T, VW>(go, r * cols + j * VW, o);
        }
      }
    }
  }
  if (part) slices_fold(smem + 32, rpb, part, cols);
}

// ============================================================================== LayerNorm

template <typename T, int VW>
__global__ void __launch_bounds__(1024) ln_fwd_kernel(const T* __restrict__ x, const T* __restrict__ gamma,
                                                     const T* __restrict__ beta, T* __restrict__ y,
                                                     float* __restrict__ mean_out, float* __restrict__ rstd_out,
                                                     int64_t rows, int64_t cols, float eps, int tpr) {
  pdl_begin();
  __shared__ float red[32];
  const int rpb = blockDim.x / tpr, l = threadIdx.x % tpr;
  const int64_t nvec = cols / VW;
  for (int64_t r0 = int64_t(blockIdx.x) * rpb; r0 < rows; r0 += int64_t(gridDim.x) * rpb) {
    const int64_t r = r0 + threadIdx.x / tpr;
    const bool act = r < rows;
    Raw<T, VW> v[NV];
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t j = l + int64_t(k) * tpr;
      if (act && j < nvec) v[k].load(x + r * cols + j * VW); else v[k].zero();
    }
    prefetch_next_row<T, VW>(x, r + int64_t(gridDim.x) * rpb, rows, cols, l, tpr);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
#pragma unroll
      for (int e = 0; e < VW; ++e) s += v[k].get(e);
    }
    const float mu = group_reduce<false>(s, tpr, red) / float(cols);
    float q = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t j = l + int64_t(k) * tpr;
      if (j < nvec)
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          const float c = v[k].get(e) - mu;
          q += c * c;
        }
    }
    const float var = group_reduce<false>(q, tpr, red) / float(cols);
    const float rs = 1.f / sqrtf(var + eps);
    if (act && l == 0) { mean_out[r] = mu; rstd_out[r] = rs; }
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t j = l + int64_t(k) * tpr;
      if (act && j < nvec) {
        float gm[VW], bt[VW], o[VW];
        load_vec<T, VW>(gamma + j * VW, gm);
        load_vec<T, VW>(beta + j * VW, bt);
#pragma unroll
        for (int e = 0; e < VW; ++e) o[e] = (v[k].get(e) - mu) * rs * gm[e] + bt[e];
        store_vec<T, VW>(y + r * cols + j * VW, o);
      }
    }
  }
}

// LayerNorm backward, one row group per row: NVT vectors per thread.  The next row's d, x and
// statistics are loaded into registers while this row is reduced and written (measured: 8192 ×
// 2048 bf16 with a float32 residual gradient 70.5 → 62.5 µs; 8192 × 768 unchanged), and each
// row's old residual gradient (acc_dx) is prefetched into L1 with them, so the accumulate after
// the two row reductions does not start a second trip to L2.  A row of 8 KB or more also has the
// row after next prefetched into L2.  dγ and dβ partials stay in registers for the thread's fixed
// columns across all of its rows; the row groups' partials meet in shared memory once, at the
// end, and are folded in group order.
template <typename T, typename TD, int VW, int NVT, int MAXT>
__global__ void __launch_bounds__(MAXT, MAXT <= 256 ? 2 : 1) ln_bwd_kernel(const T* __restrict__ d, const T* __restrict__ x,
                                                     const T* __restrict__ gamma, const float* __restrict__ mean,
                                                     const float* __restrict__ rstd, TD* dx, float* __restrict__ part_g,
                                                     float* __restrict__ part_b, int64_t rows, int64_t cols,
                                                     int tpr, int acc_dx, GradOut go) {
  pdl_begin();
  extern __shared__ float smem[];
  float* red = smem;
  const int rpb = blockDim.x / tpr, l = threadIdx.x % tpr, grp = threadIdx.x / tpr;
  const int64_t nvec = cols / VW;
  float ag[NVT][VW], ab[NVT][VW];
#pragma unroll
  for (int k = 0; k < NVT; ++k)
#pragma unroll
    for (int e = 0; e < VW; ++e) ag[k][e] = ab[k][e] = 0.f;
  const float inv_n = 1.f / float(cols);
  const int64_t step = int64_t(gridDim.x) * rpb;
  const bool pf = cols * int64_t(sizeof(T)) >= 8192;
  // The group's rows r, r + step, ...: the next row's d, x and statistics are loaded (and its
  // residual gradient prefetched into L1) while this row is reduced and written, so each warp
  // keeps two rows' loads in flight.
  Raw<T, VW> vd[NVT], vx[NVT];
  float mu = 0.f, rs = 0.f;
  auto fetch = [&](int64_t rr, Raw<T, VW> (&a)[NVT], Raw<T, VW> (&b)[NVT], float& m, float& s) {
    const bool act = rr < rows;
#pragma unroll
    for (int k = 0; k < NVT; ++k) {
      const int64_t j = l + int64_t(k) * tpr;
      if (act && j < nvec) {
        a[k].load(d + rr * cols + j * VW);
        b[k].load(x + rr * cols + j * VW);
        if (dx && acc_dx) prefetch_l1(dx + rr * cols + j * VW);
      } else {
        a[k].zero(); b[k].zero();
      }
    }
    m = act ? mean[rr] : 0.f;
    s = act ? rstd[rr] : 0.f;
  };
  fetch(int64_t(blockIdx.x) * rpb + grp, vd, vx, mu, rs);
  for (int64_t r0 = int64_t(blockIdx.x) * rpb; r0 < rows; r0 += step) {
    const int64_t r = r0 + grp;
    const bool act = r < rows;
    if (pf && r + 2 * step < rows) {
      const int64_t rn = r + 2 * step;
#pragma unroll
      for (int k = 0; k < NVT; ++k) {
        const int64_t j = l + int64_t(k) * tpr;
        if (j < nvec) {
          prefetch_l2(d + rn * cols + j * VW);
          prefetch_l2(x + rn * cols + j * VW);
          if (dx && acc_dx) prefetch_l2(dx + rn * cols + j * VW);
        }
      }
    }
    Raw<T, VW> nd[NVT], nx[NVT];
    float nmu, nrs;
    fetch(r + step, nd, nx, nmu, nrs);
    float sg = 0.f, sgx = 0.f;
#pragma unroll
    for (int k = 0; k < NVT; ++k) {
      const int64_t j = l + int64_t(k) * tpr;
      Raw<T, VW> gm;  // γ is re-read from L1 rather than held in registers
      if (j < nvec) gm.load(gamma + j * VW); else gm.zero();
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        const float g = vd[k].get(e) * gm.get(e);
        sg += g;
        sgx += g * (vx[k].get(e) - mu) * rs;
      }
    }
    const float mg = group_reduce<false>(sg, tpr, red) * inv_n;
    const float mgx = group_reduce<false>(sgx, tpr, red) * inv_n;
#pragma unroll
    for (int k = 0; k < NVT; ++k) {
      const int64_t j = l + int64_t(k) * tpr;
      if (act && j < nvec) {
        Raw<T, VW> gm;
        gm.load(gamma + j * VW);
        float o[VW];
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          const float xh = (vx[k].get(e) - mu) * rs, dv = vd[k].get(e);
          o[e] = rs * (dv * gm.get(e) - mg - xh * mgx);
          ag[k][e] = fmaf(dv, xh, ag[k][e]);
          ab[k][e] += dv;
        }
        if (dx) {
          TD* p = dx + r * cols + j * VW;
          if (acc_dx) {
            float old[VW];
            load_vec<TD, VW>(p, old);
#pragma unroll
            for (int e = 0; e < VW; ++e) o[e] += old[e];
          }
          store_vec<TD, VW>(p, o);
          if (go.g) grad_out_store<T, VW>(go, r * cols + j * VW, o);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < NVT; ++k) {
      vd[k] = nd[k];
      vx[k] = nx[k];
    }
    mu = nmu;
    rs = nrs;
  }
  if (part_g || part_b) {
    __syncthreads();  // the reductions' scratch and the slices share shared memory
    float* sgp = smem + 32 + int64_t(grp) * cols;
    float* sbp = smem + 32 + int64_t(rpb + grp) * cols;
#pragma unroll
    for (int k = 0; k < NVT; ++k) {
      const int64_t j = l + int64_t(k) * tpr;
      if (j < nvec)
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          sgp[j * VW + e] = ag[k][e];
          sbp[j * VW + e] = ab[k][e];
        }
    }
  }
  if (part_g) slices_fold(smem + 32, rpb, part_g, cols);
  if (part_b) slices_fold(smem + 32 + int64_t(rpb) * cols, rpb, part_b, cols);
}

// Residual dropout-add fused with the next pre-norm: s = h + (keep(seed, i) ? a·dscale : 0) (plain h + a
// when drop is 0) is stored in T, and the norm of the stored s follows in the same pass, with the
// expressions and accumulation order of rms_fwd_kernel / ln_fwd_kernel, so y and the statistics are
// those of the two separate kernels.
template <typename T, int VW, bool LN>
__global__ void __launch_bounds__(1024) add_norm_fwd_kernel(const T* __restrict__ h, const T* __restrict__ a,
                                                            T* __restrict__ sum, const T* __restrict__ gamma,
                                                            const T* __restrict__ beta, T* __restrict__ y,
                                                            float* __restrict__ st0, float* __restrict__ st1,
                                                            int64_t rows, int64_t cols, float eps, int tpr, int drop,
                                                            float p, float dscale, uint64_t seed) {
  pdl_begin();
  __shared__ float red[32];
  const int rpb = blockDim.x / tpr, l = threadIdx.x % tpr;
  const int64_t nvec = cols / VW;
  for (int64_t r0 = int64_t(blockIdx.x) * rpb; r0 < rows; r0 += int64_t(gridDim.x) * rpb) {
    const int64_t r = r0 + threadIdx.x / tpr;
    const bool act = r < rows;
    float f[NV][VW];
    float s1 = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t j = l + int64_t(k) * tpr;
      if (act && j < nvec) {
        Raw<T, VW> hv, av;
        hv.load(h + r * cols + j * VW);
        av.load(a + r * cols + j * VW);
        float o[VW];
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          const float ae = av.get(e);
          o[e] = hv.get(e) + (drop ? (dropout_keep(seed, uint64_t(r * cols + j * VW + e), p) ? ae * dscale : 0.f) : ae);
        }
        store_vec<T, VW>(sum + r * cols + j * VW, o);
#pragma unroll
        for (int e = 0; e < VW; ++e) f[k][e] = to_f(from_f<T>(o[e]));  // the stored value
      } else {
#pragma unroll
        for (int e = 0; e < VW; ++e) f[k][e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        if constexpr (LN) s1 += f[k][e];
        else s1 += f[k][e] * f[k][e];
      }
    }
    if constexpr (LN) {
      const float mu = group_reduce<false>(s1, tpr, red) / float(cols);
      float q = 0.f;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int64_t j = l + int64_t(k) * tpr;
        if (j < nvec)
#pragma unroll
          for (int e = 0; e < VW; ++e) {
            const float c = f[k][e] - mu;
            q += c * c;
          }
      }
      const float var = group_reduce<false>(q, tpr, red) / float(cols);
      const float rs = 1.f / sqrtf(var + eps);
      if (act && l == 0) { st0[r] = mu; st1[r] = rs; }
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int64_t j = l + int64_t(k) * tpr;
        if (act && j < nvec) {
          float gm[VW], bt[VW], o[VW];
          load_vec<T, VW>(gamma + j * VW, gm);
          load_vec<T, VW>(beta + j * VW, bt);
#pragma unroll
          for (int e = 0; e < VW; ++e) o[e] = (f[k][e] - mu) * rs * gm[e] + bt[e];
          store_vec<T, VW>(y + r * cols + j * VW, o);
        }
      }
    } else {
      const float ss = group_reduce<false>(s1, tpr, red);
      const float ir = 1.f / sqrtf(ss / float(cols) + eps);
      if (act && l == 0) st0[r] = ir;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int64_t j = l + int64_t(k) * tpr;
        if (act && j < nvec) {
          float gm[VW], o[VW];
          load_vec<T, VW>(gamma + j * VW, gm);
#pragma unroll
          for (int e = 0; e < VW; ++e) o[e] = f[k][e] * ir * gm[e];
          store_vec<T, VW>(y + r * cols + j * VW, o);
        }
      }
    }
  }
}

// ============================================================================== column sums

// part[nb][cols] → out[cols] (dtype TO).  Block (32, 32): threadIdx.x picks a column of a
// 32-column slab, threadIdx.y a slice of partial rows (y, y+32, ...), summed as four running sums
// over b ≡ 0, 1, 2, 3 (mod 4) of the slice so the loads overlap; the sums, then the 32 slice sums,
// are added in a fixed order, so the result does not depend on timing.  blockIdx.y selects one of
// two (part, out) jobs, so two column sums of a kernel finalize in one launch.
struct ColsumJob {
  const float* part;
  void* out;
};
template <typename TO>
__global__ void __launch_bounds__(1024) colsum_finalize(ColsumJob j0, ColsumJob j1, int nb, int64_t cols, int acc) {
  pdl_begin();
  __shared__ float red[32][33];
  const ColsumJob jb = blockIdx.y ? j1 : j0;
  const float* part = jb.part;
  TO* out = static_cast<TO*>(jb.out);
  const int64_t c = int64_t(blockIdx.x) * 32 + threadIdx.x;
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
  if (c < cols) {
    int b = threadIdx.y;
    for (; b + 96 < nb; b += 128) {
      s0 += part[int64_t(b) * cols + c];
      s1 += part[int64_t(b + 32) * cols + c];
      s2 += part[int64_t(b + 64) * cols + c];
      s3 += part[int64_t(b + 96) * cols + c];
    }
    if (b < nb) s0 += part[int64_t(b) * cols + c];
    if (b + 32 < nb) s1 += part[int64_t(b + 32) * cols + c];
    if (b + 64 < nb) s2 += part[int64_t(b + 64) * cols + c];
  }
  red[threadIdx.y][threadIdx.x] = (s0 + s1) + (s2 + s3);
  __syncthreads();
  for (int w = 16; w > 0; w >>= 1) {
    if (threadIdx.y < w) red[threadIdx.y][threadIdx.x] += red[threadIdx.y + w][threadIdx.x];
    __syncthreads();
  }
  if (threadIdx.y == 0 && c < cols) {
    float r = red[0][threadIdx.x];
    if (acc) r += to_f(out[c]);
    out[c] = from_f<TO>(r);
  }
}

// Finalizes one or two column sums (out1 may be null) of `nb` partial rows each.
static int finalize(const float* part, int nb, int64_t cols, void* out, int dt, int acc, cudaStream_t s,
                    const float* part1 = nullptr, void* out1 = nullptr) {
  const dim3 grid(unsigned(ceil_div(cols, 32)), out1 ? 2u : 1u);
  const dim3 block(32, 32);
  const ColsumJob j0{part, out}, j1{part1, out1};
  if (dt == XT_F32) launch(colsum_finalize<float>, grid, block, 0, s, j0, j1, nb, cols, acc);
  else launch(colsum_finalize<bf16>, grid, block, 0, s, j0, j1, nb, cols, acc);
  return check_launch("column-sum finalize");
}

constexpr int kColChunkRows = 64;  // rows per partial in the plain column sum

static int colsum_chunks(int64_t rows) { return int(ceil_div(rows, kColChunkRows)); }

// Plain column sum of d [rows, cols] into one partial row per 64-row chunk (and an optional copy
// dx = d, or dx += d).  A block of 8 warps owns a slab of 32 vectors of VW columns (512 bytes of
// a row per warp access) and one chunk: warp w sums rows w, w + 8, ... of the chunk, four rows in
// flight per thread, and the eight warp sums are added in warp order, so the partials do not
// depend on timing.  VW = 1 is the form for ragged or misaligned rows.
template <typename T, int VW>
__global__ void __launch_bounds__(256) colsum_stage1(const T* __restrict__ d, T* dx, int acc_dx,
                                                     float* __restrict__ part, int64_t rows, int64_t cols) {
  pdl_begin();
  __shared__ float red[8][32 * VW];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t c = (int64_t(blockIdx.x) * 32 + lane) * VW;
  const int64_t r0 = int64_t(blockIdx.y) * kColChunkRows;
  const int64_t r1 = r0 + kColChunkRows < rows ? r0 + kColChunkRows : rows;
  float s[VW];
#pragma unroll
  for (int e = 0; e < VW; ++e) s[e] = 0.f;
  if (c < cols) {
    auto row = [&](int64_t r, const float (&v)[VW]) {
      if (dx) {
        if (acc_dx) {
          float o[VW];
          load_vec<T, VW>(dx + r * cols + c, o);
#pragma unroll
          for (int e = 0; e < VW; ++e) o[e] += v[e];
          store_vec<T, VW>(dx + r * cols + c, o);
        } else {
          store_vec<T, VW>(dx + r * cols + c, v);
        }
      }
#pragma unroll
      for (int e = 0; e < VW; ++e) s[e] += v[e];
    };
    int64_t r = r0 + warp;
    for (; r + 24 < r1; r += 32) {
      float v[4][VW];
#pragma unroll
      for (int k = 0; k < 4; ++k) load_vec<T, VW>(d + (r + 8 * k) * cols + c, v[k]);
#pragma unroll
      for (int k = 0; k < 4; ++k) row(r + 8 * k, v[k]);
    }
    for (; r < r1; r += 8) {
      float v[VW];
      load_vec<T, VW>(d + r * cols + c, v);
      row(r, v);
    }
  }
#pragma unroll
  for (int e = 0; e < VW; ++e) red[warp][lane * VW + e] = s[e];
  __syncthreads();
  for (int t = threadIdx.x; t < 32 * VW; t += blockDim.x) {
    const int64_t cc = int64_t(blockIdx.x) * 32 * VW + t;
    float a = red[0][t];
#pragma unroll
    for (int w = 1; w < 8; ++w) a += red[w][t];
    if (cc < cols) part[int64_t(blockIdx.y) * cols + cc] = a;
  }
}

// ============================================================================== softmax

// Causal rows: the row with query index q reads columns [0, vis) with vis = min(q + 1, cols)
// and writes [0, ext): ext = cols, or, in mode 2, the end of q's 128-wide key block (the extent
// the probability-times-value product reads), columns in [vis, ext) written as zeros.
// Column arithmetic is 32-bit (a row holds at most 32768 elements); the visibility test is
// one integer per 16-byte vector, and only the vector that straddles `vis` is masked per element.
__device__ __forceinline__ int row_query(int64_t r, int64_t q_len, bool small) {
  return small ? int(uint32_t(r) % uint32_t(q_len)) : int(r % q_len);
}
__device__ __forceinline__ int causal_vis(int causal, int q, int cols) {
  return causal ? (q + 1 < cols ? q + 1 : cols) : cols;
}
__device__ __forceinline__ int causal_ext(int causal, int q, int cols) {
  if (causal != 2) return cols;
  const int e = ((q >> 7) + 1) << 7;
  return e < cols ? e : cols;
}

template <typename T, int VW>
__global__ void __launch_bounds__(1024) softmax_fwd_kernel(const T* __restrict__ x, T* __restrict__ y, int64_t rows,
                                                          int cols, int causal, int64_t q_len, int tpr) {
  pdl_begin();
  __shared__ float red[32];
  const int rpb = blockDim.x / tpr, l = threadIdx.x % tpr;
  const bool small = rows <= INT32_MAX && q_len <= INT32_MAX;
  for (int64_t r0 = int64_t(blockIdx.x) * rpb; r0 < rows; r0 += int64_t(gridDim.x) * rpb) {
    const int64_t r = r0 + threadIdx.x / tpr;
    const bool act = r < rows;
    const int q = act ? row_query(r, q_len, small) : 0;
    const int vis = act ? causal_vis(causal, q, cols) : 0;
    const T* xr = x + (act ? r : 0) * int64_t(cols);
    float f[NV][VW];
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int c0 = (l + k * tpr) * VW;
      const int lim = vis - c0;   // visible elements of this vector (<= 0: none, >= VW: all)
      if (lim >= VW) {
        Raw<T, VW> v;
        v.load(xr + c0);
#pragma unroll
        for (int e = 0; e < VW; ++e) f[k][e] = v.get(e);
      } else if (lim > 0) {
        Raw<T, VW> v;
        v.load(xr + c0);
#pragma unroll
        for (int e = 0; e < VW; ++e) f[k][e] = e < lim ? v.get(e) : -INFINITY;
      } else {
#pragma unroll
        for (int e = 0; e < VW; ++e) f[k][e] = -INFINITY;
      }
#pragma unroll
      for (int e = 0; e < VW; ++e) m = fmaxf(m, f[k][e]);
    }
    prefetch_next_row<T, VW>(x, r + int64_t(gridDim.x) * rpb, rows, cols, l, tpr);
    m = group_reduce<true>(m, tpr, red);
    // exp(x − m) = 2^(x·log2 e − m·log2 e): one fma and one exp2 per element; masked
    // elements hold −inf and give exactly 0
    const float ml = act ? m * kLog2e : 0.f;
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        f[k][e] = exp2f(fmaf(f[k][e], kLog2e, -ml));
        s += f[k][e];
      }
    s = group_reduce<false>(s, tpr, red);
    if (!act) continue;
    const float inv = 1.f / s;
    const int ext = causal_ext(causal, q, cols);
    T* yr = y + r * int64_t(cols);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int c0 = (l + k * tpr) * VW;
      if (c0 < ext) {
        float o[VW];
#pragma unroll
        for (int e = 0; e < VW; ++e) o[e] = f[k][e] * inv;
        store_vec<T, VW>(yr + c0, o);
      }
    }
  }
}

// MAXT: the launch's block size bound; 256-thread launches get registers for two packed
// row shares without spilling.
template <typename T, int VW, int MAXT>
__global__ void __launch_bounds__(MAXT, MAXT <= 256 ? 2 : 1) softmax_bwd_kernel(
    const T* __restrict__ d, const T* __restrict__ y, T* dx, int64_t rows, int cols, int causal, int64_t q_len,
    int tpr, int acc) {
  pdl_begin();
  __shared__ float red[32];
  const int rpb = blockDim.x / tpr, l = threadIdx.x % tpr;
  const bool small = rows <= INT32_MAX && q_len <= INT32_MAX;
  for (int64_t r0 = int64_t(blockIdx.x) * rpb; r0 < rows; r0 += int64_t(gridDim.x) * rpb) {
    const int64_t r = r0 + threadIdx.x / tpr;
    const bool act = r < rows;
    const int q = act ? row_query(r, q_len, small) : 0;
    const int vis = act ? causal_vis(causal, q, cols) : 0;
    const int64_t base = (act ? r : 0) * int64_t(cols);
    // packed vectors stay in registers; elements at or past `vis` are zeroed in place, so
    // they add nothing to Σ d·y and come out as y·(d − s) = 0
    Raw<T, VW> vd[NV], vy[NV];
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int c0 = (l + k * tpr) * VW;
      const int lim = vis - c0;
      if (lim > 0) {
        vd[k].load(d + base + c0);
        vy[k].load(y + base + c0);
        if (lim < VW) { vd[k].keep_first(lim); vy[k].keep_first(lim); }
      } else {
        vd[k].zero(); vy[k].zero();
      }
#pragma unroll
      for (int e = 0; e < VW; ++e) s = fmaf(vd[k].get(e), vy[k].get(e), s);
    }
    prefetch_next_row<T, VW>(d, r + int64_t(gridDim.x) * rpb, rows, cols, l, tpr);
    prefetch_next_row<T, VW>(y, r + int64_t(gridDim.x) * rpb, rows, cols, l, tpr);
    s = group_reduce<false>(s, tpr, red);
    if (!act) continue;
    const int ext = causal_ext(causal, q, cols);
    T* p = dx + base;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int c0 = (l + k * tpr) * VW;
      if (c0 < ext) {
        float o[VW];
#pragma unroll
        for (int e = 0; e < VW; ++e) o[e] = fmaf(vy[k].get(e), vd[k].get(e) - s, 0.f);
        if (acc) {
          float old[VW];
          load_vec<T, VW>(p + c0, old);
#pragma unroll
          for (int e = 0; e < VW; ++e) o[e] += old[e];
        }
        store_vec<T, VW>(p + c0, o);
      }
    }
  }
}

// ============================================================================== cross-entropy

// Streaming online log-sum-exp over one row per row group; writes lse[r] and nll[r].
template <typename T, int VW>
__global__ void __launch_bounds__(1024) ce_fwd_kernel(const T* __restrict__ x, const int32_t* __restrict__ tgt,
                                                     float* __restrict__ lse, float* __restrict__ nll, int64_t rows,
                                                     int64_t V, int tpr, uint32_t* flag) {
  pdl_begin();
  __shared__ float red_m[32], red_s[32];
  const int rpb = blockDim.x / tpr, l = threadIdx.x % tpr;
  const int64_t nvec = V / VW;
  for (int64_t r0 = int64_t(blockIdx.x) * rpb; r0 < rows; r0 += int64_t(gridDim.x) * rpb) {
    const int64_t r = r0 + threadIdx.x / tpr;
    const bool act = r < rows;
    // per thread: running max m and s = Σ exp(x − m); s is rescaled only when a vector raises
    // the max, so each logit costs one hardware exp2 (ex2.approx, relative error ~2⁻²²)
    // four vectors per step, all four loads issued before any is used
    float m = -INFINITY, s = 0.f;
    if (act) {
      const T* row = x + r * V;
      for (int64_t j0 = l; j0 < nvec; j0 += 4 * int64_t(tpr)) {
        float v[4][VW];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t j = j0 + int64_t(u) * tpr;
          if (j < nvec) load_vec<T, VW>(row + j * VW, v[u]);
          else
#pragma unroll
            for (int e = 0; e < VW; ++e) v[u][e] = -INFINITY;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float vm = v[u][0];
#pragma unroll
          for (int e = 1; e < VW; ++e) vm = fmaxf(vm, v[u][e]);
          if (vm > m) {
            s = (m == -INFINITY) ? 0.f : s * fast_exp2((m - vm) * kLog2e);
            m = vm;
          }
          const float ml = m * kLog2e;
          float vs = 0.f;
#pragma unroll
          for (int e = 0; e < VW; ++e) vs += fast_exp2(fmaf(v[u][e], kLog2e, -ml));
          s += vs;
        }
      }
    }
    // row-group merge of (m, s): warp shuffle, then shared memory across warps
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
      lse_merge(m, s, m2, s2);
    }
    if (tpr > 32) {
      const int warp = threadIdx.x >> 5, wpg = tpr >> 5, g0 = (warp / wpg) * wpg;
      __syncthreads();
      if ((threadIdx.x & 31) == 0) { red_m[warp] = m; red_s[warp] = s; }
      __syncthreads();
      m = red_m[g0]; s = red_s[g0];
      for (int w = 1; w < wpg; ++w) lse_merge(m, s, red_m[g0 + w], red_s[g0 + w]);
    }
    if (act && l == 0) {
      const float L = m + logf(s);
      lse[r] = L;
      const int32_t t = tgt[r];
      if (t < 0 || int64_t(t) >= V) {
        flag_error(flag, XT_DEVERR_INDEX);
        nll[r] = __int_as_float(0x7fc00000);
      } else {
        nll[r] = L - to_f(x[r * V + t]);
      }
    }
  }
}

// loss = Σ nll / rows in a fixed order (one block).
__global__ void ce_loss_kernel(const float* __restrict__ nll, int64_t rows, float* loss) {
  pdl_begin();
  __shared__ float red[32];
  float acc = 0.f;
  for (int64_t i = threadIdx.x; i < rows; i += blockDim.x) acc += nll[i];
  acc = warp_sum(acc);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < int(blockDim.x >> 5); ++w) s += red[w];
    *loss = s / float(rows);
  }
}

// dx = (upstream / rows)·(exp(x − lse) − onehot(t)).  Blocks walk rows; threads walk a
// row's vectors (no per-element index division).
template <typename T, typename TG, int VW>
__global__ void __launch_bounds__(256) ce_bwd_kernel(const T* x, const int32_t* __restrict__ tgt,
                                                    const float* __restrict__ lse, const float* __restrict__ upstream,
                                                    TG* dx, int64_t rows, int64_t V, int acc, uint32_t* flag) {
  pdl_begin();
  const float sc = *upstream / float(rows);
  const int64_t nvec = V / VW;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const float Ll = lse[r] * kLog2e;
    const int32_t t = tgt[r];
    const bool bad = t < 0 || int64_t(t) >= V;
    if (bad && threadIdx.x == 0) flag_error(flag, XT_DEVERR_INDEX);
    const T* xr = x + r * V;
    TG* dr = dx + r * V;
    for (int64_t j = threadIdx.x; j < nvec; j += blockDim.x) {
      const int64_t c = j * VW;
      float xv[VW], o[VW];
      load_vec<T, VW>(xr + c, xv);
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        const float p = fast_exp2(fmaf(xv[e], kLog2e, -Ll));
        o[e] = bad ? __int_as_float(0x7fc00000) : sc * (p - (c + e == t ? 1.f : 0.f));
      }
      if (acc) {
        float old[VW];
        load_vec<TG, VW>(dr + c, old);
#pragma unroll
        for (int e = 0; e < VW; ++e) o[e] += old[e];
      }
      store_vec<TG, VW>(dr + c, o);
    }
  }
}

// Forward and backward of the mean cross-entropy in one pass over the logits (training, the
// loss being the graph's root): one block per row at a time holds the row in shared memory
// (read from HBM once), forms max, Σ exp(x − max) and lse from it, writes lse[r] and
// nll[r] = lse − x[t], then dx = (upstream / rows)·(exp(x − lse) − onehot(t)) (dx may be x).
constexpr int kCeFusedThreads = 512;

template <typename T, typename TG>
__global__ void __launch_bounds__(kCeFusedThreads) ce_fused_kernel(const T* x, const int32_t* __restrict__ tgt,
                                                                   float* __restrict__ lse, float* __restrict__ nll,
                                                                   const float* __restrict__ upstream, TG* dx,
                                                                   int64_t rows, int64_t V, uint32_t* flag) {
  pdl_begin();
  extern __shared__ __align__(16) uint8_t ce_row_raw[];
  T* row_s = reinterpret_cast<T*>(ce_row_raw);
  __shared__ float red[kCeFusedThreads / 32];
  constexpr int VW = 16 / sizeof(T);
  const float sc = *upstream / float(rows);
  const int64_t nvec = V / VW;  // V % VW == 0 (checked on the host)
  auto block_reduce = [&](float v, bool is_max) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float w = __shfl_xor_sync(0xffffffffu, v, o);
      v = is_max ? fmaxf(v, w) : v + w;
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = red[0];
    for (int i = 1; i < kCeFusedThreads / 32; ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
    return r;
  };
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const T* xr = x + r * V;
    // 1. the row into shared memory (16-byte vectors, several in flight), running max
    float m = -INFINITY;
    for (int64_t j = threadIdx.x; j < nvec; j += kCeFusedThreads) {
      const uint4 u = __ldcs(reinterpret_cast<const uint4*>(xr) + j);
      reinterpret_cast<uint4*>(row_s)[j] = u;
      float v[VW];
      load_vec<T, VW>(reinterpret_cast<const T*>(&u), v);
#pragma unroll
      for (int e = 0; e < VW; ++e) m = fmaxf(m, v[e]);
    }
    m = block_reduce(m, true);
    // the block's next row is asked of L2 now, so its copy into shared memory after this row's
    // two passes over shared memory and its gradient stores does not wait on DRAM
    if (r + gridDim.x < rows) {
      const T* xn = x + (r + gridDim.x) * V;
      for (int64_t j = int64_t(threadIdx.x) * 8; j < nvec; j += int64_t(kCeFusedThreads) * 8)
        prefetch_l2(reinterpret_cast<const uint4*>(xn) + j);
    }
    // 2. Σ exp(x − max) from shared memory
    const float ml = m * kLog2e;
    float s = 0.f;
    for (int64_t j = threadIdx.x; j < nvec; j += kCeFusedThreads) {
      float v[VW];
      load_vec<T, VW>(row_s + j * VW, v);
#pragma unroll
      for (int e = 0; e < VW; ++e) s += fast_exp2(fmaf(v[e], kLog2e, -ml));
    }
    s = block_reduce(s, false);
    const float L = m + logf(s);
    const int32_t t = tgt[r];
    const bool bad = t < 0 || int64_t(t) >= V;
    if (threadIdx.x == 0) {
      lse[r] = L;
      if (bad) {
        flag_error(flag, XT_DEVERR_INDEX);
        nll[r] = __int_as_float(0x7fc00000);
      } else {
        nll[r] = L - to_f(row_s[t]);
      }
    }
    // 3. the gradient from shared memory
    const float Ll = L * kLog2e;
    TG* dr = dx + r * V;
    for (int64_t j = threadIdx.x; j < nvec; j += kCeFusedThreads) {
      const int64_t c = j * VW;
      float v[VW], o[VW];
      load_vec<T, VW>(row_s + c, v);
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        const float pr = fast_exp2(fmaf(v[e], kLog2e, -Ll));
        o[e] = bad ? __int_as_float(0x7fc00000) : sc * (pr - (c + e == t ? 1.f : 0.f));
      }
      store_vec<TG, VW>(dr + c, o);
    }
    __syncthreads();  // the next row overwrites the shared row
  }
}

// ============================================================================== RoPE

__global__ void rope_table_kernel(float* table, int S, int hd, double base, int pos_offset) {
  pdl_begin();
  const int h = hd / 2;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < S * h; idx += gridDim.x * blockDim.x) {
    const int s = idx / h, i = idx - s * h;
    const double th = double(pos_offset + s) * pow(base, -2.0 * double(i) / double(hd));
    double sn, cs;
    sincos(th, &sn, &cs);
    table[idx] = float(cs);
    table[S * h + idx] = float(sn);
  }
}

// BWD = false: y_i = x_i c − x_{i+h} s; y_{i+h} = x_{i+h} c + x_i s
// BWD = true:  dx_i = d_i c + d_{i+h} s; dx_{i+h} = d_{i+h} c − d_i s
template <typename T, bool BWD, int VW>
__global__ void __launch_bounds__(256) rope_kernel(const T* x, T* y, const float* __restrict__ table, int B, int S,
                                                  int H, int hd, int64_t ld, int acc) {
  pdl_begin();
  const int h = hd / 2;
  const int per_head = h / VW;
  const int64_t total = int64_t(B) * S * H * per_head;
  const float* ct = table;
  const float* st = table + int64_t(S) * h;
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < total; v += int64_t(gridDim.x) * blockDim.x) {
    const int64_t tok_head = v / per_head;
    const int i0 = int(v - tok_head * per_head) * VW;
    const int64_t tok = tok_head / H;
    const int head = int(tok_head - tok * H);
    const int s = int(tok % S);
    const int64_t off = tok * ld + int64_t(head) * hd + i0;
    float a[VW], b[VW], c[VW], sn[VW], o1[VW], o2[VW];
    load_vec<T, VW>(x + off, a);
    load_vec<T, VW>(x + off + h, b);
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      c[e] = ct[int64_t(s) * h + i0 + e];
      sn[e] = st[int64_t(s) * h + i0 + e];
    }
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      if (BWD) {
        o1[e] = a[e] * c[e] + b[e] * sn[e];
        o2[e] = b[e] * c[e] - a[e] * sn[e];
      } else {
        o1[e] = a[e] * c[e] - b[e] * sn[e];
        o2[e] = b[e] * c[e] + a[e] * sn[e];
      }
    }
    if (acc) {
      float p1[VW], p2[VW];
      load_vec<T, VW>(y + off, p1);
      load_vec<T, VW>(y + off + h, p2);
#pragma unroll
      for (int e = 0; e < VW; ++e) { o1[e] += p1[e]; o2[e] += p2[e]; }
    }
    store_vec<T, VW>(y + off, o1);
    store_vec<T, VW>(y + off + h, o2);
  }
}

// ============================================================================== embedding

template <typename T, int VW>
__global__ void __launch_bounds__(256) embed_fwd_kernel(const int32_t* __restrict__ ids, const T* __restrict__ E,
                                                       const T* __restrict__ P, T* __restrict__ h, int64_t T_,
                                                       int S, int64_t d, int64_t V, uint32_t* flag) {
  pdl_begin();
  const int64_t per = d / VW;
  const int64_t total = T_ * per;
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < total; v += int64_t(gridDim.x) * blockDim.x) {
    const int64_t t = v / per, c = (v - t * per) * VW;
    const int32_t id = ids[t];
    float o[VW];
    if (id < 0 || int64_t(id) >= V) {
      if (c == 0) flag_error(flag, XT_DEVERR_INDEX);
#pragma unroll
      for (int e = 0; e < VW; ++e) o[e] = __int_as_float(0x7fc00000);
    } else {
      load_vec<T, VW>(E + int64_t(id) * d + c, o);
      if (P) {
        float p[VW];
        load_vec<T, VW>(P + int64_t(t % S) * d + c, p);
#pragma unroll
        for (int e = 0; e < VW; ++e) o[e] += p[e];
      }
    }
    store_vec<T, VW>(h + t * d + c, o);
  }
}

constexpr int kSortMax = 16384;
constexpr int kEmbThreads = 512;

// dE[v] (+)= Σ_{t: ids[t] = v} dh[t], the sum formed in float32 in ascending t and then added
// to dE[v].  Block b owns the ids [b·per, (b+1)·per): it lists, in ascending t, the tokens
// whose id falls in its range (each warp compacts a contiguous range of t with ballots, the
// warps' lists joined in warp order: two block barriers in all), then warp w takes the ids
// v0 + w, v0 + w + warps, …: for each it walks the list in order and sums the rows of the
// tokens with that id, 8 columns per lane per pass (lane-interleaved, coalesced).  Ids outside
// [0, V) set XT_DEVERR_INDEX (block 0) and are skipped.  No sort and no atomics.
template <typename TH, typename TG>
__global__ void __launch_bounds__(kEmbThreads) embed_bwd_kernel(const int32_t* __restrict__ ids,
                                                                const TH* __restrict__ dh, TG* dE, int T_,
                                                                int64_t d, int64_t V, int64_t per, uint32_t* flag) {
  pdl_begin();
  extern __shared__ int emb_list[];   // [T] token indices, then [T] their ids
  __shared__ int warp_base[kEmbThreads / 32];
  __shared__ int total;
  int* lt = emb_list;
  int* lid = emb_list + T_;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  constexpr int NW = kEmbThreads / 32;
  const int64_t v0 = int64_t(blockIdx.x) * per;
  const int64_t v1 = v0 + per < V ? v0 + per : V;
  // Warp w lists the tokens of its own contiguous range [w·cw, (w + 1)·cw) that fall in this
  // block's id range: a count pass, one barrier for the warps' offsets (ranges in warp order, so
  // the list is in ascending t), then a write pass; the ids are loaded once, before either pass.
  const int cw = ((T_ + NW - 1) / NW + 31) & ~31;
  const int t_begin = w * cw;
  constexpr int kPer = kSortMax / kEmbThreads;  // rounds of 32 ids a warp can have
  int32_t idv[kPer];
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int t = t_begin + r * 32 + lane;
    idv[r] = (r * 32 < cw && t < T_) ? __ldg(ids + t) : -1;
  }
  auto match = [&](int r) {
    const int32_t id = idv[r];
    return id >= 0 && int64_t(id) < V && int64_t(id) >= v0 && int64_t(id) < v1;
  };
  int cnt = 0;
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    if (r * 32 >= cw) break;
    const int t = t_begin + r * 32 + lane;
    if (blockIdx.x == 0 && t < T_ && (idv[r] < 0 || int64_t(idv[r]) >= V)) flag_error(flag, XT_DEVERR_INDEX);
    cnt += __popc(__ballot_sync(0xffffffffu, match(r)));
  }
  if (lane == 0) warp_base[w] = cnt;
  __syncthreads();
  int pos = 0, all = 0;
  for (int i = 0; i < NW; ++i) {
    const int c = warp_base[i];
    pos += i < w ? c : 0;
    all += c;
  }
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    if (r * 32 >= cw) break;
    const bool m = match(r);
    const unsigned bal = __ballot_sync(0xffffffffu, m);
    if (m) {
      const int k = pos + __popc(bal & ((1u << lane) - 1u));
      lt[k] = t_begin + r * 32 + lane;
      lid[k] = idv[r];
    }
    pos += __popc(bal);
  }
  if (threadIdx.x == 0) total = all;
  __syncthreads();
  const int count = total;
  for (int64_t v = v0 + w; v < v1; v += NW) {
    for (int64_t c0 = 0; c0 < d; c0 += 32 * 8) {
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.f;
      bool any = false;
      for (int k = 0; k < count; ++k) {
        if (lid[k] != int(v)) continue;
        any = true;
        const TH* row = dh + int64_t(lt[k]) * d;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int64_t c = c0 + lane + 32 * e;
          if (c < d) acc[e] += to_f(row[c]);
        }
      }
      if (!any) break;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int64_t c = c0 + lane + 32 * e;
        if (c < d) {
          TG* q = dE + v * d + c;
          *q = from_f<TG>(to_f(*q) + acc[e]);
        }
      }
    }
  }
}

// dP[s] (+)= Σ_b dh[b·S + s]
template <typename TH, typename TG>
__global__ void __launch_bounds__(256) embed_pos_kernel(const TH* __restrict__ dh, TG* dP, int64_t T_, int S, int64_t d,
                                                       int acc) {
  pdl_begin();
  const int64_t nb = T_ / S;
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < int64_t(S) * d; v += int64_t(gridDim.x) * blockDim.x) {
    const int64_t s = v / d, c = v - s * d;
    float a = 0.f;
    for (int64_t b = 0; b < nb; ++b) a += to_f(dh[(b * S + s) * d + c]);
    if (acc) a += to_f(dP[v]);
    dP[v] = from_f<TG>(a);
  }
}

// ============================================================================== launch helpers

#define XT_ROW_DISPATCH(dt, vec, ...)                         \
  do {                                                        \
    if ((dt) == XT_F32) {                                     \
      using T = float;                                        \
      if (vec) { constexpr int VW = 4; __VA_ARGS__; }         \
      else { constexpr int VW = 1; __VA_ARGS__; }             \
    } else {                                                  \
      using T = bf16;                                         \
      if (vec) { constexpr int VW = 8; __VA_ARGS__; }         \
      else { constexpr int VW = 1; __VA_ARGS__; }             \
    }                                                         \
  } while (0)

constexpr int kBwdMaxTpr = 512;  // backward row kernels hold two rows + partials in registers

// (T, TD) pairs for the norm backward: dx in the activation dtype, or fp32 from bf16.
#define XT_NORM_BWD_DISPATCH(dt, dt_dx, vec, ...)                              \
  do {                                                                         \
    if ((dt) == XT_F32) {                                                      \
      using T = float; using TD = float;                                       \
      if (vec) { constexpr int VW = 4; __VA_ARGS__; }                          \
      else { constexpr int VW = 1; __VA_ARGS__; }                              \
    } else if ((dt_dx) == XT_BF16) {                                           \
      using T = bf16; using TD = bf16;                                         \
      if (vec) { constexpr int VW = 8; __VA_ARGS__; }                          \
      else { constexpr int VW = 1; __VA_ARGS__; }                              \
    } else {                                                                   \
      using T = bf16; using TD = float;                                        \
      if (vec) { constexpr int VW = 8; __VA_ARGS__; }                          \
      else { constexpr int VW = 1; __VA_ARGS__; }                              \
    }                                                                          \
  } while (0)

// LayerNorm backward plan: a bf16 row that the default plan gives four vectors per thread runs
// with twice the threads and two vectors each instead, since four vectors of bf16 plus both
// sets of (dγ, dβ) partials do not fit in the 128 registers of two resident blocks, as long as
// that stays within 256-thread blocks (a 512-thread row, one block per SM, measured slower than
// the spilling plan).
static RowPlan ln_bwd_plan(int64_t cols, int vw) {
  RowPlan pl = plan_rows(cols, vw, kBwdMaxTpr);
  if (pl.ok && vw == 8 && ceil_div(ceil_div(cols, vw), pl.tpr) == NV) {
    const RowPlan p2 = plan_rows(cols, vw, kBwdMaxTpr, 2);
    if (p2.ok && p2.threads <= 256) pl = p2;
  }
  return pl;
}

static size_t norm_ws_floats(int64_t rows, int64_t cols, int vw, bool ln = false) {
  RowPlan pl = ln ? ln_bwd_plan(cols, vw) : plan_rows(cols, vw, kBwdMaxTpr);
  if (!pl.ok) return 0;
  return size_t(bwd_blocks(rows, pl.rpb)) * size_t(cols);
}

}  // namespace xt

// ==================================================================================== C ABI
using namespace xt;

extern "C" {

int xt_norm_bwd_workspace_size(int64_t rows, int64_t cols, size_t* bytes) {
  XT_REQUIRE(rows >= 0 && cols > 0 && bytes, "xt_norm_bwd_workspace_size: bad arguments");
  // the scalar path (vector width 1) has the most row groups per block: take the max
  size_t f = norm_ws_floats(rows, cols, 1);
  for (const size_t fv : {norm_ws_floats(rows, cols, 4), norm_ws_floats(rows, cols, 8),
                          norm_ws_floats(rows, cols, 8, true)})
    if (fv > f) f = fv;
  *bytes = 2 * f * sizeof(float);
  return XT_OK;
}

int xt_rms_norm_fwd(const void* x, const void* gamma, void* y, float* inv_rms, int64_t rows, int64_t cols,
                    float eps, int dt, void* stream) {
  XT_REQUIRE(valid_dtype(dt), "xt_rms_norm_fwd: bad dtype");
  XT_REQUIRE(rows >= 0 && cols > 0, "xt_rms_norm_fwd: bad sizes");
  XT_REQUIRE(rows == 0 || (x && gamma && y && inv_rms), "xt_rms_norm_fwd: NULL pointer");
  if (rows == 0) return XT_OK;
  const bool vec = rows_vec_ok(cols, dt, {x, gamma, y});
  RowPlan pl = plan_rows(cols, vec ? (dt == XT_BF16 ? 8 : 4) : 1);
  if (!pl.ok) return fail(XT_ERR_UNSUPPORTED, "xt_rms_norm_fwd: row too long (%lld)", (long long)cols);
  cudaStream_t s = as_stream(stream);
  const int grid = row_grid(rows, pl.rpb);
  XT_ROW_DISPATCH(dt, vec, (launch(rms_fwd_kernel<T, VW>, grid, pl.threads, 0, s, 
                               static_cast<const T*>(x), static_cast<const T*>(gamma), static_cast<T*>(y), inv_rms,
                               rows, cols, eps, pl.tpr)));
  return check_launch("xt_rms_norm_fwd");
}

static int rms_bwd_impl(const void* d, const void* x, const void* gamma, const float* inv_rms, void* dx, void* dgamma,
                        int64_t rows, int64_t cols, int dt, int dt_dx, int dt_param, void* ws, int acc_dx, int acc_param,
                        void* stream, GradOut go) {
  XT_REQUIRE(valid_dtype(dt) && valid_dtype(dt_dx) && valid_dtype(dt_param), "xt_rms_norm_bwd: bad dtype");
  XT_REQUIRE(dt_dx == dt || (dt == XT_BF16 && dt_dx == XT_F32), "xt_rms_norm_bwd: dx dtype must be dt or f32");
  XT_REQUIRE(rows >= 0 && cols > 0, "xt_rms_norm_bwd: bad sizes");
  XT_REQUIRE(rows == 0 || (d && x && gamma && inv_rms), "xt_rms_norm_bwd: NULL input");
  XT_REQUIRE(!dgamma || ws, "xt_rms_norm_bwd: dgamma needs a workspace");
  cudaStream_t s = as_stream(stream);
  if (rows == 0) {
    if (dgamma && !acc_param)
      if (cudaMemsetAsync(dgamma, 0, size_t(cols) * dtype_size(dt_param), s) != cudaSuccess)
        return check_launch("xt_rms_norm_bwd");
    return XT_OK;
  }
  const bool vec = rows_vec_ok(cols, dt, {d, x, gamma, dx});
  RowPlan pl = plan_rows(cols, vec ? (dt == XT_BF16 ? 8 : 4) : 1, kBwdMaxTpr);
  if (!pl.ok) return fail(XT_ERR_UNSUPPORTED, "xt_rms_norm_bwd: row too long (%lld)", (long long)cols);
  const int nb = bwd_blocks(rows, pl.rpb);
  float* part = dgamma ? static_cast<float*>(ws) : nullptr;
  const size_t smem = (32 + size_t(pl.rpb) * size_t(cols)) * sizeof(float);
  if (smem > 200 * 1024) return fail(XT_ERR_UNSUPPORTED, "xt_rms_norm_bwd: row too long");
  XT_NORM_BWD_DISPATCH(dt, dt_dx, vec, {
    auto k = pl.threads <= 256 ? rms_bwd_kernel<T, TD, VW, 256> : rms_bwd_kernel<T, TD, VW, 512>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    launch(k, nb, pl.threads, smem, s, static_cast<const T*>(d), static_cast<const T*>(x), static_cast<const T*>(gamma),
                                   inv_rms, static_cast<TD*>(dx), part, rows, cols, pl.tpr, acc_dx, go);
  });
  XT_TRY(check_launch("xt_rms_norm_bwd"));
  if (dgamma) return finalize(part, nb, cols, dgamma, dt_param, acc_param, s);
  return XT_OK;
}

int xt_rms_norm_bwd(const void* d, const void* x, const void* gamma, const float* inv_rms, void* dx, void* dgamma,
                    int64_t rows, int64_t cols, int dt, int dt_dx, int dt_param, void* ws, int acc_dx, int acc_param,
                    void* stream) {
  return rms_bwd_impl(d, x, gamma, inv_rms, dx, dgamma, rows, cols, dt, dt_dx, dt_param, ws, acc_dx, acc_param, stream,
                      GradOut{});
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// Allocation-free RMSNorm backward.  Its per-block dγ partial rows live in this file-scope
// device array instead of caller workspace; every GPU that loads libxt holds the 4 MiB until
// the process exits.  Host code may not hand the array's name to a kernel (on the host it is
// only a stand-in for the symbol): the device address is looked up per device with
// cudaGetSymbolAddress, once, and cached.
namespace {
constexpr int kNoAllocMaxBlocks = 128;
constexpr int64_t kNoAllocMaxCols = 8192;
__device__ __align__(256) float g_rms_bwd_scratch[kNoAllocMaxBlocks * kNoAllocMaxCols];
constexpr int kNoAllocDevices = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kNoAllocDevices] = {};

int noalloc_scratch(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocDevices)
    return fail(XT_ERR_CUDA, "xt_rms_norm_bwd_noalloc: no usable current device");
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_rms_bwd_scratch);
    if (e != cudaSuccess)
      return fail(XT_ERR_CUDA, "xt_rms_norm_bwd_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return XT_OK;
}
}  // namespace

extern "C" {

int xt_rms_norm_bwd_noalloc(const void* d, const void* x, const void* gamma, const float* inv_rms, void* dx,
                            void* dgamma, int64_t rows, int64_t cols, int dt, int dt_dx, int dt_param, int acc_dx,
                            int acc_param, void* stream) {
  XT_REQUIRE(valid_dtype(dt) && valid_dtype(dt_dx) && valid_dtype(dt_param), "xt_rms_norm_bwd_noalloc: bad dtype");
  XT_REQUIRE(dt_dx == dt || (dt == XT_BF16 && dt_dx == XT_F32), "xt_rms_norm_bwd_noalloc: dx dtype must be dt or f32");
  XT_REQUIRE(rows >= 0 && cols > 0, "xt_rms_norm_bwd_noalloc: bad sizes");
  XT_REQUIRE(rows == 0 || (d && x && gamma && inv_rms), "xt_rms_norm_bwd_noalloc: NULL input");
  if (cols > kNoAllocMaxCols)
    return fail(XT_ERR_UNSUPPORTED, "xt_rms_norm_bwd_noalloc: cols = %lld exceeds the fixed scratch limit of %lld",
                (long long)cols, (long long)kNoAllocMaxCols);
  cudaStream_t s = as_stream(stream);
  if (rows == 0) {
    if (dgamma && !acc_param)
      if (cudaMemsetAsync(dgamma, 0, size_t(cols) * dtype_size(dt_param), s) != cudaSuccess)
        return check_launch("xt_rms_norm_bwd_noalloc");
    return XT_OK;
  }
  float* part = nullptr;
  if (dgamma) XT_TRY(noalloc_scratch(&part));
  const bool vec = rows_vec_ok(cols, dt, {d, x, gamma, dx});
  RowPlan pl = plan_rows(cols, vec ? (dt == XT_BF16 ? 8 : 4) : 1, kBwdMaxTpr);
  if (!pl.ok) return fail(XT_ERR_UNSUPPORTED, "xt_rms_norm_bwd_noalloc: row too long (%lld)", (long long)cols);
  int nb = bwd_blocks(rows, pl.rpb);
  if (nb > kNoAllocMaxBlocks) nb = kNoAllocMaxBlocks;   // each block loops over its share of rows
  const size_t smem = (32 + size_t(pl.rpb) * size_t(cols)) * sizeof(float);
  XT_NORM_BWD_DISPATCH(dt, dt_dx, vec, {
    auto k = pl.threads <= 256 ? rms_bwd_kernel<T, TD, VW, 256> : rms_bwd_kernel<T, TD, VW, 512>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    launch(k, nb, pl.threads, smem, s, static_cast<const T*>(d), static_cast<const T*>(x), static_cast<const T*>(gamma),
                                   inv_rms, static_cast<TD*>(dx), part, rows, cols, pl.tpr, acc_dx, GradOut{});
  });
  XT_TRY(check_launch("xt_rms_norm_bwd_noalloc"));
  if (dgamma) return finalize(part, nb, cols, dgamma, dt_param, acc_param, s);
  return XT_OK;
}

int xt_layernorm_fwd(const void* x, const void* gamma, const void* beta, void* y, float* mean, float* rstd,
                     int64_t rows, int64_t cols, float eps, int dt, void* stream) {
  XT_REQUIRE(valid_dtype(dt), "xt_layernorm_fwd: bad dtype");
  XT_REQUIRE(rows >= 0 && cols > 0, "xt_layernorm_fwd: bad sizes");
  XT_REQUIRE(rows == 0 || (x && gamma && beta && y && mean && rstd), "xt_layernorm_fwd: NULL pointer");
  if (rows == 0) return XT_OK;
  const bool vec = rows_vec_ok(cols, dt, {x, gamma, beta, y});
  RowPlan pl = plan_rows(cols, vec ? (dt == XT_BF16 ? 8 : 4) : 1);
  if (!pl.ok) return fail(XT_ERR_UNSUPPORTED, "xt_layernorm_fwd: row too long");
  cudaStream_t s = as_stream(stream);
  const int grid = row_grid(rows, pl.rpb);
  XT_ROW_DISPATCH(dt, vec, (launch(ln_fwd_kernel<T, VW>, grid, pl.threads, 0, s, 
                               static_cast<const T*>(x), static_cast<const T*>(gamma), static_cast<const T*>(beta),
                               static_cast<T*>(y), mean, rstd, rows, cols, eps, pl.tpr)));
  return check_launch("xt_layernorm_fwd");
}

static int ln_bwd_impl(const void* d, const void* x, const void* gamma, const float* mean, const float* rstd, void* dx,
                       void* dgamma, void* dbeta, int64_t rows, int64_t cols, int dt, int dt_dx, int dt_param, void* ws,
                       int acc_dx, int acc_param, void* stream, GradOut go) {
  XT_REQUIRE(valid_dtype(dt) && valid_dtype(dt_dx) && valid_dtype(dt_param), "xt_layernorm_bwd: bad dtype");
  XT_REQUIRE(dt_dx == dt || (dt == XT_BF16 && dt_dx == XT_F32), "xt_layernorm_bwd: dx dtype must be dt or f32");
  XT_REQUIRE(rows >= 0 && cols > 0, "xt_layernorm_bwd: bad sizes");
  XT_REQUIRE(rows == 0 || (d && x && gamma && mean && rstd), "xt_layernorm_bwd: NULL input");
  XT_REQUIRE(!(dgamma || dbeta) || ws, "xt_layernorm_bwd: parameter grads need a workspace");
  cudaStream_t s = as_stream(stream);
  if (rows == 0) {
    for (void* p : {dgamma, dbeta})
      if (p && !acc_param && cudaMemsetAsync(p, 0, size_t(cols) * dtype_size(dt_param), s) != cudaSuccess)
        return check_launch("xt_layernorm_bwd");
    return XT_OK;
  }
  const bool vec = rows_vec_ok(cols, dt, {d, x, gamma, dx});
  RowPlan pl = ln_bwd_plan(cols, vec ? (dt == XT_BF16 ? 8 : 4) : 1);
  if (!pl.ok) return fail(XT_ERR_UNSUPPORTED, "xt_layernorm_bwd: row too long");
  // two blocks per SM are resident (128 registers × 256 threads), and the partials live in
  // registers across rows: more blocks would only add partial rows to fold
  int nb = bwd_blocks(rows, pl.rpb);
  if (nb > 2 * num_sms()) nb = 2 * num_sms();
  float* part_g = dgamma ? static_cast<float*>(ws) : nullptr;
  float* part_b = dbeta ? static_cast<float*>(ws) + size_t(nb) * size_t(cols) : nullptr;
  const size_t smem = (32 + 2 * size_t(pl.rpb) * size_t(cols)) * sizeof(float);
  if (smem > 200 * 1024) return fail(XT_ERR_UNSUPPORTED, "xt_layernorm_bwd: row too long");
  const int64_t nvt = ceil_div(ceil_div(cols, pl.vw), pl.tpr);  // vectors per thread (1..NV)
  XT_NORM_BWD_DISPATCH(dt, dt_dx, vec, {
    void (*k)(const T*, const T*, const T*, const float*, const float*, TD*, float*, float*, int64_t, int64_t, int,
              int, GradOut) = nullptr;
    const bool narrow = pl.threads <= 256;
    switch (nvt) {
      case 1: k = narrow ? ln_bwd_kernel<T, TD, VW, 1, 256> : ln_bwd_kernel<T, TD, VW, 1, 512>; break;
      case 2: k = narrow ? ln_bwd_kernel<T, TD, VW, 2, 256> : ln_bwd_kernel<T, TD, VW, 2, 512>; break;
      case 3: k = narrow ? ln_bwd_kernel<T, TD, VW, 3, 256> : ln_bwd_kernel<T, TD, VW, 3, 512>; break;
      default: k = narrow ? ln_bwd_kernel<T, TD, VW, 4, 256> : ln_bwd_kernel<T, TD, VW, 4, 512>; break;
    }
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    launch(k, nb, pl.threads, smem, s, static_cast<const T*>(d), static_cast<const T*>(x), static_cast<const T*>(gamma),
                                   mean, rstd, static_cast<TD*>(dx), part_g, part_b, rows, cols, pl.tpr, acc_dx, go);
  });
  XT_TRY(check_launch("xt_layernorm_bwd"));
  if (dgamma && dbeta) return finalize(part_g, nb, cols, dgamma, dt_param, acc_param, s, part_b, dbeta);
  if (dgamma) return finalize(part_g, nb, cols, dgamma, dt_param, acc_param, s);
  if (dbeta) return finalize(part_b, nb, cols, dbeta, dt_param, acc_param, s);
  return XT_OK;
}

int xt_layernorm_bwd(const void* d, const void* x, const void* gamma, const float* mean, const float* rstd, void* dx,
                     void* dgamma, void* dbeta, int64_t rows, int64_t cols, int dt, int dt_dx, int dt_param, void* ws,
                     int acc_dx, int acc_param, void* stream) {
  return ln_bwd_impl(d, x, gamma, mean, rstd, dx, dgamma, dbeta, rows, cols, dt, dt_dx, dt_param, ws, acc_dx, acc_param,
                     stream, GradOut{});
}

int xt_dropout_add_norm_fwd(const void* h, const void* a, void* sum, const void* gamma, const void* beta, void* y,
                            float* stat0, float* stat1, int64_t rows, int64_t cols, float p, uint64_t seed,
                            int training, int norm, float eps, int dt, void* stream) {
  XT_REQUIRE(valid_dtype(dt), "xt_dropout_add_norm_fwd: bad dtype");
  XT_REQUIRE(norm == XT_NORM_RMS || norm == XT_NORM_LN, "xt_dropout_add_norm_fwd: bad norm");
  XT_REQUIRE(rows >= 0 && cols > 0, "xt_dropout_add_norm_fwd: bad sizes");
  XT_REQUIRE(p >= 0.f && p < 1.f, "xt_dropout_add_norm_fwd: p must be in [0, 1)");
  XT_REQUIRE(rows == 0 || (h && a && sum && gamma && y && stat0 && (norm == XT_NORM_RMS || (beta && stat1))),
             "xt_dropout_add_norm_fwd: NULL pointer");
  if (rows == 0) return XT_OK;
  const bool vec = rows_vec_ok(cols, dt, {h, a, sum, gamma, beta, y});
  RowPlan pl = plan_rows(cols, vec ? (dt == XT_BF16 ? 8 : 4) : 1);
  if (!pl.ok) return fail(XT_ERR_UNSUPPORTED, "xt_dropout_add_norm_fwd: row too long");
  cudaStream_t s = as_stream(stream);
  const int grid = row_grid(rows, pl.rpb);
  const int drop = (training && p > 0.f) ? 1 : 0;
  const float dscale = float(1.0 / (1.0 - double(p)));
  if (norm == XT_NORM_LN)
    XT_ROW_DISPATCH(dt, vec, (launch(add_norm_fwd_kernel<T, VW, true>, grid, pl.threads, 0, s, static_cast<const T*>(h),
                                     static_cast<const T*>(a), static_cast<T*>(sum), static_cast<const T*>(gamma),
                                     static_cast<const T*>(beta), static_cast<T*>(y), stat0, stat1, rows, cols, eps,
                                     pl.tpr, drop, p, dscale, seed)));
  else
    XT_ROW_DISPATCH(dt, vec, (launch(add_norm_fwd_kernel<T, VW, false>, grid, pl.threads, 0, s, static_cast<const T*>(h),
                                     static_cast<const T*>(a), static_cast<T*>(sum), static_cast<const T*>(gamma),
                                     static_cast<const T*>(beta), static_cast<T*>(y), stat0, stat1, rows, cols, eps,
                                     pl.tpr, drop, p, dscale, seed)));
  return check_launch("xt_dropout_add_norm_fwd");
}

int xt_norm_bwd_dropout(int norm, const void* d, const void* x, const void* gamma, const float* stat0,
                        const float* stat1, void* dx, void* dgamma, void* dbeta, void* g, int64_t rows, int64_t cols,
                        int dt, int dt_dx, int dt_param, void* ws, int acc_dx, int acc_param, float p, uint64_t seed,
                        int training, void* stream) {
  XT_REQUIRE(norm == XT_NORM_RMS || norm == XT_NORM_LN, "xt_norm_bwd_dropout: bad norm");
  XT_REQUIRE(dx && g, "xt_norm_bwd_dropout: dx and g are required");
  XT_REQUIRE(p >= 0.f && p < 1.f, "xt_norm_bwd_dropout: p must be in [0, 1)");
  if (!aligned16(g)) return fail(XT_ERR_ALIGNMENT, "xt_norm_bwd_dropout: g must be 16-byte aligned");
  GradOut go{g, p, float(1.0 / (1.0 - double(p))), seed, (training && p > 0.f) ? 1 : 0};
  if (norm == XT_NORM_RMS)
    return rms_bwd_impl(d, x, gamma, stat0, dx, dgamma, rows, cols, dt, dt_dx, dt_param, ws, acc_dx, acc_param,
                        stream, go);
  return ln_bwd_impl(d, x, gamma, stat0, stat1, dx, dgamma, dbeta, rows, cols, dt, dt_dx, dt_param, ws, acc_dx,
                     acc_param, stream, go);
}

int xt_colsum_workspace_size(int64_t rows, int64_t cols, size_t* bytes) {
  XT_REQUIRE(rows >= 0 && cols >= 0 && bytes, "xt_colsum_workspace_size: bad arguments");
  *bytes = size_t(colsum_chunks(rows)) * size_t(cols) * sizeof(float);
  return XT_OK;
}

int xt_add_bias_bwd(const void* d, void* dx, void* dbias, int64_t rows, int64_t cols, int dt, int dt_bias, void* ws,
                    int acc_dx, int acc_dbias, void* stream) {
  XT_REQUIRE(valid_dtype(dt) && valid_dtype(dt_bias), "xt_add_bias_bwd: bad dtype");
  XT_REQUIRE(rows >= 0 && cols > 0, "xt_add_bias_bwd: bad sizes");
  XT_REQUIRE(rows == 0 || d, "xt_add_bias_bwd: d is NULL");
  XT_REQUIRE(dbias && ws, "xt_add_bias_bwd: dbias and ws are required");
  cudaStream_t s = as_stream(stream);
  if (rows == 0) {
    if (!acc_dbias && cudaMemsetAsync(dbias, 0, size_t(cols) * dtype_size(dt_bias), s) != cudaSuccess)
      return check_launch("xt_add_bias_bwd");
    return XT_OK;
  }
  const int nch = colsum_chunks(rows);
  float* part = static_cast<float*>(ws);
  if (nch > 65535) return fail(XT_ERR_UNSUPPORTED, "xt_add_bias_bwd: too many rows");
  const int vw = dt == XT_F32 ? 4 : 8;
  const bool vec = cols % vw == 0 && aligned16(d) && (!dx || aligned16(dx));
  const int64_t slab = 32 * (vec ? vw : 1);
  const int64_t slabs = ceil_div(cols, slab);
  if (slabs > INT32_MAX) return fail(XT_ERR_UNSUPPORTED, "xt_add_bias_bwd: too many columns");
  const dim3 grid{unsigned(slabs), unsigned(nch)};
  if (dt == XT_F32) {
    auto D = static_cast<const float*>(d);
    auto DX = static_cast<float*>(dx);
    if (vec) launch(colsum_stage1<float, 4>, grid, 256, 0, s, D, DX, acc_dx, part, rows, cols);
    else launch(colsum_stage1<float, 1>, grid, 256, 0, s, D, DX, acc_dx, part, rows, cols);
  } else {
    auto D = static_cast<const bf16*>(d);
    auto DX = static_cast<bf16*>(dx);
    if (vec) launch(colsum_stage1<bf16, 8>, grid, 256, 0, s, D, DX, acc_dx, part, rows, cols);
    else launch(colsum_stage1<bf16, 1>, grid, 256, 0, s, D, DX, acc_dx, part, rows, cols);
  }
  XT_TRY(check_launch("xt_add_bias_bwd"));
  return finalize(part, nch, cols, dbias, dt_bias, acc_dbias, s);
}

int xt_softmax_fwd(const void* x, void* y, int64_t rows, int64_t cols, int causal, int64_t q_len, int dt,
                   void* stream) {
  XT_REQUIRE(valid_dtype(dt), "xt_softmax_fwd: bad dtype");
  XT_REQUIRE(rows >= 0 && cols > 0 && causal >= 0 && causal <= 2, "xt_softmax_fwd: bad arguments");
  XT_REQUIRE(!causal || q_len > 0, "xt_softmax_fwd: causal needs q_len > 0");
  XT_REQUIRE(rows == 0 || (x && y), "xt_softmax_fwd: NULL pointer");
  if (rows == 0) return XT_OK;
  const bool vec = rows_vec_ok(cols, dt, {x, y});
  RowPlan pl = plan_rows(cols, vec ? (dt == XT_BF16 ? 8 : 4) : 1);
  if (!pl.ok) return fail(XT_ERR_UNSUPPORTED, "xt_softmax_fwd: row too long");
  cudaStream_t s = as_stream(stream);
  const int grid = row_grid(rows, pl.rpb);
  XT_ROW_DISPATCH(dt, vec, (launch(softmax_fwd_kernel<T, VW>, grid, pl.threads, 0, s, 
                               static_cast<const T*>(x), static_cast<T*>(y), rows, int(cols), causal, q_len, pl.tpr)));
  return check_launch("xt_softmax_fwd");
}

int xt_softmax_bwd(const void* d, const void* y, void* dx, int64_t rows, int64_t cols, int causal, int64_t q_len,
                   int dt, int acc, void* stream) {
  XT_REQUIRE(valid_dtype(dt), "xt_softmax_bwd: bad dtype");
  XT_REQUIRE(rows >= 0 && cols > 0 && causal >= 0 && causal <= 2, "xt_softmax_bwd: bad arguments");
  XT_REQUIRE(!causal || q_len > 0, "xt_softmax_bwd: causal needs q_len > 0");
  XT_REQUIRE(rows == 0 || (d && y && dx), "xt_softmax_bwd: NULL pointer");
  if (rows == 0) return XT_OK;
  const bool vec = rows_vec_ok(cols, dt, {d, y, dx});
  RowPlan pl = plan_rows(cols, vec ? (dt == XT_BF16 ? 8 : 4) : 1);
  if (!pl.ok) return fail(XT_ERR_UNSUPPORTED, "xt_softmax_bwd: row too long");
  cudaStream_t s = as_stream(stream);
  const int grid = row_grid(rows, pl.rpb);
  const bool narrow = pl.threads <= 256;
  XT_ROW_DISPATCH(dt, vec, (launch(narrow ? softmax_bwd_kernel<T, VW, 256> : softmax_bwd_kernel<T, VW, 1024>, grid,
                                   pl.threads, 0, s, static_cast<const T*>(d), static_cast<const T*>(y),
                                   static_cast<T*>(dx), rows, int(cols), causal, q_len, pl.tpr, acc)));
  return check_launch("xt_softmax_bwd");
}

int xt_cross_entropy_workspace_size(int64_t rows, size_t* bytes) {
  XT_REQUIRE(rows >= 0 && bytes, "xt_cross_entropy_workspace_size: bad arguments");
  *bytes = size_t(rows > 0 ? rows : 1) * sizeof(float);
  return XT_OK;
}

int xt_cross_entropy_fwd(const void* logits, const int32_t* targets, float* lse, float* loss, int64_t rows, int64_t V,
                         int dt, void* ws, void* stream) {
  XT_REQUIRE(valid_dtype(dt), "xt_cross_entropy_fwd: bad dtype");
  XT_REQUIRE(rows > 0 && V > 0, "xt_cross_entropy_fwd: bad sizes");
  XT_REQUIRE(logits && targets && lse && loss && ws, "xt_cross_entropy_fwd: NULL pointer");
  cudaStream_t s = as_stream(stream);
  const bool vec = rows_vec_ok(V, dt, {logits});
  const int vw = vec ? (dt == XT_BF16 ? 8 : 4) : 1;
  // streaming: threads per row sized so each thread handles ~8 vectors
  int tpr = next_pow2(ceil_div(ceil_div(V, vw), 8));
  if (tpr < 32) tpr = 32;
  if (tpr > 512) tpr = 512;
  const int threads = tpr < 256 ? 256 : tpr;
  const int rpb = threads / tpr;
  const int grid = row_grid(rows, rpb);
  float* nll = static_cast<float*>(ws);
  uint32_t* flag = errflag();
  XT_ROW_DISPATCH(dt, vec, (launch(ce_fwd_kernel<T, VW>, grid, threads, 0, s, static_cast<const T*>(logits), targets,
                                                                         lse, nll, rows, V, tpr, flag)));
  XT_TRY(check_launch("xt_cross_entropy_fwd"));
  launch(ce_loss_kernel, 1, 1024, 0, s, nll, rows, loss);
  return check_launch("xt_cross_entropy_fwd loss");
}

int xt_cross_entropy_bwd(const void* logits, const int32_t* targets, const float* lse, const float* upstream,
                         void* dlogits, int64_t rows, int64_t V, int dt, int dt_grad, int acc, void* stream) {
  XT_REQUIRE(valid_dtype(dt) && valid_dtype(dt_grad), "xt_cross_entropy_bwd: bad dtype");
  XT_REQUIRE(rows > 0 && V > 0, "xt_cross_entropy_bwd: bad sizes");
  XT_REQUIRE(logits && targets && lse && upstream && dlogits, "xt_cross_entropy_bwd: NULL pointer");
  XT_REQUIRE(!(logits == dlogits && dt != dt_grad), "xt_cross_entropy_bwd: in-place needs equal dtypes");
  cudaStream_t s = as_stream(stream);
  uint32_t* flag = errflag();
  const bool vec = V % 8 == 0 && aligned16(logits) && aligned16(dlogits);
  int64_t grid = rows;
  if (grid > int64_t(num_sms()) * 16) grid = int64_t(num_sms()) * 16;
  const int g = int(grid < 1 ? 1 : grid);
#define XT_CE_BWD(TI, TG)                                                                                  \
  do {                                                                                                     \
    if (vec) launch(ce_bwd_kernel<TI, TG, 8>, g, 256, 0, s, static_cast<const TI*>(logits), targets, lse, upstream, \
                                                        static_cast<TG*>(dlogits), rows, V, acc, flag);    \
    else launch(ce_bwd_kernel<TI, TG, 1>, g, 256, 0, s, static_cast<const TI*>(logits), targets, lse, upstream,     \
                                                    static_cast<TG*>(dlogits), rows, V, acc, flag);        \
  } while (0)
  if (dt == XT_F32 && dt_grad == XT_F32) XT_CE_BWD(float, float);
  else if (dt == XT_BF16 && dt_grad == XT_BF16) XT_CE_BWD(bf16, bf16);
  else if (dt == XT_BF16 && dt_grad == XT_F32) XT_CE_BWD(bf16, float);
  else XT_CE_BWD(float, bf16);
#undef XT_CE_BWD
  return check_launch("xt_cross_entropy_bwd");
}

static bool ce_fused_fits(int64_t V, int dt) {
  const size_t e = dtype_size(dt);
  return valid_dtype(dt) && V % int64_t(16 / e) == 0 && size_t(V) * e <= size_t(200) * 1024;
}

int xt_cross_entropy_fwd_bwd(const void* logits, const int32_t* targets, float* lse, float* loss, const float* upstream,
                             void* dlogits, int64_t rows, int64_t V, int dt, int dt_grad, void* ws, void* stream) {
  XT_REQUIRE(valid_dtype(dt) && valid_dtype(dt_grad), "xt_cross_entropy_fwd_bwd: bad dtype");
  XT_REQUIRE(rows > 0 && V > 0, "xt_cross_entropy_fwd_bwd: bad sizes");
  XT_REQUIRE(logits && targets && lse && loss && upstream && dlogits && ws, "xt_cross_entropy_fwd_bwd: NULL pointer");
  XT_REQUIRE(!(logits == dlogits && dt != dt_grad), "xt_cross_entropy_fwd_bwd: in-place needs equal dtypes");
  cudaStream_t s = as_stream(stream);
  const bool vec_ok = V % int64_t(16 / dtype_size(dt)) == 0 && aligned16(logits) && aligned16(dlogits);
  if (vec_ok && (!ce_fused_fits(V, dt) || dt != dt_grad) && ce_split_cluster(V, dt) > 0)
    // wide rows, or a gradient of another dtype: the chunked one-pass kernel (rows split
    // across a cluster of CTAs when wide); rows of up to 200 KB written in place keep the
    // one-CTA-per-row kernel below, which measured faster in place (0.65 against 0.62 of HBM
    // at 8192 × 50304 bf16)
    return ce_split_run(logits, targets, lse, loss, nullptr, upstream, dlogits, rows, V, dt, dt_grad, 0, 0.f, 0.f, ws,
                        s);
  if (!vec_ok || !ce_fused_fits(V, dt) || dt != dt_grad) {
    // rows without 16-byte vectors: the forward then the backward
    XT_TRY(xt_cross_entropy_fwd(logits, targets, lse, loss, rows, V, dt, ws, stream));
    return xt_cross_entropy_bwd(logits, targets, lse, upstream, dlogits, rows, V, dt, dt_grad, 0, stream);
  }
  const size_t smem = size_t(V) * dtype_size(dt);
  int64_t grid = rows;
  const int64_t cap = int64_t(num_sms()) * 2;
  if (grid > cap) grid = cap;
  float* nll = static_cast<float*>(ws);
  uint32_t* flag = errflag();
  if (dt == XT_BF16) {
    cudaFuncSetAttribute(ce_fused_kernel<bf16, bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    launch(ce_fused_kernel<bf16, bf16>, int(grid), kCeFusedThreads, smem, s, static_cast<const bf16*>(logits),
           targets, lse, nll, upstream, static_cast<bf16*>(dlogits), rows, V, flag);
  } else {
    cudaFuncSetAttribute(ce_fused_kernel<float, float>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    launch(ce_fused_kernel<float, float>, int(grid), kCeFusedThreads, smem, s, static_cast<const float*>(logits),
           targets, lse, nll, upstream, static_cast<float*>(dlogits), rows, V, flag);
  }
  XT_TRY(check_launch("xt_cross_entropy_fwd_bwd"));
  launch(ce_loss_kernel, 1, 1024, 0, s, static_cast<const float*>(nll), rows, loss);
  return check_launch("xt_cross_entropy_fwd_bwd loss");
}

int xt_rope_table(float* table, int S, int hd, double base, int pos_offset, void* stream) {
  XT_REQUIRE(table && S > 0 && hd > 0 && hd % 2 == 0 && base > 0, "xt_rope_table: bad arguments");
  const int n = S * (hd / 2);
  launch(rope_table_kernel, (n + 255) / 256, 256, 0, as_stream(stream), table, S, hd, base, pos_offset);
  return check_launch("xt_rope_table");
}

static int rope_run(bool bwd, const void* x, void* y, const float* table, int B, int S, int H, int hd, int64_t ld,
                    int dt, int acc, void* stream) {
  XT_REQUIRE(valid_dtype(dt), "rope: bad dtype");
  XT_REQUIRE(B >= 0 && S > 0 && H > 0 && hd > 0 && hd % 2 == 0 && ld >= int64_t(H) * hd, "rope: bad sizes");
  XT_REQUIRE(B == 0 || (x && y && table), "rope: NULL pointer");
  if (B == 0) return XT_OK;
  cudaStream_t s = as_stream(stream);
  const int vw = dt == XT_BF16 ? 8 : 4;
  const size_t e = dtype_size(dt);
  const bool vec = (hd / 2) % vw == 0 && (ld * e) % 16 == 0 && aligned16(x) && aligned16(y);
  const int64_t total = int64_t(B) * S * H * (hd / 2) / (vec ? vw : 1);
  int64_t grid = ceil_div(total, 256);
  if (grid > int64_t(num_sms()) * 16) grid = int64_t(num_sms()) * 16;
  XT_ROW_DISPATCH(dt, vec, {
    if (bwd)
      launch(rope_kernel<T, true, VW>, int(grid), 256, 0, s, static_cast<const T*>(x), static_cast<T*>(y), table, B, S, H,
                                                         hd, ld, acc);
    else
      launch(rope_kernel<T, false, VW>, int(grid), 256, 0, s, static_cast<const T*>(x), static_cast<T*>(y), table, B, S,
                                                          H, hd, ld, acc);
  });
  return check_launch("rope");
}

int xt_rope_fwd(const void* x, void* y, const float* table, int B, int S, int H, int hd, int64_t ld, int dt,
                void* stream) {
  return rope_run(false, x, y, table, B, S, H, hd, ld, dt, 0, stream);
}

int xt_rope_bwd(const void* d, void* dx, const float* table, int B, int S, int H, int hd, int64_t ld, int dt, int acc,
                void* stream) {
  XT_REQUIRE(!(acc && d == dx), "xt_rope_bwd: accumulate cannot be in place");
  return rope_run(true, d, dx, table, B, S, H, hd, ld, dt, acc, stream);
}

int xt_embedding_workspace_size(int64_t T, size_t* bytes) {
  XT_REQUIRE(T >= 0 && bytes, "xt_embedding_workspace_size: bad arguments");
  *bytes = 16;  // kept for the interface; the backward needs no scratch
  return XT_OK;
}

int xt_embedding_fwd(const int32_t* ids, const void* E, const void* P, void* h, int64_t T_, int S, int64_t d,
                     int64_t V, int dt, void* stream) {
  XT_REQUIRE(valid_dtype(dt), "xt_embedding_fwd: bad dtype");
  XT_REQUIRE(T_ >= 0 && d > 0 && V > 0 && (!P || S > 0), "xt_embedding_fwd: bad sizes");
  XT_REQUIRE(T_ == 0 || (ids && E && h), "xt_embedding_fwd: NULL pointer");
  if (T_ == 0) return XT_OK;
  cudaStream_t s = as_stream(stream);
  const bool vec = rows_vec_ok(d, dt, {E, P, h});
  const int64_t work = T_ * d / (vec ? (dt == XT_BF16 ? 8 : 4) : 1);
  int64_t grid = ceil_div(work, 256);
  if (grid > int64_t(num_sms()) * 16) grid = int64_t(num_sms()) * 16;
  uint32_t* flag = errflag();
  XT_ROW_DISPATCH(dt, vec, (launch(embed_fwd_kernel<T, VW>, int(grid), 256, 0, s, 
                               ids, static_cast<const T*>(E), static_cast<const T*>(P), static_cast<T*>(h), T_, S, d,
                               V, flag)));
  return check_launch("xt_embedding_fwd");
}

int xt_embedding_bwd(const int32_t* ids, const void* dh, void* dE, void* dP, int64_t T, int S, int64_t d, int64_t V,
                     int dt_dh, int dt_grad, void* ws, int acc, void* stream) {
  XT_REQUIRE(valid_dtype(dt_dh) && valid_dtype(dt_grad), "xt_embedding_bwd: bad dtype");
  XT_REQUIRE(T >= 0 && d > 0 && V > 0 && (!dP || (S > 0 && T % S == 0)), "xt_embedding_bwd: bad sizes");
  XT_REQUIRE(T <= kSortMax, "xt_embedding_bwd: T > %d is not supported", kSortMax);
  XT_REQUIRE(dE && (T == 0 || (ids && dh)), "xt_embedding_bwd: NULL pointer");
  XT_REQUIRE(V < (int64_t(1) << 31), "xt_embedding_bwd: V too large");
  cudaStream_t s = as_stream(stream);
  if (!acc) {
    if (cudaMemsetAsync(dE, 0, size_t(V) * size_t(d) * dtype_size(dt_grad), s) != cudaSuccess)
      return check_launch("xt_embedding_bwd zero");
  }
  if (T == 0) return XT_OK;
  const int64_t blocks = V < int64_t(num_sms()) * 4 ? V : int64_t(num_sms()) * 4;
  const int64_t per = ceil_div(V, blocks);
  const size_t smem = size_t(T) * 2 * sizeof(int);
#define XT_EMB(TH, TG)                                                                                      \
  do {                                                                                                      \
    cudaFuncSetAttribute(embed_bwd_kernel<TH, TG>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));  \
    launch(embed_bwd_kernel<TH, TG>, unsigned(ceil_div(V, per)), kEmbThreads, smem, s, ids,                 \
           static_cast<const TH*>(dh), static_cast<TG*>(dE), int(T), d, V, per, errflag());                 \
    XT_TRY(check_launch("xt_embedding_bwd"));                                                               \
    if (dP) {                                                                                               \
      int64_t gp = ceil_div(int64_t(S) * d, 256);                                                           \
      launch(embed_pos_kernel<TH, TG>, unsigned(gp), 256, 0, s, static_cast<const TH*>(dh), static_cast<TG*>(dP), \
                                                            T, S, d, acc);                                  \
    }                                                                                                       \
  } while (0)
  if (dt_dh == XT_F32 && dt_grad == XT_F32) XT_EMB(float, float);
  else if (dt_dh == XT_BF16 && dt_grad == XT_BF16) XT_EMB(bf16, bf16);
  else if (dt_dh == XT_BF16 && dt_grad == XT_F32) XT_EMB(bf16, float);
  else XT_EMB(float, bf16);
#undef XT_EMB
  return check_launch("xt_embedding_bwd");
}

}  // extern "C"
