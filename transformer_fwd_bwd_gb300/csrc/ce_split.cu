// Cross-entropy forward + backward in one pass over logits rows too wide for one CTA's shared
// memory ([AE] op table row cross_entropy, § Cross-entropy 反向推导; the large-vocabulary loss
// head), and the fused three-consumer loss of [AE] § 梯度累加's fan-out example.
//
// A cluster of CL CTAs owns a row at a time; CTA q holds the row's q-th chunk of columns in
// shared memory (bulk copies, completion on an mbarrier; with two chunk buffers the next
// row's copy runs while this row is reduced and written), forms its chunk's max m_q and
// s_q = Σ exp(x − m_q), sends (m_q, s_q) to every CTA of the cluster through distributed shared
// memory, and after one cluster barrier merges the CL pairs in rank order (the same order in
// every CTA, so all agree bit for bit) into lse = M + log S.  The gradient of its chunk is then
// written from shared memory: the logits are read from HBM once and the gradient written once.
//
// Optional extra terms (the fan-out): with row sums requested, each CTA also writes Σx and Σx²
// of its chunk, and the gradient gains alpha + beta·x, i.e. the gradient of
// c_lin·Σx + c_sq·Σx∘x with alpha = c_lin, beta = 2·c_sq; every term is scaled by the
// upstream gradient.
#include <mutex>

#include "common.cuh"
#include "gemm_kernel.cuh"
#include "internal.cuh"

namespace xt {
namespace ce {

using gemm::cluster_ctarank;
using gemm::cluster_sync_all;
using gemm::mapa_shared;
using gemm::mbar_init;
using gemm::mbar_wait;
using gemm::smem_u32;

constexpr int kThreads = 512;
constexpr float kLog2e = 1.4426950408889634f;
// largest chunk of one row held by one CTA
constexpr size_t kMaxChunkBytes = size_t(200) * 1024;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16-byte vector of T as floats
template <typename T>
__device__ __forceinline__ void unpack(const uint4& u, float (&v)[16 / sizeof(T)]);
template <>
__device__ __forceinline__ void unpack<float>(const uint4& u, float (&v)[4]) {
  v[0] = __uint_as_float(u.x);
  v[1] = __uint_as_float(u.y);
  v[2] = __uint_as_float(u.z);
  v[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void unpack<bf16>(const uint4& u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Stores VW float gradients (VW = 4 or 8) as TG at p, adding p's old contents when acc.
template <typename TG, int VW>
__device__ __forceinline__ void store_grad(TG* p, const float (&o)[VW], int acc) {
  if constexpr (sizeof(TG) == 4) {
#pragma unroll
    for (int e = 0; e < VW; e += 4) {
      float4 q = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
      if (acc) {
        const float4 old = *reinterpret_cast<const float4*>(p + e);
        q.x += old.x; q.y += old.y; q.z += old.z; q.w += old.w;
      }
      *reinterpret_cast<float4*>(p + e) = q;
    }
  } else {
    // VW bf16 values: 16 bytes for VW = 8, 8 bytes for VW = 4 (float32 logits)
    float v[VW];
#pragma unroll
    for (int e = 0; e < VW; ++e) v[e] = o[e];
    uint32_t w[VW / 2];
    if (acc) {
      if constexpr (VW == 8) {
        const uint4 old = *reinterpret_cast<const uint4*>(p);
        w[0] = old.x; w[1] = old.y; w[2] = old.z; w[3] = old.w;
      } else {
        const uint2 old = *reinterpret_cast<const uint2*>(p);
        w[0] = old.x; w[1] = old.y;
      }
#pragma unroll
      for (int i = 0; i < VW / 2; ++i) {
        v[2 * i] += __uint_as_float(w[i] << 16);
        v[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
      }
    }
#pragma unroll
    for (int i = 0; i < VW / 2; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    if constexpr (VW == 8) *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    else *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
  }
}

// Block-wide reduction (max or sum) of one float per thread; every thread gets the result.
__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < kThreads / 32; ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
  return r;
}

struct Args {
  int64_t rows, V, chunk;  // chunk: columns per CTA (a multiple of the vector width)
  const int32_t* tgt;
  float* lse;
  float* nll;
  float* row_sums;         // null, or [rows][CL][2]: Σx and Σx² of each CTA's chunk
  const float* upstream;   // upstream gradient of the loss (device scalar): scales every term
  int acc;
  float alpha, beta;       // extra gradient alpha + beta·x before the upstream scale (0, 0: none)
  uint32_t* flag;
  uint64_t wait_ns;
};

// CL CTAs per row (clusters of CL along x); T logits, TG gradient (may alias the logits).  NB
// chunk buffers: with two, the next row's chunk is copied in while this row's is reduced and
// its gradient written.
template <typename T, typename TG, int CL, int NB>
__global__ void __launch_bounds__(kThreads, 2) ce_split_kernel(const T* x, TG* dx, const Args a) {
  pdl_begin();
  constexpr int VW = 16 / sizeof(T);
  extern __shared__ __align__(128) uint8_t raw[];
  __shared__ float red[kThreads / 32];
  __shared__ float xch[2][CL][2];  // (m, s) of every rank, double-buffered by row parity
  __shared__ __align__(8) uint64_t bar[NB];
  const int rank = CL > 1 ? int(cluster_ctarank()) : 0;
  const int cid = int(blockIdx.x) / CL, ncl = int(gridDim.x) / CL;
  const int64_t c0 = int64_t(rank) * a.chunk;
  const int64_t c1 = c0 + a.chunk < a.V ? c0 + a.chunk : a.V;
  const int64_t n = c1 > c0 ? c1 - c0 : 0;  // this CTA's columns (a multiple of VW)
  const int64_t nvec = n / VW;
  const uint32_t bytes = uint32_t(n * int64_t(sizeof(T)));
  const size_t buf_bytes = size_t(a.chunk) * sizeof(T);
  if (threadIdx.x == 0) {
    for (int b = 0; b < NB; ++b) mbar_init(smem_u32(&bar[b]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // every CTA of the cluster has started (its shared memory exists) before the first remote store
  if constexpr (CL > 1) cluster_sync_all();
  else __syncthreads();
  // the chunk of row r into buffer b: one bulk copy per 64 KB, completion on bar[b]
  auto load = [&](int64_t r, int b) {
    if (threadIdx.x != 0 || n == 0) return;
    const uint32_t ba = smem_u32(&bar[b]);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(x + r * a.V + c0);
    const uint32_t dst = smem_u32(raw + size_t(b) * buf_bytes);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(ba), "r"(bytes) : "memory");
    for (uint32_t off = 0; off < bytes; off += 65536u) {
      const uint32_t len = bytes - off < 65536u ? bytes - off : 65536u;
      asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                       dst + off),
                   "l"(src + off), "r"(len), "r"(ba)
                   : "memory");
    }
  };
  const float up = *a.upstream;
  const float sc = up / float(a.rows), alpha = up * a.alpha, beta = up * a.beta;
  if (int64_t(cid) < a.rows) load(cid, 0);
  int it = 0;
  for (int64_t r = cid; r < a.rows; r += ncl, ++it) {
    const int b = NB == 2 ? (it & 1) : 0;
    // two buffers: the next row's chunk into the other buffer; one buffer: this row's chunk
    // (the first row's was issued before the loop).  Either buffer's last reader finished
    // before the __syncthreads that ended the previous row.
    if constexpr (NB == 2) {
      if (r + ncl < a.rows) load(r + ncl, b ^ 1);
    } else {
      if (it > 0) load(r, 0);
    }
    if (n > 0) {
      const uint32_t ph = uint32_t(NB == 2 ? (it >> 1) & 1 : it & 1);
      if (!mbar_wait(smem_u32(&bar[b]), ph, a.wait_ns)) {
        // report, then still wait for the copy before the buffer is read or reused
        flag_error(a.flag, XT_DEVERR_TIMEOUT);
        mbar_wait(smem_u32(&bar[b]), ph);
      }
    }
    const T* row_s = reinterpret_cast<const T*>(raw + size_t(b) * buf_bytes);
    // 1. chunk max, Σx, Σx² from shared memory
    float m = -INFINITY, sx = 0.f, sq = 0.f;
    for (int64_t j = threadIdx.x; j < nvec; j += kThreads) {
      float v[VW];
      unpack<T>(reinterpret_cast<const uint4*>(row_s)[j], v);
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        m = fmaxf(m, v[e]);
        sx += v[e];
        sq = fmaf(v[e], v[e], sq);
      }
    }
    m = block_reduce(m, true, red);
    if (a.row_sums) {
      sx = block_reduce(sx, false, red);
      sq = block_reduce(sq, false, red);
      if (threadIdx.x == 0) {
        a.row_sums[(r * CL + rank) * 2] = sx;
        a.row_sums[(r * CL + rank) * 2 + 1] = sq;
      }
    }
    // 2. s = Σ exp(x − m) over the chunk
    const float ml = m * kLog2e;
    float s = 0.f;
    if (m != -INFINITY) {
      for (int64_t j = threadIdx.x; j < nvec; j += kThreads) {
        float v[VW];
        unpack<T>(reinterpret_cast<const uint4*>(row_s)[j], v);
#pragma unroll
        for (int e = 0; e < VW; ++e) s += ex2f(fmaf(v[e], kLog2e, -ml));
      }
    }
    s = block_reduce(s, false, red);
    // 3. every rank's (m, s) to every CTA, one cluster barrier, merge in rank order
    float M = m, S = s;
    if constexpr (CL > 1) {
      if (threadIdx.x < CL) {
        const uint32_t dst = mapa_shared(smem_u32(&xch[it & 1][rank][0]), uint32_t(threadIdx.x));
        asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(dst), "f"(m), "f"(s) : "memory");
      }
      cluster_sync_all();
      M = -INFINITY;
#pragma unroll
      for (int q = 0; q < CL; ++q) M = fmaxf(M, xch[it & 1][q][0]);
      S = 0.f;
#pragma unroll
      for (int q = 0; q < CL; ++q) {
        const float mq = xch[it & 1][q][0];
        if (mq != -INFINITY) S += xch[it & 1][q][1] * ex2f((mq - M) * kLog2e);
      }
    }
    const float L = M + logf(S);
    const int32_t t = a.tgt[r];
    const bool bad = t < 0 || int64_t(t) >= a.V;
    if (threadIdx.x == 0) {
      if (rank == 0) a.lse[r] = L;
      if (bad) {
        if (rank == 0) {
          flag_error(a.flag, XT_DEVERR_INDEX);
          a.nll[r] = __int_as_float(0x7fc00000);
        }
      } else if (int64_t(t) >= c0 && int64_t(t) < c1) {
        a.nll[r] = L - to_f(row_s[t - c0]);
      }
    }
    // 4. the gradient of this chunk from shared memory
    const float Ll = L * kLog2e;
    TG* dr = dx + r * a.V + c0;
    for (int64_t j = threadIdx.x; j < nvec; j += kThreads) {
      float v[VW], o[VW];
      unpack<T>(reinterpret_cast<const uint4*>(row_s)[j], v);
      const int64_t c = c0 + j * VW;
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        const float p = ex2f(fmaf(v[e], kLog2e, -Ll));
        o[e] = bad ? __int_as_float(0x7fc00000) : fmaf(beta, v[e], sc * (p - (c + e == t ? 1.f : 0.f)) + alpha);
      }
      store_grad<TG, VW>(dr + j * VW, o, a.acc);
    }
    __syncthreads();  // this buffer is free for the copy of the row after next
  }
}

// loss = Σ nll / rows; with row sums, sums[0] = Σ Σx and sums[1] = Σ Σx² over rows and ranks,
// each in a fixed order (one block), and sums[2] = loss + c_lin·sums[0] + c_sq·sums[1].
__global__ void ce_split_loss(const float* __restrict__ nll, const float* __restrict__ row_sums, int64_t rows, int cl,
                              float c_lin, float c_sq, float* loss, float* sums) {
  pdl_begin();
  __shared__ float red[3][32];
  float acc[3] = {0.f, 0.f, 0.f};
  for (int64_t i = threadIdx.x; i < rows; i += blockDim.x) {
    acc[0] += nll[i];
    if (row_sums)
      for (int q = 0; q < cl; ++q) {
        acc[1] += row_sums[(i * cl + q) * 2];
        acc[2] += row_sums[(i * cl + q) * 2 + 1];
      }
  }
#pragma unroll
  for (int k = 0; k < 3; ++k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
    if ((threadIdx.x & 31) == 0) red[k][threadIdx.x >> 5] = acc[k];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float t[3] = {0.f, 0.f, 0.f};
    for (int w = 0; w < int(blockDim.x >> 5); ++w)
      for (int k = 0; k < 3; ++k) t[k] += red[k][w];
    const float ce = t[0] / float(rows);
    *loss = ce;
    if (sums) {
      sums[0] = t[1];
      sums[1] = t[2];
      sums[2] = ce + c_lin * t[1] + c_sq * t[2];
    }
  }
}

// Clusters of CL that can be resident at once with `smem` bytes of chunk buffers.
template <typename T, typename TG, int CL, int NB>
static int capacity(size_t smem) {
  auto k = ce_split_kernel<T, TG, CL, NB>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (CL > 1 && cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(num_sms() / CL * CL));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <typename T, typename TG, int CL, int NB>
static int run_cl(const void* x, void* dx, const Args& a, cudaStream_t s) {
  const size_t smem = size_t(NB) * size_t(a.chunk) * sizeof(T);
  const int cap = capacity<T, TG, CL, NB>(smem);
  if (cap < 1) return fail(XT_ERR_UNSUPPORTED, "cross-entropy: no cluster of %d CTAs with %zu bytes fits", CL, smem);
  const int64_t clusters = a.rows < cap ? a.rows : cap;
  auto k = ce_split_kernel<T, TG, CL, NB>;
  if (CL > 1)
    launch_clustered(k, dim3(unsigned(clusters * CL)), dim3(kThreads), smem, s, CL, static_cast<const T*>(x),
                     static_cast<TG*>(dx), a);
  else
    launch(k, dim3(unsigned(clusters)), dim3(kThreads), smem, s, static_cast<const T*>(x), static_cast<TG*>(dx), a);
  return check_launch("cross-entropy (split rows)");
}

template <typename T, typename TG>
static int run_t(const void* x, void* dx, const Args& a, int cl, int nb, cudaStream_t s) {
  const int key = cl * 10 + nb;
  switch (key) {
    case 11: return run_cl<T, TG, 1, 1>(x, dx, a, s);
    case 12: return run_cl<T, TG, 1, 2>(x, dx, a, s);
    case 21: return run_cl<T, TG, 2, 1>(x, dx, a, s);
    case 22: return run_cl<T, TG, 2, 2>(x, dx, a, s);
    case 41: return run_cl<T, TG, 4, 1>(x, dx, a, s);
    case 42: return run_cl<T, TG, 4, 2>(x, dx, a, s);
    case 81: return run_cl<T, TG, 8, 1>(x, dx, a, s);
    case 82: return run_cl<T, TG, 8, 2>(x, dx, a, s);
    default: return fail(XT_ERR_UNSUPPORTED, "cross-entropy: cluster of %d with %d buffers", cl, nb);
  }
}

// 1.0f on the device: the upstream gradient of a loss at the root of the graph.
__device__ float g_one = 1.0f;

}  // namespace ce

static const float* one_scalar() {
  static std::mutex mu;
  static const float* ptr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, ce::g_one) != cudaSuccess) return nullptr;
    ptr[dev] = static_cast<const float*>(p);
  }
  return ptr[dev];
}

// The row split: the smallest cluster (1, 2, 4, 8) whose per-CTA chunk fits half of
// kMaxChunkBytes, so that two CTAs share an SM (one copying its chunk in while the other
// reduces or writes; measured faster than one CTA with two chunk buffers), else the smallest
// whose chunk fits kMaxChunkBytes (one CTA per SM); one chunk buffer; 0 if none fits.
static int64_t chunk_of(int64_t V, int cl, int dt) {
  const int64_t vw = 16 / int64_t(dtype_size(dt));
  return ceil_div(ceil_div(V, cl), vw) * vw;
}

// Measurement override (xt_ce_set_split): a fixed cluster size and buffer count, 0 = automatic.
static int g_force_cl = 0, g_force_nb = 0;

int ce_split_cluster(int64_t V, int dt, int* nb) {
  const size_t e = dtype_size(dt);
  if (g_force_cl && size_t(g_force_nb) * size_t(chunk_of(V, g_force_cl, dt)) * e <= ce::kMaxChunkBytes) {
    if (nb) *nb = g_force_nb;
    return g_force_cl;
  }
  if (nb) *nb = 1;
  for (int cl = 1; cl <= 8; cl *= 2)
    if (2 * size_t(chunk_of(V, cl, dt)) * e <= ce::kMaxChunkBytes) return cl;
  for (int cl = 1; cl <= 8; cl *= 2)
    if (size_t(chunk_of(V, cl, dt)) * e <= ce::kMaxChunkBytes) return cl;
  return 0;
}

// One pass of the cross-entropy forward + backward over rows split across a cluster; the
// workspace holds nll [rows] then, when sums != null, the row sums [rows][cl][2].
int ce_split_run(const void* logits, const int32_t* targets, float* lse, float* loss, float* sums,
                 const float* upstream, void* dlogits, int64_t rows, int64_t V, int dt, int dt_grad, int acc,
                 float c_lin, float c_sq, void* ws, cudaStream_t s) {
  int nb = 1;
  const int cl = ce_split_cluster(V, dt, &nb);
  if (cl == 0) return fail(XT_ERR_UNSUPPORTED, "cross-entropy: rows of %lld columns are too wide", (long long)V);
  const int64_t vw = 16 / int64_t(dtype_size(dt));
  if (V % vw || !aligned16(logits) || !aligned16(dlogits))
    return fail(XT_ERR_ALIGNMENT, "cross-entropy (split rows): V a multiple of %lld, 16-byte aligned buffers",
                (long long)vw);
  ce::Args a{};
  a.rows = rows;
  a.V = V;
  a.chunk = chunk_of(V, cl, dt);
  a.tgt = targets;
  a.lse = lse;
  a.nll = static_cast<float*>(ws);
  a.row_sums = sums ? static_cast<float*>(ws) + rows : nullptr;
  a.upstream = upstream;
  a.acc = acc;
  a.alpha = c_lin;
  a.beta = 2.f * c_sq;
  a.flag = errflag();
  a.wait_ns = wait_limit_ns();
  int st;
  if (dt == XT_BF16)
    st = dt_grad == XT_BF16 ? ce::run_t<bf16, bf16>(logits, dlogits, a, cl, nb, s)
                            : ce::run_t<bf16, float>(logits, dlogits, a, cl, nb, s);
  else
    st = dt_grad == XT_BF16 ? ce::run_t<float, bf16>(logits, dlogits, a, cl, nb, s)
                            : ce::run_t<float, float>(logits, dlogits, a, cl, nb, s);
  XT_TRY(st);
  launch(ce::ce_split_loss, 1, 1024, 0, s, static_cast<const float*>(ws), static_cast<const float*>(a.row_sums), rows,
         cl, c_lin, c_sq, loss, sums);
  return check_launch("cross-entropy (split rows) loss");
}

}  // namespace xt

using namespace xt;

extern "C" {

int xt_ce_set_split(int cl, int nb) {
  XT_REQUIRE((cl == 0 && nb == 0) || ((cl == 1 || cl == 2 || cl == 4 || cl == 8) && (nb == 1 || nb == 2)),
             "xt_ce_set_split: cl in {1, 2, 4, 8} and nb in {1, 2}, or both 0");
  g_force_cl = cl;
  g_force_nb = nb;
  return XT_OK;
}

int xt_cross_entropy_fanout_workspace_size(int64_t rows, size_t* bytes) {
  XT_REQUIRE(rows >= 0 && bytes, "xt_cross_entropy_fanout_workspace_size: bad arguments");
  *bytes = size_t(rows > 0 ? rows : 1) * sizeof(float) * (1 + 2 * 8);
  return XT_OK;
}

int xt_cross_entropy_fanout_fwd_bwd(const void* logits, const int32_t* targets, float c_lin, float c_sq,
                                    const float* upstream, float* lse, float* loss, float* sums, void* grad, int acc,
                                    int64_t rows, int64_t V, int dt, void* ws, size_t ws_bytes, void* stream) {
  XT_REQUIRE(valid_dtype(dt), "xt_cross_entropy_fanout_fwd_bwd: bad dtype");
  XT_REQUIRE(rows > 0 && V > 0, "xt_cross_entropy_fanout_fwd_bwd: bad sizes");
  XT_REQUIRE(logits && targets && lse && loss && sums && grad && ws, "xt_cross_entropy_fanout_fwd_bwd: NULL pointer");
  XT_REQUIRE(grad != logits, "xt_cross_entropy_fanout_fwd_bwd: the gradient is float32, not in place");
  size_t need = 0;
  xt_cross_entropy_fanout_workspace_size(rows, &need);
  XT_REQUIRE(ws_bytes >= need, "xt_cross_entropy_fanout_fwd_bwd: workspace of %zu bytes, %zu needed", ws_bytes, need);
  const float* up = upstream ? upstream : one_scalar();
  if (!up) return fail(XT_ERR_CUDA, "xt_cross_entropy_fanout_fwd_bwd: no device constant");
  return ce_split_run(logits, targets, lse, loss, sums, up, grad, rows, V, dt, XT_F32, acc, c_lin, c_sq, ws,
                      as_stream(stream));
}

}  // extern "C"
