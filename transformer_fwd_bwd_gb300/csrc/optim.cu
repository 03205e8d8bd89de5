// Training-step tail after the backward: microbatch averaging, global gradient-norm clipping
// and the AdamW update, over a list of parameter tensors.
//
// [BP] § Ackumulation över mikrobatcher: the backward adds every microbatch's gradients into
// the buffers; the sum is scaled by 1 / n_microbatches before one optimizer step.
// [BP] § Parningsdisciplinen: gradient clipping runs as a partial and a final gradient-norm
// reduction followed by a gradient scale.
// [BP] § Optimiser-tillståndet: AdamW keeps a first moment m and a second moment v per weight.
//
// Every tensor is cut into tiles of kTile elements (a tile never spans two tensors).  Pass 1
// writes each tile's Σ (s·g)² (s = grad_scale) to a partial; pass 2 (one block) adds the
// partials in index order in float64 and turns the norm into the gradient factor
// s·min(1, max_norm / (norm + 1e-6)); pass 3 applies AdamW with that factor.  Fixed orders
// throughout: the step is deterministic.
#include <cmath>

#include "internal.cuh"

namespace xt {
namespace {

constexpr int kTile = 4096;          // elements per tile
constexpr int kThreads = 256;        // 16 elements per thread per tile
constexpr int kMaxTensors = 128;     // tensors per launch (the table travels in the kernel parameters)

struct Table {
  float* p[kMaxTensors];
  const float* g[kMaxTensors];
  float* m[kMaxTensors];
  float* v[kMaxTensors];
  void* sh[kMaxTensors];
  int64_t n[kMaxTensors];
  int tile0[kMaxTensors + 1];  // first tile of each tensor; tile0[count] = the group's tiles
  int count;
  int part0;                   // this group's first partial in the workspace
};

// Tensor of tile t: the last i with tile0[i] ≤ t.
__device__ __forceinline__ int tensor_of(const Table& tb, int t) {
  int lo = 0, hi = tb.count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tb.tile0[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Σ over the block's threads of x, in a fixed order (shared-memory tree).
__device__ __forceinline__ float block_sum(float x, float* sh) {
  sh[threadIdx.x] = x;
  __syncthreads();
  for (int w = kThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) sh[threadIdx.x] += sh[threadIdx.x + w];
    __syncthreads();
  }
  const float r = sh[0];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kThreads) grad_sq_tiles(const Table tb, float scale, float* __restrict__ part) {
  pdl_begin();
  __shared__ float sh[kThreads];
  const int tiles = tb.tile0[tb.count];
  for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int k = tensor_of(tb, t);
    const int64_t base = int64_t(t - tb.tile0[k]) * kTile;
    const int64_t len = tb.n[k] - base < kTile ? tb.n[k] - base : kTile;
    const float* g = tb.g[k] + base;
    float acc = 0.f;
    if (len == kTile && ((reinterpret_cast<uintptr_t>(g) & 15u) == 0)) {
#pragma unroll
      for (int u = 0; u < kTile / (4 * kThreads); ++u) {
        const float4 x = reinterpret_cast<const float4*>(g)[u * kThreads + threadIdx.x];
        const float a = x.x * scale, b = x.y * scale, c = x.z * scale, d = x.w * scale;
        acc = fmaf(a, a, acc); acc = fmaf(b, b, acc); acc = fmaf(c, c, acc); acc = fmaf(d, d, acc);
      }
    } else {
      for (int64_t i = threadIdx.x; i < len; i += kThreads) {
        const float a = g[i] * scale;
        acc = fmaf(a, a, acc);
      }
    }
    const float s = block_sum(acc, sh);
    if (threadIdx.x == 0) part[tb.part0 + t] = s;
  }
}

// One block: norm = √Σ partials (float64, index order); factor = scale·min(1, max_norm/(norm+1e-6)).
__global__ void __launch_bounds__(1024) grad_norm_final(const float* __restrict__ part, int n, float scale,
                                                        float max_norm, float* __restrict__ factor,
                                                        float* __restrict__ norm_out) {
  pdl_begin();
  __shared__ double sh[1024];
  double acc = 0.0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) acc += double(part[i]);
  sh[threadIdx.x] = acc;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) sh[threadIdx.x] += sh[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double norm = sqrt(sh[0]);
    double c = 1.0;
    if (max_norm > 0.f) c = fmin(1.0, double(max_norm) / (norm + 1e-6));
    *factor = float(double(scale) * c);
    if (norm_out) *norm_out = float(norm);
  }
}

struct AdamHyper {
  float lr, beta1, beta2, eps, decay;  // decay = 1 − lr·λ
  float inv_bc1, inv_bc2;              // 1 / (1 − β₁ᵗ), 1 / (1 − β₂ᵗ)
  float fixed_factor;                  // the gradient factor when `factor` is null
};

template <typename TS>
__device__ __forceinline__ void adam_one(float& p, float g, float& m, float& v, const AdamHyper& h) {
  m = fmaf(h.beta1, m, (1.f - h.beta1) * g);
  v = fmaf(h.beta2, v, (1.f - h.beta2) * g * g);
  const float mhat = m * h.inv_bc1;
  const float vhat = v * h.inv_bc2;
  p = p * h.decay - h.lr * (mhat / (sqrtf(vhat) + h.eps));
}

template <typename TS>
__global__ void __launch_bounds__(kThreads) adamw_tiles(const Table tb, const AdamHyper h,
                                                        const float* __restrict__ factor) {
  pdl_begin();
  const float f = factor ? *factor : h.fixed_factor;
  const int tiles = tb.tile0[tb.count];
  for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int k = tensor_of(tb, t);
    const int64_t base = int64_t(t - tb.tile0[k]) * kTile;
    const int64_t len = tb.n[k] - base < kTile ? tb.n[k] - base : kTile;
    float* p = tb.p[k] + base;
    const float* g = tb.g[k] + base;
    float* m = tb.m[k] + base;
    float* v = tb.v[k] + base;
    TS* sh = tb.sh[k] ? static_cast<TS*>(tb.sh[k]) + base : nullptr;
    const bool vec = len == kTile && ((reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(g) |
                                       reinterpret_cast<uintptr_t>(m) | reinterpret_cast<uintptr_t>(v)) & 15u) == 0;
    if (vec) {
#pragma unroll 2
      for (int u = 0; u < kTile / (4 * kThreads); ++u) {
        const int i4 = u * kThreads + threadIdx.x;
        float4 P = reinterpret_cast<float4*>(p)[i4];
        const float4 G = reinterpret_cast<const float4*>(g)[i4];
        float4 M = reinterpret_cast<float4*>(m)[i4];
        float4 V = reinterpret_cast<float4*>(v)[i4];
        adam_one<TS>(P.x, G.x * f, M.x, V.x, h);
        adam_one<TS>(P.y, G.y * f, M.y, V.y, h);
        adam_one<TS>(P.z, G.z * f, M.z, V.z, h);
        adam_one<TS>(P.w, G.w * f, M.w, V.w, h);
        reinterpret_cast<float4*>(p)[i4] = P;
        reinterpret_cast<float4*>(m)[i4] = M;
        reinterpret_cast<float4*>(v)[i4] = V;
        if (sh) {
          sh[4 * i4] = from_f<TS>(P.x);
          sh[4 * i4 + 1] = from_f<TS>(P.y);
          sh[4 * i4 + 2] = from_f<TS>(P.z);
          sh[4 * i4 + 3] = from_f<TS>(P.w);
        }
      }
    } else {
      for (int64_t i = threadIdx.x; i < len; i += kThreads) {
        float P = p[i], M = m[i], V = v[i];
        adam_one<TS>(P, g[i] * f, M, V, h);
        p[i] = P;
        m[i] = M;
        v[i] = V;
        if (sh) sh[i] = from_f<TS>(P);
      }
    }
  }
}

// Groups of up to kMaxTensors tensors with their tile offsets; returns the total tile count.
int64_t plan(int n, const int64_t* numel, int group, int first, Table& tb, int part0) {
  tb.count = 0;
  tb.part0 = part0;
  int tiles = 0;
  for (int i = first; i < n && tb.count < group; ++i) {
    tb.tile0[tb.count] = tiles;
    tb.n[tb.count] = numel[i];
    tiles += int(ceil_div(numel[i], kTile));
    ++tb.count;
  }
  tb.tile0[tb.count] = tiles;
  return tiles;
}

int64_t total_tiles(int n, const int64_t* numel) {
  int64_t t = 0;
  for (int i = 0; i < n; ++i) t += ceil_div(numel[i], kTile);
  return t;
}

}  // namespace
}  // namespace xt

using namespace xt;

extern "C" {

int xt_adamw_workspace_size(int n, const int64_t* numel, size_t* bytes) {
  XT_REQUIRE(bytes && n >= 0 && (n == 0 || numel), "xt_adamw_workspace_size: bad arguments");
  for (int i = 0; i < n; ++i) XT_REQUIRE(numel[i] >= 0, "xt_adamw_workspace_size: negative size");
  *bytes = ((size_t(total_tiles(n, numel)) * 4 + 255) & ~size_t(255)) + 256;
  return XT_OK;
}

int xt_adamw_step(const xt_adamw_config* cfg, int n, float* const* param, const float* const* grad, float* const* m,
                  float* const* v, void* const* shadow, int shadow_dtype, const int64_t* numel, float* norm_out,
                  void* ws, size_t ws_bytes, void* stream) {
  XT_REQUIRE(cfg != nullptr, "xt_adamw_step: cfg is NULL");
  XT_REQUIRE(n >= 0, "xt_adamw_step: n < 0");
  if (n == 0) return XT_OK;
  XT_REQUIRE(param && grad && m && v && numel, "xt_adamw_step: NULL table");
  XT_REQUIRE(cfg->step >= 1, "xt_adamw_step: step must be >= 1");
  XT_REQUIRE(cfg->beta1 >= 0.f && cfg->beta1 < 1.f && cfg->beta2 >= 0.f && cfg->beta2 < 1.f,
             "xt_adamw_step: betas must be in [0, 1)");
  XT_REQUIRE(cfg->eps > 0.f && cfg->lr >= 0.f && cfg->weight_decay >= 0.f, "xt_adamw_step: bad hyperparameters");
  XT_REQUIRE(shadow == nullptr || valid_dtype(shadow_dtype), "xt_adamw_step: bad shadow dtype");
  for (int i = 0; i < n; ++i) {
    XT_REQUIRE(numel[i] >= 0, "xt_adamw_step: negative size");
    if (numel[i] == 0) continue;
    XT_REQUIRE(param[i] && grad[i] && m[i] && v[i], "xt_adamw_step: NULL tensor %d", i);
    XT_REQUIRE(ceil_div(numel[i], kTile) < (int64_t(1) << 30), "xt_adamw_step: tensor too large");
  }
  const int64_t tiles = total_tiles(n, numel);
  XT_REQUIRE(tiles < (int64_t(1) << 30), "xt_adamw_step: too many elements");
  const bool need_norm = cfg->max_grad_norm > 0.f || norm_out != nullptr;
  size_t need = 0;
  XT_TRY(xt_adamw_workspace_size(n, numel, &need));
  if (need_norm) XT_REQUIRE(ws && ws_bytes >= need, "xt_adamw_step: workspace too small (%zu < %zu)", ws_bytes, need);
  cudaStream_t s = as_stream(stream);
  float* part = static_cast<float*>(ws);
  float* factor = need_norm ? reinterpret_cast<float*>(static_cast<char*>(ws) + need - 256) : nullptr;
  const int grid_cap = num_sms() * 8;
  auto fill = [&](Table& tb, int first) {
    for (int j = 0; j < tb.count; ++j) {
      const int i = first + j;
      tb.p[j] = param[i];
      tb.g[j] = grad[i];
      tb.m[j] = m[i];
      tb.v[j] = v[i];
      tb.sh[j] = shadow ? shadow[i] : nullptr;
    }
  };
  if (need_norm) {
    int part0 = 0;
    for (int first = 0; first < n; first += kMaxTensors) {
      Table tb{};
      const int64_t t = plan(n, numel, kMaxTensors, first, tb, part0);
      fill(tb, first);
      if (t > 0) {
        launch(grad_sq_tiles, int(t < grid_cap ? t : grid_cap), kThreads, 0, s, tb, cfg->grad_scale, part);
        XT_TRY(check_launch("xt_adamw_step (norm partials)"));
      }
      part0 += int(t);
    }
    launch(grad_norm_final, 1, 1024, 0, s, static_cast<const float*>(part), int(tiles), cfg->grad_scale,
           cfg->max_grad_norm, factor, norm_out);
    XT_TRY(check_launch("xt_adamw_step (norm)"));
  }
  AdamHyper h{};
  h.lr = cfg->lr;
  h.beta1 = cfg->beta1;
  h.beta2 = cfg->beta2;
  h.eps = cfg->eps;
  h.decay = float(1.0 - double(cfg->lr) * double(cfg->weight_decay));
  h.inv_bc1 = float(1.0 / (1.0 - std::pow(double(cfg->beta1), double(cfg->step))));
  h.inv_bc2 = float(1.0 / (1.0 - std::pow(double(cfg->beta2), double(cfg->step))));
  h.fixed_factor = cfg->grad_scale;
  for (int first = 0; first < n; first += kMaxTensors) {
    Table tb{};
    const int64_t t = plan(n, numel, kMaxTensors, first, tb, 0);
    fill(tb, first);
    if (t == 0) continue;
    const int grid = int(t < grid_cap ? t : grid_cap);
    if (shadow && shadow_dtype == XT_BF16)
      launch(adamw_tiles<bf16>, grid, kThreads, 0, s, tb, h, static_cast<const float*>(factor));
    else
      launch(adamw_tiles<float>, grid, kThreads, 0, s, tb, h, static_cast<const float*>(factor));
    XT_TRY(check_launch("xt_adamw_step (update)"));
  }
  return XT_OK;
}

}  // extern "C"
