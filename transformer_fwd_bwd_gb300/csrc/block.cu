// Native block stack: the whole forward and backward of the pre-norm transformer stack
// enqueued on one stream from one call, from the same kernels the per-op entry points run.
//
// [BP] § Framåtgåendet: h = embed(ids); per layer h = h + attn(norm h), h = h + mlp(norm h);
// logits = norm(h) @ embedᵀ; loss = cross_entropy(logits, targets).
// [DO] § dropout 接在哪（wiring）: residual dropout at the attention and FFN outputs with the
// per-site seeds base ⊕ layer ⊕ {0xA77, 0xF70}.
// [AE] § Attention 用组合: attention = matmul(softmax(scale(matmul(Q, Kᵀ))), V), either as the
// fused tile-by-tile kernels (bf16, head_dim 64) or as causal-tile GEMMs around an in-place
// softmax; the backward follows the same composition.
// [BP] § Ackumulation över mikrobatcher: the backward adds into every gradient buffer.
//
// The residual-stream gradient is kept in float32 whatever the activation dtype (it sums the
// fan-out of every residual add and norm); everything else is stored in the activation dtype
// with float32 statistics.
//
// The backward puts the weight-gradient GEMMs (dW = Xᵀ·dY, off the path that carries the
// gradient down the stack) on a second stream of the same device, forked and joined with events
// around the buffers they read, so they run beside the data-gradient GEMMs, the attention
// backward and the row kernels instead of between them.
#include <algorithm>
#include <map>
#include <mutex>
#include <vector>

#include "internal.cuh"

namespace xt {
namespace {

constexpr uint64_t kSiteAttn = 0xA77, kSiteFfn = 0xF70;

// Bump allocator over the caller's workspace; with base == nullptr it only measures.
struct Arena {
  char* base;
  size_t off = 0;
  void* take(size_t bytes) {
    off = (off + 255) & ~size_t(255);
    void* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  }
};

struct Dims {
  int64_t B, S, d, H, hd, F, V, L, T, UP, e;
  int dt, gdt;
  bool rms, swiglu;
  bool fused;      // attention through xt_attention_fwd / xt_attention_bwd
  bool recompute;  // layer activations recomputed in the backward from the layer input
};

bool fused_supported(const xt_block_config& c) { return c.dtype == XT_BF16 && c.hd == 64 && c.d % 8 == 0; }

Dims dims_of(const xt_block_config& c) {
  Dims m{};
  m.B = c.B; m.S = c.S; m.d = c.d; m.H = c.H; m.hd = c.hd; m.F = c.F; m.V = c.V; m.L = c.n_layers;
  m.T = m.B * m.S;
  m.swiglu = c.mlp == XT_MLP_SWIGLU;
  m.rms = c.norm == XT_NORM_RMS;
  m.UP = m.swiglu ? 2 * m.F : m.F;
  m.dt = c.dtype;
  m.gdt = c.grad_dtype;
  m.e = int64_t(dtype_size(c.dtype));
  m.fused = c.attention == XT_ATTN_FUSED || (c.attention == XT_ATTN_AUTO && fused_supported(c));
  m.recompute = c.recompute != 0;
  return m;
}

// ------------------------------------------------------------------------------ GEMM shapes

xt_matmul_desc base_desc(int dt, int dt_c) {
  xt_matmul_desc g{};
  g.batch_outer = g.batch_inner = 1;
  g.dtype_ab = dt;
  g.dtype_c = dt_c;
  g.alpha = 1.f;
  return g;
}
// y[T, out] = x[T, in] @ W[in, out]
xt_matmul_desc lin_fwd(const Dims& m, int64_t in, int64_t out) {
  xt_matmul_desc g = base_desc(m.dt, m.dt);
  g.M = int(m.T); g.N = int(out); g.K = int(in);
  g.lda = in; g.ldb = out; g.ldc = out;
  return g;
}
// dW[in, out] += x[T, in]ᵀ @ dy[T, out]
xt_matmul_desc lin_dw(const Dims& m, int64_t in, int64_t out) {
  xt_matmul_desc g = base_desc(m.dt, m.gdt);
  g.M = int(in); g.N = int(out); g.K = int(m.T);
  g.trans_a = 1; g.lda = in; g.ldb = out; g.ldc = out;
  g.accumulate = 1;
  return g;
}
// dx[T, in] = dy[T, out] @ W[in, out]ᵀ
xt_matmul_desc lin_dx(const Dims& m, int64_t in, int64_t out) {
  xt_matmul_desc g = base_desc(m.dt, m.dt);
  g.M = int(m.T); g.N = int(in); g.K = int(out);
  g.trans_b = 1; g.lda = out; g.ldb = out; g.ldc = in;
  return g;
}
// Per (batch, head) blocks: q, k, v are column blocks of qkv [T, 3d]; P / dP are [B, H, S, S];
// o / do are [T, d] with head h at columns h·hd.
xt_matmul_desc att(const Dims& m, int64_t M, int64_t N, int64_t K, int ta, int tb, int64_t lda, int64_t ldb,
                   int64_t ldc, int64_t sao, int64_t sai, int64_t sbo, int64_t sbi, int64_t sco, int64_t sci,
                   float alpha, int causal) {
  xt_matmul_desc g = base_desc(m.dt, m.dt);
  g.M = int(M); g.N = int(N); g.K = int(K);
  g.trans_a = ta; g.trans_b = tb;
  g.lda = lda; g.ldb = ldb; g.ldc = ldc;
  g.batch_outer = int(m.B); g.batch_inner = int(m.H);
  g.stride_a_outer = sao; g.stride_a_inner = sai;
  g.stride_b_outer = sbo; g.stride_b_inner = sbi;
  g.stride_c_outer = sco; g.stride_c_inner = sci;
  g.alpha = alpha;
  g.causal = causal;
  return g;
}
float att_scale(const Dims& m) { return float(1.0 / sqrt(double(m.hd))); }
int64_t QS(const Dims& m) { return m.S * 3 * m.d; }    // batch stride of q/k/v blocks
int64_t PS(const Dims& m) { return m.H * m.S * m.S; }  // batch stride of P
int64_t OS(const Dims& m) { return m.S * m.d; }        // batch stride of o
// scores = α q kᵀ (tiles above the diagonal block skipped)
xt_matmul_desc att_scores(const Dims& m) {
  return att(m, m.S, m.S, m.hd, 0, 1, 3 * m.d, 3 * m.d, m.S, QS(m), m.hd, QS(m), m.hd, PS(m), m.S * m.S,
             att_scale(m), 1);
}
// o = P v
xt_matmul_desc att_pv(const Dims& m) {
  return att(m, m.S, m.hd, m.S, 0, 0, m.S, 3 * m.d, m.d, PS(m), m.S * m.S, QS(m), m.hd, OS(m), m.hd, 1.f, 2);
}
// dP = do vᵀ
xt_matmul_desc att_dp(const Dims& m) {
  return att(m, m.S, m.S, m.hd, 0, 1, m.d, 3 * m.d, m.S, OS(m), m.hd, QS(m), m.hd, PS(m), m.S * m.S, 1.f, 1);
}
// dV = Pᵀ do
xt_matmul_desc att_dv(const Dims& m) {
  return att(m, m.S, m.hd, m.S, 1, 0, m.S, m.d, 3 * m.d, PS(m), m.S * m.S, OS(m), m.hd, QS(m), m.hd, 1.f, 3);
}
// dQ = α dS k
xt_matmul_desc att_dq(const Dims& m) {
  return att(m, m.S, m.hd, m.S, 0, 0, m.S, 3 * m.d, 3 * m.d, PS(m), m.S * m.S, QS(m), m.hd, QS(m), m.hd,
             att_scale(m), 2);
}
// dK = α dSᵀ q
xt_matmul_desc att_dk(const Dims& m) {
  return att(m, m.S, m.hd, m.S, 1, 0, m.S, 3 * m.d, 3 * m.d, PS(m), m.S * m.S, QS(m), m.hd, QS(m), m.hd,
             att_scale(m), 3);
}
// logits[T, V] = hf[T, d] @ E[V, d]ᵀ
xt_matmul_desc logits_fwd(const Dims& m) {
  xt_matmul_desc g = base_desc(m.dt, m.dt);
  g.M = int(m.T); g.N = int(m.V); g.K = int(m.d);
  g.trans_b = 1; g.lda = m.d; g.ldb = m.d; g.ldc = m.V;
  return g;
}
// dE[V, d] += dlogits[T, V]ᵀ @ hf[T, d]
xt_matmul_desc logits_de(const Dims& m) {
  xt_matmul_desc g = base_desc(m.dt, m.gdt);
  g.M = int(m.V); g.N = int(m.d); g.K = int(m.T);
  g.trans_a = 1; g.lda = m.V; g.ldb = m.d; g.ldc = m.d;
  g.accumulate = 1;
  return g;
}
// dhf[T, d] = dlogits[T, V] @ E[V, d]
xt_matmul_desc logits_dhf(const Dims& m) {
  xt_matmul_desc g = base_desc(m.dt, m.dt);
  g.M = int(m.T); g.N = int(m.d); g.K = int(m.V);
  g.lda = m.V; g.ldb = m.d; g.ldc = m.d;
  return g;
}

size_t max_matmul_ws(const Dims& m) {
  const xt_matmul_desc all[] = {
      lin_fwd(m, m.d, 3 * m.d), lin_fwd(m, m.d, m.d), lin_fwd(m, m.d, m.UP), lin_fwd(m, m.F, m.d),
      lin_dw(m, m.d, 3 * m.d), lin_dw(m, m.d, m.d), lin_dw(m, m.d, m.UP), lin_dw(m, m.F, m.d),
      lin_dx(m, m.d, 3 * m.d), lin_dx(m, m.d, m.d), lin_dx(m, m.d, m.UP), lin_dx(m, m.F, m.d),
      logits_fwd(m), logits_de(m), logits_dhf(m)};
  const xt_matmul_desc composed[] = {att_scores(m), att_pv(m), att_dp(m), att_dv(m), att_dq(m), att_dk(m)};
  size_t mx = 0;
  for (const auto& g : all) mx = std::max(mx, matmul_workspace(g));
  if (!m.fused)
    for (const auto& g : composed) mx = std::max(mx, matmul_workspace(g));
  return mx;
}

// ------------------------------------------------------------------------------ buffers

struct Bufs {
  // P[l]: the layer's probabilities [B, H, S, S] (composed attention) or its softmax
  // normaliser lse, float32 [B, H, S] (fused attention)
  std::vector<void*> h_in, x1, qkv, P, o, h_mid, x2, up, mact;
  std::vector<void*> o_lo;  // fused attention: o's bf16 rounding residual (the backward's D uses o + o_lo)
  std::vector<float*> st1, st2;
  void *h_final, *hf, *logits, *tmp;
  float *stf, *lse, *rope, *dh, *one;
  void *gA, *gB, *dm, *dgu, *dP, *dqkv;
  void *ws_norm, *ws_ce, *ws_emb, *ws_mm, *ws_mm2;  // ws_mm2: the weight-gradient stream's matmul scratch
  size_t ws_mm_bytes, dP_bytes = 0;
  size_t total;
};

int carve(const Dims& m, void* base, Bufs& b) {
  Arena a{static_cast<char*>(base)};
  const int64_t T = m.T, d = m.d, e = m.e;
  const size_t act = size_t(T * d * e);
  // the matmul scratch first: its leading stream-K flag words are the workspace's first bytes
  b.ws_mm_bytes = max_matmul_ws(m);
  b.ws_mm = a.take(b.ws_mm_bytes);
  b.ws_mm2 = a.take(b.ws_mm_bytes);  // its flag words are zero on a zeroed workspace, as ws_mm's
  b.h_in.resize(m.L); b.x1.resize(m.L); b.qkv.resize(m.L); b.P.resize(m.L); b.o.resize(m.L);
  b.h_mid.resize(m.L); b.x2.resize(m.L); b.up.resize(m.L); b.mact.resize(m.L);
  b.st1.resize(m.L); b.st2.resize(m.L); b.o_lo.assign(m.L, nullptr);
  // With recompute every layer but its input shares one set of activation buffers: the forward
  // overwrites them layer by layer and the backward refills them for the layer it is at.
  for (int64_t l = 0; l < m.L; ++l) {
    b.h_in[l] = a.take(act);
    if (m.recompute && l > 0) {
      b.x1[l] = b.x1[0]; b.st1[l] = b.st1[0]; b.qkv[l] = b.qkv[0]; b.P[l] = b.P[0]; b.o[l] = b.o[0];
      b.o_lo[l] = b.o_lo[0]; b.h_mid[l] = b.h_mid[0]; b.x2[l] = b.x2[0]; b.st2[l] = b.st2[0];
      b.up[l] = b.up[0]; b.mact[l] = b.mact[0];
      continue;
    }
    b.x1[l] = a.take(act);
    b.st1[l] = static_cast<float*>(a.take(size_t(2 * T) * 4));
    b.qkv[l] = a.take(size_t(T * 3 * d * e));
    b.P[l] = a.take(m.fused ? size_t(m.B * m.H * m.S) * 4 : size_t(m.B * m.H * m.S * m.S * e));
    b.o[l] = a.take(act);
    if (m.fused) b.o_lo[l] = a.take(act);
    b.h_mid[l] = a.take(act);
    b.x2[l] = a.take(act);
    b.st2[l] = static_cast<float*>(a.take(size_t(2 * T) * 4));
    b.up[l] = a.take(size_t(T * m.UP * e));
    b.mact[l] = a.take(size_t(T * m.F * e));
  }
  b.h_final = a.take(act);
  b.hf = a.take(act);
  b.stf = static_cast<float*>(a.take(size_t(2 * T) * 4));
  b.logits = a.take(size_t(T * m.V * e));
  b.lse = static_cast<float*>(a.take(size_t(T) * 4));
  b.tmp = a.take(act);
  b.rope = static_cast<float*>(a.take(size_t(m.S * m.hd) * 4));
  b.dh = static_cast<float*>(a.take(size_t(T * d) * 4));
  b.one = static_cast<float*>(a.take(16));
  b.gA = a.take(act);
  b.gB = a.take(act);
  b.dm = a.take(size_t(T * m.F * e));
  b.dgu = a.take(size_t(T * m.UP * e));
  if (m.fused) {  // the attention backward's D = Σ dO∘O per row
    size_t ab = 0;
    XT_TRY(xt_attention_bwd_workspace_size(int(m.B), int(m.S), int(m.H), &ab));
    b.dP = a.take(ab);
    b.dP_bytes = ab;
  } else {
    b.dP = a.take(size_t(m.B * m.H * m.S * m.S * e));
  }
  b.dqkv = a.take(size_t(T * 3 * d * e));
  size_t nb = 0, cb = 0, eb = 0;
  XT_TRY(xt_norm_bwd_workspace_size(T, d, &nb));
  XT_TRY(xt_cross_entropy_workspace_size(T, &cb));
  XT_TRY(xt_embedding_workspace_size(T, &eb));
  b.ws_norm = a.take(nb);
  b.ws_ce = a.take(cb);
  b.ws_emb = a.take(eb);
  b.total = a.off + 256;
  return XT_OK;
}

int validate(const xt_block_config* c) {
  XT_REQUIRE(c != nullptr, "block: cfg is NULL");
  XT_REQUIRE(c->B > 0 && c->S > 0 && c->d > 0 && c->H > 0 && c->hd > 0 && c->F > 0 && c->V > 0 && c->n_layers > 0,
             "block: sizes must be positive");
  XT_REQUIRE(int64_t(c->H) * c->hd == c->d, "block: H·hd must equal d");
  XT_REQUIRE(c->norm == XT_NORM_RMS || c->norm == XT_NORM_LN, "block: bad norm");
  XT_REQUIRE(c->mlp == XT_MLP_SWIGLU || c->mlp == XT_MLP_GELU, "block: bad mlp");
  XT_REQUIRE(c->causal == 1, "block: attention must be causal");
  XT_REQUIRE(!c->rope || c->hd % 2 == 0, "block: RoPE needs an even head_dim");
  XT_REQUIRE(valid_dtype(c->dtype) && valid_dtype(c->grad_dtype), "block: bad dtype");
  XT_REQUIRE(c->p >= 0.f && c->p < 1.f, "block: dropout p must be in [0, 1)");
  XT_REQUIRE(int64_t(c->B) * c->S <= 16384, "block: B·S above 16384 tokens is not supported");
  XT_REQUIRE(c->attention >= XT_ATTN_AUTO && c->attention <= XT_ATTN_FUSED, "block: bad attention mode");
  XT_REQUIRE(c->recompute == 0 || c->recompute == 1, "block: recompute must be 0 or 1");
  if (c->attention == XT_ATTN_FUSED && !fused_supported(*c))
    return fail(XT_ERR_UNSUPPORTED, "block: fused attention needs bf16, head_dim 64 and d a multiple of 8");
  return XT_OK;
}

int check_params(const xt_block_config& c, const xt_block_params* p, bool grads) {
  XT_REQUIRE(p != nullptr, "block: params is NULL");
  XT_REQUIRE(p->E && p->g1 && p->Wqkv && p->Wo && p->g2 && p->W_up && p->W_down && p->gf,
             "block: a weight pointer is NULL");
  XT_REQUIRE(!c.learned_pos || p->P, "block: learned positions need P");
  XT_REQUIRE(c.norm == XT_NORM_RMS || (p->b1 && p->b2 && p->bf), "block: LayerNorm needs b1, b2, bf");
  if (grads) {
    XT_REQUIRE(p->dE && p->dg1 && p->dWqkv && p->dWo && p->dg2 && p->dW_up && p->dW_down && p->dgf,
               "block: a gradient pointer is NULL");
    XT_REQUIRE(!c.learned_pos || p->dP, "block: learned positions need dP");
    XT_REQUIRE(c.norm == XT_NORM_RMS || (p->db1 && p->db2 && p->dbf), "block: LayerNorm needs db1, db2, dbf");
  }
  return XT_OK;
}

__global__ void set_scalar(float* p, float v) {
  pdl_begin(); *p = v; }

uint64_t site_seed(const xt_block_config& c, int64_t l, uint64_t site) { return c.base_seed ^ uint64_t(l) ^ site; }

char* off(void* p, int64_t elems, int64_t e) { return static_cast<char*>(p) + elems * e; }

int g_overlap = 1;  // xt_block_set_overlap

// The weight-gradient stream of the current device and its events: [0] fork, [1..4] the last
// dW_down / dW_up / dWo / dWqkv done, [5] all done.  Created once per device (the first
// xt_block_workspace_size or xt_block_bwd call), never destroyed.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t ev[6] = {};
};
int side_stream(SideStream** out) {
  static std::mutex mu;
  static std::map<int, SideStream> per_device;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(XT_ERR_CUDA, "block: cudaGetDevice failed");
  std::lock_guard<std::mutex> lock(mu);
  SideStream& ss = per_device[dev];
  if (!ss.s) {
    if (cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess)
      return fail(XT_ERR_CUDA, "block: cannot create the weight-gradient stream");
    for (auto& e : ss.ev)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
        return fail(XT_ERR_CUDA, "block: cannot create the weight-gradient stream's events");
  }
  *out = &ss;
  return XT_OK;
}

int norm_fwd(const xt_block_config& c, const Dims& m, const void* x, const void* g, const void* b, void* y, float* st,
             void* stream) {
  if (m.rms) return xt_rms_norm_fwd(x, g, y, st, m.T, m.d, c.eps, m.dt, stream);
  return xt_layernorm_fwd(x, g, b, y, st, st + m.T, m.T, m.d, c.eps, m.dt, stream);
}

// sum = h + dropout(a), y = norm(sum) in one pass (xt_dropout_add_norm_fwd).
int add_norm_fwd(const xt_block_config& c, const Dims& m, const void* h, const void* a, void* sum, const void* g,
                 const void* b, void* y, float* st, uint64_t seed, bool drop, void* stream) {
  return xt_dropout_add_norm_fwd(h, a, sum, g, b, y, st, m.rms ? nullptr : st + m.T, m.T, m.d, c.p, seed, drop,
                                 m.rms ? XT_NORM_RMS : XT_NORM_LN, c.eps, m.dt, stream);
}

// The norm backward into dh (float32, += when acc_dx) that also writes g = dropout_bwd(dh) for the
// residual dropout site before it (xt_norm_bwd_dropout); parameter grads +=.
int norm_bwd_g(const xt_block_config& c, const Dims& m, const void* dy, const void* x, const void* g, const float* st,
               float* dh, void* dg, void* db, int acc_dx, void* gout, uint64_t seed, bool drop, const Bufs& b,
               void* stream) {
  return xt_norm_bwd_dropout(m.rms ? XT_NORM_RMS : XT_NORM_LN, dy, x, g, st, m.rms ? nullptr : st + m.T, dh, dg, db,
                             gout, m.T, m.d, m.dt, XT_F32, m.gdt, b.ws_norm, acc_dx, 1, c.p, seed, drop, stream);
}

// dh (float32) += norm backward of dy; parameter grads += as well.
int norm_bwd(const Dims& m, const void* dy, const void* x, const void* g, const float* st, float* dh, void* dg,
             void* db, int acc_dx, const Bufs& b, void* stream) {
  if (m.rms)
    return xt_rms_norm_bwd(dy, x, g, st, dh, dg, m.T, m.d, m.dt, XT_F32, m.gdt, b.ws_norm, acc_dx, 1, stream);
  return xt_layernorm_bwd(dy, x, g, st, st + m.T, dh, dg, db, m.T, m.d, m.dt, XT_F32, m.gdt, b.ws_norm, acc_dx, 1,
                          stream);
}

// Layer l's forward from its input up to the MLP activation (x1 … mact), into the layer's
// buffers.  The forward forms x1 = norm1(h_in) in the previous layer's fused add + norm (or, for
// layer 0, before the loop); the recompute (with_norm1) forms it here with the plain norm,
// which gives the same bits (the fused pass normalises the stored sum).
int layer_front(const xt_block_config& c, const Dims& m, const xt_block_params* prm, const Bufs& b, int64_t l,
                bool with_norm1, void* stream) {
  cudaStream_t s = as_stream(stream);
  const int64_t T = m.T, d = m.d, e = m.e;
  const bool drop = c.training && c.p > 0.f;
  if (with_norm1)
    XT_TRY(norm_fwd(c, m, b.h_in[l], prm->g1[l], prm->b1 ? prm->b1[l] : nullptr, b.x1[l], b.st1[l], stream));
  // attention sub-block
  XT_TRY(matmul(lin_fwd(m, d, 3 * d), b.x1[l], prm->Wqkv[l], b.qkv[l], b.ws_mm, b.ws_mm_bytes, s));
  if (c.rope)  // q and k blocks are 2H consecutive heads of each qkv row
    XT_TRY(xt_rope_fwd(b.qkv[l], b.qkv[l], b.rope, int(m.B), int(m.S), int(2 * m.H), int(m.hd), 3 * d, m.dt, stream));
  if (m.fused) {
    XT_TRY(xt_attention_fwd(b.qkv[l], off(b.qkv[l], d, e), off(b.qkv[l], 2 * d, e), 3 * d, b.o[l], b.o_lo[l], d,
                            static_cast<float*>(b.P[l]), int(m.B), int(m.S), int(m.H), int(m.hd), 1, m.dt, stream));
  } else {
    XT_TRY(matmul(att_scores(m), b.qkv[l], off(b.qkv[l], d, e), b.P[l], b.ws_mm, b.ws_mm_bytes, s));
    XT_TRY(xt_softmax_fwd(b.P[l], b.P[l], m.B * m.H * m.S, m.S, 2, m.S, m.dt, stream));
    XT_TRY(matmul(att_pv(m), b.P[l], off(b.qkv[l], 2 * d, e), b.o[l], b.ws_mm, b.ws_mm_bytes, s));
  }
  XT_TRY(matmul(lin_fwd(m, d, d), b.o[l], prm->Wo[l], b.tmp, b.ws_mm, b.ws_mm_bytes, s));
  // residual dropout-add, then the MLP sub-block's pre-norm, in one pass
  XT_TRY(add_norm_fwd(c, m, b.h_in[l], b.tmp, b.h_mid[l], prm->g2[l], prm->b2 ? prm->b2[l] : nullptr, b.x2[l],
                      b.st2[l], site_seed(c, l, kSiteAttn), drop, stream));
  // MLP sub-block
  XT_TRY(matmul(lin_fwd(m, d, m.UP), b.x2[l], prm->W_up[l], b.up[l], b.ws_mm, b.ws_mm_bytes, s));
  if (m.swiglu)
    XT_TRY(xt_swiglu_fwd(b.up[l], off(b.up[l], m.F, e), m.UP, b.mact[l], m.F, T, m.F, m.dt, stream));
  else
    XT_TRY(xt_gelu_fwd(b.up[l], b.mact[l], T * m.F, m.dt, stream));
  return XT_OK;
}

}  // namespace
}  // namespace xt

using namespace xt;

extern "C" {

int xt_block_workspace_size(const xt_block_config* cfg, size_t* bytes) {
  XT_TRY(validate(cfg));
  XT_REQUIRE(bytes, "xt_block_workspace_size: bytes is NULL");
  Bufs b;
  XT_TRY(carve(dims_of(*cfg), nullptr, b));
  *bytes = b.total;
  // the weight-gradient stream is created here when a device is present, before any stream
  // capture the caller may start (xt_block_bwd creates it otherwise)
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) == cudaSuccess && ndev > 0) {
    SideStream* ss = nullptr;
    XT_TRY(side_stream(&ss));
  } else {
    cudaGetLastError();  // no device: a size query only
  }
  return XT_OK;
}

int xt_block_fwd(const xt_block_config* cfg, const xt_block_params* prm, const int32_t* ids, const int32_t* targets,
                 float* loss, void* ws, void* stream) {
  XT_TRY(validate(cfg));
  const xt_block_config& c = *cfg;
  XT_TRY(check_params(c, prm, false));
  XT_REQUIRE(ids && targets && loss && ws, "xt_block_fwd: NULL pointer");
  const Dims m = dims_of(c);
  Bufs b;
  XT_TRY(carve(m, ws, b));
  cudaStream_t s = as_stream(stream);
  const int64_t T = m.T, d = m.d;
  const bool drop = c.training && c.p > 0.f;
  if (c.rope) XT_TRY(xt_rope_table(b.rope, int(m.S), int(m.hd), c.rope_base, 0, stream));
  XT_TRY(xt_embedding_fwd(ids, prm->E, c.learned_pos ? prm->P : nullptr, b.h_in[0], T, int(m.S), d, m.V, m.dt, stream));
  // the first pre-norm; every later one is fused with the residual add before it
  XT_TRY(norm_fwd(c, m, b.h_in[0], prm->g1[0], prm->b1 ? prm->b1[0] : nullptr, b.x1[0], b.st1[0], stream));
  for (int64_t l = 0; l < m.L; ++l) {
    XT_TRY(layer_front(c, m, prm, b, l, false, stream));
    XT_TRY(matmul(lin_fwd(m, m.F, d), b.mact[l], prm->W_down[l], b.tmp, b.ws_mm, b.ws_mm_bytes, s));
    // residual dropout-add, then the next layer's first pre-norm (or the final norm)
    if (l + 1 < m.L)
      XT_TRY(add_norm_fwd(c, m, b.h_mid[l], b.tmp, b.h_in[l + 1], prm->g1[l + 1], prm->b1 ? prm->b1[l + 1] : nullptr,
                          b.x1[l + 1], b.st1[l + 1], site_seed(c, l, kSiteFfn), drop, stream));
    else
      XT_TRY(add_norm_fwd(c, m, b.h_mid[l], b.tmp, b.h_final, prm->gf, prm->bf, b.hf, b.stf,
                          site_seed(c, l, kSiteFfn), drop, stream));
  }
  XT_TRY(matmul(logits_fwd(m), b.hf, prm->E, b.logits, b.ws_mm, b.ws_mm_bytes, s));
  // The loss is the graph's root and the backward seeds it with 1, so the forward forms the
  // loss and dlogits in one pass over the logits (dlogits overwrite them in place).
  launch(set_scalar, 1, 1, 0, s, b.one, 1.f);
  XT_TRY(check_launch("xt_block_fwd"));
  return xt_cross_entropy_fwd_bwd(b.logits, targets, b.lse, loss, b.one, b.logits, T, m.V, m.dt, m.dt, b.ws_ce,
                                  stream);
}

int xt_block_bwd(const xt_block_config* cfg, const xt_block_params* prm, const int32_t* ids, const int32_t* targets,
                 void* ws, void* stream) {
  XT_TRY(validate(cfg));
  const xt_block_config& c = *cfg;
  XT_TRY(check_params(c, prm, true));
  XT_REQUIRE(ids && targets && ws, "xt_block_bwd: NULL pointer");
  const Dims m = dims_of(c);
  Bufs b;
  XT_TRY(carve(m, ws, b));
  cudaStream_t s = as_stream(stream);
  const int64_t T = m.T, d = m.d, e = m.e;
  const bool drop = c.training && c.p > 0.f;
  // Weight gradients go to the side stream s2 (with its own matmul scratch) unless activations
  // are recomputed: then the layers share one set of activation buffers, which the next layer's
  // recompute overwrites while a dW of this layer could still be reading them.
  const bool side = !m.recompute && g_overlap;
  SideStream* ss = nullptr;
  if (side) XT_TRY(side_stream(&ss));
  cudaStream_t s2 = side ? ss->s : s;
  void* ws2 = side ? b.ws_mm2 : b.ws_mm;
  bool recorded[5] = {false, false, false, false, false};
  auto cuda_ok = [](cudaError_t e) { return e == cudaSuccess ? XT_OK : fail(XT_ERR_CUDA, "block: %s", cudaGetErrorString(e)); };
  // s2 waits for what s has enqueued so far (the dW's operands are written)
  auto fork = [&]() -> int {
    if (!side) return XT_OK;
    XT_TRY(cuda_ok(cudaEventRecord(ss->ev[0], s)));
    return cuda_ok(cudaStreamWaitEvent(s2, ss->ev[0], 0));
  };
  auto done = [&](int k) -> int {
    if (!side) return XT_OK;
    recorded[k] = true;
    return cuda_ok(cudaEventRecord(ss->ev[k], s2));
  };
  // s waits until dW k (the latest one enqueued) has read its operands, before overwriting them
  auto join = [&](int k) -> int {
    if (!side || !recorded[k]) return XT_OK;
    return cuda_ok(cudaStreamWaitEvent(s, ss->ev[k], 0));
  };
  enum { kDown = 1, kUp = 2, kO = 3, kQkv = 4 };
  // dlogits are in the logits buffer (written by the forward's cross-entropy pass) → tied
  // embedding and final norm; dE (the embedding's weight gradient) on s2, read again only by
  // the embedding backward after the final join
  XT_TRY(fork());
  XT_TRY(matmul(logits_de(m), b.logits, b.hf, prm->dE, ws2, b.ws_mm_bytes, s2));
  XT_TRY(matmul(logits_dhf(m), b.logits, prm->E, b.gA, b.ws_mm, b.ws_mm_bytes, s));
  // Each norm backward also writes the gradient the residual dropout before it passes on: the
  // MLP sub-block reads its df from gB, the attention sub-block its input gradient from gA.
  XT_TRY(norm_bwd_g(c, m, b.gA, b.h_final, prm->gf, b.stf, b.dh, prm->dgf, prm->dbf, 0, b.gB,
                    site_seed(c, m.L - 1, kSiteFfn), drop, b, stream));
  for (int64_t l = m.L - 1; l >= 0; --l) {
    // activation recompute: the layer's forward again from its saved input (the gradients in
    // gA / gB and dh are untouched by it)
    if (m.recompute) XT_TRY(layer_front(c, m, prm, b, l, true, stream));
    // MLP sub-block: df = dropout'(dh) (in gB); dW_down += mᵀ df; dm = df W_downᵀ; activation'; ...
    XT_TRY(fork());
    XT_TRY(matmul(lin_dw(m, m.F, d), b.mact[l], b.gB, prm->dW_down[l], ws2, b.ws_mm_bytes, s2));
    XT_TRY(done(kDown));
    XT_TRY(matmul(lin_dx(m, m.F, d), b.gB, prm->W_down[l], b.dm, b.ws_mm, b.ws_mm_bytes, s));
    XT_TRY(join(kUp));  // the layer above's dW_up has read dgu
    if (m.swiglu)
      XT_TRY(xt_swiglu_bwd(b.dm, m.F, b.up[l], off(b.up[l], m.F, e), m.UP, b.dgu, off(b.dgu, m.F, e), m.UP, T, m.F,
                           m.dt, 0, stream));
    else
      XT_TRY(xt_gelu_bwd(b.dm, b.up[l], b.dgu, T * m.F, m.dt, 0, stream));
    XT_TRY(fork());
    XT_TRY(matmul(lin_dw(m, d, m.UP), b.x2[l], b.dgu, prm->dW_up[l], ws2, b.ws_mm_bytes, s2));
    XT_TRY(done(kUp));
    XT_TRY(join(kDown));  // dW_down has read gB
    XT_TRY(matmul(lin_dx(m, d, m.UP), b.dgu, prm->W_up[l], b.gB, b.ws_mm, b.ws_mm_bytes, s));
    XT_TRY(norm_bwd_g(c, m, b.gB, b.h_mid[l], prm->g2[l], b.st2[l], b.dh, prm->dg2[l],
                      prm->db2 ? prm->db2[l] : nullptr, 1, b.gA, site_seed(c, l, kSiteAttn), drop, b, stream));
    // attention sub-block (its input gradient dropout'(dh) is in gA)
    XT_TRY(fork());
    XT_TRY(matmul(lin_dw(m, d, d), b.o[l], b.gA, prm->dWo[l], ws2, b.ws_mm_bytes, s2));
    XT_TRY(done(kO));
    XT_TRY(matmul(lin_dx(m, d, d), b.gA, prm->Wo[l], b.gB, b.ws_mm, b.ws_mm_bytes, s));
    XT_TRY(join(kQkv));  // the layer above's dWqkv has read dqkv
    if (m.fused) {
      XT_TRY(xt_attention_bwd(b.qkv[l], off(b.qkv[l], d, e), off(b.qkv[l], 2 * d, e), 3 * d, b.o[l], b.o_lo[l], b.gB,
                              d, static_cast<const float*>(b.P[l]), b.dqkv, off(b.dqkv, d, e), off(b.dqkv, 2 * d, e),
                              3 * d, b.dP, b.dP_bytes, int(m.B), int(m.S), int(m.H), int(m.hd), 1, m.dt, stream));
    } else {
      XT_TRY(matmul(att_dp(m), b.gB, off(b.qkv[l], 2 * d, e), b.dP, b.ws_mm, b.ws_mm_bytes, s));
      XT_TRY(xt_softmax_bwd(b.dP, b.P[l], b.dP, m.B * m.H * m.S, m.S, 2, m.S, m.dt, 0, stream));
      XT_TRY(matmul(att_dv(m), b.P[l], b.gB, off(b.dqkv, 2 * d, e), b.ws_mm, b.ws_mm_bytes, s));
      XT_TRY(matmul(att_dq(m), b.dP, off(b.qkv[l], d, e), b.dqkv, b.ws_mm, b.ws_mm_bytes, s));
      XT_TRY(matmul(att_dk(m), b.dP, b.qkv[l], off(b.dqkv, d, e), b.ws_mm, b.ws_mm_bytes, s));
    }
    if (c.rope)
      XT_TRY(xt_rope_bwd(b.dqkv, b.dqkv, b.rope, int(m.B), int(m.S), int(2 * m.H), int(m.hd), 3 * d, m.dt, 0, stream));
    XT_TRY(fork());
    XT_TRY(matmul(lin_dw(m, d, 3 * d), b.x1[l], b.dqkv, prm->dWqkv[l], ws2, b.ws_mm_bytes, s2));
    XT_TRY(done(kQkv));
    XT_TRY(join(kO));  // dWo has read gA
    XT_TRY(matmul(lin_dx(m, d, 3 * d), b.dqkv, prm->Wqkv[l], b.gA, b.ws_mm, b.ws_mm_bytes, s));
    if (l > 0)
      XT_TRY(norm_bwd_g(c, m, b.gA, b.h_in[l], prm->g1[l], b.st1[l], b.dh, prm->dg1[l],
                        prm->db1 ? prm->db1[l] : nullptr, 1, b.gB, site_seed(c, l - 1, kSiteFfn), drop, b, stream));
    else
      XT_TRY(norm_bwd(m, b.gA, b.h_in[l], prm->g1[l], b.st1[l], b.dh, prm->dg1[l], prm->db1 ? prm->db1[l] : nullptr,
                      1, b, stream));
  }
  // every weight gradient is in before the embedding backward adds into dE and the call returns
  if (side) {
    XT_TRY(cuda_ok(cudaEventRecord(ss->ev[5], s2)));
    XT_TRY(cuda_ok(cudaStreamWaitEvent(s, ss->ev[5], 0)));
  }
  return xt_embedding_bwd(ids, b.dh, prm->dE, c.learned_pos ? prm->dP : nullptr, T, int(m.S), d, m.V, XT_F32, m.gdt,
                          b.ws_emb, 1, stream);
}

int xt_block_set_overlap(int on) {
  XT_REQUIRE(on == 0 || on == 1, "xt_block_set_overlap: on must be 0 or 1");
  g_overlap = on;
  return XT_OK;
}

int xt_block_zero_grads(const xt_block_config* cfg, const xt_block_params* prm, void* stream) {
  XT_TRY(validate(cfg));
  const xt_block_config& c = *cfg;
  XT_TRY(check_params(c, prm, true));
  const Dims m = dims_of(c);
  cudaStream_t s = as_stream(stream);
  const size_t g = dtype_size(m.gdt);
  auto z = [&](void* p, int64_t n) -> int {
    if (p && cudaMemsetAsync(p, 0, size_t(n) * g, s) != cudaSuccess) return check_launch("xt_block_zero_grads");
    return XT_OK;
  };
  XT_TRY(z(prm->dE, m.V * m.d));
  if (c.learned_pos) XT_TRY(z(prm->dP, m.S * m.d));
  for (int64_t l = 0; l < m.L; ++l) {
    XT_TRY(z(prm->dg1[l], m.d));
    XT_TRY(z(prm->dg2[l], m.d));
    if (!m.rms) {
      XT_TRY(z(prm->db1[l], m.d));
      XT_TRY(z(prm->db2[l], m.d));
    }
    XT_TRY(z(prm->dWqkv[l], m.d * 3 * m.d));
    XT_TRY(z(prm->dWo[l], m.d * m.d));
    XT_TRY(z(prm->dW_up[l], m.d * m.UP));
    XT_TRY(z(prm->dW_down[l], m.F * m.d));
  }
  XT_TRY(z(prm->dgf, m.d));
  if (!m.rms) XT_TRY(z(prm->dbf, m.d));
  return XT_OK;
}

}  // extern "C"
