// Fused attention for sm_103a: per (batch, head), scores = Q Kᵀ·α, P = softmax(scores) under
// the causal mask, O = P V ([AE] § Attention 用组合 gives the composition; this computes the
// same result tile by tile, so the S × S probabilities never reach global memory).
//
// Forward (one CTA per SM, persistent, two independent streams of 128-query tiles, heaviest
// first; each stream has its own warps, buffers and work items, so one stream's MMA round trips
// overlap the other's softmax):
//   warps 0 / 2  TMA producer: Q tile once per work item, K and V tiles through 2-slot rings;
//   warps 1 / 3  MMA issuer (warp 1 also owns TMEM): S_j = Q K_jᵀ into the stream's TMEM score
//                buffer (issued once the softmax warps have loaded S_{j−1}), then O += P_j V_j
//                into the stream's TMEM accumulator;
//   warps 4..7 / 8..11  one query row per thread (TMEM lane): load the score row, mask, running
//                max, exp2, running sum, write P_j as bf16 into shared memory in the 128-byte-
//                swizzled K-major layout the MMA reads; rescale O in TMEM when the running max
//                grows by more than 2^8 (otherwise the stale max is kept: O and the sum share it,
//                so O / l is exact either way); at the end O / l goes out through a TMA store and
//                the row's natural-log normaliser lse = log Σ exp(scores) is saved for the backward.
//
// Backward (deterministic, no atomics): D = rowsum(dO ∘ O); then one kernel per 128-key tile
// that recomputes Pᵀ = exp(K Qᵀ·α − lse) and dPᵀ = V dOᵀ and accumulates dV = Pᵀ dO and
// dK = α·dSᵀ Q over the query tiles, and one kernel per 128-query tile that recomputes P and dP
// and accumulates dQ = α·dS K over the key tiles, with dS = P ∘ (dP − D).
//
// Every mbarrier wait is bounded (%globaltimer); on expiry the CTA records XT_DEVERR_TIMEOUT,
// all roles stop, the producer waits (bounded) for its copies in flight and TMEM is freed.
#include <cudaTypedefs.h>

#include <cmath>

#include "gemm.cuh"

namespace xt {
namespace attn {

using namespace gemm;

constexpr int HD = 64;                     // head dimension the kernels are built for
constexpr int BT = 128;                    // query / key tile
// Backward kernels: warp 0 TMA, warp 1 MMA, warps 2..9 rows — two warps per TMEM lane quadrant,
// each owning 64 of a tile's 128 columns (the backward's P and dS are elementwise, so the halves
// never need each other's values).
constexpr int kThreadsBwd = 320;
constexpr int TILE = BT * 128;             // one 128-row × 64-element bf16 tile: 16 KB
constexpr int PT = 2 * TILE;               // 128 × 128 bf16 operand: two 64-wide K chunks
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.f;            // log2 growth of the running max that forces a rescale

struct FwdParams {
  int B, H, S, nq, items, causal;
  float sc;     // α·log2 e
  float* lse;   // [B, H, S], natural log
  int o_lo;     // 1: also store O − bf16(O) rounded to bf16 (through tmOlo)
  uint32_t* flag;
  uint64_t wait_ns;  // limit of the waits on work; draining the CTA's own copies / MMAs keeps the default
};

// Work item i → (b, h, query tile); with a causal mask, the longest rows come first.
struct Item {
  int b, h, qt, nkv;
};
__device__ __forceinline__ Item decode(int i, int B, int H, int nq, int causal) {
  const int bh_n = B * H;
  Item it;
  const int t = i / bh_n, bh = i - t * bh_n;
  it.qt = causal ? nq - 1 - t : t;
  it.b = bh / H;
  it.h = bh - it.b * H;
  it.nkv = causal ? it.qt + 1 : nq;
  return it;
}

// Work item of round r for this CTA: rounds alternate direction over the CTAs (a boustrophedon),
// so with items ordered longest first the CTAs' totals even out (95 % balance for the causal
// 1024-token case against 84 % for plain round-robin).
__device__ __forceinline__ int snake_item(int r) {
  const int G = int(gridDim.x), c = int(blockIdx.x);
  return r * G + ((r & 1) ? G - 1 - c : c);
}

// Row r (0..127) of a 128-row operand in the 128-byte-swizzled K-major layout: 16-byte unit u of
// the 64-element chunk c sits at chunk base + r·128 + ((u ^ (r & 7)) << 4).
__device__ __forceinline__ uint32_t swz(uint32_t base, int r, int c, int u) {
  return base + uint32_t(c) * TILE + uint32_t(r) * 128 + (uint32_t(u ^ (r & 7)) << 4);
}
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Pins the computation of r[] before the next volatile asm (an mbarrier wait): the compiler may
// otherwise sink pure register arithmetic past the wait, serialising it behind the tensor core
// instead of overlapping the two.  Emits no instruction.
template <int N>
__device__ __forceinline__ void keep_before(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// 2^x with the hardware approximation (ex2.approx.ftz: relative error ~2⁻²², −inf → +0,
// results below 2⁻¹²⁶ flushed to 0); the probabilities it feeds are rounded to bf16.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait taken by a whole warp (the decision is warp-uniform).  It polls with test_wait: the
// row warps' waits for S, dP and the accumulators are handoffs on each tile's MMA chain, and a
// suspended try_wait wakes later than the next poll sees the phase flip (dK/dV + dQ backward
// 120.2 -> 118.2 us at B 8, S 1024, 12 heads x 64).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  return __all_sync(0xffffffffu, mbar_wait_spin(bar, parity, limit_ns));
}

// ------------------------------------------------------------------------------ forward


// setmaxnreg: a warp group gives registers back to the pool or takes them from it (all four
// warps of the group execute it).
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// The forward with two independent query-tile streams per CTA: each stream has its own TMA
// producer (warps 0 / 2), MMA issuer (warps 1 / 3), four softmax warps (4–7 / 8–11), TMEM score
// buffer and O accumulator, Q tile, two-slot K / V rings and P tile, and its own work items
// (virtual CTA 2·blockIdx + stream of a grid twice as wide).  A stream's softmax warps wait for
// their scores while the other stream's compute, so the per-tile MMA round trips of one stream
// overlap the other's exp and P stores.  With one score buffer per stream, S_{j+1} is computed
// as soon as the softmax warps have loaded S_j.  The epilogue stages O (and O_lo) in the warp's
// own rows of the P tile once the last P V is done.
constexpr int kThreadsFwd = 384;
constexpr int KV_SLOTS = 2;
constexpr uint32_t kFwdRegsCtl = 72, kFwdRegsRows = 216;  // 128·72 + 256·216 = 384·168
struct FwdSmem {
  static constexpr int Q = 0;
  static constexpr int K = Q + TILE;
  static constexpr int V = K + KV_SLOTS * TILE;
  static constexpr int P = V + KV_SLOTS * TILE;
  static constexpr int STREAM = P + PT;           // 112 KB per stream
  static constexpr int BARS = 2 * STREAM;
  static constexpr int BYTES = 1024 + BARS + 512;
};

__global__ void __launch_bounds__(kThreadsFwd, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                     const __grid_constant__ CUtensorMap tmOlo, const FwdParams p) {
  pdl_begin();
  constexpr uint32_t IDESC_S = instr_desc_bf16(128, 128, false, false);
  constexpr uint32_t IDESC_PV = instr_desc_bf16(128, HD, false, true);
  constexpr uint32_t TCOLS = 512;  // stream s: S [256 s, 256 s + 128), O [256 s + 128, 256 s + 192)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  // per stream, 16 slots: q_full, q_empty, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full,
  // s_free, p_full, p_free, mma_done
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + FwdSmem::BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int st = 0; st < 2; ++st) {
      uint64_t* b = bars + 16 * st;
      for (int i = 0; i < 15; ++i) mbar_init(smem_u32(&b[i]), (i == 11 || i == 12) ? 4 : 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  auto give_up = [&]() {
    *abort_flag = 1;
    flag_error(p.flag, XT_DEVERR_TIMEOUT);
  };
  const int VG = 2 * int(gridDim.x);
  // work item of round r for virtual CTA vc (rounds alternate direction, longest items first)
  auto vitem = [&](int r, int vc) { return r * VG + ((r & 1) ? VG - 1 - vc : vc); };

  const int wg = warp >> 2;
  if (wg == 0) {
    regs_dec<kFwdRegsCtl>();
    const int st = warp >> 1;
    const int vc = 2 * int(blockIdx.x) + st;
    uint64_t* b = bars + 16 * st;
    uint64_t *q_full = b, *q_empty = b + 1, *k_full = b + 2, *k_empty = b + 4, *v_full = b + 6, *v_empty = b + 8;
    uint64_t *s_full = b + 10, *s_free = b + 11, *p_full = b + 12, *p_free = b + 13, *mma_done = b + 14;
    const uint32_t base = sb + uint32_t(st * FwdSmem::STREAM);
    if ((warp & 1) == 0 && lane == 0) {
      // -------------------------------------------------------------- TMA producer
      int ks = 0, vs = 0, nk = 0, nv = 0, nqi = 0;
      uint32_t kph = 0, vph = 0;
      bool ok = true;
      #pragma unroll 1
      for (int r = 0; r * VG < p.items && ok && !*abort_flag; ++r) {
        const int i = vitem(r, vc);
        if (i >= p.items) continue;
        const Item it = decode(i, p.B, p.H, p.nq, p.causal);
        if (!mbar_wait(smem_u32(q_empty), (nqi & 1) ^ 1, p.wait_ns)) { ok = false; break; }
        mbar_expect_tx(smem_u32(q_full), TILE);
        tma_load_4d(base + FwdSmem::Q, &tmQ, smem_u32(q_full), 0, it.h, it.qt * BT, it.b);
        ++nqi;
        #pragma unroll 1
        for (int j = 0; j < it.nkv; ++j) {
          if (*abort_flag) { ok = false; break; }
          if (!mbar_wait(smem_u32(&k_empty[ks]), kph ^ 1, p.wait_ns)) { ok = false; break; }
          mbar_expect_tx(smem_u32(&k_full[ks]), TILE);
          tma_load_4d(base + FwdSmem::K + ks * TILE, &tmK, smem_u32(&k_full[ks]), 0, it.h, j * BT, it.b);
          ++nk;
          if (++ks == KV_SLOTS) { ks = 0; kph ^= 1; }
          if (!mbar_wait(smem_u32(&v_empty[vs]), vph ^ 1, p.wait_ns)) { ok = false; break; }
          mbar_expect_tx(smem_u32(&v_full[vs]), TILE);
          tma_load_4d(base + FwdSmem::V + vs * TILE, &tmV, smem_u32(&v_full[vs]), 0, it.h, j * BT, it.b);
          ++nv;
          if (++vs == KV_SLOTS) { vs = 0; vph ^= 1; }
        }
      }
      if (!ok) give_up();
      // bounded wait for the fills that may still be in flight
      bool drained = true;
      if (nqi > 0) drained &= mbar_wait(smem_u32(q_full), (nqi - 1) & 1);
      for (int n = 0; n < (nk < KV_SLOTS ? nk : KV_SLOTS); ++n) {
        if (--ks < 0) { ks = KV_SLOTS - 1; kph ^= 1; }
        drained &= mbar_wait(smem_u32(&k_full[ks]), kph);
      }
      for (int n = 0; n < (nv < KV_SLOTS ? nv : KV_SLOTS); ++n) {
        if (--vs < 0) { vs = KV_SLOTS - 1; vph ^= 1; }
        drained &= mbar_wait(smem_u32(&v_full[vs]), vph);
      }
      if (!drained) give_up();
    } else if ((warp & 1) == 1 && lane == 0) {
      // -------------------------------------------------------------- MMA issuer
      const uint32_t tS = tbase + uint32_t(256 * st), tO = tS + 128;
      int ks = 0, vs = 0, nqi = 0;
      uint32_t kph = 0, vph = 0;
      uint32_t g = 0;  // score tiles issued so far (phases of the single S and P buffers)
      bool ok = true;
      auto issue_pv = [&](uint32_t gg, bool first) -> bool {
        if (!mbar_wait_spin(smem_u32(p_full), gg & 1, p.wait_ns)) return false;
        if (!mbar_wait_spin(smem_u32(&v_full[vs]), vph, p.wait_ns)) return false;
        tc_fence_after();
        const uint32_t ps = base + FwdSmem::P;
        const uint32_t vsm = base + FwdSmem::V + vs * TILE;
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk) {
          const uint64_t ad = smem_desc(ps + (kk >> 2) * TILE + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc(vsm + kk * 16 * 128, TILE, 1024);
          tc_mma<false>(tO, ad, bd, IDESC_PV, (!first || kk > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&v_empty[vs]));
        tc_commit(smem_u32(p_free));
        if (++vs == KV_SLOTS) { vs = 0; vph ^= 1; }
        return true;
      };
      #pragma unroll 1
      for (int r = 0; r * VG < p.items && ok && !*abort_flag; ++r) {
        const int i = vitem(r, vc);
        if (i >= p.items) continue;
        const Item it = decode(i, p.B, p.H, p.nq, p.causal);
        if (!mbar_wait_spin(smem_u32(q_full), nqi & 1, p.wait_ns)) { ok = false; break; }
        ++nqi;
        tc_fence_after();
        #pragma unroll 1
        for (int j = 0; j < it.nkv; ++j, ++g) {
          if (*abort_flag || !mbar_wait_spin(smem_u32(&k_full[ks]), kph, p.wait_ns) ||
              !mbar_wait_spin(smem_u32(s_free), (g & 1) ^ 1, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t ksm = base + FwdSmem::K + ks * TILE;
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk)
            tc_mma<false>(tS, smem_desc(base + FwdSmem::Q + kk * 32, 16, 1024), smem_desc(ksm + kk * 32, 16, 1024),
                          IDESC_S, kk > 0 ? 1u : 0u);
          tc_commit(smem_u32(&k_empty[ks]));
          tc_commit(smem_u32(s_full));
          if (j == it.nkv - 1) tc_commit(smem_u32(q_empty));
          if (++ks == KV_SLOTS) { ks = 0; kph ^= 1; }
          if (j >= 1 && !issue_pv(g - 1, j == 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (!issue_pv(g - 1, it.nkv == 1)) { ok = false; break; }
      }
      if (!ok) give_up();
      // every MMA issued has completed (also after a give-up) before TMEM is released
      tc_commit(smem_u32(mma_done));
      if (!mbar_wait(smem_u32(mma_done), 0)) give_up();
    }
  } else {
    regs_inc<kFwdRegsRows>();
    // ---------------------------------------------------------------- softmax / epilogue
    const int st = wg - 1;
    const int vc = 2 * int(blockIdx.x) + st;
    uint64_t* b = bars + 16 * st;
    uint64_t *s_full = b + 10, *s_free = b + 11, *p_full = b + 12, *p_free = b + 13;
    const uint32_t base = sb + uint32_t(st * FwdSmem::STREAM);
    const uint32_t tS = tbase + uint32_t(256 * st), tO = tS + 128;
    const int qw = warp & 3;            // TMEM lanes [32 qw, 32 qw + 32)
    const int rr = qw * 32 + lane;      // row within the query tile
    const uint32_t lane_off = uint32_t(qw * 32) << 16;
    // O and O_lo are staged in this warp's own rows of the P tile (chunk 0 and chunk 1)
    const uint32_t stage = base + FwdSmem::P + uint32_t(qw) * 4096;
    uint32_t g = 0;
    #pragma unroll 1
    for (int r = 0; r * VG < p.items; ++r) {
      const int i = vitem(r, vc);
      if (i >= p.items) continue;
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const Item it = decode(i, p.B, p.H, p.nq, p.causal);
      const int row = it.qt * BT + rr;
      float m = -INFINITY;  // running max of the raw scores (Q·K, before α)
      float l = 0.f;        // running Σ 2^((s − m)·sc)
      bool ok = true;
      #pragma unroll 1
      for (int j = 0; j < it.nkv; ++j, ++g) {
        if (!warp_wait(smem_u32(s_full), g & 1, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        uint32_t r[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tS + lane_off + uint32_t(c * 32), *reinterpret_cast<uint32_t(*)[32]>(r + 32 * c));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(s_free));
        // keys at or past `lim` (relative to this tile) are masked
        const int lim = (p.causal ? min(row + 1, p.S) : p.S) - j * BT;
        if (lim < BT) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= lim) r[c] = __float_as_uint(-INFINITY);
        }
        float mx[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) mx[t] = __uint_as_float(r[t]);
#pragma unroll
        for (int c = 8; c < 128; ++c) mx[c & 7] = fmaxf(mx[c & 7], __uint_as_float(r[c]));
        const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        const float m_new = fmaxf(m, mt);
        const bool need = m_new > m && (m == -INFINITY || (m_new - m) * p.sc > kRescale);
        // P V of the previous tile is complete before P is rewritten (and before O is rescaled)
        if (!warp_wait(smem_u32(p_free), (g & 1) ^ 1, p.wait_ns)) { ok = false; break; }
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // O holds Σ 2^((s − m)·sc)·v with the old m: bring it to m_new
          tc_fence_after();
          const float a = need ? exp2f((m - m_new) * p.sc) : 1.f;
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + lane_off + uint32_t(c * 32), o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
            tmem_st32(tO + lane_off + uint32_t(c * 32), o);
          }
          tmem_st_wait();
        }
        if (need) {
          l = (m == -INFINITY) ? 0.f : l * exp2f((m - m_new) * p.sc);
          m = m_new;
        }
        const float ms = (m == -INFINITY) ? 0.f : m * p.sc;
        if (j == 0) {  // the previous item's O stores have read this warp's rows of the P tile
          if (lane == 0) bulk_wait_read_0();
          __syncwarp();
        }
        const uint32_t ps = base + FwdSmem::P;
        float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // 8 independent partial sums
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int un = 0; un < 8; ++un) {
            float e[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              e[t] = ex2(fmaf(__uint_as_float(r[c * 64 + un * 8 + t]), p.sc, -ms));
              ls[t] += e[t];
            }
            st_shared_v4(swz(ps, rr, c, un), pack_bf16(e[0], e[1]), pack_bf16(e[2], e[3]), pack_bf16(e[4], e[5]),
                         pack_bf16(e[6], e[7]));
          }
        l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(p_full));
      }
      if (!ok) {
        if (lane == 0) give_up();
        break;
      }
      // ---- epilogue: O / l after the last P V
      if (!warp_wait(smem_u32(p_free), (g - 1) & 1, p.wait_ns)) {
        if (lane == 0) give_up();
        break;
      }
      tc_fence_after();
      uint32_t o[64];
      tmem_ld32(tO + lane_off, *reinterpret_cast<uint32_t(*)[32]>(o));
      tmem_ld32(tO + lane_off + 32, *reinterpret_cast<uint32_t(*)[32]>(o + 32));
      tmem_ld_wait();
      tc_fence_before();
      const float inv = 1.f / l;
      // O rounded to bf16, and (optionally) the rounding residual O − bf16(O) rounded to bf16
#pragma unroll
      for (int un = 0; un < 8; ++un) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = __uint_as_float(o[8 * un + 2 * e]) * inv, bb = __uint_as_float(o[8 * un + 2 * e + 1]) * inv;
          hi[e] = pack_bf16(a, bb);
          const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&hi[e]);
          lo[e] = pack_bf16(a - __low2float(h), bb - __high2float(h));
        }
        const uint32_t off = uint32_t(lane) * 128 + (uint32_t(un ^ (lane & 7)) << 4);
        st_shared_v4(stage + off, hi[0], hi[1], hi[2], hi[3]);
        if (p.o_lo) st_shared_v4(stage + TILE + off, lo[0], lo[1], lo[2], lo[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_4d(&tmO, stage, 0, it.h, it.qt * BT + qw * 32, it.b);
        if (p.o_lo) tma_store_4d(&tmOlo, stage + TILE, 0, it.h, it.qt * BT + qw * 32, it.b);
        bulk_commit();
      }
      if (row < p.S) p.lse[(int64_t(it.b) * p.H + it.h) * p.S + row] = (m * p.sc + log2f(l)) * kLn2;
    }
    if (lane == 0) bulk_wait_all();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, TCOLS);
  }
}

// ------------------------------------------------------------------------------ backward

struct BwdParams {
  int B, H, S, nq, items, causal;
  float sc;          // α·log2 e
  float alpha;       // α = 1/√hd
  const float* lse;  // [B, H, S] natural log, from the forward
  const float* D;    // [B, H, S] rowsum(dO ∘ O)
  uint32_t* flag;
  uint64_t wait_ns;  // limit of the waits on work; draining the CTA's own copies / MMAs keeps the default
};

// D[b, h, s] = Σ_c dO[t, h·hd + c]·O[t, h·hd + c], t = b·S + s: 8 threads per (t, h), four
// (t, h) rows per warp; the loop runs warp-uniformly so the shuffles see every lane.  With the
// forward's residual O_lo, O = O_hi + O_lo to ~2⁻¹⁶ and D agrees with Σ_c P·dP of the recomputed
// P and dP, so the rows of dS = P∘(dP − D) sum to ~0 as they must; the bf16 O alone would leave
// a bias of its rounding (2⁻⁹ relative) in every row of dS.
__global__ void attn_delta_kernel(const bf16* __restrict__ o, const bf16* __restrict__ o_lo,
                                  const bf16* __restrict__ dO, int64_t ld_o, int B, int S, int H,
                                  float* __restrict__ D) {
  pdl_begin();
  const int64_t n = int64_t(B) * S * H;
  const int lane = threadIdx.x & 31, sub = lane & 7;
  const int64_t warp0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t base = warp0 * 4; base < n; base += nwarps * 4) {
    const int64_t r = base + (lane >> 3);
    const bool act = r < n;
    float acc = 0.f;
    int64_t t = 0;
    int h = 0;
    if (act) {
      t = r / H;
      h = int(r - t * H);
      const int64_t off = t * ld_o + int64_t(h) * HD + sub * 8;
      float a[8], b[8];
      Vec<bf16>::load(o + off, a);
      Vec<bf16>::load(dO + off, b);
      if (o_lo) {
        float c[8];
        Vec<bf16>::load(o_lo + off, c);
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] += c[e];
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) acc = fmaf(a[e], b[e], acc);
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if (act && sub == 0) {
      const int64_t bb = t / S, ss = t - bb * S;
      D[(bb * H + h) * S + ss] = acc;
    }
  }
}

// Work item of the key-tile kernel: (b, h, key tile kt); query tiles kt.. (causal) or all.
__device__ __forceinline__ Item decode_kv(int i, int B, int H, int nq, int causal) {
  const int bh_n = B * H;
  Item it;
  const int t = i / bh_n, bh = i - t * bh_n;
  it.qt = t;  // the key tile
  it.b = bh / H;
  it.h = bh - it.b * H;
  it.nkv = causal ? nq - t : nq;  // number of query tiles
  return it;
}

// Staged TMA store of one warp's 32 rows × 64 bf16 (values × scale) from TMEM columns [col, col + 64).
__device__ __forceinline__ void store_rows(uint32_t taddr, float scale, uint32_t stage, int lane,
                                           const CUtensorMap* tm, int h, int y, int b) {
  uint32_t o[64];
  tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(o));
  tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(o + 32));
  tmem_ld_wait();
#pragma unroll
  for (int un = 0; un < 8; ++un)
    st_shared_v4(stage + uint32_t(lane) * 128 + (uint32_t(un ^ (lane & 7)) << 4),
                 pack_bf16(__uint_as_float(o[8 * un]) * scale, __uint_as_float(o[8 * un + 1]) * scale),
                 pack_bf16(__uint_as_float(o[8 * un + 2]) * scale, __uint_as_float(o[8 * un + 3]) * scale),
                 pack_bf16(__uint_as_float(o[8 * un + 4]) * scale, __uint_as_float(o[8 * un + 5]) * scale),
                 pack_bf16(__uint_as_float(o[8 * un + 6]) * scale, __uint_as_float(o[8 * un + 7]) * scale));
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_4d(tm, stage, 0, h, y, b);
    bulk_commit();
  }
}

struct KvSmem {
  static constexpr int K = 0;
  static constexpr int V = K + TILE;
  static constexpr int QD = V + TILE;            // 2 slots × (Q tile, dO tile)
  static constexpr int P = QD + 2 * 2 * TILE;    // Pᵀ  [keys × queries]
  static constexpr int DS = P + PT;              // dSᵀ [keys × queries]
  static constexpr int STAGE = DS + PT;          // 4 warps × (dV, dK) × 4 KB
  static constexpr int VEC = STAGE + 8 * 4096;   // 2 slots × (lse·log2 e, D) × 128 floats
  static constexpr int BARS = VEC + 2 * 2 * 512;
  static constexpr int BYTES = 1024 + BARS + 256;
};

// dK, dV for one 128-key tile per work item: thread = key row; Sᵀ = K Qᵀ and dPᵀ = V dOᵀ per
// query tile, Pᵀ = 2^(Sᵀ·sc − lse2[q]) (0 where q < key or q ≥ S), dSᵀ = Pᵀ ∘ (dPᵀ − D[q]);
// dV += Pᵀ dO and dK += dSᵀ Q accumulate in TMEM; dK is scaled by α on the way out.
__global__ void __launch_bounds__(kThreadsBwd, 1)
    attn_bwd_kv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV,
                       const BwdParams p) {
  pdl_begin();
  constexpr uint32_t IDESC_S = instr_desc_bf16(128, 128, false, false);
  constexpr uint32_t IDESC_O = instr_desc_bf16(128, HD, false, true);
  constexpr uint32_t TCOLS = 512;  // Sᵀ0 [0,128), Sᵀ1 [128,256), dPᵀ [256,384), dV [384,448), dK [448,512)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + KvSmem::BARS);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + 1;
  uint64_t* qd_full = bars + 2;     // [2]
  uint64_t* qd_empty = bars + 4;    // [2]
  uint64_t* s_full = bars + 6;      // [2]
  uint64_t* s_free = bars + 8;      // [2]
  uint64_t* dp_full = bars + 10;
  uint64_t* dp_free = bars + 11;
  uint64_t* p_full = bars + 12;
  uint64_t* p_free = bars + 13;
  uint64_t* ds_full = bars + 14;
  uint64_t* ds_free = bars + 15;
  uint64_t* vec_full = bars + 16;   // [2] the query tile's lse / D rows are in shared memory
  uint64_t* mma_done = bars + 18;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 19);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* vec = reinterpret_cast<float*>(smem + KvSmem::VEC);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(kv_full), 1);
    mbar_init(smem_u32(kv_empty), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&qd_full[b]), 1);
      mbar_init(smem_u32(&qd_empty[b]), 1);
      mbar_init(smem_u32(&s_full[b]), 1);
      mbar_init(smem_u32(&s_free[b]), 8);
    }
    mbar_init(smem_u32(dp_full), 1);
    mbar_init(smem_u32(dp_free), 8);
    mbar_init(smem_u32(p_full), 8);
    mbar_init(smem_u32(p_free), 1);
    mbar_init(smem_u32(ds_full), 8);
    mbar_init(smem_u32(ds_free), 1);
    mbar_init(smem_u32(&vec_full[0]), 256);
    mbar_init(smem_u32(&vec_full[1]), 256);
    mbar_init(smem_u32(mma_done), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmDO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t tDP = tbase + 256, tDV = tbase + 384, tDK = tbase + 448;

  auto give_up = [&]() {
    *abort_flag = 1;
    flag_error(p.flag, XT_DEVERR_TIMEOUT);
  };

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------------------- TMA producer
      int slot = 0, nkv = 0, nqd = 0;
      uint32_t ph = 0;
      bool ok = true;
      #pragma unroll 1
      for (int r = 0; r * int(gridDim.x) < p.items && ok && !*abort_flag; ++r) {
        const int i = snake_item(r);
        if (i >= p.items) continue;
        const Item it = decode_kv(i, p.B, p.H, p.nq, p.causal);
        if (!mbar_wait(smem_u32(kv_empty), (nkv & 1) ^ 1, p.wait_ns)) { ok = false; break; }
        mbar_expect_tx(smem_u32(kv_full), 2 * TILE);
        tma_load_4d(sb + KvSmem::K, &tmK, smem_u32(kv_full), 0, it.h, it.qt * BT, it.b);
        tma_load_4d(sb + KvSmem::V, &tmV, smem_u32(kv_full), 0, it.h, it.qt * BT, it.b);
        ++nkv;
        const int q_first = p.causal ? it.qt : 0;
        #pragma unroll 1
        for (int j = 0; j < it.nkv; ++j) {
          if (*abort_flag || !mbar_wait(smem_u32(&qd_empty[slot]), ph ^ 1, p.wait_ns)) { ok = false; break; }
          const uint32_t fb = smem_u32(&qd_full[slot]);
          mbar_expect_tx(fb, 2 * TILE);
          const uint32_t dst = sb + KvSmem::QD + slot * 2 * TILE;
          tma_load_4d(dst, &tmQ, fb, 0, it.h, (q_first + j) * BT, it.b);
          tma_load_4d(dst + TILE, &tmDO, fb, 0, it.h, (q_first + j) * BT, it.b);
          ++nqd;
          if (++slot == 2) { slot = 0; ph ^= 1; }
        }
      }
      if (!ok) give_up();
      bool drained = true;
      if (nkv > 0) drained &= mbar_wait(smem_u32(kv_full), (nkv - 1) & 1);
      for (int n = 0; n < (nqd < 2 ? nqd : 2); ++n) {
        if (--slot < 0) { slot = 1; ph ^= 1; }
        drained &= mbar_wait(smem_u32(&qd_full[slot]), ph);
      }
      if (!drained) give_up();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------------- MMA issuer
      int nkv = 0;
      uint32_t g = 0;  // query tiles processed so far (ring slot, buffers and phases)
      bool ok = true;
      auto slot_addr = [&](uint32_t gg) { return sb + KvSmem::QD + uint32_t(gg & 1) * 2 * TILE; };
      auto issue_s = [&](uint32_t gg) -> bool {  // Sᵀ = K Qᵀ into buffer gg & 1
        const int b = int(gg & 1);
        const uint32_t u = gg >> 1;
        if (!mbar_wait_spin(smem_u32(&qd_full[b]), u & 1, p.wait_ns) || !mbar_wait_spin(smem_u32(&s_free[b]), (u & 1) ^ 1, p.wait_ns)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          tc_mma<false>(tbase + uint32_t(b * 128), smem_desc(sb + KvSmem::K + kk * 32, 16, 1024),
                        smem_desc(slot_addr(gg) + kk * 32, 16, 1024), IDESC_S, kk > 0 ? 1u : 0u);
        tc_commit(smem_u32(&s_full[b]));
        return true;
      };
      auto issue_dp = [&](uint32_t gg) -> bool {  // dPᵀ = V dOᵀ
        if (!mbar_wait_spin(smem_u32(dp_free), (gg & 1) ^ 1, p.wait_ns)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          tc_mma<false>(tDP, smem_desc(sb + KvSmem::V + kk * 32, 16, 1024),
                        smem_desc(slot_addr(gg) + TILE + kk * 32, 16, 1024), IDESC_S, kk > 0 ? 1u : 0u);
        tc_commit(smem_u32(dp_full));
        return true;
      };
      auto issue_dv = [&](uint32_t gg, bool first) -> bool {
        if (!mbar_wait_spin(smem_u32(p_full), gg & 1, p.wait_ns)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)  // dV += Pᵀ dO (dO tile read MN-major)
          tc_mma<false>(tDV, smem_desc(sb + KvSmem::P + (kk >> 2) * TILE + (kk & 3) * 32, 16, 1024),
                        smem_desc(slot_addr(gg) + TILE + kk * 2048, TILE, 1024), IDESC_O, (!first || kk > 0) ? 1u : 0u);
        tc_commit(smem_u32(p_free));
        return true;
      };
      auto issue_dk = [&](uint32_t gg, bool first) -> bool {
        if (!mbar_wait_spin(smem_u32(ds_full), gg & 1, p.wait_ns)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)  // dK += dSᵀ Q (Q tile read MN-major)
          tc_mma<false>(tDK, smem_desc(sb + KvSmem::DS + (kk >> 2) * TILE + (kk & 3) * 32, 16, 1024),
                        smem_desc(slot_addr(gg) + kk * 2048, TILE, 1024), IDESC_O, (!first || kk > 0) ? 1u : 0u);
        tc_commit(smem_u32(ds_free));
        tc_commit(smem_u32(&qd_empty[gg & 1]));
        return true;
      };
      #pragma unroll 1
      for (int r = 0; r * int(gridDim.x) < p.items && ok && !*abort_flag; ++r) {
        const int i = snake_item(r);
        if (i >= p.items) continue;
        const Item it = decode_kv(i, p.B, p.H, p.nq, p.causal);
        if (!mbar_wait_spin(smem_u32(kv_full), nkv & 1, p.wait_ns)) { ok = false; break; }
        ++nkv;
        tc_fence_after();
        const uint32_t g0 = g;
        if (!issue_s(g0) || !issue_dp(g0)) { ok = false; break; }
        #pragma unroll 1
        for (int j = 0; j < it.nkv; ++j) {
          // next tile's dPᵀ goes ahead of this tile's dK, so it is computed while the row warps
          // form dSᵀ (its buffer is free once they have loaded this tile's dPᵀ)
          const uint32_t gg = g0 + uint32_t(j);
          if (*abort_flag) { ok = false; break; }
          if (j + 1 < it.nkv && !issue_s(gg + 1)) { ok = false; break; }
          if (!issue_dv(gg, j == 0)) { ok = false; break; }
          if (j + 1 < it.nkv && !issue_dp(gg + 1)) { ok = false; break; }
          if (!issue_dk(gg, j == 0)) { ok = false; break; }
        }
        if (!ok) break;
        tc_commit(smem_u32(kv_empty));
        g = g0 + uint32_t(it.nkv);
      }
      if (!ok) give_up();
      // every MMA issued has completed (also after a give-up) before TMEM is released
      tc_commit(smem_u32(mma_done));
      if (!mbar_wait(smem_u32(mma_done), 0)) give_up();
    }
  } else {
    // ---------------------------------------------------------------- Pᵀ / dSᵀ rows, epilogue
    const int qw = warp & 3;
    const int half = (warp - 2) >> 2;  // this warp's 64 query columns: [64·half, 64·half + 64)
    const int col0 = 64 * half;
    const int rr = qw * 32 + lane;     // key row within the tile
    const uint32_t lane_off = uint32_t(qw * 32) << 16;
    const uint32_t stage = sb + KvSmem::STAGE + uint32_t(qw) * 8192;
    uint32_t g = 0;
    #pragma unroll 1
    for (int r = 0; r * int(gridDim.x) < p.items; ++r) {
      const int i = snake_item(r);
      if (i >= p.items) continue;
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const Item it = decode_kv(i, p.B, p.H, p.nq, p.causal);
      const int q_first = p.causal ? it.qt : 0;
      const int64_t bh = int64_t(it.b) * p.H + it.h;
      // this thread's entry of a query tile's lse·log2 e (half 0) or D (half 1), read one tile ahead
      auto vec_entry = [&](int jj) -> float {
        const int q = (q_first + jj) * BT + rr;
        if (half == 0) return q < p.S ? p.lse[bh * p.S + q] * kLog2e : INFINITY;
        return q < p.S ? p.D[bh * p.S + q] : 0.f;
      };
      float vnext = vec_entry(0);
      bool ok = true;
      #pragma unroll 1
      for (int j = 0; j < it.nkv; ++j, ++g) {
        const int b = int(g & 1);
        const uint32_t u = g >> 1;
        // this query tile's lse·log2 e and D, shared by the row warps through slot g & 1 (a
        // thread refills a slot only after every thread has arrived for the tile in between,
        // i.e. has finished reading it)
        float* lv = vec + b * 256;
        lv[half * 128 + rr] = vnext;
        if (j + 1 < it.nkv) vnext = vec_entry(j + 1);
        mbar_arrive(smem_u32(&vec_full[b]));
        if (!warp_wait(smem_u32(&vec_full[b]), u & 1, p.wait_ns)) { ok = false; break; }
        if (!warp_wait(smem_u32(&s_full[b]), u & 1, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        uint32_t r[64];  // this warp's 64 columns of the row
#pragma unroll
        for (int c = 0; c < 2; ++c)
          tmem_ld32(tbase + lane_off + uint32_t(b * 128 + col0 + c * 32), *reinterpret_cast<uint32_t(*)[32]>(r + 32 * c));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s_free[b]));
        // Pᵀ[key rr][query col0 + c]; the diagonal tile hides queries before this key
        const int first = ((p.causal && q_first + j == it.qt) ? rr : 0) - col0;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float e = ex2(fmaf(__uint_as_float(r[c]), p.sc, -lv[col0 + c]));
          r[c] = __float_as_uint(c < first ? 0.f : e);
        }
        keep_before(r);
        if (!warp_wait(smem_u32(p_free), (g & 1) ^ 1, p.wait_ns)) { ok = false; break; }
#pragma unroll
        for (int un = 0; un < 8; ++un) {
          const int c0 = un * 8;
          st_shared_v4(swz(sb + KvSmem::P, rr, half, un),
                       pack_bf16(__uint_as_float(r[c0]), __uint_as_float(r[c0 + 1])),
                       pack_bf16(__uint_as_float(r[c0 + 2]), __uint_as_float(r[c0 + 3])),
                       pack_bf16(__uint_as_float(r[c0 + 4]), __uint_as_float(r[c0 + 5])),
                       pack_bf16(__uint_as_float(r[c0 + 6]), __uint_as_float(r[c0 + 7])));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(p_full));
        // dSᵀ = Pᵀ ∘ (dPᵀ − D), 32 query columns at a time
        if (!warp_wait(smem_u32(dp_full), g & 1, p.wait_ns) || !warp_wait(smem_u32(ds_free), (g & 1) ^ 1, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        uint32_t d[64];  // both dPᵀ chunks in flight before one wait
        tmem_ld32(tDP + lane_off + uint32_t(col0), *reinterpret_cast<uint32_t(*)[32]>(d));
        tmem_ld32(tDP + lane_off + uint32_t(col0 + 32), *reinterpret_cast<uint32_t(*)[32]>(d + 32));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(dp_free));
#pragma unroll
        for (int un = 0; un < 8; ++un) {
          float ds[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const int cc = un * 8 + t;
            ds[t] = __uint_as_float(r[cc]) * (__uint_as_float(d[cc]) - lv[128 + col0 + cc]);
          }
          st_shared_v4(swz(sb + KvSmem::DS, rr, half, un), pack_bf16(ds[0], ds[1]), pack_bf16(ds[2], ds[3]),
                       pack_bf16(ds[4], ds[5]), pack_bf16(ds[6], ds[7]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(ds_full));
      }
      if (!ok) {
        if (lane == 0) give_up();
        break;
      }
      // ---- epilogue: dV, α·dK once the last tile's MMAs are done (one warp per quadrant; the
      // other half's next arrival on p_full comes after this, so the next item's first dV / dK
      // MMAs cannot overwrite the accumulators before they are read)
      if (half != 0) continue;
      if (!warp_wait(smem_u32(ds_free), (g - 1) & 1, p.wait_ns)) {
        if (lane == 0) give_up();
        break;
      }
      tc_fence_after();
      if (lane == 0) bulk_wait_read_0();
      __syncwarp();
      const int y = it.qt * BT + qw * 32;
      store_rows(tDV + lane_off, 1.f, stage, lane, &tmDV, it.h, y, it.b);
      store_rows(tDK + lane_off, p.alpha, stage + 4096, lane, &tmDK, it.h, y, it.b);
      tc_fence_before();
    }
    if (lane == 0) bulk_wait_all();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, TCOLS);
  }
}

// dQ with two streams per CTA: one 128-query tile per work item, its key tiles split between the
// streams (stream 0 the even ones, stream 1 the odd ones).  Each stream has an MMA issuer (warps
// 1 / 2), four row warps (4–7 / 8–11: one query row per thread, all 128 key columns), a TMEM
// buffer that holds S and then dP of its current key tile, a dQ accumulator, and a dS tile in
// shared memory; the Q / dO tiles and a three-slot K / V ring (tiles in key order, filled by
// warp 0) are shared.  Per key tile: S = Q Kᵀ; the rows load S and form P = 2^(S·sc − lse2)
// (masked), in registers; dP = dO Vᵀ into the same buffer; the rows form dS = P ∘ (dP − D), 32
// columns at a time, into the stream's dS tile; dQ_s += dS K.  One stream's MMA round trips
// overlap the other's row work.  At the end of an item stream 0's rows add the two accumulators
// (in stream order, so the sum does not depend on timing), scale by α and store dQ.
constexpr int kThreadsQ2 = 384;
constexpr int Q2_RING = 3;
constexpr uint32_t kQ2RegsCtl = 72, kQ2RegsRows = 216;  // 128·72 + 256·216 = 384·168
struct Q2Smem {
  static constexpr int Q = 0;
  static constexpr int DO = Q + TILE;
  static constexpr int KV = DO + TILE;               // Q2_RING slots × (K tile, V tile)
  static constexpr int DS = KV + Q2_RING * 2 * TILE;  // 2 streams × dS [queries × keys]
  static constexpr int BARS = DS + 2 * PT;
  static constexpr int BYTES = 1024 + BARS + 512;
};

__global__ void __launch_bounds__(kThreadsQ2, 1)
    attn_bwd_q_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                      const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  pdl_begin();
  constexpr uint32_t IDESC_S = instr_desc_bf16(128, 128, false, false);
  constexpr uint32_t IDESC_O = instr_desc_bf16(128, HD, false, true);
  constexpr uint32_t TCOLS = 512;  // stream s: S / dP [256 s, 256 s + 128), dQ [256 s + 128, 256 s + 192)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  // q_full, q_empty, kv_full[3], kv_empty[3], per stream s (8 + 8 s): s_full, s_read, dp_full,
  // ds_full, ds_free, acc_full, mma_done; acc_free
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Q2Smem::BARS);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* kv_full = bars + 2;
  uint64_t* kv_empty = bars + 5;
  uint64_t* acc_free = bars + 24;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 26);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    mbar_init(smem_u32(q_empty), 2);  // one arrival per stream
    for (int s = 0; s < Q2_RING; ++s) {
      mbar_init(smem_u32(&kv_full[s]), 1);
      mbar_init(smem_u32(&kv_empty[s]), 1);
    }
    for (int st = 0; st < 2; ++st) {
      uint64_t* b = bars + 8 + 8 * st;
      mbar_init(smem_u32(&b[0]), 1);  // s_full
      mbar_init(smem_u32(&b[1]), 4);  // s_read
      mbar_init(smem_u32(&b[2]), 1);  // dp_full
      mbar_init(smem_u32(&b[3]), 4);  // ds_full
      mbar_init(smem_u32(&b[4]), 1);  // ds_free
      mbar_init(smem_u32(&b[5]), 1);  // acc_full
      mbar_init(smem_u32(&b[6]), 1);  // mma_done
    }
    mbar_init(smem_u32(acc_free), 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmDO);
    prefetch_tmap(&tmDQ);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  auto give_up = [&]() {
    *abort_flag = 1;
    flag_error(p.flag, XT_DEVERR_TIMEOUT);
  };
  const int wg = warp >> 2;
  if (wg == 0) {
    regs_dec<kQ2RegsCtl>();
    if (warp == 0 && lane == 0) {
      // -------------------------------------------------------------- TMA producer
      int nqi = 0;
      uint32_t gt = 0;  // K / V tiles loaded so far
      bool ok = true;
      #pragma unroll 1
      for (int r = 0; r * int(gridDim.x) < p.items && ok && !*abort_flag; ++r) {
        const int i = snake_item(r);
        if (i >= p.items) continue;
        const Item it = decode(i, p.B, p.H, p.nq, p.causal);
        if (!mbar_wait(smem_u32(q_empty), (nqi & 1) ^ 1, p.wait_ns)) { ok = false; break; }
        mbar_expect_tx(smem_u32(q_full), 2 * TILE);
        tma_load_4d(sb + Q2Smem::Q, &tmQ, smem_u32(q_full), 0, it.h, it.qt * BT, it.b);
        tma_load_4d(sb + Q2Smem::DO, &tmDO, smem_u32(q_full), 0, it.h, it.qt * BT, it.b);
        ++nqi;
        #pragma unroll 1
        for (int j = 0; j < it.nkv; ++j, ++gt) {
          const int slot = int(gt % Q2_RING);
          if (*abort_flag || !mbar_wait(smem_u32(&kv_empty[slot]), ((gt / Q2_RING) & 1) ^ 1, p.wait_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&kv_full[slot]);
          mbar_expect_tx(fb, 2 * TILE);
          const uint32_t dst = sb + Q2Smem::KV + uint32_t(slot) * 2 * TILE;
          tma_load_4d(dst, &tmK, fb, 0, it.h, j * BT, it.b);
          tma_load_4d(dst + TILE, &tmV, fb, 0, it.h, j * BT, it.b);
        }
      }
      if (!ok) give_up();
      // bounded wait for the fills that may still be in flight
      bool drained = true;
      if (nqi > 0) drained &= mbar_wait(smem_u32(q_full), (nqi - 1) & 1);
      for (uint32_t n = 0; n < (gt < Q2_RING ? gt : uint32_t(Q2_RING)); ++n) {
        const uint32_t g = gt - 1 - n;
        drained &= mbar_wait(smem_u32(&kv_full[g % Q2_RING]), (g / Q2_RING) & 1);
      }
      if (!drained) give_up();
    } else if ((warp == 1 || warp == 2) && lane == 0) {
      // -------------------------------------------------------------- MMA issuer, stream warp − 1
      const int st = warp - 1;
      uint64_t* b = bars + 8 + 8 * st;
      const uint32_t tS = tbase + uint32_t(256 * st), tDQ = tS + 128;
      const uint32_t dsb = sb + Q2Smem::DS + uint32_t(st) * PT;
      uint32_t t = 0, gt0 = 0;  // this stream's tiles so far; K / V tiles of the items before this one
      int k = 0;                // items so far
      bool ok = true;
      #pragma unroll 1
      for (int r = 0; r * int(gridDim.x) < p.items && ok && !*abort_flag; ++r) {
        const int i = snake_item(r);
        if (i >= p.items) continue;
        const Item it = decode(i, p.B, p.H, p.nq, p.causal);
        if (!mbar_wait_spin(smem_u32(q_full), k & 1, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        bool first = true;
        #pragma unroll 1
        for (int j = st; j < it.nkv; j += 2, ++t) {
          const uint32_t gt = gt0 + uint32_t(j);
          const int slot = int(gt % Q2_RING);
          const uint32_t kvs = sb + Q2Smem::KV + uint32_t(slot) * 2 * TILE;
          if (*abort_flag || !mbar_wait_spin(smem_u32(&kv_full[slot]), (gt / Q2_RING) & 1, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk)  // S = Q Kᵀ
            tc_mma<false>(tS, smem_desc(sb + Q2Smem::Q + kk * 32, 16, 1024), smem_desc(kvs + kk * 32, 16, 1024),
                          IDESC_S, kk > 0 ? 1u : 0u);
          tc_commit(smem_u32(&b[0]));
          if (!mbar_wait_spin(smem_u32(&b[1]), t & 1, p.wait_ns)) { ok = false; break; }  // the rows have loaded S
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk)  // dP = dO Vᵀ into the same columns
            tc_mma<false>(tS, smem_desc(sb + Q2Smem::DO + kk * 32, 16, 1024),
                          smem_desc(kvs + TILE + kk * 32, 16, 1024), IDESC_S, kk > 0 ? 1u : 0u);
          tc_commit(smem_u32(&b[2]));
          if (!mbar_wait_spin(smem_u32(&b[3]), t & 1, p.wait_ns)) { ok = false; break; }  // dS written, dP read
          if (first && !mbar_wait_spin(smem_u32(acc_free), (k & 1) ^ 1, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BT / 16; ++kk)  // dQ_s += dS K (K tile read MN-major)
            tc_mma<false>(tDQ, smem_desc(dsb + (kk >> 2) * TILE + (kk & 3) * 32, 16, 1024),
                          smem_desc(kvs + kk * 2048, TILE, 1024), IDESC_O, (!first || kk > 0) ? 1u : 0u);
          tc_commit(smem_u32(&b[4]));
          tc_commit(smem_u32(&kv_empty[slot]));
          first = false;
        }
        if (!ok) break;
        // this stream is done with the item: its accumulator is final, Q and dO are free to it
        if (!first) {
          tc_commit(smem_u32(&b[5]));
          tc_commit(smem_u32(q_empty));
        } else {
          mbar_arrive(smem_u32(&b[5]));
          mbar_arrive(smem_u32(q_empty));
        }
        gt0 += uint32_t(it.nkv);
        ++k;
      }
      if (!ok) give_up();
      // every MMA issued has completed (also after a give-up) before TMEM is released
      tc_commit(smem_u32(&b[6]));
      if (!mbar_wait(smem_u32(&b[6]), 0)) give_up();
    }
  } else {
    regs_inc<kQ2RegsRows>();
    // ---------------------------------------------------------------- P / dS rows, epilogue
    const int st = wg - 1;
    uint64_t* b = bars + 8 + 8 * st;
    const uint32_t tS = tbase + uint32_t(256 * st);
    const uint32_t dsb = sb + Q2Smem::DS + uint32_t(st) * PT;
    const int qw = warp & 3;
    const int rr = qw * 32 + lane;  // query row within the tile
    const uint32_t lane_off = uint32_t(qw * 32) << 16;
    // stream 0 stages α·dQ in its warp's own 32 rows of its dS tile (chunk 0)
    const uint32_t stage = sb + Q2Smem::DS + uint32_t(qw) * 4096;
    uint32_t t = 0;
    int k = 0;
    #pragma unroll 1
    for (int r = 0; r * int(gridDim.x) < p.items; ++r) {
      const int i = snake_item(r);
      if (i >= p.items) continue;
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const Item it = decode(i, p.B, p.H, p.nq, p.causal);
      const int row = it.qt * BT + rr;
      const int64_t bh = int64_t(it.b) * p.H + it.h;
      const float lse2 = row < p.S ? p.lse[bh * p.S + row] * kLog2e : INFINITY;
      const float Dr = row < p.S ? p.D[bh * p.S + row] : 0.f;
      bool ok = true;
      #pragma unroll 1
      for (int j = st; j < it.nkv; j += 2, ++t) {
        if (!warp_wait(smem_u32(&b[0]), t & 1, p.wait_ns)) { ok = false; break; }
        tc_fence_after();
        uint32_t pr[128];  // S, then P, of this row's 128 keys
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tS + lane_off + uint32_t(c * 32), *reinterpret_cast<uint32_t(*)[32]>(pr + 32 * c));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&b[1]));
        const int lim = (p.causal ? min(row + 1, p.S) : p.S) - j * BT;  // keys at or past lim are masked
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const float e = ex2(fmaf(__uint_as_float(pr[c]), p.sc, -lse2));
          pr[c] = __float_as_uint(c < lim ? e : 0.f);
        }
        keep_before(pr);
        if (!warp_wait(smem_u32(&b[2]), t & 1, p.wait_ns) || !warp_wait(smem_u32(&b[4]), (t & 1) ^ 1, p.wait_ns)) {
          ok = false;
          break;
        }
        if (st == 0 && j == 0) {  // the previous item's dQ stores have read this warp's rows of the tile
          if (lane == 0) bulk_wait_read_0();
          __syncwarp();
        }
        tc_fence_after();
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {  // dS = P ∘ (dP − D), 32 keys at a time
          uint32_t d[32];
          tmem_ld32(tS + lane_off + uint32_t(c4 * 32), d);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float ds[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int cc = c4 * 32 + u * 8 + e;
              ds[e] = __uint_as_float(pr[cc]) * (__uint_as_float(d[u * 8 + e]) - Dr);
            }
            st_shared_v4(swz(dsb, rr, c4 >> 1, (c4 & 1) * 4 + u), pack_bf16(ds[0], ds[1]), pack_bf16(ds[2], ds[3]),
                         pack_bf16(ds[4], ds[5]), pack_bf16(ds[6], ds[7]));
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&b[3]));
      }
      if (!ok) {
        if (lane == 0) give_up();
        break;
      }
      if (st == 0) {
        // ---- epilogue: α·(dQ_0 + dQ_1) once both streams are done with the item
        uint64_t* b1 = bars + 16;
        if (!warp_wait(smem_u32(&b[5]), k & 1, p.wait_ns) || !warp_wait(smem_u32(&b1[5]), k & 1, p.wait_ns)) {
          if (lane == 0) give_up();
          break;
        }
        tc_fence_after();
        uint32_t o[64];
        tmem_ld32(tbase + 128 + lane_off, *reinterpret_cast<uint32_t(*)[32]>(o));
        tmem_ld32(tbase + 160 + lane_off, *reinterpret_cast<uint32_t(*)[32]>(o + 32));
        tmem_ld_wait();
        if (it.nkv > 1) {  // stream 1 holds the odd key tiles' sum
          uint32_t o1[32];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            tmem_ld32(tbase + 256 + 128 + uint32_t(c * 32) + lane_off, o1);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[c * 32 + e] = __float_as_uint(__uint_as_float(o[c * 32 + e]) + __uint_as_float(o1[e]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(acc_free));
#pragma unroll
        for (int un = 0; un < 8; ++un)
          st_shared_v4(stage + uint32_t(lane) * 128 + (uint32_t(un ^ (lane & 7)) << 4),
                       pack_bf16(__uint_as_float(o[8 * un]) * p.alpha, __uint_as_float(o[8 * un + 1]) * p.alpha),
                       pack_bf16(__uint_as_float(o[8 * un + 2]) * p.alpha, __uint_as_float(o[8 * un + 3]) * p.alpha),
                       pack_bf16(__uint_as_float(o[8 * un + 4]) * p.alpha, __uint_as_float(o[8 * un + 5]) * p.alpha),
                       pack_bf16(__uint_as_float(o[8 * un + 6]) * p.alpha, __uint_as_float(o[8 * un + 7]) * p.alpha));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_4d(&tmDQ, stage, 0, it.h, it.qt * BT + qw * 32, it.b);
          bulk_commit();
        }
      }
      ++k;
    }
    if (lane == 0) bulk_wait_all();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, TCOLS);
  }
}

// ------------------------------------------------------------------------------ host side

// [B, S, H, hd] view of a row-major [B·S, ld] matrix whose head h occupies columns h·hd..:
// dims (innermost first) hd, H, S, B; box 64 × 1 × rows × 1, 128-byte swizzle.
static int head_map(CUtensorMap* tm, const void* base, int64_t ld, int B, int S, int H, int rows) {
  auto enc = encode_fn();
  if (!enc) return fail(XT_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[4] = {cuuint64_t(HD), cuuint64_t(H), cuuint64_t(S), cuuint64_t(B)};
  cuuint64_t strides[3] = {cuuint64_t(HD * 2), cuuint64_t(ld * 2), cuuint64_t(int64_t(S) * ld * 2)};
  cuuint32_t box[4] = {HD, 1, cuuint32_t(rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(XT_ERR_CUDA, "attention: cuTensorMapEncodeTiled failed (%d)", int(r));
  return XT_OK;
}

static int check_common(const char* fn, int B, int S, int H, int hd, int causal, int dt, int64_t ld_in,
                        int64_t ld_out, std::initializer_list<const void*> ptrs) {
  XT_REQUIRE(B >= 0 && S >= 0 && H >= 0, "%s: negative size", fn);
  XT_REQUIRE(causal == 0 || causal == 1, "%s: causal must be 0 or 1", fn);
  if (dt != XT_BF16) return fail(XT_ERR_UNSUPPORTED, "%s: only bf16 is supported", fn);
  if (hd != HD) return fail(XT_ERR_UNSUPPORTED, "%s: head_dim must be %d", fn, HD);
  XT_REQUIRE(ld_in >= int64_t(H) * hd && ld_out >= int64_t(H) * hd, "%s: row stride smaller than H·hd", fn);
  if ((ld_in % 8) || (ld_out % 8)) return fail(XT_ERR_ALIGNMENT, "%s: row strides must be multiples of 8", fn);
  for (const void* q : ptrs) {
    if (B * S * H == 0) break;
    XT_REQUIRE(q != nullptr, "%s: NULL pointer", fn);
    if (!aligned16(q)) return fail(XT_ERR_ALIGNMENT, "%s: pointers must be 16-byte aligned", fn);
  }
  return XT_OK;
}

// Raises a kernel's dynamic shared-memory limit once (`done` is the call site's flag).
static int set_smem(const void* k, int bytes, bool& done, const char* what) {
  if (done) return XT_OK;
  const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return fail(XT_ERR_CUDA, "%s: shared memory attribute: %s", what, cudaGetErrorString(e));
  done = true;
  return XT_OK;
}

}  // namespace attn
}  // namespace xt

using namespace xt;
using namespace xt::attn;

extern "C" {

int xt_attention_fwd(const void* q, const void* k, const void* v, int64_t ld_qkv, void* o, void* o_lo, int64_t ld_o,
                     float* lse, int B, int S, int H, int hd, int causal, int dt, void* stream) {
  XT_TRY(check_common("xt_attention_fwd", B, S, H, hd, causal, dt, ld_qkv, ld_o, {q, k, v, o, lse}));
  if (o_lo && !aligned16(o_lo)) return fail(XT_ERR_ALIGNMENT, "xt_attention_fwd: o_lo must be 16-byte aligned");
  if (int64_t(B) * S * H == 0) return XT_OK;
  CUtensorMap tq, tk, tv, to, tolo;
  XT_TRY(head_map(&tq, q, ld_qkv, B, S, H, BT));
  XT_TRY(head_map(&tk, k, ld_qkv, B, S, H, BT));
  XT_TRY(head_map(&tv, v, ld_qkv, B, S, H, BT));
  XT_TRY(head_map(&to, o, ld_o, B, S, H, 32));
  XT_TRY(head_map(&tolo, o_lo ? o_lo : o, ld_o, B, S, H, 32));
  FwdParams p{};
  p.B = B;
  p.H = H;
  p.S = S;
  p.nq = int(ceil_div(S, BT));
  p.items = B * H * p.nq;
  p.causal = causal;
  p.sc = float(1.0 / std::sqrt(double(hd)) * 1.4426950408889634);
  p.lse = lse;
  p.o_lo = o_lo != nullptr;
  p.flag = errflag();
  p.wait_ns = wait_limit_ns();
  static bool smem_set = false;
  static int regs = -1;
  XT_TRY(set_smem(reinterpret_cast<const void*>(attn_fwd_kernel), FwdSmem::BYTES, smem_set, "xt_attention_fwd"));
  if (regs < 0) {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, attn_fwd_kernel) != cudaSuccess)
      return fail(XT_ERR_CUDA, "xt_attention_fwd: cudaFuncGetAttributes failed");
    regs = fa.numRegs;
  }
  // the warp groups' register split (kFwdRegsCtl + 2 × kFwdRegsRows per 128 threads) adds up to
  // the 168 per thread the kernel is launched with; any other count could never be met
  if (regs != 168)
    return fail(XT_ERR_UNSUPPORTED, "xt_attention_fwd: forward kernel built with %d registers, not 168", regs);
  const int pairs = (p.items + 1) / 2;  // two query-tile streams per CTA
  const int grid = pairs < num_sms() ? pairs : num_sms();
  launch(attn_fwd_kernel, grid, kThreadsFwd, FwdSmem::BYTES, as_stream(stream), tq, tk, tv, to, tolo, p);
  return check_launch("xt_attention_fwd");
}

int xt_attention_bwd_workspace_size(int B, int S, int H, size_t* bytes) {
  XT_REQUIRE(B >= 0 && S >= 0 && H >= 0 && bytes, "xt_attention_bwd_workspace_size: bad arguments");
  *bytes = (size_t(B) * size_t(S) * size_t(H) * 4 + 255) & ~size_t(255);
  return XT_OK;
}

int xt_attention_bwd(const void* q, const void* k, const void* v, int64_t ld_qkv, const void* o, const void* o_lo,
                     const void* d_o, int64_t ld_o, const float* lse, void* dq, void* dk, void* dv, int64_t ld_dqkv,
                     void* ws, size_t ws_bytes, int B, int S, int H, int hd, int causal, int dt, void* stream) {
  XT_TRY(check_common("xt_attention_bwd", B, S, H, hd, causal, dt, ld_qkv, ld_o,
                      {q, k, v, o, d_o, lse, dq, dk, dv, ws}));
  XT_REQUIRE(ld_dqkv >= int64_t(H) * hd, "xt_attention_bwd: ld_dqkv smaller than H·hd");
  if (ld_dqkv % 8) return fail(XT_ERR_ALIGNMENT, "xt_attention_bwd: ld_dqkv must be a multiple of 8");
  if (int64_t(B) * S * H == 0) return XT_OK;
  size_t need = 0;
  xt_attention_bwd_workspace_size(B, S, H, &need);
  XT_REQUIRE(ws_bytes >= need, "xt_attention_bwd: workspace too small (%zu < %zu)", ws_bytes, need);
  cudaStream_t s = as_stream(stream);
  float* D = static_cast<float*>(ws);
  {
    const int64_t threads = int64_t(B) * S * H * 8;
    int64_t blocks = ceil_div(threads, 256);
    const int64_t cap = int64_t(num_sms()) * 32;  // one (t, h) row per 8 threads up to 1.2 M rows
    if (blocks > cap) blocks = cap;
    if (o_lo && !aligned16(o_lo)) return fail(XT_ERR_ALIGNMENT, "xt_attention_bwd: o_lo must be 16-byte aligned");
    launch(attn_delta_kernel, int(blocks), 256, 0, s, static_cast<const bf16*>(o), static_cast<const bf16*>(o_lo),
                                                   static_cast<const bf16*>(d_o), ld_o, B, S, H, D);
    XT_TRY(check_launch("xt_attention_bwd (delta)"));
  }
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
  XT_TRY(head_map(&tq, q, ld_qkv, B, S, H, BT));
  XT_TRY(head_map(&tk, k, ld_qkv, B, S, H, BT));
  XT_TRY(head_map(&tv, v, ld_qkv, B, S, H, BT));
  XT_TRY(head_map(&tdo, d_o, ld_o, B, S, H, BT));
  XT_TRY(head_map(&tdq, dq, ld_dqkv, B, S, H, 32));
  XT_TRY(head_map(&tdk, dk, ld_dqkv, B, S, H, 32));
  XT_TRY(head_map(&tdv, dv, ld_dqkv, B, S, H, 32));
  BwdParams p{};
  p.B = B;
  p.H = H;
  p.S = S;
  p.nq = int(ceil_div(S, BT));
  p.items = B * H * p.nq;
  p.causal = causal;
  p.alpha = float(1.0 / std::sqrt(double(hd)));
  p.sc = float(1.0 / std::sqrt(double(hd)) * 1.4426950408889634);
  p.lse = lse;
  p.D = D;
  p.flag = errflag();
  p.wait_ns = wait_limit_ns();
  const int grid = p.items < num_sms() ? p.items : num_sms();
  static bool kv_set = false, q_set = false;
  XT_TRY(set_smem(reinterpret_cast<const void*>(attn_bwd_kv_kernel), KvSmem::BYTES, kv_set, "xt_attention_bwd"));
  XT_TRY(set_smem(reinterpret_cast<const void*>(attn_bwd_q_kernel), Q2Smem::BYTES, q_set, "xt_attention_bwd"));
  static int q_regs = -1;
  if (q_regs < 0) {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, attn_bwd_q_kernel) != cudaSuccess)
      return fail(XT_ERR_CUDA, "xt_attention_bwd: cudaFuncGetAttributes failed");
    q_regs = fa.numRegs;
  }
  // the dQ kernel's register split (kQ2RegsCtl + 2 × kQ2RegsRows per 128 threads) adds up to the
  // 168 per thread it is launched with
  if (q_regs != 168)
    return fail(XT_ERR_UNSUPPORTED, "xt_attention_bwd: dQ kernel built with %d registers, not 168", q_regs);
  launch(attn_bwd_kv_kernel, grid, kThreadsBwd, KvSmem::BYTES, s, tq, tk, tv, tdo, tdk, tdv, p);
  XT_TRY(check_launch("xt_attention_bwd (dK, dV)"));
  launch(attn_bwd_q_kernel, grid, kThreadsQ2, Q2Smem::BYTES, s, tq, tk, tv, tdo, tdq, p);
  return check_launch("xt_attention_bwd (dQ)");
}

}  // extern "C"
