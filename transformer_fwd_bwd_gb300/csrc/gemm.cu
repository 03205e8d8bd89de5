// Host side of the tensor-core GEMM: TMA tensor maps, tile-shape choice, launch, and the
// matmul C ABI ([AE] op table row matmul: C = A@B; dA = d@Bᵀ, dB = Aᵀ@d).
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "gemm.cuh"
#include "internal.cuh"

namespace xt {
namespace gemm {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Operand as the kernel sees it: `mn` rows (M or N) by K, either K contiguous (K-major) or
// MN contiguous (MN-major), with two batch levels.
int make_operand_map(CUtensorMap* tm, const Operand& o, int kind, int box_mn, int k_atom_count) {
  auto enc = encode_fn();
  if (!enc) return fail(XT_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const int64_t e = kind == kTf32 ? 4 : kind == kFp8 ? 1 : 2;
  const uint32_t atom = uint32_t(128 / e);
  cuuint64_t dims[4];
  cuuint64_t strides[3];
  cuuint32_t box[4];
  cuuint32_t estr[4] = {1, 1, 1, 1};
  if (!o.mn_major) {
    dims[0] = cuuint64_t(o.K);
    dims[1] = cuuint64_t(o.mn);
    box[0] = atom;
    box[1] = uint32_t(box_mn);
  } else {
    dims[0] = cuuint64_t(o.mn);
    dims[1] = cuuint64_t(o.K);
    box[0] = atom;
    box[1] = atom * uint32_t(k_atom_count);  // BK rows of K
  }
  dims[2] = cuuint64_t(o.batch_inner);
  dims[3] = cuuint64_t(o.batch_outer);
  box[2] = 1;
  box[3] = 1;
  const int64_t row_bytes = o.ld * e;
  strides[0] = cuuint64_t(row_bytes);
  strides[1] = cuuint64_t(o.batch_inner > 1 ? o.s_inner * e : row_bytes);
  strides[2] = cuuint64_t(o.batch_outer > 1 ? o.s_outer * e : row_bytes);
  const CUtensorMapDataType dt = kind == kTf32  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : kind == kFp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(tm, dt, 4, const_cast<void*>(o.ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(XT_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return XT_OK;
}

// Tile width, K split and schedule from a per-tile time model: rounds of persistent CTAs × the
// time of one tile at the SM's share of the tensor peak, scaled by the measured relative
// efficiency of the tile width (narrow tiles move more operand bytes per FLOP), plus for a K
// split the fixed-order reduction of the partial slices by a second kernel.  Two stream-K
// forms (in-kernel fixup, one partial tile written and read per shared tile piece):
//   - over every SM: each CTA an equal share of the k-block iterations, so no SM idles in a
//     last round; the CTAs sit at staggered K offsets, so only when the operands stay
//     resident in L2 (≤ 80 MB);
//   - lockstep K slices: tiles × s CTAs (≤ the SMs), each one K slice of one tile, every CTA
//     at the same K offsets as the others of its slice (operand tiles shared through L2 as
//     by whole tiles).
// Splits and stream-K need a workspace and a non-causal problem; the K split one batch.
//
// The constants were fitted to CUDA-graph timings of the 12-layer stack's fifteen GEMM shapes
// under every (kernel, tile width, schedule) combination on a GB300: the model's pick is then
// within 0.6 µs of the fastest measured one on each shape.  The paired kernel's factors were
// raised once it staged two K atoms per stage (8192 × 2304 × 768 in whole 256-wide tiles and
// 8192 × 768 × 2304 in whole 192-wide tiles, graph-timed, give ≈ 1.15 and ≈ 1.0).
static double tile_eff(int bn) { return bn >= 256 ? 1.0 : bn >= 192 ? 0.95 : bn >= 128 ? 0.64 : 0.35; }
// The same for the paired kernel's 256-row tiles (relative to the single-CTA BN 256 rate):
// each CTA stages 128 rows of A and bn / 2 rows of B per k-block, 2/3 of the single kernel's
// bytes per FLOP at bn 256, with six pipeline stages instead of four.
static double pair_eff(int bn) { return bn >= 256 ? 1.15 : bn >= 192 ? 1.0 : 0.75; }

// Schedule override (xt_gemm_set_schedule): 0 the model's choice, 1 whole tiles only, 2 a K
// split where one is allowed, 3 stream-K over every SM where allowed, 4 stream-K in lockstep
// K slices where allowed.
static int g_schedule = 0;
// Paired-kernel override (xt_gemm_set_pairing): 0 the model's choice, 1 never, 2 wherever allowed,
// 3 the multicast form of the paired kernel wherever allowed (else as 2).
static int g_pairing = 0;
// Tile-width override (xt_gemm_set_tile): 0 the model's choice, else that BN wherever it is a
// candidate.
static int g_tile = 0;

// Fixup time of a stream-K tile shared by `parts` CTAs: one latency plus one pass per partial.
static double sk_fixup_time(int64_t parts) { return 0.7e-6 + 1.2e-6 * double(parts - 1); }

Choice choose(bool tf32, int64_t M, int64_t N, int64_t K, int64_t batches, int causal, bool allow_split,
              bool fp8, bool b_mn) {
  const bool pair_ok = !tf32 && !fp8 && causal == 0 && g_pairing != 1;
  if (fp8) allow_split = false;  // fp8: whole tiles only
  const int mode = allow_split ? g_schedule : 1;
  if (mode == 1) allow_split = false;
  const int cands_bf16[4] = {64, 128, 192, 256};
  const int cands_tf32[2] = {64, 128};
  const int cands_fp8[2] = {128, 256};
  // paired tiles stage BN / 2 rows of B per CTA: whole 64-element swizzle atoms when B is read
  // MN-major (BN 128, 256), any multiple of 16 rows K-major (also BN 192)
  const int cands_pair[3] = {128, 192, 256};
  const int sms = num_sms();
  const int bk1 = fp8 ? 128 : tf32 ? 32 : 64;  // K elements per 128-byte atom
  const double per_sm = fp8 ? 22.4e12 : tf32 ? 5.6e12 : 11.2e12;
  const double e = fp8 ? 1.0 : tf32 ? 4.0 : 2.0;
  Choice best{fp8 ? cands_fp8[0] : tf32 ? cands_tf32[0] : cands_bf16[0], 1, 0, 0};
  double best_t = 1e300;

  // forced modes: the forced kind of candidate first, whole tiles when it is not allowed
  auto weigh = [&](double t, int kind, int cg, int mc = 1) {  // kind 1 tiles, 2 K split, 3 stream-K all units, 4 lockstep
    if (mode >= 2) t *= (kind == mode) ? 1e-6 : (kind == 1 ? 1.0 : 1e6);
    if (g_pairing >= 2 && cg == 2) t *= 1e-12;
    if (g_pairing == 3 && mc == 2) t *= 1e-12;
    return t;
  };
  auto tile_weight = [&](int bn) { return g_tile != 0 && bn != g_tile ? 1e18 : 1.0; };
  auto offer = [&](double t, Choice ch) {
    if (t < best_t * 0.999) {
      best_t = t;
      best = ch;
    }
  };
  for (int cg = 1; cg <= 2; ++cg) {
    // units: CTAs, or CTA pairs that can be resident together (stream-K waits need every unit resident)
    const int units = cg == 1 ? sms : (pair_ok ? pair_capacity() : 0);
    if (units < 1) continue;
    const int bm = BM * cg;
    const int bk = bk1 * k_atoms(cg);  // K per stage of this kernel
    const int64_t kbt = ceil_div(K, bk);
    const int* c = cg == 2 ? cands_pair : fp8 ? cands_fp8 : tf32 ? cands_tf32 : cands_bf16;
    const int nc = cg == 2 ? 3 : fp8 || tf32 ? 2 : 4;
    const double rate = per_sm * cg;  // per unit
    const bool sk_ok = allow_split && causal == 0 && units * cg <= kSkMaxCtas;
    for (int i = 0; i < nc; ++i) {
      const int bn = c[i];
      if (i > 0 && c[i - 1] >= N) break;  // wider tiles only add padding
      if (cg == 2 && bn == 192 && b_mn) continue;
      const double eff = cg == 2 ? pair_eff(bn) : tile_eff(bn);
      int64_t tiles = ceil_div(M, bm) * ceil_div(N, bn) * batches;
      if (causal == 1) tiles = (tiles + 1) / 2;
      const double t_kb = 2.0 * bm * bn * bk / (rate * eff);
      for (int s = 1; s <= 8; s *= 2) {
        if (s > 1 && (!allow_split || batches != 1 || causal != 0 || N % 4 != 0)) break;
        if (s > 1 && kbt < 4 * s) break;
        const double rounds = double(ceil_div(tiles * s, units));
        const double t_tile = 2.0 * bm * bn * (double(K) / s) / (rate * eff) + 1.5e-6;
        double t = rounds * t_tile;
        if (s > 1) t += double(s + 1) * double(M) * double(N) * 4.0 / 5e12 + 2e-6;
        Choice ch{bn, s, 0, 0};
        ch.cg = cg;
        offer(weigh(t, s > 1 ? 2 : 1, cg) * tile_weight(bn), ch);
      }
      // multicast pairs (only when forced: graph-timed against the plain pairs at BN 256 they
      // were slower on every shape of the 12-layer stack, 38.2 against 29.2 µs at 8192 × 3072 ×
      // 768 and 504 against 379 µs on the logits): whole 256-wide tiles, an even number of
      // 256-row tiles (the two pairs of a cluster take vertically adjacent ones), in clusters
      // that can be resident at once
      const int64_t num_m = ceil_div(M, bm);
      if (g_pairing == 3 && cg == 2 && bn == 256 && causal == 0 && num_m % 2 == 0 && (mode == 0 || mode == 1)) {
        const int mcu = mc_capacity();
        if (mcu > 0) {
          const double rounds = double(ceil_div(tiles / 2, mcu));
          const double t = rounds * (2.0 * bm * bn * double(K) / (rate * eff) + 1.5e-6);
          Choice ch{bn, 1, 0, 0};
          ch.cg = 2;
          ch.mc = 2;
          offer(weigh(t, 1, cg, 2) * tile_weight(bn), ch);
        }
      }
      if (!sk_ok) continue;
      const int64_t iters = tiles * kbt;
      const double operands = double(M + N) * double(batches) * double(K) * e;
      if (iters >= units && tiles % units != 0 && (operands <= 80e6 || mode == 3)) {
        const double share = double(iters) / units;
        const int64_t parts = int64_t(std::ceil(double(kbt) / share)) + 1;
        // + 3 µs: the measured cost per launch beyond the model (staggered tiles, partial
        // stores, the exposed fixup)
        const double t = std::ceil(share) * t_kb + (double(tiles) / units + 1.0) * 1.5e-6 + sk_fixup_time(parts) + 3e-6;
        Choice ch{bn, 1, 1, units * cg};
        ch.cg = cg;
        offer(weigh(t, 3, cg) * tile_weight(bn), ch);
      }
      for (int64_t sl = 2; sl <= 8 && tiles * sl <= units && kbt >= 2 * sl; ++sl) {
        const double t = double(ceil_div(kbt, sl)) * t_kb + 1.5e-6 + sk_fixup_time(sl);
        Choice ch{bn, 1, 2, int(tiles * sl) * cg};
        ch.cg = cg;
        offer(weigh(t, 4, cg) * tile_weight(bn), ch);
      }
    }
  }
  return best;
}

size_t split_bytes(const Choice& c, int64_t M, int64_t N) {
  if (c.sk) return size_t(c.grid) * BM * size_t(c.bn) * 4;
  if (c.splits <= 1) return 0;
  return (size_t(c.splits) * size_t(M) * size_t(N) * 4 + 255) & ~size_t(255);
}

// C (+)= Σ_s part[s] in split order (deterministic); part is [splits][M][N] float32.
// ts (may be null): this launch's timestamp slots, (start, end) %globaltimer per block.
template <typename TC>
__global__ void splitk_reduce(const float* __restrict__ part, int splits, int64_t M, int64_t N, TC* C, int64_t ldc,
                              int acc, unsigned long long* ts) {
  pdl_begin();
  if (ts && threadIdx.x == 0) ts[2 * blockIdx.x] = global_ns();
  const int64_t n4 = N / 4, total = M * n4, slice = M * N;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t m = i / n4, c = (i - m * n4) * 4;
    float4 a = *reinterpret_cast<const float4*>(part + m * N + c);
    for (int k = 1; k < splits; ++k) {
      const float4 b = *reinterpret_cast<const float4*>(part + k * slice + m * N + c);
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    TC* out = C + m * ldc + c;
    float v[4] = {a.x, a.y, a.z, a.w};
    if (acc)
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] += to_f(out[e]);
#pragma unroll
    for (int e = 0; e < 4; ++e) out[e] = from_f<TC>(v[e]);
  }
  if (ts) {
    __syncthreads();
    if (threadIdx.x == 0) ts[2 * blockIdx.x + 1] = global_ns();
  }
}

// An output as the epilogue's TMA stores see it: boxes of 32 rows × 128 bytes, 128-byte swizzle.
static int make_output_map(CUtensorMap* tm, void* base, bool bf16, int64_t M, int64_t N, int64_t ldc, int bi, int bo,
                           int64_t s_inner, int64_t s_outer) {
  auto enc = encode_fn();
  if (!enc) return fail(XT_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const int64_t e = bf16 ? 2 : 4;
  const int64_t row_bytes = ldc * e;
  cuuint64_t dims[4] = {cuuint64_t(N), cuuint64_t(M), cuuint64_t(bi), cuuint64_t(bo)};
  cuuint64_t strides[3] = {cuuint64_t(row_bytes), cuuint64_t(bi > 1 ? s_inner * e : row_bytes),
                           cuuint64_t(bo > 1 ? s_outer * e : row_bytes)};
  cuuint32_t box[4] = {uint32_t(128 / e), 32, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(tm, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(XT_ERR_CUDA, "cuTensorMapEncodeTiled (C) failed (%d)", int(r));
  return XT_OK;
}

int run(const Problem& pb, cudaStream_t s) {
  const bool tf32 = pb.tf32;
  const int64_t batches = int64_t(pb.batch_outer) * pb.batch_inner;
  Choice ch = choose(tf32, pb.M, pb.N, pb.K, batches, pb.causal, pb.act == 0, pb.fp8, pb.B.mn_major);
  if ((ch.splits > 1 || ch.sk) && (pb.split_ws == nullptr || split_bytes(ch, pb.M, pb.N) > pb.split_ws_bytes ||
                                   (ch.sk && pb.sk_flags == nullptr)))
    ch = choose(tf32, pb.M, pb.N, pb.K, batches, pb.causal, false, pb.fp8, pb.B.mn_major);
  if (pb.act) ch = Choice{256, 1, 0, 0};  // the GELU epilogues are built for BN 256 only
  const int bn = ch.bn;
  const int cg = ch.cg;
  const bool split = ch.splits > 1;
  CUtensorMap ta, tb, tc, tc2;
  memset(&tc2, 0, sizeof(tc2));
  if (pb.act == 1) XT_TRY(make_output_map(&tc2, pb.C2, true, pb.M, pb.N, pb.ldc, 1, 1, 0, 0));
  const int kind = pb.fp8 ? kFp8 : tf32 ? kTf32 : kBf16;
  XT_TRY(make_operand_map(&ta, pb.A, kind, BM, k_atoms(cg)));
  // a pair's CTA stages half of B's rows; a multicast pair's CTA loads half of those
  XT_TRY(make_operand_map(&tb, pb.B, kind, bn / cg / ch.mc, k_atoms(cg)));
  // TMA epilogue for every output except a bf16 C that is accumulated into (TMA reduce-add is
  // used for float32 only; bf16 accumulation keeps the direct read-modify-write stores).  A K
  // split stores float32 partial tiles into [splits][M][N] slices instead.
  const bool tma_store = split || !(pb.c_bf16 && pb.accumulate);
  memset(&tc, 0, sizeof(tc));
  if (split)
    XT_TRY(make_output_map(&tc, pb.split_ws, false, pb.M, pb.N, pb.N, ch.splits, 1, pb.M * pb.N, 0));
  else if (tma_store)
    XT_TRY(make_output_map(&tc, pb.C, pb.c_bf16, pb.M, pb.N, pb.ldc, pb.batch_inner, pb.batch_outer, pb.sc_inner,
                           pb.sc_outer));
  Params p{};
  p.M = int(pb.M);
  p.N = int(pb.N);
  p.K = int(pb.K);
  p.num_m = int(ceil_div(pb.M, int64_t(BM) * cg));
  p.num_n = int(ceil_div(pb.N, bn));
  p.batch_inner = split ? ch.splits : pb.batch_inner;
  p.batches = split ? ch.splits : pb.batch_inner * pb.batch_outer;
  p.splitk = ch.splits;
  const int bk = (pb.fp8 ? 128 : tf32 ? 32 : 64) * k_atoms(cg);
  p.kb_per_split = int(ceil_div(ceil_div(pb.K, bk), ch.splits));
  p.causal = pb.causal;
  p.accumulate = split ? 0 : pb.accumulate;
  p.c_bf16 = split ? 0 : pb.c_bf16;
  p.tma_store = tma_store ? 1 : 0;
  p.alpha = pb.alpha;
  p.C = pb.C;
  p.ldc = pb.ldc;
  p.sc_inner = pb.sc_inner;
  p.sc_outer = pb.sc_outer;
  p.act = pb.act;
  p.aux = static_cast<const bf16*>(pb.aux);
  p.ld_aux = pb.ldc;
  p.flag = errflag();
  p.wait_ns = wait_limit_ns();
  p.scale_a = pb.scale_a;
  p.scale_b = pb.scale_b;
  const int64_t tiles = int64_t(p.num_m) * p.num_n * p.batches;  // a K split counts its slices
  if (tiles > int64_t(1) << 30) return fail(XT_ERR_UNSUPPORTED, "matmul: too many tiles");
  int grid;
  if (ch.mc == 2) {
    const int units = mc_capacity();
    if (units < 1) return fail(XT_ERR_CUDA, "gemm: no cluster of two pairs can be resident");
    if (p.num_m % 2 || p.sk || p.splitk > 1) return fail(XT_ERR_INVALID_ARG, "gemm: bad multicast schedule");
    const int64_t groups = tiles / 2;
    grid = 4 * int(groups < units ? groups : units);
  } else if (cg == 2) {
    const int units = pair_capacity();
    if (units < 1) return fail(XT_ERR_CUDA, "gemm: no CTA pair can be resident");
    grid = 2 * int(tiles < units ? tiles : units);
  } else {
    grid = int(tiles < num_sms() ? tiles : num_sms());
  }
  if (grid < 1) grid = 1;
  if (ch.sk) {
    p.sk = 1;
    p.kb_tile = int(ceil_div(pb.K, bk));
    p.sk_iters = tiles * p.kb_tile;
    p.sk_part = static_cast<float*>(pb.split_ws);
    p.sk_flag = pb.sk_flags;
    grid = ch.grid;  // ≤ the resident units and ≤ the iterations: every unit resident, every share non-empty
  }
  const bool amn = pb.A.mn_major, bmn = pb.B.mn_major;
  // algorithmic FLOPs: the unmasked work only for the causal modes
  const double nb = double(batches);  // problem batches (a K split does not add work)
  double flops = 2.0 * double(pb.M) * double(pb.N) * double(pb.K) * nb;
  if (pb.causal == 1) flops = 2.0 * double(pb.K) * double(pb.M) * double(pb.M + 1) / 2.0 * nb;
  if (pb.causal >= 2) flops = 2.0 * double(pb.N) * double(pb.M) * double(pb.M + 1) / 2.0 * nb;
  void* tok = nullptr;
  // record: causal mode, or 10 × K splits, or 1000 for stream-K over every SM, 1000 + slices
  // for stream-K in lockstep K slices
  // (the tile width of a paired launch is recorded as 1000 + BN, of a multicast pair as 2000 + BN)
  const int shape[8] = {p.M, p.N, p.K, split ? ch.splits : p.batches, cg == 2 ? 1000 * ch.mc + bn : bn, int(amn), int(bmn),
                        ch.sk == 1 ? 1000 : ch.sk == 2 ? 1000 + int(ch.grid / cg / tiles) :
                        split ? 10 * ch.splits : p.causal};
  unsigned long long* ts = nullptr;
  const bool prof = gemm_profile_begin(flops, shape, &ts, &tok) && grid <= kProfGemmSlots;
  p.prof_ts = prof ? ts : nullptr;
  int rgrid = 0;
  int st = pb.fp8    ? launch_fp8(bn, ta, tb, tc, tc2, p, grid, s)
           : tf32    ? launch_tf32(bn, amn, bmn, ta, tb, tc, tc2, p, grid, s)
           : pb.act ? launch_bf16_act(pb.act, amn, bmn, ta, tb, tc, tc2, p, grid, s)
           : cg == 2 ? launch_bf16_pair(bn, ch.mc, amn, bmn, ta, tb, tc, tc2, p, grid, s)
                    : launch_bf16(bn, amn, bmn, ta, tb, tc, tc2, p, grid, s);
  if (st == XT_OK && split) {
    const int64_t work = pb.M * (pb.N / 4);
    int64_t g = ceil_div(work, 256);
    if (g > int64_t(num_sms()) * 8) g = int64_t(num_sms()) * 8;
    const float* part = static_cast<const float*>(pb.split_ws);
    unsigned long long* rts = prof && g <= kProfSlots - kProfGemmSlots ? ts + 2 * kProfGemmSlots : nullptr;
    rgrid = rts ? int(g) : 0;
    if (pb.c_bf16)
      launch(splitk_reduce<bf16>, int(g), 256, 0, s, part, ch.splits, pb.M, pb.N, static_cast<bf16*>(pb.C), pb.ldc,
                                                 pb.accumulate, rts);
    else
      launch(splitk_reduce<float>, int(g), 256, 0, s, part, ch.splits, pb.M, pb.N, static_cast<float*>(pb.C), pb.ldc,
                                                  pb.accumulate, rts);
    st = check_launch("gemm K-split reduce");
  }
  if (prof) gemm_profile_grids(tok, grid, rgrid);
  return st;
}

}  // namespace gemm

// ------------------------------------------------------------------------------ tf32 staging
// The tf32 MMA is fed K-major operands only: an fp32 operand stored MN-major (MN
// contiguous) is first copied, transposed, into K-major scratch (rows of round_up(K, 4)
// floats) by a tiled shared-memory transpose.  bf16 operands are read MN-major directly.

static int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }
static size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

static size_t stage_bytes(const gemm::Operand& o) {
  if (!o.mn_major) return 0;
  return align256(size_t(o.batch_inner) * size_t(o.batch_outer) * size_t(o.mn) * size_t(round_up(o.K, 4)) * 4);
}

__global__ void transpose_to_kmajor(const float* __restrict__ src, int64_t ld, int64_t s_inner, int64_t s_outer,
                                    int bi, int64_t mn, int64_t K, float* __restrict__ dst, int64_t ldk) {
  pdl_begin();
  __shared__ float tile[32][33];
  const int z = blockIdx.z;
  const int zo = z / bi, zi = z - zo * bi;
  const float* S = src + int64_t(zo) * s_outer + int64_t(zi) * s_inner;
  float* D = dst + int64_t(z) * mn * ldk;
  const int64_t i0 = int64_t(blockIdx.x) * 32, k0 = int64_t(blockIdx.y) * 32;
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int64_t k = k0 + r, i = i0 + threadIdx.x;
    tile[r][threadIdx.x] = (k < K && i < mn) ? S[k * ld + i] : 0.f;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += blockDim.y) {
    const int64_t i = i0 + r, k = k0 + threadIdx.x;
    if (i < mn && k < ldk) D[i * ldk + k] = tile[threadIdx.x][r];
  }
}

// Rewrites `o` (fp32, MN-major) to point at a K-major copy carved from ws.
static int stage_operand(gemm::Operand& o, char*& ws, size_t& left, cudaStream_t s) {
  const size_t need = stage_bytes(o);
  if (need > left) return fail(XT_ERR_INVALID_ARG, "matmul: workspace too small (tf32 staging)");
  const int64_t ldk = round_up(o.K, 4);
  const int batches = o.batch_inner * o.batch_outer;
  if (batches > 65535) return fail(XT_ERR_UNSUPPORTED, "matmul: too many batches for tf32 staging");
  dim3 grid(unsigned(ceil_div(o.mn, 32)), unsigned(ceil_div(ldk, 32)), unsigned(batches));
  launch(transpose_to_kmajor, grid, dim3(32, 8), 0, s, static_cast<const float*>(o.ptr), o.ld, o.s_inner, o.s_outer,
                                                    o.batch_inner, o.mn, o.K, reinterpret_cast<float*>(ws), ldk);
  XT_TRY(check_launch("matmul tf32 staging"));
  o.ptr = ws;
  o.mn_major = false;
  o.ld = ldk;
  o.s_inner = o.mn * ldk;
  o.s_outer = int64_t(o.batch_inner) * o.mn * ldk;
  ws += need;
  left -= need;
  return XT_OK;
}

static gemm::Operand operand_a(const xt_matmul_desc* d, const void* A) {
  return gemm::Operand{A, d->trans_a == 1, d->M, d->K, d->lda, d->stride_a_inner, d->stride_a_outer,
                       d->batch_inner, d->batch_outer};
}
// op(B) is K×N; the kernel's B operand is N rows by K: K-major iff B is stored [N, K].
static gemm::Operand operand_b(const xt_matmul_desc* d, const void* B) {
  return gemm::Operand{B, d->trans_b == 0, d->N, d->K, d->ldb, d->stride_b_inner, d->stride_b_outer,
                       d->batch_inner, d->batch_outer};
}

// Workspace: the stream-K flag words (zero between calls), then fp32 staging copies, then
// K-split or stream-K partial tiles.
static size_t matmul_ws(const xt_matmul_desc* d) {
  if (d->M == 0 || d->N == 0 || d->K == 0) return 0;
  size_t b = gemm::kSkFlagBytes;
  if (d->dtype_ab == XT_F32) b += stage_bytes(operand_a(d, nullptr)) + stage_bytes(operand_b(d, nullptr));
  const gemm::Choice ch = gemm::choose(d->dtype_ab == XT_F32, d->M, d->N, d->K,
                                       int64_t(d->batch_outer) * d->batch_inner, d->causal, true, false,
                                       d->trans_b == 0);
  return b + gemm::split_bytes(ch, d->M, d->N);
}

// Validates and runs C[M,N] (+)= alpha · op(A) @ op(B) for one matmul descriptor.
static int matmul_run(const xt_matmul_desc* d, const void* A, const void* B, void* C, void* ws, size_t ws_bytes,
                      cudaStream_t s, int act = 0, void* C2 = nullptr, const void* aux = nullptr) {
  XT_REQUIRE(d != nullptr, "matmul: desc is NULL");
  if (act) {
    XT_REQUIRE(d->dtype_ab == XT_BF16 && d->dtype_c == XT_BF16, "matmul gelu: bf16 operands and output only");
    XT_REQUIRE(!d->accumulate && !d->causal && d->batch_outer == 1 && d->batch_inner == 1,
               "matmul gelu: one batch, no accumulate, no causal mode");
    if (d->N % 64) return fail(XT_ERR_UNSUPPORTED, "matmul gelu: N must be a multiple of 64");
    const void* extra = act == 1 ? C2 : aux;
    XT_REQUIRE(d->M == 0 || d->N == 0 || extra != nullptr, "matmul gelu: %s is NULL", act == 1 ? "Y" : "X");
    if (extra && !aligned16(extra)) return fail(XT_ERR_ALIGNMENT, "matmul gelu: Y / X must be 16-byte aligned");
    XT_REQUIRE(d->K > 0 || d->M == 0 || d->N == 0, "matmul gelu: K must be positive");
  }
  XT_REQUIRE(d->M >= 0 && d->N >= 0 && d->K >= 0, "matmul: negative size");
  XT_REQUIRE(d->batch_outer >= 1 && d->batch_inner >= 1, "matmul: batch counts must be >= 1");
  XT_REQUIRE(valid_dtype(d->dtype_ab) && valid_dtype(d->dtype_c), "matmul: bad dtype");
  XT_REQUIRE(d->causal >= 0 && d->causal <= 3, "matmul: bad causal mode");
  XT_REQUIRE(d->trans_a == 0 || d->trans_a == 1, "matmul: trans_a must be 0 or 1");
  XT_REQUIRE(d->trans_b == 0 || d->trans_b == 1, "matmul: trans_b must be 0 or 1");
  if (d->M == 0 || d->N == 0) return XT_OK;
  XT_REQUIRE(C != nullptr, "matmul: C is NULL");
  XT_REQUIRE(d->ldc >= d->N, "matmul: ldc < N");
  const int64_t ec = int64_t(dtype_size(d->dtype_c));
  if (!aligned16(C) || (d->ldc * ec) % 16 || (d->batch_inner > 1 && (d->stride_c_inner * ec) % 16) ||
      (d->batch_outer > 1 && (d->stride_c_outer * ec) % 16))
    return fail(XT_ERR_ALIGNMENT, "matmul: C, ldc and C batch strides must be 16-byte aligned");
  if (d->K == 0) {
    if (!d->accumulate) {
      for (int zo = 0; zo < d->batch_outer; ++zo)
        for (int zi = 0; zi < d->batch_inner; ++zi) {
          char* c0 = static_cast<char*>(C) + (zo * d->stride_c_outer + zi * d->stride_c_inner) * ec;
          if (cudaMemset2DAsync(c0, size_t(d->ldc * ec), 0, size_t(d->N * ec), size_t(d->M), s) != cudaSuccess)
            return check_launch("matmul K = 0");
        }
    }
    return XT_OK;
  }
  XT_REQUIRE(A && B, "matmul: A or B is NULL");
  const int64_t e = int64_t(dtype_size(d->dtype_ab));
  XT_REQUIRE(d->lda >= (d->trans_a ? d->M : d->K), "matmul: lda too small");
  XT_REQUIRE(d->ldb >= (d->trans_b ? d->K : d->N), "matmul: ldb too small");
  if (!aligned16(A) || !aligned16(B) || (d->lda * e) % 16 || (d->ldb * e) % 16 ||
      (d->batch_inner > 1 && ((d->stride_a_inner * e) % 16 || (d->stride_b_inner * e) % 16)) ||
      (d->batch_outer > 1 && ((d->stride_a_outer * e) % 16 || (d->stride_b_outer * e) % 16)))
    return fail(XT_ERR_ALIGNMENT, "matmul: A, B, lda, ldb and A/B batch strides must be 16-byte aligned");
  if (d->causal) XT_REQUIRE(d->M == d->N || d->causal >= 2, "matmul: causal mode 1 needs a square output");
  gemm::Problem pb{};
  pb.tf32 = d->dtype_ab == XT_F32;
  pb.M = d->M;
  pb.N = d->N;
  pb.K = d->K;
  pb.batch_inner = d->batch_inner;
  pb.batch_outer = d->batch_outer;
  pb.A = operand_a(d, A);
  pb.B = operand_b(d, B);
  char* w = static_cast<char*>(ws);
  size_t left = ws ? ws_bytes : 0;
  pb.sk_flags = nullptr;
  if (left >= gemm::kSkFlagBytes) {
    pb.sk_flags = reinterpret_cast<uint32_t*>(w);
    w += gemm::kSkFlagBytes;
    left -= gemm::kSkFlagBytes;
  } else {
    left = 0;  // too small to hold the flags: no workspace is used
  }
  if (pb.tf32 && (pb.A.mn_major || pb.B.mn_major)) {
    XT_REQUIRE(ws != nullptr, "matmul: fp32 operands read MN-major need a workspace");
    if (pb.A.mn_major) XT_TRY(stage_operand(pb.A, w, left, s));
    if (pb.B.mn_major) XT_TRY(stage_operand(pb.B, w, left, s));
  }
  pb.split_ws = left ? w : nullptr;  // what remains holds K-split partials, if used
  pb.split_ws_bytes = left;
  pb.C = C;
  pb.ldc = d->ldc;
  pb.sc_inner = d->stride_c_inner;
  pb.sc_outer = d->stride_c_outer;
  pb.c_bf16 = d->dtype_c == XT_BF16;
  pb.alpha = d->alpha;
  pb.accumulate = d->accumulate;
  pb.causal = d->causal;
  pb.act = act;
  pb.C2 = C2;
  pb.aux = aux;
  return gemm::run(pb, s);
}

}  // namespace xt

using namespace xt;

extern "C" {

int xt_gemm_set_schedule(int mode) {
  XT_REQUIRE(mode >= 0 && mode <= 4, "xt_gemm_set_schedule: mode must be 0..4");
  gemm::g_schedule = mode;
  return XT_OK;
}

int xt_gemm_set_tile(int bn) {
  XT_REQUIRE(bn == 0 || bn == 64 || bn == 128 || bn == 192 || bn == 256, "xt_gemm_set_tile: bn must be 0, 64, 128, 192 or 256");
  gemm::g_tile = bn;
  return XT_OK;
}

int xt_gemm_set_pairing(int mode) {
  XT_REQUIRE(mode >= 0 && mode <= 3, "xt_gemm_set_pairing: mode must be 0..3");
  gemm::g_pairing = mode;
  return XT_OK;
}

int xt_matmul_workspace_size(const xt_matmul_desc* desc, size_t* bytes) {
  XT_REQUIRE(desc && bytes, "xt_matmul_workspace_size: NULL pointer");
  *bytes = matmul_ws(desc);
  return XT_OK;
}

int xt_matmul_fwd(const xt_matmul_desc* desc, const void* A, const void* B, void* C, void* ws, size_t ws_bytes,
                  void* stream) {
  return matmul_run(desc, A, B, C, ws, ws_bytes, as_stream(stream));
}

int xt_matmul_gelu_fwd(const xt_matmul_desc* desc, const void* A, const void* B, void* C, void* Y, void* ws,
                       size_t ws_bytes, void* stream) {
  return matmul_run(desc, A, B, C, ws, ws_bytes, as_stream(stream), 1, Y, nullptr);
}

int xt_matmul_gelu_bwd(const xt_matmul_desc* desc, const void* A, const void* B, const void* X, void* C, void* ws,
                       size_t ws_bytes, void* stream) {
  return matmul_run(desc, A, B, C, ws, ws_bytes, as_stream(stream), 2, nullptr, X);
}

}  // extern "C"

// The two GEMMs of the matmul backward, as descriptors over (dC, A, B).
struct BwdPlan {
  xt_matmul_desc ga, gb;
  int a_first_is_dc, b_first_is_dc;  // operand order of each GEMM
};

static BwdPlan bwd_plan(const xt_matmul_desc& f, int dt_grad_a, int dt_grad_b, int acc_a, int acc_b) {
  BwdPlan pl{};
  {
    xt_matmul_desc& g = pl.ga;
    g.batch_outer = f.batch_outer;
    g.batch_inner = f.batch_inner;
    g.dtype_ab = f.dtype_ab;
    g.dtype_c = dt_grad_a;
    g.accumulate = acc_a;
    g.alpha = f.alpha;
    if (!f.trans_a) {  // dA [M,K] = dC [M,N] @ op(B)ᵀ
      g.M = f.M; g.N = f.K; g.K = f.N;
      g.trans_a = 0; g.lda = f.ldc; g.stride_a_inner = f.stride_c_inner; g.stride_a_outer = f.stride_c_outer;
      g.trans_b = f.trans_b ? 0 : 1; g.ldb = f.ldb; g.stride_b_inner = f.stride_b_inner; g.stride_b_outer = f.stride_b_outer;
      g.ldc = f.lda; g.stride_c_inner = f.stride_a_inner; g.stride_c_outer = f.stride_a_outer;
      pl.a_first_is_dc = 1;
    } else {  // A stored [K,M]: dA = op(B) @ dCᵀ
      g.M = f.K; g.N = f.M; g.K = f.N;
      g.trans_a = f.trans_b; g.lda = f.ldb; g.stride_a_inner = f.stride_b_inner; g.stride_a_outer = f.stride_b_outer;
      g.trans_b = 1; g.ldb = f.ldc; g.stride_b_inner = f.stride_c_inner; g.stride_b_outer = f.stride_c_outer;
      g.ldc = f.lda; g.stride_c_inner = f.stride_a_inner; g.stride_c_outer = f.stride_a_outer;
      pl.a_first_is_dc = 0;
    }
  }
  {
    xt_matmul_desc& g = pl.gb;
    g.batch_outer = f.batch_outer;
    g.batch_inner = f.batch_inner;
    g.dtype_ab = f.dtype_ab;
    g.dtype_c = dt_grad_b;
    g.accumulate = acc_b;
    g.alpha = f.alpha;
    if (!f.trans_b) {  // dB [K,N] = op(A)ᵀ @ dC
      g.M = f.K; g.N = f.N; g.K = f.M;
      g.trans_a = f.trans_a ? 0 : 1; g.lda = f.lda; g.stride_a_inner = f.stride_a_inner; g.stride_a_outer = f.stride_a_outer;
      g.trans_b = 0; g.ldb = f.ldc; g.stride_b_inner = f.stride_c_inner; g.stride_b_outer = f.stride_c_outer;
      g.ldc = f.ldb; g.stride_c_inner = f.stride_b_inner; g.stride_c_outer = f.stride_b_outer;
      pl.b_first_is_dc = 0;
    } else {  // B stored [N,K]: dB = dCᵀ @ op(A)
      g.M = f.N; g.N = f.K; g.K = f.M;
      g.trans_a = 1; g.lda = f.ldc; g.stride_a_inner = f.stride_c_inner; g.stride_a_outer = f.stride_c_outer;
      g.trans_b = f.trans_a; g.ldb = f.lda; g.stride_b_inner = f.stride_a_inner; g.stride_b_outer = f.stride_a_outer;
      g.ldc = f.ldb; g.stride_c_inner = f.stride_b_inner; g.stride_c_outer = f.stride_b_outer;
      pl.b_first_is_dc = 1;
    }
  }
  return pl;
}

extern "C" {

int xt_matmul_bwd_workspace_size(const xt_matmul_desc* desc, size_t* bytes) {
  XT_REQUIRE(desc && bytes, "xt_matmul_bwd_workspace_size: NULL pointer");
  const BwdPlan pl = bwd_plan(*desc, XT_F32, XT_F32, 0, 0);
  const size_t a = matmul_ws(&pl.ga), b = matmul_ws(&pl.gb);
  *bytes = a > b ? a : b;
  return XT_OK;
}

int xt_matmul_bwd(const xt_matmul_desc* desc, const void* A, const void* B, const void* dC, void* dA, void* dB,
                  int dt_grad_a, int dt_grad_b, int acc_a, int acc_b, void* ws, size_t ws_bytes, void* stream) {
  XT_REQUIRE(desc != nullptr, "xt_matmul_bwd: desc is NULL");
  XT_REQUIRE(desc->causal == 0, "xt_matmul_bwd: causal must be 0");
  XT_REQUIRE(!dA || valid_dtype(dt_grad_a), "xt_matmul_bwd: bad dt_grad_a");
  XT_REQUIRE(!dB || valid_dtype(dt_grad_b), "xt_matmul_bwd: bad dt_grad_b");
  cudaStream_t s = as_stream(stream);
  const BwdPlan pl = bwd_plan(*desc, dt_grad_a, dt_grad_b, acc_a, acc_b);
  // the two GEMMs run in stream order, so they can share one workspace
  if (dA) {
    if (pl.a_first_is_dc) XT_TRY(matmul_run(&pl.ga, dC, B, dA, ws, ws_bytes, s));
    else XT_TRY(matmul_run(&pl.ga, B, dC, dA, ws, ws_bytes, s));
  }
  if (dB) {
    if (pl.b_first_is_dc) XT_TRY(matmul_run(&pl.gb, dC, A, dB, ws, ws_bytes, s));
    else XT_TRY(matmul_run(&pl.gb, A, dC, dB, ws, ws_bytes, s));
  }
  return XT_OK;
}

}  // extern "C"

namespace xt {
int matmul(const xt_matmul_desc& d, const void* A, const void* B, void* C, void* ws, size_t ws_bytes,
           cudaStream_t s) {
  return matmul_run(&d, A, B, C, ws, ws_bytes, s);
}
size_t matmul_workspace(const xt_matmul_desc& d) { return matmul_ws(&d); }

}  // namespace xt
