// Tensor-core GEMM for sm_103a: tcgen05.mma with the accumulator in tensor memory (TMEM),
// operands staged in shared memory by TMA (cp.async.bulk.tensor, 128-byte swizzle),
// an mbarrier pipeline of STAGES slots, and a persistent tile loop.
//
// Roles (192 threads): warp 0 lane 0 issues TMA loads; warp 1 allocates TMEM and its
// lane 0 issues the MMAs; warps 2..5 drain the accumulator (tcgen05.ld) and store C.
// TMEM holds two accumulators of BN fp32 columns so the epilogue of tile i overlaps the
// MMAs of tile i+1.  Each epilogue warp stages its 32 rows × 128 bytes of C in a
// double-buffered, 128-byte-swizzled shared-memory tile and writes it with a TMA bulk tensor
// store (for accumulation into fp32 C: a TMA reduce-add, performed in L2 without reading C).
//
// Every mbarrier wait is bounded (%globaltimer); on expiry the CTA records
// XT_DEVERR_TIMEOUT in the device flag, every role stops issuing work, the producer waits
// (bounded) for its copies in flight, and TMEM is released before the CTA exits.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace xt {
namespace gemm {

constexpr int BM = 128;
// Operand kinds (the KIND template parameter): bf16 (tcgen05 kind::f16), tf32 (kind::tf32) and
// fp8 e4m3 (kind::f8f6f4).  One MMA instruction consumes 32 bytes of K of each operand row.
constexpr int kBf16 = 0, kTf32 = 1, kFp8 = 2;
constexpr int kThreads = 192;
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct Params {
  int M, N, K;
  int num_m, num_n;
  int batch_inner, batches;  // batches = outer × inner
  int splitk;                // > 1: batch_inner is the K split; partial tiles go to C slices
  int kb_per_split;
  int causal;
  int accumulate;
  int c_bf16;
  int tma_store;  // 1: epilogue writes through TMA (C described by tmC); 0: direct stores
  float alpha;
  void* C;
  int64_t ldc, sc_inner, sc_outer;
  // GELU epilogue (bf16 C, TMA stores, one batch): 1 = also store gelu(C) through tmC2;
  // 2 = C = (alpha·A@B) ∘ gelu'(aux), aux bf16 [M, N] with row stride ld_aux
  int act;
  const bf16* aux;
  int64_t ld_aux;
  uint32_t* flag;
  // Stream-K schedule (sk = 1): CTA c computes the k-block iterations [⌊c·I/G⌋, ⌊(c+1)·I/G⌋) of
  // the tiles × kb_tile iteration space (I = sk_iters ≥ G = gridDim.x ≤ the SMs), so every CTA
  // does the same amount of MMA work whatever the tile count (G = the SMs), or every CTA one
  // K slice of one tile with all CTAs at the same K offsets (G = tiles × slices).  A CTA whose share starts inside a tile
  // writes that piece's raw fp32 accumulator to slot c of sk_part ([G][BM·BN] floats) and sets
  // sk_flag[4c + q] = tile + 1 for each TMEM lane quadrant q; the CTA that computes the tile's
  // first k-blocks (the last piece of its own share) waits for those flags, adds the slots in
  // CTA order (a fixed order: deterministic), clears the flags and stores C.
  int sk;
  int kb_tile;
  int64_t sk_iters;
  float* sk_part;
  uint32_t* sk_flag;
  // per-tensor factors (device floats, may be null) multiplying alpha: the dequantization
  // factors of fp8 operands
  const float* scale_a;
  const float* scale_b;
  // measurement (may be null): (start, end) %globaltimer words per CTA, at 2·blockIdx.x
  unsigned long long* prof_ts;
  // limit of the waits on work (xt_set_wait_limit_ns); the waits that drain a CTA's own copies
  // and MMAs before it exits keep kTimeoutNs
  uint64_t wait_ns;
};

// ------------------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of parity `parity`; false when `limit_ns` expired.  Limits of a
// millisecond or more use the suspending try_wait; a shorter limit (set for tests of the
// give-up paths) polls with the non-blocking test_wait, so that a wait cannot outlast it by a
// suspension.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = kTimeoutNs) {
  if (limit_ns >= 1000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
      if (mbar_try_wait(bar, parity)) return true;
      if (globaltimer() - t0 > limit_ns) return false;
    }
  }
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_test_wait(bar, parity)) return true;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

// test_wait with acquire at cluster scope: pairs with a remote mbarrier.arrive.release.cluster
// (the paired kernel's relayed stage arrivals).
__device__ __forceinline__ bool mbar_test_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_spin_cl(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_test_wait_cl(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_test_wait_cl(bar, parity)) return true;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

// Bounded wait that polls with the non-blocking test_wait: the waiting thread sees the phase
// flip on its next poll instead of after a suspended try_wait wakes, for the MMA issuer's waits
// on landed operand stages (a few per tile, each on the tensor core's critical path).
__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_test_wait(bar, parity)) return true;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], "
      "[%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
// Shared → global tensor store / reduce-add of one box; completion tracked by bulk groups.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* tm, uint32_t src, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
__device__ __forceinline__ void tma_reduce_add_4d(const CUtensorMap* tm, uint32_t src, int c0, int c1, int c2, int c3) {
  asm volatile("cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most one committed bulk group is still reading its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrives on `bar` once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// One MMA: D (+)= A·Bᵀ over 32 bytes of K.  CG = 2 issues the paired-CTA form: the issuing
// (even) CTA and its peer each supply 128 rows of A and half of B's rows from the same
// shared-memory offsets, and each peer's TMEM receives its own 128 rows of D.
template <int KIND, int CG = 1>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accum) {
#define XT_TC_MMA(GROUP, K_)                                                                       \
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"                                 \
               "tcgen05.mma.cta_group::" GROUP ".kind::" K_ " [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem), \
               "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)                                      \
               : "memory")
  if constexpr (CG == 2) {
    if constexpr (KIND == kFp8) XT_TC_MMA("2", "f8f6f4");
    else if constexpr (KIND == kTf32) XT_TC_MMA("2", "tf32");
    else XT_TC_MMA("2", "f16");
  } else {
    if constexpr (KIND == kFp8) XT_TC_MMA("1", "f8f6f4");
    else if constexpr (KIND == kTf32) XT_TC_MMA("1", "tf32");
    else XT_TC_MMA("1", "f16");
  }
#undef XT_TC_MMA
}

// ------------------------------------------------------------- paired-CTA (cluster of two) forms
// All tcgen05 instructions of one kernel use the same cta_group; the pair kernel uses these.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Every thread of both CTAs; release / acquire orders shared-memory writes (barrier inits)
// before the peer's first remote access.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on an mbarrier given by its shared::cluster address (possibly in the peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
// Tile load whose completion is signalled on an mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int c0, int c1,
                                                 int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
// Tile load multicast to the CTAs of `mask` (cluster ranks): the box lands at the same
// shared-memory offset in each of them, and each one's mbarrier at the offset of `bar` receives
// the bytes that landed in it.
__device__ __forceinline__ void tma_load_4d_mc(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int c0, int c1,
                                               int c2, int c3, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster [%0], "
      "[%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "h"(mask)
      : "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_alloc_cg(uint32_t dst_smem, uint32_t ncols) {
  if constexpr (CG == 2)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
  else
    tmem_alloc(dst_smem, ncols);
}
template <int CG>
__device__ __forceinline__ void tmem_relinquish_cg() {
  if constexpr (CG == 2) asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  else tmem_relinquish();
}
template <int CG>
__device__ __forceinline__ void tmem_dealloc_cg(uint32_t taddr, uint32_t ncols) {
  if constexpr (CG == 2)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  else
    tmem_dealloc(taddr, ncols);
}
// Arrives on `bar` once this thread's earlier tcgen05 operations have completed: CG = 2 on the
// barrier at that offset in each CTA of `mask` (cluster ranks; a pair's two CTAs by default),
// CG = 1 on this CTA's barrier only.
template <int CG>
__device__ __forceinline__ void tc_commit_cg(uint32_t bar, uint16_t mask = 3) {
  if constexpr (CG == 2) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
  } else {
    tc_commit(bar);
  }
}
// 32 lanes × 32 consecutive fp32 columns: thread t of the warp receives row (lane base + t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 lanes × 32 consecutive fp32 columns written from registers (the layout of tmem_ld32).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Wait until every committed bulk group has finished reading its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Shared-memory matrix descriptor (sm_100 format): start address, leading- and stride-
// dimension byte offsets (all >> 4), descriptor version 1 at bit 46, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor for kind::f16 / kind::tf32 / kind::f8f6f4: fp32 accumulator, A/B
// types (bf16 = 1, tf32 = 2, e4m3 = 0), operand majorness (1 = MN-major), N >> 3, M >> 4.
template <int KIND, int N, bool A_MN, bool B_MN, int M = BM>
__host__ __device__ constexpr uint32_t instr_desc() {
  constexpr uint32_t t = KIND == kTf32 ? 2u : KIND == kFp8 ? 0u : 1u;
  return (1u << 4) | (t << 7) | (t << 10) | ((A_MN ? 1u : 0u) << 15) | ((B_MN ? 1u : 0u) << 16) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// bf16 × bf16 → fp32 instruction descriptor for an M × N tile.
__host__ __device__ constexpr uint32_t instr_desc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

template <int BN>
constexpr uint32_t tmem_cols() {
  return 2 * BN <= 32 ? 32 : 2 * BN <= 64 ? 64 : 2 * BN <= 128 ? 128 : 2 * BN <= 256 ? 256 : 512;
}

// K per stage, in 128-byte swizzle atoms: a K-major operand is staged as that many chunks of
// [rows × 128 B] (one TMA box each), an MN-major one as [BK rows × 128 B] chunks along MN.  The
// paired kernel takes two (half the mbarrier round trips per tile, three stages); the single-CTA
// kernel one (its wide tiles would keep only two stages of two).
__host__ __device__ constexpr int k_atoms(int cg) { return cg == 2 ? 2 : 1; }

// CG = 2: a CTA pair computes a (2·BM) × BN tile; each CTA stages its own BM rows of A and
// BN / 2 rows of B.
template <int KIND, int BN, int CG = 1>
struct Cfg {
  static constexpr int E = KIND == kTf32 ? 4 : KIND == kFp8 ? 1 : 2;
  static constexpr int KA = k_atoms(CG);     // 128-byte K atoms per stage
  static constexpr int BK = KA * 128 / E;    // K elements per stage
  static constexpr int ATOM = 128 / E;       // MN (or K) elements per 128-byte swizzle row
  static constexpr int UK = 32 / E;          // K per MMA instruction (32 bytes)
  static constexpr int A_BYTES = BM * 128 * KA;
  static constexpr int B_BYTES = BN / CG * 128 * KA;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (192 * 1024) / STAGE_BYTES > 8 ? 8 : (192 * 1024) / STAGE_BYTES;
  static constexpr int STAGING_BYTES = 4 * 2 * 4096;  // 4 epilogue warps × 2 buffers × 32 rows × 128 B
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES + STAGING_BYTES + BAR_BYTES;
};

struct TileInfo {
  int m0, n0, zi, zo, kb_begin, kb_end;
  int ozi, ozo;  // batch coordinates of the operands (0 for a K split)
  bool skip;
};

template <int BK>
__device__ __forceinline__ TileInfo tile_info(int t, const Params& p) {
  TileInfo ti;
  const int per = p.num_m * p.num_n;
  const int z = t / per;
  const int r = t - z * per;
  const int nb = r / p.num_m;
  const int mb = r - nb * p.num_m;  // m fastest: concurrent CTAs share B tiles
  ti.m0 = mb * BM;
  ti.n0 = nb * 0;  // set by caller (BN known there)
  ti.zo = z / p.batch_inner;
  ti.zi = z - ti.zo * p.batch_inner;
  ti.kb_begin = 0;
  ti.kb_end = (p.K + BK - 1) / BK;
  if (p.causal == 2) {
    const int e = (ti.m0 + BM + BK - 1) / BK;
    if (e < ti.kb_end) ti.kb_end = e;
  } else if (p.causal == 3) {
    ti.kb_begin = ti.m0 / BK;
  }
  ti.ozi = ti.zi;
  ti.ozo = ti.zo;
  if (p.splitk > 1) {  // K split: zi selects the range of K blocks and the output slice
    ti.kb_begin = ti.zi * p.kb_per_split;
    const int e = ti.kb_begin + p.kb_per_split;
    if (e < ti.kb_end) ti.kb_end = e;
    ti.ozi = 0;
    ti.ozo = 0;
  }
  ti.skip = false;
  (void)nb;
  return ti;
}

// The pieces (tile, k-block range) a CTA computes, in order: whole tiles blockIdx.x + i·gridDim.x,
// or under stream-K the parts of the tiles its contiguous share of iterations covers.
struct Cursor {
  int64_t it, end;
};
// `u` of `nu` schedule units: a CTA, or a CTA pair of the paired kernel.
__device__ __forceinline__ Cursor cursor_begin(const Params& p, int u, int nu) {
  Cursor c;
  if (p.sk) {
    c.it = int64_t(u) * p.sk_iters / nu;
    c.end = int64_t(u + 1) * p.sk_iters / nu;
  } else {
    c.it = u;
    c.end = 0;
  }
  return c;
}
// Next piece, false when none is left; kb0 = kb1 = -1 for a whole tile of the plain schedule.
__device__ __forceinline__ bool cursor_next(Cursor& c, const Params& p, int total, int nu, int& t, int& kb0,
                                            int& kb1) {
  if (!p.sk) {
    if (c.it >= total) return false;
    t = int(c.it);
    c.it += nu;
    kb0 = kb1 = -1;
    return true;
  }
  if (c.it >= c.end) return false;
  t = int(c.it / p.kb_tile);
  kb0 = int(c.it - int64_t(t) * p.kb_tile);
  const int64_t room = c.end - c.it;
  kb1 = room < int64_t(p.kb_tile - kb0) ? kb0 + int(room) : p.kb_tile;
  c.it += kb1 - kb0;
  return true;
}
// Stream-K: the unit whose share holds iteration x, i.e. the largest c with ⌊c·I/G⌋ ≤ x.
__device__ __forceinline__ int sk_cta_of(int64_t x, const Params& p, int nu) {
  return int(((x + 1) * int64_t(nu) - 1) / p.sk_iters);
}

// Stream-K fixup of a tile's accumulator in TMEM (columns tacc .. tacc + BN of this warp's
// lanes): adds the partial accumulators of CTAs first..last, in CTA order, 32 columns at a
// time (tcgen05.ld, add, tcgen05.st), with the loads of the group two ahead in flight.  Slot
// layout: float4 (g·8 + j)·BM + row holds columns 32·g + 4·j .. +4 of the row, so a warp's
// loads and stores each cover 512 contiguous bytes.
// Slot of unit cc: cc·CG + rank (each CTA of a pair keeps its own rows' partial).
template <int BN, int CG = 1>
__device__ __forceinline__ void sk_fixup(uint32_t tacc, const Params& p, int first, int last, int rank, int row) {
  constexpr int NG = BN / 32;
  for (int cc = first; cc <= last; ++cc) {
    const float4* src = reinterpret_cast<const float4*>(p.sk_part) + size_t(cc * CG + rank) * (BM * BN / 4) + row;
    float4 v[2][8];
#pragma unroll
    for (int g = 0; g < 2 && g < NG; ++g)
#pragma unroll
      for (int j = 0; j < 8; ++j) v[g][j] = __ldcg(src + size_t(g * 8 + j) * BM);
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      uint32_t a[32];
      tmem_ld32(tacc + uint32_t(g * 32), a);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        a[4 * j] = __float_as_uint(__uint_as_float(a[4 * j]) + v[g & 1][j].x);
        a[4 * j + 1] = __float_as_uint(__uint_as_float(a[4 * j + 1]) + v[g & 1][j].y);
        a[4 * j + 2] = __float_as_uint(__uint_as_float(a[4 * j + 2]) + v[g & 1][j].z);
        a[4 * j + 3] = __float_as_uint(__uint_as_float(a[4 * j + 3]) + v[g & 1][j].w);
      }
      if (g + 2 < NG)
#pragma unroll
        for (int j = 0; j < 8; ++j) v[g & 1][j] = __ldcg(src + size_t((g + 2) * 8 + j) * BM);
      tmem_st32(tacc + uint32_t(g * 32), a);
    }
    tmem_st_wait();
  }
}

// ACT: the epilogue's GELU mode (Params::act), a template parameter so the plain GEMMs carry
// none of its code.
//
// CG = 2 (launched as clusters of two CTAs): each pair computes (2·BM) × BN tiles with the
// paired MMA.  The even CTA's lane issues every MMA; each CTA's producer loads its own BM rows
// of A and BN / 2 rows of B into its own shared memory and signals the even CTA's full barrier
// (which expects both CTAs' bytes); each MMA group's commit arrives on the stage's empty
// barrier of both CTAs and, per tile, on both CTAs' accumulator-full barriers; both CTAs'
// epilogues (each draining its own 128 TMEM lanes) arrive on the even CTA's accumulator-empty
// barrier.  Schedule units (Params::num_m tiles of 2·BM rows, stream-K shares) are pairs.
//
// MC = 2 (clusters of four CTAs, two pairs; whole tiles of a plain schedule only): the two pairs
// compute vertically adjacent tiles (pair i of the cluster the 2·BM rows of tile 2j + i of a
// tile group), so both need the same B rows.  Each CTA loads half of its B rows and multicasts
// it to the CTA at the same place in the other pair: every CTA's B stage is filled by two
// loads, one from each pair, and a pair reads half the B bytes from L2 that it would alone.  A
// stage of B in a pair's odd CTA completes on that CTA's own full barrier (a multicast signals
// the barrier in each receiving CTA), and the odd CTA's warp 1 relays it to the even CTA's full
// barrier, which then counts two arrivals; the MMAs' commits free a stage in all four CTAs
// (each empty barrier counts one commit per pair).
template <int KIND, int BN, bool A_MN, bool B_MN, int ACT = 0, int CG = 1, int MC = 1>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmC2, const Params p) {
  static_assert(CG == 1 || (CG == 2 && ACT == 0 && BN % 32 == 0), "paired tiles: plain epilogue, BN / 2 whole atoms");
  static_assert(MC == 1 || (MC == 2 && CG == 2 && BN == 256), "multicast pairs: 256-wide paired tiles");
  // The set-up below (barriers, tensor-map prefetch, TMEM) reads nothing a preceding kernel
  // writes, so it runs before the programmatic-launch wait.
  using C_ = Cfg<KIND, BN, CG>;
  constexpr int BK = C_::BK, ATOM = C_::ATOM, UK = C_::UK, STAGES = C_::STAGES;
  constexpr uint32_t IDESC = instr_desc<KIND, BN, A_MN, B_MN, BM * CG>();
  constexpr uint32_t TCOLS = tmem_cols<BN>();
  constexpr int BNH = BN / CG;  // B rows staged by one CTA
  constexpr int CL = CG * MC;   // CTAs per cluster
  // rank: this CTA's place in its pair; pidx: the pair's place in the cluster; leader: the
  // cluster rank of the pair's even CTA
  const int crank = CG == 2 ? int(cluster_ctarank()) : 0;
  const int rank = crank & 1;
  const int pidx = MC == 2 ? crank >> 1 : 0, leader = MC == 2 ? crank & ~1 : 0;
  const int unit = int(blockIdx.x) / CL, units = int(gridDim.x) / CL;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + STAGES * C_::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + C_::STAGING_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = bars + 2 * STAGES + 2;
  uint64_t* mma_done = bars + 2 * STAGES + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), MC == 2 && rank == 0 ? 2 : 1);  // + the odd CTA's relayed arrival
      mbar_init(smem_u32(&empty[s]), MC);                            // one commit per pair
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), 4 * CG);
    }
    mbar_init(smem_u32(mma_done), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (p.tma_store) prefetch_tmap(&tmC);
    if (ACT == 1) prefetch_tmap(&tmC2);
  }
  if (warp == 1) {
    tmem_alloc_cg<CG>(smem_u32(tmem_slot), TCOLS);
    tmem_relinquish_cg<CG>();
  }
  tc_fence_before();
  if constexpr (CG == 2) cluster_sync_all();  // the peer's barriers exist before any remote arrive
  else __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  pdl_wait();  // the operands (and C, when accumulating) are the preceding kernels' outputs
  pdl_trigger();
  if (p.prof_ts && threadIdx.x == 0) p.prof_ts[2 * blockIdx.x] = global_ns();

  // schedule items: tiles, or with MC = 2 tile groups (two vertically adjacent tiles)
  const int total = p.num_m * p.num_n * p.batches / MC;

  // ti.m0: this CTA's first row (tile row + rank·BM); ti.n0: the tile's first column.
  auto info = [&](int t, int kb0, int kb1) {
    if constexpr (MC == 2) {  // group t → this pair's tile (m-groups fastest, as tiles are)
      const int nmg = p.num_m / 2, per_g = nmg * p.num_n;
      const int z = t / per_g, r = t - z * per_g;
      const int nb = r / nmg, mg = r - nb * nmg;
      t = z * (p.num_m * p.num_n) + nb * p.num_m + 2 * mg + pidx;
    }
    TileInfo ti = tile_info<BK>(t, p);
    const int per = p.num_m * p.num_n;
    const int r = t - (t / per) * per;
    if constexpr (CG == 2) ti.m0 = ti.m0 * 2 + rank * BM;
    ti.n0 = (r / p.num_m) * BN;
    if (p.causal == 1 && ti.n0 >= ti.m0 + BM) ti.skip = true;
    if (kb0 >= 0) {  // a stream-K piece
      ti.kb_begin = kb0;
      ti.kb_end = kb1;
    }
    return ti;
  };

  auto give_up = [&]() {
    *abort_flag = 1;
    flag_error(p.flag, XT_DEVERR_TIMEOUT);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      Cursor cur = cursor_begin(p, unit, units);
      int t, kb0, kb1;
      // load: one box into this CTA's stage, completing on the stage's full barrier (the even
      // CTA's for a pair)
      auto load = [&](uint32_t dst, const CUtensorMap* tm, uint32_t fb, int c0, int c1, int c2, int c3) {
        if constexpr (CG == 2) tma_load_4d_pair(dst, tm, fb, c0, c1, c2, c3);
        else tma_load_4d(dst, tm, fb, c0, c1, c2, c3);
      };
      while (!*abort_flag && cursor_next(cur, p, total, units, t, kb0, kb1)) {
        const TileInfo ti = info(t, kb0, kb1);
        if (ti.skip) continue;
        const int nb0 = ti.n0 + rank * BNH;  // this CTA's rows of B
        for (int kb = ti.kb_begin; kb < ti.kb_end; ++kb) {
          if (*abort_flag) break;
          if (!mbar_wait_spin(smem_u32(&empty[stage]), phase ^ 1, p.wait_ns)) { give_up(); break; }
          const uint32_t fb_own = smem_u32(&full[stage]);
          uint32_t fb = fb_own;
          if constexpr (MC == 2) mbar_expect_tx(fb_own, rank == 0 ? 2 * C_::A_BYTES + C_::B_BYTES : C_::B_BYTES);
          else if (rank == 0) mbar_expect_tx(fb, CG * C_::STAGE_BYTES);
          if constexpr (CG == 2) fb = mapa_shared(fb, leader);
          const uint32_t a_s = smem_u32(smem + stage * C_::STAGE_BYTES);
          const uint32_t b_s = a_s + C_::A_BYTES;
          const int k0 = kb * BK;
          if constexpr (!A_MN) {
#pragma unroll
            for (int c = 0; c < C_::KA; ++c) load(a_s + c * (BM * 128), &tmA, fb, k0 + c * ATOM, ti.m0, ti.ozi, ti.ozo);
          } else {
#pragma unroll
            for (int j = 0; j < BM / ATOM; ++j)
              load(a_s + j * (BK * 128), &tmA, fb, ti.m0 + j * ATOM, k0, ti.ozi, ti.ozo);
          }
          if constexpr (MC == 2) {
            // this CTA's half of its B rows, to itself and to its place in the other pair
            const uint16_t mask = uint16_t((1u << rank) | (1u << (rank + 2)));
            if constexpr (!B_MN) {
#pragma unroll
              for (int c = 0; c < C_::KA; ++c)
                tma_load_4d_mc(b_s + c * (BNH * 128) + pidx * (BNH / 2 * 128), &tmB, fb_own, k0 + c * ATOM,
                               nb0 + pidx * (BNH / 2), ti.ozi, ti.ozo, mask);
            } else {
              static_assert(!B_MN || BNH == 2 * ATOM, "MN-major B: one atom-wide box per pair");
              tma_load_4d_mc(b_s + pidx * (BK * 128), &tmB, fb_own, nb0 + pidx * ATOM, k0, ti.ozi, ti.ozo, mask);
            }
          } else if constexpr (!B_MN) {
#pragma unroll
            for (int c = 0; c < C_::KA; ++c) load(b_s + c * (BNH * 128), &tmB, fb, k0 + c * ATOM, nb0, ti.ozi, ti.ozo);
          } else {
#pragma unroll
            for (int j = 0; j < BNH / ATOM; ++j)
              load(b_s + j * (BK * 128), &tmB, fb, nb0 + j * ATOM, k0, ti.ozi, ti.ozo);
          }
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      // Wait (bounded) for the copies that may still be in flight: the last min(STAGES, issued)
      // fills, so no TMA write lands in shared memory after the CTA exits.  A pair's full
      // barriers live in the even CTA and count both CTAs' bytes: the even CTA waits for both,
      // and the cluster barrier before exit keeps the odd CTA resident until then.
      const int pending = rank != 0 ? 0 : issued < STAGES ? issued : STAGES;
      for (int i = 0; i < pending; ++i) {
        if (--stage < 0) { stage = STAGES - 1; phase ^= 1; }
        if (!mbar_wait(smem_u32(&full[stage]), phase)) { give_up(); break; }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int ab = 0;
      uint32_t aphase = 0;
      bool any = false;
      Cursor cur = cursor_begin(p, unit, units);
      int t, kb0, kb1;
      // The next piece's coordinates are worked out while the current tile's first MMAs run, so
      // the tensor pipe does not wait on this thread's index arithmetic between tiles.
      bool have = cursor_next(cur, p, total, units, t, kb0, kb1);
      TileInfo ti_next;
      if (have) ti_next = info(t, kb0, kb1);
      while (have && !*abort_flag) {
        const TileInfo ti = ti_next;
        bool fetched = false;
        auto fetch = [&]() {
          have = cursor_next(cur, p, total, units, t, kb0, kb1);
          if (have) ti_next = info(t, kb0, kb1);
          fetched = true;
        };
        if (ti.skip || ti.kb_end <= ti.kb_begin) {
          fetch();
          continue;
        }
        if (!mbar_wait_spin(smem_u32(&tempty[ab]), aphase ^ 1, p.wait_ns)) { give_up(); break; }
        tc_fence_after();
        const uint32_t d_tmem = tbase + uint32_t(ab * BN);
        bool ok = true;
        for (int kb = ti.kb_begin; kb < ti.kb_end; ++kb) {
          const bool landed = MC == 2 ? mbar_wait_spin_cl(smem_u32(&full[stage]), phase, p.wait_ns)
                                      : mbar_wait_spin(smem_u32(&full[stage]), phase, p.wait_ns);
          if (*abort_flag || !landed) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_s = smem_u32(smem + stage * C_::STAGE_BYTES);
          const uint32_t b_s = a_s + C_::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk) {
            // K-major: K step kk lies in atom kk / (ATOM / UK) at byte (kk % (ATOM / UK))·32
            constexpr int PA = ATOM / UK;
            const uint64_t ad = A_MN ? smem_desc(a_s + kk * UK * 128, BK * 128, 1024)
                                     : smem_desc(a_s + (kk / PA) * (BM * 128) + (kk % PA) * UK * C_::E, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc(b_s + kk * UK * 128, BK * 128, 1024)
                                     : smem_desc(b_s + (kk / PA) * (BNH * 128) + (kk % PA) * UK * C_::E, 16, 1024);
            tc_mma<KIND, CG>(d_tmem, ad, bd, IDESC, (kb > ti.kb_begin || kk > 0) ? 1u : 0u);
          }
          any = true;
          // frees the smem slot(s) once these MMAs finish: a multicast stage in all four CTAs
          tc_commit_cg<CG>(smem_u32(&empty[stage]), MC == 2 ? uint16_t(0xF) : uint16_t(3));
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
          if (!fetched) fetch();
        }
        if (!ok) { give_up(); break; }
        tc_commit_cg<CG>(smem_u32(&tfull[ab]), uint16_t(3u << leader));  // accumulator ready for the epilogue(s)
        if (++ab == 2) { ab = 0; aphase ^= 1; }
      }
      // every MMA issued has completed (also after a give-up) before TMEM is released
      if (any) {
        tc_commit_cg<CG>(smem_u32(mma_done), uint16_t(3u << leader));  // (the odd CTA's arrival is unused)
        if (!mbar_wait(smem_u32(mma_done), 0)) give_up();
      }
    } else if (MC == 2 && lane == 0 && rank == 1) {
      // ------------------------------------------------ relay of the odd CTA's B stages
      // The multicast halves of this CTA's B rows complete on its own full barrier; each
      // completed stage is passed on to the even CTA's full barrier, where the MMA issuer waits.
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t full_at = mapa_shared(smem_u32(&full[0]), leader);
      Cursor cur = cursor_begin(p, unit, units);
      int t, kb0, kb1;
      bool ok = true;
      while (ok && !*abort_flag && cursor_next(cur, p, total, units, t, kb0, kb1)) {
        const TileInfo ti = info(t, kb0, kb1);
        if (ti.skip) continue;
        for (int kb = ti.kb_begin; kb < ti.kb_end; ++kb) {
          if (*abort_flag || !mbar_wait_spin(smem_u32(&full[stage]), phase, p.wait_ns)) { ok = false; break; }
          mbar_arrive_cluster(full_at + uint32_t(stage * 8));
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) give_up();
    }
  } else {
    // -------------------------------------------------------------------- epilogue
    // Every decision below is warp-uniform: tcgen05.ld is a .sync.aligned instruction.
    const int q = warp & 3;  // this warp may read TMEM lanes [32q, 32q + 32)
    // alpha times the operands' per-tensor factors (exactly alpha when there are none)
    const float alpha = p.alpha * (p.scale_a ? __ldg(p.scale_a) : 1.f) * (p.scale_b ? __ldg(p.scale_b) : 1.f);
    int ab = 0;
    uint32_t aphase = 0;
    uint32_t chunk = 0;  // staged stores issued by this warp (selects the staging buffer)
    const int self = (unit * MC + pidx) * CG + rank;  // this CTA's stream-K slot and flags
    // this warp's share of freeing accumulator ab: a pair's barrier is in the even CTA
    const uint32_t tempty0 = smem_u32(&tempty[0]);
    const uint32_t tempty_at = CG == 2 ? mapa_shared(tempty0, leader) : tempty0;
    auto release_acc = [&](int b) {
      if (CG == 2 && rank != 0) mbar_arrive_cluster(tempty_at + uint32_t(b * 8));
      else mbar_arrive(tempty0 + uint32_t(b * 8));
    };
    Cursor cur = cursor_begin(p, unit, units);
    int t, kb0, kb1;
    while (cursor_next(cur, p, total, units, t, kb0, kb1)) {
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const TileInfo ti = info(t, kb0, kb1);
      if (ti.skip) continue;
      const int row = ti.m0 + q * 32 + lane;
      const bool empty_k = ti.kb_end <= ti.kb_begin;
      // stream-K piece kind: 1 = a later part of the tile (partial to its slot), 2 = the tile's
      // first k-blocks with later parts in units unit + 1 .. sk_last (adds their partials)
      const int kind = kb0 > 0 ? 1 : (kb0 == 0 && kb1 < p.kb_tile) ? 2 : 0;
      if (!empty_k) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull[ab]), aphase, p.wait_ns));
        if (!ok) {
          if (lane == 0) give_up();
          break;
        }
        tc_fence_after();
      }
      if (kind == 1) {
        float4* slot = reinterpret_cast<float4*>(p.sk_part) + size_t(self) * (BM * BN / 4);
        const int rowt = q * 32 + lane;
#pragma unroll 1
        for (int g = 0; g < BN / 32; ++g) {
          uint32_t r[32];
          tmem_ld32(tbase + (uint32_t(q * 32) << 16) + uint32_t(ab * BN + g * 32), r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            slot[size_t(g * 8 + j) * BM + rowt] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                              __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release_acc(ab);
        if (++ab == 2) { ab = 0; aphase ^= 1; }
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(p.sk_flag + self * 4 + q, uint32_t(t + 1));
        continue;
      }
      int sk_last = 0;
      if (kind == 2) {
        sk_last = sk_cta_of(int64_t(t) * p.kb_tile + p.kb_tile - 1, p, units);
        bool ok = true;
        for (int cc = unit + 1; cc <= sk_last && ok; ++cc) {
          const uint32_t* f = p.sk_flag + (cc * CG + rank) * 4 + q;
          if (ld_acquire_gpu(f) != uint32_t(t + 1)) {
            const uint64_t t0 = globaltimer();
            while (ld_acquire_gpu(f) != uint32_t(t + 1))
              if (globaltimer() - t0 > p.wait_ns) { ok = false; break; }
          }
        }
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) give_up();
          break;
        }
        // the flags are this launch's alone until it completes: clear them for the next one
        if (lane == 0)
          for (int cc = unit + 1; cc <= sk_last; ++cc) p.sk_flag[(cc * CG + rank) * 4 + q] = 0u;
        // the later parts' sums join this piece's accumulator in TMEM; the store paths below
        // then read the tile's full sum
        sk_fixup<BN, CG>(tbase + (uint32_t(q * 32) << 16) + uint32_t(ab * BN), p, unit + 1, sk_last, rank,
                         q * 32 + lane);
      }
      if (p.tma_store) {
        // ---- staged TMA stores: chunk = 32 rows × 128 bytes (32 fp32 or 64 bf16 columns)
        const int cw = p.c_bf16 ? 64 : 32;
        const int y = ti.m0 + q * 32;
        const bool rows_in = y < p.M;
#pragma unroll 1
        for (int c = 0; c < BN / cw; ++c) {
          const int x = ti.n0 + c * cw;
          const bool write = rows_in && x < p.N && !(empty_k && p.accumulate);
          // act 1 stores two tiles per chunk (C and gelu(C)) from both buffers; otherwise the
          // buffers alternate between chunks
          const uint32_t buf = smem_u32(staging) + uint32_t((q * 2 + (ACT == 1 ? 0 : (chunk & 1))) * 4096);
          if (lane == 0) {
            if (ACT == 1) bulk_wait_read_0();
            else bulk_wait_read_1();  // the store issued from this buffer two chunks ago has read it
          }
          __syncwarp();
          uint32_t r[64];
          if (!empty_k) {
            tmem_ld32(tbase + (uint32_t(q * 32) << 16) + uint32_t(ab * BN + c * cw), *reinterpret_cast<uint32_t(*)[32]>(r));
            if (p.c_bf16)
              tmem_ld32(tbase + (uint32_t(q * 32) << 16) + uint32_t(ab * BN + c * cw + 32),
                        *reinterpret_cast<uint32_t(*)[32]>(r + 32));
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 64; ++j) r[j] = 0u;
          }
          if (write) {
            const uint32_t row_addr = buf + uint32_t(lane) * 128;
            if (!p.c_bf16) {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                st_shared_v4(row_addr + (uint32_t(j ^ (lane & 7)) << 4),
                             __float_as_uint(__uint_as_float(r[4 * j]) * alpha),
                             __float_as_uint(__uint_as_float(r[4 * j + 1]) * alpha),
                             __float_as_uint(__uint_as_float(r[4 * j + 2]) * alpha),
                             __float_as_uint(__uint_as_float(r[4 * j + 3]) * alpha));
            } else if constexpr (ACT == 0) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[8 * j + 2 * e]) * alpha,
                                                           __uint_as_float(r[8 * j + 2 * e + 1]) * alpha);
                  w[e] = *reinterpret_cast<uint32_t*>(&h);
                }
                st_shared_v4(row_addr + (uint32_t(j ^ (lane & 7)) << 4), w[0], w[1], w[2], w[3]);
              }
            } else if constexpr (ACT == 1) {
              // the pre-activation a (rounded to bf16, the value the backward reads) and gelu(a),
              // 16 columns at a time
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                float av[16], gv[16];
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  __nv_bfloat162 hh = __floats2bfloat162_rn(__uint_as_float(r[16 * h + 2 * e]) * alpha,
                                                            __uint_as_float(r[16 * h + 2 * e + 1]) * alpha);
                  w[e] = *reinterpret_cast<uint32_t*>(&hh);
                  av[2 * e] = __low2float(hh);
                  av[2 * e + 1] = __high2float(hh);
                }
                gelu_batch<16, 0>(av, gv);
                uint32_t gw[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  __nv_bfloat162 gg = __floats2bfloat162_rn(gv[2 * e], gv[2 * e + 1]);
                  gw[e] = *reinterpret_cast<uint32_t*>(&gg);
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const int j = 2 * h + u;
                  const uint32_t off = uint32_t(lane) * 128 + (uint32_t(j ^ (lane & 7)) << 4);
                  st_shared_v4(buf + off, w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                  st_shared_v4(buf + 4096 + off, gw[4 * u], gw[4 * u + 1], gw[4 * u + 2], gw[4 * u + 3]);
                }
              }
            } else {
              // dgelu: C ∘ gelu'(a) with a read from aux (this lane's row, 64 columns from x),
              // 16 columns at a time; rows past M (a ragged last tile) are clipped by the TMA
              // store: read nothing there
              const bool row_ok = y + lane < p.M;
              const uint4* ap = reinterpret_cast<const uint4*>(p.aux + int64_t(row_ok ? y + lane : y) * p.ld_aux + x);
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                float av[16], dv[16];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const uint4 a4 = row_ok ? __ldg(ap + 2 * h + u) : make_uint4(0u, 0u, 0u, 0u);
                  const uint32_t aw[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const __nv_bfloat162 ah = *reinterpret_cast<const __nv_bfloat162*>(&aw[e]);
                    av[8 * u + 2 * e] = __low2float(ah);
                    av[8 * u + 2 * e + 1] = __high2float(ah);
                  }
                }
                gelu_batch<16, 1>(av, dv);
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  __nv_bfloat162 hh = __floats2bfloat162_rn(__uint_as_float(r[16 * h + 2 * e]) * alpha * dv[2 * e],
                                                            __uint_as_float(r[16 * h + 2 * e + 1]) * alpha * dv[2 * e + 1]);
                  w[e] = *reinterpret_cast<uint32_t*>(&hh);
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const int j = 2 * h + u;
                  st_shared_v4(row_addr + (uint32_t(j ^ (lane & 7)) << 4), w[4 * u], w[4 * u + 1], w[4 * u + 2],
                               w[4 * u + 3]);
                }
              }
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (write && lane == 0) {
            if (p.accumulate) tma_reduce_add_4d(&tmC, buf, x, y, ti.zi, ti.zo);
            else tma_store_4d(&tmC, buf, x, y, ti.zi, ti.zo);
            if (ACT == 1) tma_store_4d(&tmC2, buf + 4096, x, y, ti.zi, ti.zo);
            bulk_commit();
          }
          ++chunk;
        }
        if (!empty_k) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) release_acc(ab);
          if (++ab == 2) { ab = 0; aphase ^= 1; }
        }
        continue;
      }
      const int64_t cbase = int64_t(ti.zo) * p.sc_outer + int64_t(ti.zi) * p.sc_inner + int64_t(row) * p.ldc;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        __syncwarp();
        if (!empty_k) {
          tmem_ld32(tbase + (uint32_t(q * 32) << 16) + uint32_t(ab * BN + c * 32), r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = 0u;
        }
        const int col0 = ti.n0 + c * 32;
        if (row >= p.M || col0 >= p.N) continue;
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) * alpha;
        const bool full_cols = col0 + 32 <= p.N;
        if (!p.c_bf16) {
          float* cp = static_cast<float*>(p.C) + cbase + col0;
          if (full_cols) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              float4 o = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
              if (p.accumulate) {
                const float4 old = *reinterpret_cast<const float4*>(cp + j);
                o.x += old.x; o.y += old.y; o.z += old.z; o.w += old.w;
              }
              *reinterpret_cast<float4*>(cp + j) = o;
            }
          } else {
            const int nrem = p.N - col0;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nrem) cp[j] = v[j] + (p.accumulate ? cp[j] : 0.f);
          }
        } else {
          bf16* cp = static_cast<bf16*>(p.C) + cbase + col0;
          if (full_cols) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              float o[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) o[e] = v[j + e];
              if (p.accumulate) {
                float old[8];
                Vec<bf16>::load(cp + j, old);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] += old[e];
              }
              Vec<bf16>::store(cp + j, o);
            }
          } else {
            const int nrem = p.N - col0;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nrem) cp[j] = __float2bfloat16_rn(v[j] + (p.accumulate ? __bfloat162float(cp[j]) : 0.f));
          }
        }
      }
      if (!empty_k) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release_acc(ab);
        if (++ab == 2) { ab = 0; aphase ^= 1; }
      }
    }
    if (p.tma_store && lane == 0) bulk_wait_all();  // staging smem must outlive the stores
  }

  __syncthreads();
  // a pair: neither CTA releases TMEM or exits while the other may still signal its barriers
  // or (the even CTA's MMAs) read its shared memory and write its TMEM
  if constexpr (CG == 2) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_cg<CG>(tbase, TCOLS);
  }
  if (p.prof_ts && threadIdx.x == 0) p.prof_ts[2 * blockIdx.x + 1] = global_ns();
}

}  // namespace gemm
}  // namespace xt
