// Internal interface between the GEMM host code and its kernel instantiations.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "gemm_kernel.cuh"

namespace xt {
namespace gemm {

// One operand as the kernel reads it: `mn` rows (M for A, N for B) by K.
// mn_major = false: K contiguous (element (i, k) at ptr + i·ld + k);
// mn_major = true:  MN contiguous (element (i, k) at ptr + k·ld + i).
struct Operand {
  const void* ptr;
  bool mn_major;
  int64_t mn, K, ld, s_inner, s_outer;
  int batch_inner, batch_outer;
};

struct Problem {
  bool tf32;
  bool fp8;              // e4m3 operands (K-major), kind::f8f6f4
  const float* scale_a;  // device per-tensor factors multiplying alpha (may be null)
  const float* scale_b;
  int64_t M, N, K;
  int batch_inner, batch_outer;
  Operand A, B;
  void* C;
  int64_t ldc, sc_inner, sc_outer;
  int c_bf16;
  float alpha;
  int accumulate;
  int causal;
  void* split_ws;  // room for K-split or stream-K partial tiles (may be null)
  size_t split_ws_bytes;
  uint32_t* sk_flags;  // kSkFlagBytes of stream-K flag words, zero between calls (null: no stream-K)
  int act;         // GELU epilogue (see Params::act); 0 none
  void* C2;        // act 1: gelu(C), C's layout
  const void* aux; // act 2: the pre-activation, C's layout
};

// Tile width, K split and schedule chosen for a problem (see choose()).
struct Choice {
  int bn;
  int splits;
  int sk;      // stream-K schedule: 1 over every SM (every resident unit), 2 in lockstep K slices
  int grid;    // stream-K units: the SMs (or pairs), or tiles × K slices (lockstep)
  int cg = 1;  // 2: the paired-CTA kernel, tiles of 2·BM rows, units are CTA pairs
  int mc = 1;  // 2 (with cg 2): clusters of two pairs sharing B by multicast, units are clusters
};
Choice choose(bool tf32, int64_t M, int64_t N, int64_t K, int64_t batches, int causal, bool allow_split,
              bool fp8, bool b_mn);
size_t split_bytes(const Choice& c, int64_t M, int64_t N);

// Stream-K flag words at the head of every matmul workspace: 4 per CTA for up to kSkMaxCtas CTAs.
constexpr int kSkMaxCtas = 256;
constexpr size_t kSkFlagBytes = size_t(kSkMaxCtas) * 4 * sizeof(uint32_t);

// kind: kBf16, kTf32 or kFp8 (element size 2, 4, 1)
int make_operand_map(CUtensorMap* tm, const Operand& o, int kind, int box_mn, int k_atom_count);
// The driver's cuTensorMapEncodeTiled (null when the driver does not provide it).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();
int run(const Problem& pb, cudaStream_t s);
int launch_bf16(int bn, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                const CUtensorMap& tc2, const Params& p, int grid, cudaStream_t s);
int launch_tf32(int bn, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                const CUtensorMap& tc2, const Params& p, int grid, cudaStream_t s);
// fp8 e4m3, K-major operands, BN 128 or 256.
int launch_fp8(int bn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tc2,
               const Params& p, int grid, cudaStream_t s);
// bf16, BN 256, with the GELU epilogue `act` (1 or 2).
int launch_bf16_act(int act, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                    const CUtensorMap& tc2, const Params& p, int grid, cudaStream_t s);

template <int KIND, int BN, bool A_MN, bool B_MN, int ACT = 0, int CG = 1, int MC = 1>
int launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tc2,
               const Params& p, int grid, cudaStream_t s) {
  auto k = gemm_kernel<KIND, BN, A_MN, B_MN, ACT, CG, MC>;
  constexpr int smem = Cfg<KIND, BN, CG>::SMEM;
  static bool attr_set = false;  // per instantiation; idempotent if raced
  if (!attr_set) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return check_launch("gemm: shared memory attribute");
    if (CG == 2 && cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) != cudaSuccess)
      return check_launch("gemm: cluster attribute");
    attr_set = true;
  }
  if constexpr (CG == 2) {
    if (grid % (CG * MC)) return fail(XT_ERR_INVALID_ARG, "gemm: clustered launch needs whole clusters");
    launch_clustered(k, grid, kThreads, smem, s, CG * MC, ta, tb, tc, tc2, p);
  } else {
    launch(k, grid, kThreads, smem, s, ta, tb, tc, tc2, p);
  }
  return check_launch("gemm kernel");
}

// bf16 paired-CTA GEMM (BN 128, 256, or 192 with B K-major; plain epilogue), launched as
// clusters of two, or with mc = 2 (BN 256) as clusters of two pairs sharing B by multicast.
int launch_bf16_pair(int bn, int mc, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                     const CUtensorMap& tc, const CUtensorMap& tc2, const Params& p, int grid, cudaStream_t s);
// CTA pairs of the paired kernel that can be resident at once on the current device (0 if none).
int pair_capacity();
// Clusters of two pairs (the multicast form) that can be resident at once (0 if none).
int mc_capacity();

}  // namespace gemm
}  // namespace xt
