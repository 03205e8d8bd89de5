// bf16 GEMM on CTA pairs (tcgen05 cta_group::2, clusters of two): 256-row tiles, each CTA
// staging its own 128 rows of A and half of the tile's B rows.
#include <mutex>

#include "gemm.cuh"

namespace xt {
namespace gemm {

template <int BN>
static int pick_major_pair(bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                           const CUtensorMap& tc2, const Params& p, int grid, cudaStream_t s) {
  if (!a_mn && !b_mn) return launch_one<kBf16, BN, false, false, 0, 2>(ta, tb, tc, tc2, p, grid, s);
  if (!a_mn && b_mn) return launch_one<kBf16, BN, false, true, 0, 2>(ta, tb, tc, tc2, p, grid, s);
  if (a_mn && !b_mn) return launch_one<kBf16, BN, true, false, 0, 2>(ta, tb, tc, tc2, p, grid, s);
  return launch_one<kBf16, BN, true, true, 0, 2>(ta, tb, tc, tc2, p, grid, s);
}

template <bool A_MN, bool B_MN>
static int launch_mc(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tc2,
                     const Params& p, int grid, cudaStream_t s) {
  return launch_one<kBf16, 256, A_MN, B_MN, 0, 2, 2>(ta, tb, tc, tc2, p, grid, s);
}

int launch_bf16_pair(int bn, int mc, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                     const CUtensorMap& tc, const CUtensorMap& tc2, const Params& p, int grid, cudaStream_t s) {
  if (mc == 2) {
    if (bn != 256) return fail(XT_ERR_UNSUPPORTED, "gemm: multicast pairs need tile width 256");
    if (!a_mn && !b_mn) return launch_mc<false, false>(ta, tb, tc, tc2, p, grid, s);
    if (!a_mn && b_mn) return launch_mc<false, true>(ta, tb, tc, tc2, p, grid, s);
    if (a_mn && !b_mn) return launch_mc<true, false>(ta, tb, tc, tc2, p, grid, s);
    return launch_mc<true, true>(ta, tb, tc, tc2, p, grid, s);
  }
  switch (bn) {
    case 128: return pick_major_pair<128>(a_mn, b_mn, ta, tb, tc, tc2, p, grid, s);
    case 192:  // 96 rows of B per CTA: K-major B only
      if (b_mn) return fail(XT_ERR_UNSUPPORTED, "gemm: paired tile width 192 needs B K-major");
      return a_mn ? launch_one<kBf16, 192, true, false, 0, 2>(ta, tb, tc, tc2, p, grid, s)
                  : launch_one<kBf16, 192, false, false, 0, 2>(ta, tb, tc, tc2, p, grid, s);
    case 256: return pick_major_pair<256>(a_mn, b_mn, ta, tb, tc, tc2, p, grid, s);
    default: return fail(XT_ERR_UNSUPPORTED, "gemm: paired tile width %d", bn);
  }
}

// Every paired instantiation has the same block size and (within 1 KB) shared memory, so the
// widest one stands for all of them; `mc` selects the cluster size (2·mc CTAs).
static int capacity(int mc) {
  static std::mutex mu;
  static int cap[2][64];
  static bool known[2][64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!known[mc - 1][dev]) {
    auto k = mc == 2 ? gemm_kernel<kBf16, 256, false, false, 0, 2, 2> : gemm_kernel<kBf16, 256, false, false, 0, 2>;
    constexpr int smem = Cfg<kBf16, 256, 2>::SMEM;
    int n = 0;
    bool err = true;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = unsigned(2 * mc);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(unsigned(num_sms() & ~(2 * mc - 1)));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = smem;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      err = cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess;
    }
    if (err) {
      n = 0;
      cudaGetLastError();  // a failed query leaves no launch error behind for the next check
    }
    cap[mc - 1][dev] = n > 0 ? n : 0;
    known[mc - 1][dev] = true;
  }
  return cap[mc - 1][dev];
}

int pair_capacity() { return capacity(1); }
int mc_capacity() { return capacity(2); }

}  // namespace gemm
}  // namespace xt
