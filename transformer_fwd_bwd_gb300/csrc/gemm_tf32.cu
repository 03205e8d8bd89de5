// fp32 operands read as tf32, fp32-accumulated GEMM instantiations (tcgen05 kind::tf32).
#include "gemm.cuh"

namespace xt {
namespace gemm {

// tf32 operands are always K-major here: MN-major fp32 operands are staged K-major by the
// host side first (the tf32 MMA is fed K-major operands only).
template <int BN>
static int pick_major(bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                      const CUtensorMap& tc2, const Params& p, int grid, cudaStream_t s) {
  if (a_mn || b_mn) return fail(XT_ERR_UNSUPPORTED, "gemm: tf32 operands must be K-major");
  return launch_one<true, BN, false, false>(ta, tb, tc, tc2, p, grid, s);
}

int launch_tf32(int bn, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                const CUtensorMap& tc, const CUtensorMap& tc2, const Params& p, int grid, cudaStream_t s) {
  switch (bn) {
    case 64: return pick_major<64>(a_mn, b_mn, ta, tb, tc, tc2, p, grid, s);
    case 128: return pick_major<128>(a_mn, b_mn, ta, tb, tc, tc2, p, grid, s);
    default: return fail(XT_ERR_UNSUPPORTED, "gemm: tile width %d", bn);
  }
}

}  // namespace gemm
}  // namespace xt
