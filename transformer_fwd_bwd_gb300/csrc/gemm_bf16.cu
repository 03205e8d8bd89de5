// bf16 × bf16 → fp32-accumulated GEMM instantiations (tcgen05 kind::f16).
#include "gemm.cuh"

namespace xt {
namespace gemm {

template <int BN>
static int pick_major(bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                      const CUtensorMap& tc2, const Params& p, int grid, cudaStream_t s) {
  if (!a_mn && !b_mn) return launch_one<false, BN, false, false>(ta, tb, tc, tc2, p, grid, s);
  if (!a_mn && b_mn) return launch_one<false, BN, false, true>(ta, tb, tc, tc2, p, grid, s);
  if (a_mn && !b_mn) return launch_one<false, BN, true, false>(ta, tb, tc, tc2, p, grid, s);
  return launch_one<false, BN, true, true>(ta, tb, tc, tc2, p, grid, s);
}

int launch_bf16(int bn, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                const CUtensorMap& tc, const CUtensorMap& tc2, const Params& p, int grid, cudaStream_t s) {
  switch (bn) {
    case 64: return pick_major<64>(a_mn, b_mn, ta, tb, tc, tc2, p, grid, s);
    case 128: return pick_major<128>(a_mn, b_mn, ta, tb, tc, tc2, p, grid, s);
    case 192: return pick_major<192>(a_mn, b_mn, ta, tb, tc, tc2, p, grid, s);
    case 256: return pick_major<256>(a_mn, b_mn, ta, tb, tc, tc2, p, grid, s);
    default: return fail(XT_ERR_UNSUPPORTED, "gemm: tile width %d", bn);
  }
}

}  // namespace gemm
}  // namespace xt
