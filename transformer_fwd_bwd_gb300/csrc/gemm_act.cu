// bf16 GEMM instantiations with the GELU epilogue (BN 256): act 1 stores the pre-activation
// and its GELU, act 2 multiplies the product by GELU' of a saved pre-activation.
#include "gemm.cuh"

namespace xt {
namespace gemm {

template <int ACT>
static int pick_major_act(bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                          const CUtensorMap& tc2, const Params& p, int grid, cudaStream_t s) {
  if (!a_mn && !b_mn) return launch_one<false, 256, false, false, ACT>(ta, tb, tc, tc2, p, grid, s);
  if (!a_mn && b_mn) return launch_one<false, 256, false, true, ACT>(ta, tb, tc, tc2, p, grid, s);
  if (a_mn && !b_mn) return launch_one<false, 256, true, false, ACT>(ta, tb, tc, tc2, p, grid, s);
  return launch_one<false, 256, true, true, ACT>(ta, tb, tc, tc2, p, grid, s);
}

int launch_bf16_act(int act, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                    const CUtensorMap& tc2, const Params& p, int grid, cudaStream_t s) {
  if (act == 1) return pick_major_act<1>(a_mn, b_mn, ta, tb, tc, tc2, p, grid, s);
  if (act == 2) return pick_major_act<2>(a_mn, b_mn, ta, tb, tc, tc2, p, grid, s);
  return fail(XT_ERR_UNSUPPORTED, "gemm: epilogue mode %d", act);
}

}  // namespace gemm
}  // namespace xt
