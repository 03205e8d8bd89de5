// Host side of the tensor-core GEMM: TMA tensor maps, tile-shape choice, launch, and the
// matmul C ABI ([AE] op table row matmul: C = A@B; dA = d@Bᵀ, dB = Aᵀ@d).
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm.cuh"

namespace xt {
namespace gemm {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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
int make_operand_map(CUtensorMap* tm, const Operand& o, bool tf32, int box_mn) {
  auto enc = encode_fn();
  if (!enc) return fail(XT_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const int64_t e = tf32 ? 4 : 2;
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
    box[1] = atom;  // BK rows of K
  }
  dims[2] = cuuint64_t(o.batch_inner);
  dims[3] = cuuint64_t(o.batch_outer);
  box[2] = 1;
  box[3] = 1;
  const int64_t row_bytes = o.ld * e;
  strides[0] = cuuint64_t(row_bytes);
  strides[1] = cuuint64_t(o.batch_inner > 1 ? o.s_inner * e : row_bytes);
  strides[2] = cuuint64_t(o.batch_outer > 1 ? o.s_outer * e : row_bytes);
  CUresult r = enc(tm, tf32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                   const_cast<void*>(o.ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(XT_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return XT_OK;
}

// Tile width: fewest "wave-weighted" columns, with the lower per-FLOP efficiency of narrow
// tiles (shared-memory operand bandwidth) taken into account.
static int choose_bn(bool tf32, int64_t M, int64_t N, int64_t batches, int causal) {
  const int cands_bf16[3] = {64, 128, 256};
  const int cands_tf32[2] = {64, 128};
  const int* c = tf32 ? cands_tf32 : cands_bf16;
  const int nc = tf32 ? 2 : 3;
  const int sms = num_sms();
  int best = c[0];
  double best_cost = 1e300;
  for (int i = 0; i < nc; ++i) {
    const int bn = c[i];
    if (i > 0 && c[i - 1] >= N) break;  // wider tiles only add padding
    int64_t tiles = ceil_div(M, BM) * ceil_div(N, bn) * batches;
    if (causal == 1) tiles = (tiles + 1) / 2;
    const double waves = double(ceil_div(tiles, sms));
    const double eff = bn >= 256 ? 1.0 : bn >= 128 ? 0.9 : 0.7;
    const double cost = waves * double(bn) / eff;
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

int run(const Problem& pb, cudaStream_t s) {
  const bool tf32 = pb.tf32;
  const int bn = choose_bn(tf32, pb.M, pb.N, int64_t(pb.batch_outer) * pb.batch_inner, pb.causal);
  CUtensorMap ta, tb;
  XT_TRY(make_operand_map(&ta, pb.A, tf32, BM));
  XT_TRY(make_operand_map(&tb, pb.B, tf32, bn));
  Params p{};
  p.M = int(pb.M);
  p.N = int(pb.N);
  p.K = int(pb.K);
  p.num_m = int(ceil_div(pb.M, BM));
  p.num_n = int(ceil_div(pb.N, bn));
  p.batch_inner = pb.batch_inner;
  p.batches = pb.batch_inner * pb.batch_outer;
  p.causal = pb.causal;
  p.accumulate = pb.accumulate;
  p.c_bf16 = pb.c_bf16;
  p.alpha = pb.alpha;
  p.C = pb.C;
  p.ldc = pb.ldc;
  p.sc_inner = pb.sc_inner;
  p.sc_outer = pb.sc_outer;
  p.flag = errflag();
  const int64_t tiles = int64_t(p.num_m) * p.num_n * p.batches;
  if (tiles > int64_t(1) << 30) return fail(XT_ERR_UNSUPPORTED, "matmul: too many tiles");
  int grid = int(tiles < num_sms() ? tiles : num_sms());
  if (grid < 1) grid = 1;
  const bool amn = pb.A.mn_major, bmn = pb.B.mn_major;
  if (tf32) return launch_tf32(bn, amn, bmn, ta, tb, p, grid, s);
  return launch_bf16(bn, amn, bmn, ta, tb, p, grid, s);
}

}  // namespace gemm

// Validates and runs C[M,N] (+)= alpha · op(A) @ op(B) for one matmul descriptor.
static int matmul_run(const xt_matmul_desc* d, const void* A, const void* B, void* C, cudaStream_t s) {
  XT_REQUIRE(d != nullptr, "matmul: desc is NULL");
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
  pb.A = gemm::Operand{A, d->trans_a == 1, d->M, d->K, d->lda, d->stride_a_inner, d->stride_a_outer,
                       d->batch_inner, d->batch_outer};
  // op(B) is K×N; the kernel's B operand is N rows by K: K-major iff B is stored [N, K].
  pb.B = gemm::Operand{B, d->trans_b == 0, d->N, d->K, d->ldb, d->stride_b_inner, d->stride_b_outer,
                       d->batch_inner, d->batch_outer};
  pb.C = C;
  pb.ldc = d->ldc;
  pb.sc_inner = d->stride_c_inner;
  pb.sc_outer = d->stride_c_outer;
  pb.c_bf16 = d->dtype_c == XT_BF16;
  pb.alpha = d->alpha;
  pb.accumulate = d->accumulate;
  pb.causal = d->causal;
  return gemm::run(pb, s);
}

}  // namespace xt

using namespace xt;

extern "C" {

int xt_matmul_fwd(const xt_matmul_desc* desc, const void* A, const void* B, void* C, void* stream) {
  return matmul_run(desc, A, B, C, as_stream(stream));
}

int xt_matmul_bwd(const xt_matmul_desc* desc, const void* A, const void* B, const void* dC, void* dA, void* dB,
                  int dt_grad_a, int dt_grad_b, int acc_a, int acc_b, void* stream) {
  XT_REQUIRE(desc != nullptr, "xt_matmul_bwd: desc is NULL");
  XT_REQUIRE(desc->causal == 0, "xt_matmul_bwd: causal must be 0");
  XT_REQUIRE(!dA || valid_dtype(dt_grad_a), "xt_matmul_bwd: bad dt_grad_a");
  XT_REQUIRE(!dB || valid_dtype(dt_grad_b), "xt_matmul_bwd: bad dt_grad_b");
  const xt_matmul_desc& f = *desc;
  cudaStream_t s = as_stream(stream);
  if (dA) {
    xt_matmul_desc g{};
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
      XT_TRY(matmul_run(&g, dC, B, dA, s));
    } else {  // A stored [K,M]: dA = op(B) @ dCᵀ
      g.M = f.K; g.N = f.M; g.K = f.N;
      g.trans_a = f.trans_b; g.lda = f.ldb; g.stride_a_inner = f.stride_b_inner; g.stride_a_outer = f.stride_b_outer;
      g.trans_b = 1; g.ldb = f.ldc; g.stride_b_inner = f.stride_c_inner; g.stride_b_outer = f.stride_c_outer;
      g.ldc = f.lda; g.stride_c_inner = f.stride_a_inner; g.stride_c_outer = f.stride_a_outer;
      XT_TRY(matmul_run(&g, B, dC, dA, s));
    }
  }
  if (dB) {
    xt_matmul_desc g{};
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
      XT_TRY(matmul_run(&g, A, dC, dB, s));
    } else {  // B stored [N,K]: dB = dCᵀ @ op(A)
      g.M = f.N; g.N = f.K; g.K = f.M;
      g.trans_a = 1; g.lda = f.ldc; g.stride_a_inner = f.stride_c_inner; g.stride_a_outer = f.stride_c_outer;
      g.trans_b = f.trans_a; g.ldb = f.lda; g.stride_b_inner = f.stride_a_inner; g.stride_b_outer = f.stride_a_outer;
      g.ldc = f.ldb; g.stride_c_inner = f.stride_b_inner; g.stride_c_outer = f.stride_b_outer;
      XT_TRY(matmul_run(&g, dC, A, dB, s));
    }
  }
  return XT_OK;
}

}  // extern "C"
