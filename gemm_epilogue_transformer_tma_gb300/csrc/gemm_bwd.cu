// Backward GEMM instantiation: the second GEMM's data gradient with the
// RMSNorm backward (dh = g*acc - c*h, dg partial sums) in its epilogue.
#include "gemm_launch.cuh"

namespace coda {

namespace {
constexpr int kBN = 256;
}  // namespace

cudaError_t gemm_dgrad_rms(const LaunchCtx& c, const __nv_bfloat16* dP, const __nv_bfloat16* W2t,
                           const __nv_bfloat16* H, const __nv_bfloat16* g, const float* cvec, __nv_bfloat16* dH,
                           float* dgpart, int M, int N2, int d, const float* cpart, int Tc, const float* rstd) {
  // acc[m, k] = sum_n dP[m, n] W2t[n, k]: A = dP K-major (K = N2), B = W2t
  // stored [K][N] (MN-major).
  CUtensorMap ta, tb;
  if (!make_operand_maps(&ta, &tb, dP, false, W2t, true, M, d, N2, b_box_rows(c))) return cudaErrorInvalidValue;
  EpiDgradRms::Params ep{H, d, g, cvec, dH, d, dgpart, cpart, Tc, rstd, 1.0f / static_cast<float>(d)};
  return run_gemm<false, true, false, EpiDgradRms>(c, ta, tb, tb, M, d, N2, (d + kBN - 1) / kBN, ep);
}

}  // namespace coda

namespace coda {

cudaError_t gemm_dgrad_swiglu_bwd(const LaunchCtx& c, const __nv_bfloat16* dYb, const __nv_bfloat16* W3t,
                                  const __nv_bfloat16* z, const float* rstd, __nv_bfloat16* dP, float* cpart, int M,
                                  int d, int F, int T) {
  // dY[m, j] = sum_k dYb[m, k] W3t[k, j]: A = dYb K-major (K = d), B = W3t
  // stored [K][N] (MN-major), N = F gate columns
  CUtensorMap ta, tb;
  if (!make_operand_maps(&ta, &tb, dYb, false, W3t, true, M, F, d, b_box_rows(c))) return cudaErrorInvalidValue;
  EpiSwigluBwd::Params ep{z, rstd, dP, cpart, T, F};
  return run_gemm<false, true, false, EpiSwigluBwd>(c, ta, tb, tb, M, F, d, (F + 255) / 256, ep);
}

}  // namespace coda
