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
  EpiDgradRms::Params ep{};
  if (!make_tmap_store_bf16(&ep.dH, dH, d, M, d)) return cudaErrorInvalidValue;
  ep.H = H;
  ep.ldh = d;
  ep.g = g;
  ep.c = cvec;
  ep.dgpart = dgpart;
  ep.cpart = cpart;
  ep.Tc = Tc;
  ep.rstd = rstd;
  ep.inv_d = 1.0f / static_cast<float>(d);
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
  EpiSwigluBwd::Params ep{};
  if (!make_tmap_store_bf16(&ep.dPg, dP, F, M, 2 * static_cast<uint64_t>(F))) return cudaErrorInvalidValue;
  if (!make_tmap_store_bf16(&ep.dPu, dP + F, F, M, 2 * static_cast<uint64_t>(F))) return cudaErrorInvalidValue;
  ep.z = z;
  ep.rstd = rstd;
  ep.cpart = cpart;
  ep.T = T;
  ep.F = F;
  return run_gemm<false, true, false, EpiSwigluBwd>(c, ta, tb, tb, M, F, d, (F + 255) / 256, ep);
}

}  // namespace coda
