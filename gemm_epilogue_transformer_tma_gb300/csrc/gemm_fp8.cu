// FP8 (e4m3, per-tensor scaled) forms of the forward GEMMs with the same
// epilogue programs: GEMM1 + residual + partial RMS, GEMM2 + row scale +
// SwiGLU.  kind::f8f6f4 MMAs, 128 e4m3 elements (128 bytes) per k-block row;
// the product of the two operands' scales is applied in the epilogue.
#include "gemm_launch.cuh"

namespace coda {

namespace {
constexpr int kBN = 256;

bool make_fp8_maps(CUtensorMap* ta, CUtensorMap* tb, const uint8_t* A, const uint8_t* B, int M, int N, int K,
                   int b_rows) {
  return make_tmap_u8(ta, A, K, M, K, 128, BM) && make_tmap_u8(tb, B, K, N, K, 128, b_rows);
}
}  // namespace

cudaError_t gemm_res_prms_fp8(const LaunchCtx& c0, const uint8_t* Xq, const float* sX, const uint8_t* W1q,
                              const float* sW1, const __nv_bfloat16* R, __nv_bfloat16* H, float* psum, int M, int K1,
                              int d, int T) {
  LaunchCtx c = c0;
  c.scale_a = sX;
  c.scale_b = sW1;
  CUtensorMap ta, tb;
  if (!make_fp8_maps(&ta, &tb, Xq, W1q, M, d, K1, b_box_rows(c))) return cudaErrorInvalidValue;
  EpiResPrms::Params ep{};
  if (!make_tmap_store_bf16(&ep.H, H, d, M, d)) return cudaErrorInvalidValue;
  ep.R = R;
  ep.ldr = d;
  ep.psum = psum;
  ep.T = T;
  return run_gemm<false, false, false, EpiResPrms, true>(c, ta, tb, tb, M, d, K1, (d + kBN - 1) / kBN, ep);
}

cudaError_t gemm_rowscale_swiglu_fp8(const LaunchCtx& c0, const uint8_t* Hq, const float* sH, const uint8_t* W2q,
                                     const float* sW2, const float* rstd, __nv_bfloat16* out, __nv_bfloat16* zsave,
                                     int M, int d, int N2, bool swiglu) {
  LaunchCtx c = c0;
  c.scale_a = sH;
  c.scale_b = sW2;
  CUtensorMap ta, tb, tb2;
  if (!swiglu) {
    if (!make_fp8_maps(&ta, &tb, Hq, W2q, M, N2, d, b_box_rows(c))) return cudaErrorInvalidValue;
    EpiStore::Params ep{};
    if (!make_tmap_store_bf16(&ep.out, out, N2, M, N2)) return cudaErrorInvalidValue;
    ep.row_scale = rstd;
    return run_gemm<false, false, false, EpiStore, true>(c, ta, tb, tb, M, N2, d, (N2 + kBN - 1) / kBN, ep);
  }
  const int F = N2 / 2;
  if (!make_tmap_u8(&ta, Hq, d, M, d, 128, BM)) return cudaErrorInvalidValue;
  if (!make_tmap_u8(&tb, W2q, d, F, d, 128, kBN / 2)) return cudaErrorInvalidValue;
  if (!make_tmap_u8(&tb2, W2q + static_cast<int64_t>(F) * d, d, F, d, 128, kBN / 2)) return cudaErrorInvalidValue;
  EpiRowscaleSwiglu::Params ep{};
  if (!make_tmap_store_bf16(&ep.out, out, F, M, F)) return cudaErrorInvalidValue;
  if (zsave != nullptr) {
    if (!make_tmap_store_bf16(&ep.zg, zsave, F, M, N2)) return cudaErrorInvalidValue;
    if (!make_tmap_store_bf16(&ep.zu, zsave + F, F, M, N2)) return cudaErrorInvalidValue;
  }
  ep.save_z = zsave != nullptr;
  ep.rstd = rstd;
  ep.F = F;
  return run_gemm<false, false, true, EpiRowscaleSwiglu, true>(c, ta, tb, tb2, M, F, d,
                                                               (F + kBN / 2 - 1) / (kBN / 2), ep);
}

}  // namespace coda
