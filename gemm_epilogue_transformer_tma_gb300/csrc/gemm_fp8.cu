// FP8 (per-tensor scaled e4m3 / e5m2) forms of the GEMMs with the same
// epilogue programs: GEMM1 + residual + partial RMS, GEMM2 + row scale +
// SwiGLU, and the plain store used by the backward.  kind::f8f6f4 MMAs, 128
// 8-bit elements (128 bytes) per k-block row; the product of the two
// operands' scales is applied in the epilogue.
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

// Tensor map of an 8-bit operand: K-major [rows][K] with boxes of 128 K x
// box_rows, or MN-major [K][mn] with boxes of 128 (M/N) x 128 (K).
bool make_f8_operand_map(CUtensorMap* m, const uint8_t* p, bool mn_major, int mn, int K, int box_rows) {
  if (!mn_major) return make_tmap_u8(m, p, K, mn, K, 128, box_rows);
  return make_tmap_u8(m, p, mn, K, mn, 128, 128);
}

cudaError_t gemm_store_fp8(const LaunchCtx& c0, const uint8_t* A, bool a_mn, int a_fmt, const float* sA,
                           const uint8_t* B, bool b_mn, int b_fmt, const float* sB, __nv_bfloat16* C, int M, int N,
                           int K, const float* row_scale, const __nv_bfloat16* col_scale) {
  LaunchCtx c = c0;
  c.scale_a = sA;
  c.scale_b = sB;
  c.f8_fmt = f8_format_bits(a_fmt, b_fmt);
  CUtensorMap ta, tb;
  if (!make_f8_operand_map(&ta, A, a_mn, M, K, BM)) return cudaErrorInvalidValue;
  if (!make_f8_operand_map(&tb, B, b_mn, N, K, b_box_rows(c))) return cudaErrorInvalidValue;
  EpiStore::Params ep{};
  if (!make_tmap_store_bf16(&ep.out, C, N, M, N)) return cudaErrorInvalidValue;
  ep.row_scale = row_scale;
  ep.col_scale = col_scale;
  const int tn = (N + kBN - 1) / kBN;
  if (!a_mn && !b_mn) return run_gemm<false, false, false, EpiStore, true>(c, ta, tb, tb, M, N, K, tn, ep);
  if (!a_mn && b_mn) return run_gemm<false, true, false, EpiStore, true>(c, ta, tb, tb, M, N, K, tn, ep);
  if (a_mn && b_mn) return run_gemm<true, true, false, EpiStore, true>(c, ta, tb, tb, M, N, K, tn, ep);
  return cudaErrorNotSupported;  // MN-major A with K-major B is not used on this path
}

cudaError_t gemm_dgrad_rms_fp8(const LaunchCtx& c0, const uint8_t* dPq, int dp_fmt, const float* sdP,
                               const uint8_t* W2q, int w_fmt, const float* sW2, const __nv_bfloat16* H,
                               const __nv_bfloat16* g, const float* cvec, __nv_bfloat16* dH, float* dgpart, int M,
                               int N2, int d) {
  LaunchCtx c = c0;
  c.scale_a = sdP;
  c.scale_b = sW2;
  c.f8_fmt = f8_format_bits(dp_fmt, w_fmt);
  // acc[m, k] = sum_n dP[m, n] W2t[n, k]: A = dP codes K-major (K = N2), B =
  // W2t codes stored [K][N] (MN-major)
  CUtensorMap ta, tb;
  if (!make_f8_operand_map(&ta, dPq, false, M, N2, BM)) return cudaErrorInvalidValue;
  if (!make_f8_operand_map(&tb, W2q, true, d, N2, b_box_rows(c))) return cudaErrorInvalidValue;
  EpiDgradRms::Params ep{};
  if (!make_tmap_store_bf16(&ep.dH, dH, d, M, d)) return cudaErrorInvalidValue;
  ep.H = H;
  ep.ldh = d;
  ep.g = g;
  ep.c = cvec;
  ep.dgpart = dgpart;
  ep.inv_d = 1.0f / static_cast<float>(d);
  return run_gemm<false, true, false, EpiDgradRms, true>(c, ta, tb, tb, M, d, N2, (d + kBN - 1) / kBN, ep);
}

// LM-head statistics GEMM on e4m3 operands: logits = sH * sW * (Hq Wq^T),
// the blocked log-sum-exp epilogue as in the bf16 form.
cudaError_t gemm_ce_stats_fp8(const LaunchCtx& c0, const uint8_t* Hq, const float* sH, const uint8_t* Wq,
                              const float* sW, const int32_t* labels, float* pmax, float* psum, int32_t* parg,
                              float* zy, int M, int d, int V, int T) {
  LaunchCtx c = c0;
  c.scale_a = sH;
  c.scale_b = sW;
  c.f8_fmt = f8_format_bits(0, 0);
  CUtensorMap ta, tb;
  if (!make_fp8_maps(&ta, &tb, Hq, Wq, M, V, d, b_box_rows(c))) return cudaErrorInvalidValue;
  EpiCeStats::Params ep{labels, pmax, psum, parg, zy, T, c.status};
  return run_gemm<false, false, false, EpiCeStats, true>(c, ta, tb, tb, M, V, d, (V + kBN - 1) / kBN, ep);
}

// The recomputed logits of one vocabulary chunk on e4m3 operands, dL written
// as e5m2 codes of dL * code_inv into dLq [M][Vc].
cudaError_t gemm_ce_grad_fp8(const LaunchCtx& c0, const uint8_t* Hq, const float* sH, const uint8_t* Wq_chunk,
                             const float* sW, const int32_t* labels, const float* lse, uint8_t* dLq, float code_inv,
                             int M, int d, int Vc, int v0, float inv_M) {
  LaunchCtx c = c0;
  c.scale_a = sH;
  c.scale_b = sW;
  c.f8_fmt = f8_format_bits(0, 0);
  CUtensorMap ta, tb;
  if (!make_fp8_maps(&ta, &tb, Hq, Wq_chunk, M, Vc, d, b_box_rows(c))) return cudaErrorInvalidValue;
  EpiCeGrad::Params ep{};
  if (!make_tmap_store_u8_sw32(&ep.dL, dLq, Vc, M, Vc)) return cudaErrorInvalidValue;
  ep.labels = labels;
  ep.lse = lse;
  ep.inv_M = inv_M;
  ep.v0 = v0;
  ep.codes = 1;
  ep.code_inv = code_inv;
  return run_gemm<false, false, false, EpiCeGrad, true>(c, ta, tb, tb, M, Vc, d, (Vc + kBN - 1) / kBN, ep);
}

// The chunk's two gradient GEMMs on the e5m2 dL codes (scale s_dL, known on
// the host) and the e4m3 codes of W and H:
//   dH32 [M][d] (+)= s_dL * sW * dLq Wq_chunk    (dLq K-major, Wq_chunk [Vc][d] read MN-major)
//   dWc [Vc][d] = s_dL * sH * dLq^T Hq           (both read MN-major, K = M)
cudaError_t gemm_ce_bwd_fp8(const LaunchCtx& c0, const uint8_t* dLq, float s_dL, const uint8_t* Wq_chunk,
                            const float* sW, const uint8_t* Hq, const float* sH, float* dH32, bool accumulate,
                            __nv_bfloat16* dWc, int M, int d, int Vc) {
  LaunchCtx c = c0;
  c.scale_a = nullptr;
  c.scale_host = s_dL;
  c.scale_b = sW;
  c.f8_fmt = f8_format_bits(1, 0);
  CUtensorMap ta, tb;
  if (!make_f8_operand_map(&ta, dLq, false, M, Vc, BM)) return cudaErrorInvalidValue;
  if (!make_f8_operand_map(&tb, Wq_chunk, true, d, Vc, b_box_rows(c))) return cudaErrorInvalidValue;
  EpiStoreF32::Params e0{};
  if (!make_tmap_store_f32(&e0.out, dH32, d, M, d)) return cudaErrorInvalidValue;
  e0.beta = accumulate ? 1 : 0;
  const int tn = (d + kBN - 1) / kBN;
  cudaError_t e = run_gemm<false, true, false, EpiStoreF32, true>(c, ta, tb, tb, M, d, Vc, tn, e0);
  if (e != cudaSuccess) return e;
  c.scale_b = sH;
  if (!make_f8_operand_map(&ta, dLq, true, Vc, M, BM)) return cudaErrorInvalidValue;
  if (!make_f8_operand_map(&tb, Hq, true, d, M, b_box_rows(c))) return cudaErrorInvalidValue;
  EpiStore::Params e1{};
  if (!make_tmap_store_bf16(&e1.out, dWc, d, Vc, d)) return cudaErrorInvalidValue;
  return run_gemm<true, true, false, EpiStore, true>(c, ta, tb, tb, Vc, d, M, tn, e1);
}

}  // namespace coda
