// LM-head GEMM instantiations: blocked log-sum-exp statistics epilogue and the
// softmax-gradient epilogue (logits never leave the chip).
#include "gemm_launch.cuh"

namespace coda {

namespace {
constexpr int kBN = 256;
}  // namespace

int ce_tile_cols() { return PART_COLS; }

cudaError_t gemm_ce_stats(const LaunchCtx& c, const __nv_bfloat16* H, const __nv_bfloat16* Wt, const int32_t* labels,
                          float* pmax, float* psum, int32_t* parg, float* zy, int M, int d, int V, int T) {
  CUtensorMap ta, tb;
  if (!make_operand_maps(&ta, &tb, H, false, Wt, false, M, V, d, b_box_rows(c))) return cudaErrorInvalidValue;
  EpiCeStats::Params ep{labels, pmax, psum, parg, zy, T, c.status};
  return run_gemm<false, false, false, EpiCeStats>(c, ta, tb, tb, M, V, d, (V + kBN - 1) / kBN, ep);
}

cudaError_t gemm_ce_grad(const LaunchCtx& c, const __nv_bfloat16* H, const __nv_bfloat16* Wt_chunk,
                         const int32_t* labels, const float* lse, __nv_bfloat16* dL, int M, int d, int Vc, int v0,
                         float inv_M) {
  CUtensorMap ta, tb;
  if (!make_operand_maps(&ta, &tb, H, false, Wt_chunk, false, M, Vc, d, b_box_rows(c))) return cudaErrorInvalidValue;
  EpiCeGrad::Params ep{};
  if (!make_tmap_store_bf16(&ep.dL, dL, Vc, M, Vc)) return cudaErrorInvalidValue;
  ep.labels = labels;
  ep.lse = lse;
  ep.inv_M = inv_M;
  ep.v0 = v0;
  return run_gemm<false, false, false, EpiCeGrad>(c, ta, tb, tb, M, Vc, d, (Vc + kBN - 1) / kBN, ep);
}

}  // namespace coda
