// QKV projection GEMM with the rotary-position-embedding epilogue.
#include "gemm_launch.cuh"

namespace coda {

cudaError_t gemm_qkv_rope(const LaunchCtx& c, const __nv_bfloat16* X, const __nv_bfloat16* Wqkv_t,
                          const float* cos_t, const float* sin_t, __nv_bfloat16* qkv, int M, int d, int N,
                          int rot_cols, int S) {
  // qkv[m, n] = sum_k X[m, k] Wqkv_t[n, k]: both operands K-major
  CUtensorMap ta, tb;
  if (!make_operand_maps(&ta, &tb, X, false, Wqkv_t, false, M, N, d, b_box_rows(c))) return cudaErrorInvalidValue;
  EpiRope::Params ep{};
  if (!make_tmap_store_bf16(&ep.out, qkv, N, M, N)) return cudaErrorInvalidValue;
  ep.cos_t = cos_t;
  ep.sin_t = sin_t;
  ep.S = S;
  ep.rot_cols = rot_cols;
  return run_gemm<false, false, false, EpiRope>(c, ta, tb, tb, M, N, d, (N + 255) / 256, ep);
}

}  // namespace coda
