// Host-side launch of one gemm_tc_kernel instantiation: tile counts,
// shared-memory opt-in, persistent grid of at most one CTA per SM.
#pragma once

#include <algorithm>

#include "coda_internal.h"
#include "gemm_tc.cuh"

namespace coda {

template <int BN, int STAGES, bool A_MN, bool B_MN, bool B_DUAL, class Epi>
cudaError_t launch_gemm_kernel(const LaunchCtx& c, const CUtensorMap& ta, const CUtensorMap& tb,
                               const CUtensorMap& tb2, int M, int N, int K, int tiles_n,
                               const typename Epi::Params& ep) {
  using L = GemmSmem<BN, STAGES>;
  auto kern = gemm_tc_kernel<BN, STAGES, A_MN, B_MN, B_DUAL, Epi>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
  if (e != cudaSuccess) return e;
  GemmShape sh;
  sh.M = M;
  sh.N = N;
  sh.K = K;
  sh.tiles_m = (M + BM - 1) / BM;
  sh.tiles_n = tiles_n;
  sh.num_kb = (K + BK - 1) / BK;
  sh.group_m = 8;
  KernelCtl ctl{c.status, c.timeout_ns, c.skip_first_stage};
  const int tiles = sh.tiles_m * sh.tiles_n;
  const int grid = std::max(1, std::min(tiles, c.num_sms));
  kern<<<grid, GEMM_THREADS, L::TOTAL, c.stream>>>(ta, tb, tb2, sh, ctl, ep);
  return cudaGetLastError();
}

// Tensor maps for the two operands given their majors.
inline bool make_operand_maps(CUtensorMap* ta, CUtensorMap* tb, const __nv_bfloat16* A, bool a_mn,
                              const __nv_bfloat16* B, bool b_mn, int M, int N, int K, int BN) {
  bool ok;
  if (!a_mn)
    ok = make_tmap_bf16(ta, A, K, M, K, 64, BM);   // [M][K], box 64(K) x 128(M)
  else
    ok = make_tmap_bf16(ta, A, M, K, M, 64, 64);   // [K][M], box 64(M) x 64(K)
  if (!ok) return false;
  if (!b_mn)
    ok = make_tmap_bf16(tb, B, K, N, K, 64, BN);   // [N][K], box 64(K) x BN(N)
  else
    ok = make_tmap_bf16(tb, B, N, K, N, 64, 64);   // [K][N], box 64(N) x 64(K)
  return ok;
}

}  // namespace coda
