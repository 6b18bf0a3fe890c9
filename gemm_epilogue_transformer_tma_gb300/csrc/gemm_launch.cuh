// Host-side launch of one gemm_tc_kernel instantiation: tile counts,
// shared-memory opt-in, persistent grid of at most one CTA per SM.
#pragma once

#include <algorithm>

#include "coda_internal.h"
#include "gemm_tc.cuh"
#include "gemm_tc2.cuh"
#include "gemm_tc2w.cuh"

namespace coda {

template <int BN, int STAGES, bool A_MN, bool B_MN, bool B_DUAL, class Epi, bool FP8 = false>
cudaError_t launch_gemm_kernel(const LaunchCtx& c, const CUtensorMap& ta, const CUtensorMap& tb,
                               const CUtensorMap& tb2, int M, int N, int K, int tiles_n,
                               const typename Epi::Params& ep) {
  using L = GemmSmem<BN, STAGES, epi_stage_bytes<Epi>()>;
  auto kern = gemm_tc_kernel<BN, STAGES, A_MN, B_MN, B_DUAL, Epi, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
  if (e != cudaSuccess) return e;
  GemmShape sh;
  sh.M = M;
  sh.N = N;
  sh.K = K;
  sh.tiles_m = (M + BM - 1) / BM;
  sh.tiles_n = tiles_n;
  sh.num_kb = (K + (FP8 ? 128 : BK) - 1) / (FP8 ? 128 : BK);
  sh.group_m = 8;
  KernelCtl ctl{c.status, c.timeout_ns, c.skip_first_stage, c.scale_a, c.scale_b, c.f8_fmt, c.scale_host};
  const int tiles = sh.tiles_m * sh.tiles_n;
  sh.sk_first = tiles;  // the 1-SM kernel never splits tiles
  sh.sk_ranges = 1;
  const int grid = std::max(1, std::min(tiles, c.num_sms));
  return launch_chained(c, kern, dim3(grid), dim3(gemm_threads<Epi>()), L::TOTAL, ta, tb, tb2, sh, ctl, ep);
}

// The split of an SM-pair launch: the remainder tiles after the full waves
// (the last, partial wave) are each cut into `ranges` k-ranges, dealt
// range-major and round-robin to all clusters.  The count is the one that
// finishes the remainder in the fewest rounds, ceil(rem * ranges / clusters)
// k-ranges' time, against one whole round unsplit.  Ranges of fewer than
// kSplitMinRangeKb k-blocks are not used (the owner's reads of the other
// ranges' partials at the end of the launch would eat the gain), nor more
// than kSplitMaxRanges, nor more partial slots than the scratch has.
constexpr int kSplitMaxRanges = kMaxSplitParts + 1;
constexpr int kSplitMinRangeKb = 48;
struct SplitPlan {
  int first;   // first split tile (tiles: no split)
  int ranges;  // k-ranges per split tile (1: no split)
};
inline SplitPlan split_plan(int tiles, int num_kb, int clusters, int slots) {
  SplitPlan plan{tiles, 1};
  if (clusters < 2 || tiles < 1) return plan;
  const int rem = tiles % clusters;
  if (rem == 0) return plan;
  // rounds of ranges for the remainder, compared as best_rounds / best
  int best = 1, best_rounds = 1;
  for (int r = 2; r <= kSplitMaxRanges && num_kb / r >= kSplitMinRangeKb; ++r) {
    const int rounds = (rem * r + clusters - 1) / clusters;  // in units of 1/r of a round
    if (rounds * best < best_rounds * r) {
      best = r;
      best_rounds = rounds;
    }
  }
  if (best < 2 || rem * (best - 1) > slots) return plan;
  plan.first = tiles - rem;
  plan.ranges = best;
  return plan;
}

// Co-resident SM pairs of one pair-kernel instantiation on the current
// device (not every TPC need have both SMs enabled), queried once into
// `cached` (one slot per device, owned by the calling launcher instantiation).
inline cudaError_t pair_capacity(const void* kern, int threads, int smem, int num_sms, int (&cached)[64], int* pairs) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (cached[dev] == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    cached[dev] = std::max(1, std::min(n, num_sms / 2));
  }
  *pairs = cached[dev];
  return cudaSuccess;
}

template <int BN, int STAGES, bool A_MN, bool B_MN, bool B_DUAL, class Epi, bool FP8 = false>
cudaError_t launch_gemm2_kernel(const LaunchCtx& c, const CUtensorMap& ta, const CUtensorMap& tb,
                                const CUtensorMap& tb2, int M, int N, int K, int tiles_n,
                                const typename Epi::Params& ep) {
  using L = Gemm2Smem<BN, STAGES, epi_stage_bytes<Epi>()>;
  auto kern = gemm_tc2_kernel<BN, STAGES, A_MN, B_MN, B_DUAL, Epi, FP8, false>;
  auto kern_split = gemm_tc2_kernel<BN, STAGES, A_MN, B_MN, B_DUAL, Epi, FP8, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
  if (e != cudaSuccess) return e;
  GemmShape sh;
  sh.M = M;
  sh.N = N;
  sh.K = K;
  sh.tiles_m = (M + BM2 - 1) / BM2;
  sh.tiles_n = tiles_n;
  sh.num_kb = (K + (FP8 ? 128 : BK) - 1) / (FP8 ? 128 : BK);
  sh.group_m = 8;
  KernelCtl ctl{c.status, c.timeout_ns, c.skip_first_stage, c.scale_a, c.scale_b, c.f8_fmt, c.scale_host};
  static int cap[64] = {};        // per device, for this instantiation
  static int cap_split[64] = {};
  int pairs = 0;
  e = pair_capacity(reinterpret_cast<const void*>(kern), gemm_threads<Epi>(), L::TOTAL, c.num_sms, cap, &pairs);
  if (e != cudaSuccess) return e;
  const int tiles = sh.tiles_m * sh.tiles_n;
  sh.sk_first = tiles;
  sh.sk_ranges = 1;
  // split tiles only when a scratch is set, and only under 4-warp epilogue
  // programs (the partials are written per TMEM lane quadrant by one warp)
  if (c.sk_parts != nullptr && c.sk_flags != nullptr && Epi::kEpiWarps == 4) {
    int split_pairs = 0;
    e = pair_capacity(reinterpret_cast<const void*>(kern_split), gemm_threads<Epi>(), L::TOTAL, c.num_sms, cap_split,
                      &split_pairs);
    if (e != cudaSuccess) return e;
    const SplitPlan plan = split_plan(tiles, sh.num_kb, split_pairs, c.sk_slots);
    sh.sk_first = plan.first;
    sh.sk_ranges = plan.ranges;
    if (sh.sk_first < tiles) {
      ctl.sk_parts = c.sk_parts;
      ctl.sk_flags = c.sk_flags;
      return launch_chained(c, kern_split, dim3(2 * split_pairs), dim3(gemm_threads<Epi>()), L::TOTAL, ta, tb, tb2,
                            sh, ctl, ep);
    }
  }
  const int clusters = std::max(1, std::min(tiles, pairs));
  return launch_chained(c, kern, dim3(2 * clusters), dim3(gemm_threads<Epi>()), L::TOTAL, ta, tb, tb2, sh, ctl, ep);
}

// The wide-tile pair kernel (256 x 512 tiles, gemm_tc2w.cuh) on a persistent
// grid of all co-resident SM pairs.  tiles_n counts 256-column tiles and must
// be even.  When the last wave holds at most half as many wide tiles as there
// are pairs, its tiles run as 256-column halves.
template <bool A_MN, bool B_MN, class Epi>
cudaError_t launch_gemm2w_kernel(const LaunchCtx& c, const CUtensorMap& ta, const CUtensorMap& tb, int M, int N,
                                 int K, int tiles_n, const typename Epi::Params& ep) {
  constexpr int STAGES = 4;
  using L = Gemm2wSmem<STAGES, epi_stage_bytes<Epi>()>;
  auto kern = gemm_tc2w_kernel<STAGES, A_MN, B_MN, Epi>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
  if (e != cudaSuccess) return e;
  GemmShape sh;
  sh.M = M;
  sh.N = N;
  sh.K = K;
  sh.tiles_m = (M + BM2 - 1) / BM2;
  sh.tiles_n = tiles_n;
  sh.num_kb = (K + BK - 1) / BK;
  sh.group_m = 8;
  sh.sk_first = sh.tiles_m * sh.tiles_n;
  sh.sk_ranges = 1;
  sh.w_lead = c.wide_lead;
  static int cap[64] = {};  // per device, for this instantiation
  int pairs = 0;
  e = pair_capacity(reinterpret_cast<const void*>(kern), gemm_threads<Epi>(), L::TOTAL, c.num_sms, cap, &pairs);
  if (e != cudaSuccess) return e;
  sh.w_single_from = wide_single_from(sh.tiles_m * (tiles_n / 2), pairs);
  KernelCtl ctl{c.status, c.timeout_ns, c.skip_first_stage, c.scale_a, c.scale_b, c.f8_fmt, c.scale_host};
  return launch_chained(c, kern, dim3(2 * pairs), dim3(gemm_threads<Epi>()), L::TOTAL, ta, tb, sh, ctl, ep);
}

// An epilogue program run by 8 warps, two per TMEM lane quadrant, each on
// half of a tile's columns: the wide-tile kernel drains one accumulator half
// while the other accumulates, so the drain must be short.
template <class E>
struct Epi8 : E {
  static constexpr int kEpiWarps = 8;
};

// Epilogue programs the wide-tile kernel is instantiated for: those of the
// long-K backward GEMMs (dgrad2's RMSNorm backward, the weight gradients'
// store).
template <class Epi>
struct WideTiles {
  static constexpr bool value = false;
};
template <>
struct WideTiles<EpiStore> {
  static constexpr bool value = true;
};
template <>
struct WideTiles<EpiDgradRms> {
  static constexpr bool value = true;
};

// The 2-SM pair kernel (default) or the 1-SM kernel, 256-column tiles.
template <bool A_MN, bool B_MN, bool B_DUAL, class Epi, bool FP8 = false>
cudaError_t run_gemm(const LaunchCtx& c, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tb2, int M,
                     int N, int K, int tiles_n, const typename Epi::Params& ep) {
  static_assert(!FP8 || Epi::kAccScale, "an epilogue on 8-bit operands must dequantise the accumulator");
  if constexpr (!FP8 && !B_DUAL && WideTiles<Epi>::value && Epi::kEpiWarps == 4)
    if (wide_tiles_fit(c, K, tiles_n))
      return launch_gemm2w_kernel<A_MN, B_MN, Epi8<Epi>>(c, ta, tb, M, N, K, tiles_n, ep);
  if (c.pair) return launch_gemm2_kernel<256, 6, A_MN, B_MN, B_DUAL, Epi, FP8>(c, ta, tb, tb2, M, N, K, tiles_n, ep);
  return launch_gemm_kernel<256, 4, A_MN, B_MN, B_DUAL, Epi, FP8>(c, ta, tb, tb2, M, N, K, tiles_n, ep);
}

// Rows of one K-major B box: a whole 256-row tile (1-SM) or the half a CTA
// of the pair holds.
inline int b_box_rows(const LaunchCtx& c) { return c.pair ? 128 : 256; }

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
