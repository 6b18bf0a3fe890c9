// Grouped launches of independent GEMM pairs (the data and the weight
// gradient of one layer: the first layer of the block, in bf16 or on 8-bit
// codes, and the LM-head chunks) on the SM-pair kernel of gemm_group.cuh.  With SM pairing switched off they run
// as two launches of the 1-SM kernel.
#include <vector>

#include "gemm_group.cuh"
#include "gemm_launch.cuh"

namespace coda {

namespace {
constexpr int kStages = 6;

// k-blocks of 128 bytes of K per row: 64 bf16 or 128 8-bit codes
GemmShape pair_shape(int M, int N, int K, bool fp8 = false) {
  const int bke = fp8 ? 128 : BK;
  GemmShape sh;
  sh.M = M;
  sh.N = N;
  sh.K = K;
  sh.tiles_m = (M + BM2 - 1) / BM2;
  sh.tiles_n = (N + 255) / 256;
  sh.num_kb = (K + bke - 1) / bke;
  sh.group_m = 8;
  sh.sk_first = sh.tiles_m * sh.tiles_n;  // grouped launches never split tiles
  sh.sk_ranges = 1;
  return sh;
}

// Cost of a tile ~ its k-blocks; the heavier problem is dealt first.
GroupSched make_sched(const GemmShape& a, const GemmShape& b, int P) {
  GroupSched s;
  const int ta = a.tiles_m * a.tiles_n, tb = b.tiles_m * b.tiles_n;
  s.P = P;
  s.heavy = b.num_kb > a.num_kb ? 1 : 0;
  s.nH = s.heavy ? tb : ta;
  s.nL = s.heavy ? ta : tb;
  const int cH = a.num_kb > b.num_kb ? a.num_kb : b.num_kb;
  const int cL0 = a.num_kb > b.num_kb ? b.num_kb : a.num_kb;
  const int cL = cL0 > 0 ? cL0 : 1;
  s.q = (cH + cL / 2) / cL;
  return s;
}

template <bool A_MN0, bool B_MN0, bool A_MN1, bool B_MN1, class Epi0, class Epi1, bool FP8 = false>
cudaError_t launch_group(const LaunchCtx& c, GroupArgs<Epi0, Epi1>& g) {
  using L = Gemm2Smem<256, kStages, group_stage_bytes<Epi0, Epi1>()>;
  auto kern = gemm_tc2_group_kernel<kStages, A_MN0, B_MN0, A_MN1, B_MN1, Epi0, Epi1, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL);
  if (e != cudaSuccess) return e;
  static int max_pairs[2][64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int* mp = &max_pairs[FP8 ? 1 : 0][dev];
  if (*mp == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (c.num_sms / 2), 1, 1);
    cfg.blockDim = dim3(gemm_threads<Epi0>(), 1, 1);
    cfg.dynamicSmemBytes = L::TOTAL;
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
    *mp = std::max(1, std::min(n, c.num_sms / 2));
  }
  const int tiles = g.sh0.tiles_m * g.sh0.tiles_n + g.sh1.tiles_m * g.sh1.tiles_n;
  const int P = std::max(1, std::min(tiles, *mp));
  g.sched = make_sched(g.sh0, g.sh1, P);
  KernelCtl ctl{c.status, c.timeout_ns, c.skip_first_stage, nullptr, nullptr, FP8 ? c.f8_fmt : 0u,
                FP8 ? c.scale_host : 1.f};
  return launch_chained(c, kern, dim3(2 * P), dim3(gemm_threads<Epi0>()), L::TOTAL, g, ctl);
}
}  // namespace

cudaError_t gemm_group_store(const LaunchCtx& c, const __nv_bfloat16* dH, const __nv_bfloat16* W1t,
                             const __nv_bfloat16* X, __nv_bfloat16* dX, __nv_bfloat16* dW1t, int M, int K1, int d) {
  if (!c.pair) {
    cudaError_t e = gemm_store(c, dH, false, W1t, true, dX, M, K1, d, nullptr, nullptr);
    if (e != cudaSuccess) return e;
    return gemm_store(c, dH, true, X, true, dW1t, d, K1, M, nullptr, nullptr);
  }
  GroupArgs<EpiStore, EpiStore> ga{};
  // problem 0, dgrad: dX[M, K1] from dH [M][d] (K-major) and W1t [d][K1] (MN-major)
  if (!make_operand_maps(&ga.tmA0, &ga.tmB0, dH, false, W1t, true, M, K1, d, b_box_rows(c)))
    return cudaErrorInvalidValue;
  // problem 1, wgrad: dW1t[d, K1] = dH^T X; K' = M, A' = dH [M][d] and
  // B' = X [M][K1], both MN-major
  if (!make_operand_maps(&ga.tmA1, &ga.tmB1, dH, true, X, true, d, K1, M, b_box_rows(c)))
    return cudaErrorInvalidValue;
  ga.sh0 = pair_shape(M, K1, d);
  ga.sh1 = pair_shape(d, K1, M);
  if (!make_tmap_store_bf16(&ga.ep0.out, dX, K1, M, K1)) return cudaErrorInvalidValue;
  if (!make_tmap_store_bf16(&ga.ep1.out, dW1t, K1, d, K1)) return cudaErrorInvalidValue;
  return launch_group<false, true, true, true, EpiStore, EpiStore>(c, ga);
}

cudaError_t gemm_group_store_fp8(const LaunchCtx& c0, const uint8_t* dHq, int dh_fmt, const float* sdH,
                                 const uint8_t* W1q, const float* sW1, const uint8_t* Xq, const float* sX, int w_fmt,
                                 __nv_bfloat16* dX, __nv_bfloat16* dW1t, int M, int K1, int d) {
  if (!c0.pair) {
    cudaError_t e = gemm_store_fp8(c0, dHq, false, dh_fmt, sdH, W1q, true, w_fmt, sW1, dX, M, K1, d, nullptr, nullptr);
    if (e != cudaSuccess) return e;
    return gemm_store_fp8(c0, dHq, true, dh_fmt, sdH, Xq, true, w_fmt, sX, dW1t, d, K1, M, nullptr, nullptr);
  }
  LaunchCtx c = c0;
  c.f8_fmt = f8_format_bits(dh_fmt, w_fmt);
  GroupArgs<EpiStore, EpiStore> ga{};
  // problem 0, dgrad: dX[M, K1] from dH codes [M][d] (K-major) and W1t codes
  // [d][K1] (MN-major)
  if (!make_f8_operand_map(&ga.tmA0, dHq, false, M, d, BM) ||
      !make_f8_operand_map(&ga.tmB0, W1q, true, K1, d, b_box_rows(c)))
    return cudaErrorInvalidValue;
  // problem 1, wgrad: dW1t[d, K1] = dH^T X; K' = M, A' = dH codes [M][d] and
  // B' = X codes [M][K1], both MN-major
  if (!make_f8_operand_map(&ga.tmA1, dHq, true, d, M, BM) ||
      !make_f8_operand_map(&ga.tmB1, Xq, true, K1, M, b_box_rows(c)))
    return cudaErrorInvalidValue;
  ga.sh0 = pair_shape(M, K1, d, true);
  ga.sh1 = pair_shape(d, K1, M, true);
  if (!make_tmap_store_bf16(&ga.ep0.out, dX, K1, M, K1)) return cudaErrorInvalidValue;
  if (!make_tmap_store_bf16(&ga.ep1.out, dW1t, K1, d, K1)) return cudaErrorInvalidValue;
  ga.scale_a0 = sdH;
  ga.scale_b0 = sW1;
  ga.scale_a1 = sdH;
  ga.scale_b1 = sX;
  return launch_group<false, true, true, true, EpiStore, EpiStore, true>(c, ga);
}

cudaError_t gemm_group_ce_bwd(const LaunchCtx& c, const __nv_bfloat16* dL, const __nv_bfloat16* Wc,
                              const __nv_bfloat16* H, float* dH32, bool accumulate, __nv_bfloat16* dWc, int M, int d,
                              int Vc) {
  if (!c.pair) {
    cudaError_t e = gemm_store_f32(c, dL, false, Wc, true, dH32, M, d, Vc, accumulate);
    if (e != cudaSuccess) return e;
    return gemm_store(c, dL, true, H, true, dWc, Vc, d, M, nullptr, nullptr);
  }
  GroupArgs<EpiStoreF32, EpiStore> ga{};
  // problem 0: dH32[M, d] (+)= dL [M][Vc] (K-major) Wc [Vc][d] (MN-major)
  if (!make_operand_maps(&ga.tmA0, &ga.tmB0, dL, false, Wc, true, M, d, Vc, b_box_rows(c)))
    return cudaErrorInvalidValue;
  // problem 1: dWc[Vc, d] = dL^T H; K' = M, A' = dL [M][Vc] and B' = H [M][d],
  // both MN-major
  if (!make_operand_maps(&ga.tmA1, &ga.tmB1, dL, true, H, true, Vc, d, M, b_box_rows(c)))
    return cudaErrorInvalidValue;
  ga.sh0 = pair_shape(M, d, Vc);
  ga.sh1 = pair_shape(Vc, d, M);
  if (!make_tmap_store_f32(&ga.ep0.out, dH32, d, M, d)) return cudaErrorInvalidValue;
  ga.ep0.beta = accumulate ? 1 : 0;
  if (!make_tmap_store_bf16(&ga.ep1.out, dWc, d, Vc, d)) return cudaErrorInvalidValue;
  return launch_group<false, true, true, true, EpiStoreF32, EpiStore>(c, ga);
}

cudaError_t gemm_group_ce_bwd_fp8(const LaunchCtx& c0, const uint8_t* dLq, float s_dL, const uint8_t* Wq_chunk,
                                  const float* sW, const uint8_t* Hq, const float* sH, float* dH32, bool accumulate,
                                  __nv_bfloat16* dWc, int M, int d, int Vc) {
  if (!c0.pair) return gemm_ce_bwd_fp8(c0, dLq, s_dL, Wq_chunk, sW, Hq, sH, dH32, accumulate, dWc, M, d, Vc);
  LaunchCtx c = c0;
  c.scale_host = s_dL;               // dL's power-of-two scale, common to both problems
  c.f8_fmt = f8_format_bits(1, 0);   // e5m2 dL codes against e4m3 W / H codes
  GroupArgs<EpiStoreF32, EpiStore> ga{};
  // problem 0: dH32[M, d] (+)= dL codes [M][Vc] (K-major) W codes [Vc][d]
  // (MN-major), scale s_dL * sW
  if (!make_f8_operand_map(&ga.tmA0, dLq, false, M, Vc, BM) ||
      !make_f8_operand_map(&ga.tmB0, Wq_chunk, true, d, Vc, b_box_rows(c)))
    return cudaErrorInvalidValue;
  // problem 1: dWc[Vc, d] = dL^T H; K' = M, A' = dL codes [M][Vc] and B' = H
  // codes [M][d], both MN-major, scale s_dL * sH
  if (!make_f8_operand_map(&ga.tmA1, dLq, true, Vc, M, BM) ||
      !make_f8_operand_map(&ga.tmB1, Hq, true, d, M, b_box_rows(c)))
    return cudaErrorInvalidValue;
  ga.sh0 = pair_shape(M, d, Vc, true);
  ga.sh1 = pair_shape(Vc, d, M, true);
  if (!make_tmap_store_f32(&ga.ep0.out, dH32, d, M, d)) return cudaErrorInvalidValue;
  ga.ep0.beta = accumulate ? 1 : 0;
  if (!make_tmap_store_bf16(&ga.ep1.out, dWc, d, Vc, d)) return cudaErrorInvalidValue;
  ga.scale_a0 = nullptr;
  ga.scale_b0 = sW;
  ga.scale_a1 = nullptr;
  ga.scale_b1 = sH;
  return launch_group<false, true, true, true, EpiStoreF32, EpiStore, true>(c, ga);
}

// Host check of the grouped schedule: every tile of both problems is visited
// by exactly one cluster.  Returns 0 when it holds, else the number of
// violations.
int group_schedule_violations(int P, int heavy, int nH, int nL, int q) {
  GroupSched s;
  s.P = P;
  s.heavy = heavy;
  s.nH = nH;
  s.nL = nL;
  s.q = q;
  std::vector<int> seen0(static_cast<size_t>(heavy == 0 ? nH : nL), 0), seen1(static_cast<size_t>(heavy == 1 ? nH : nL), 0);
  int bad = 0;
  for (int c = 0; c < P; ++c) {
    int prob, t;
    for (int k = 0; group_tile(s, c, k, prob, t); ++k) {
      std::vector<int>& seen = prob == 0 ? seen0 : seen1;
      if (t < 0 || t >= static_cast<int>(seen.size()))
        ++bad;
      else
        ++seen[static_cast<size_t>(t)];
      if (k > nH + nL) {  // a cluster cannot hold more tiles than exist
        ++bad;
        break;
      }
    }
  }
  for (int v : seen0) bad += v != 1;
  for (int v : seen1) bad += v != 1;
  return bad;
}

}  // namespace coda
