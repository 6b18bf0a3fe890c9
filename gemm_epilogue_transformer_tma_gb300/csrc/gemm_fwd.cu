// Forward GEMM instantiations: GEMM1 with the residual + partial-RMS epilogue,
// GEMM2 with the deferred row scale + SwiGLU epilogue, and the plain GEMM.
#include <vector>

#include "gemm_launch.cuh"

namespace coda {

namespace {
constexpr int kBN = 256;
}  // namespace

int prms_tile_cols() { return PART_COLS; }

cudaError_t gemm_res_prms(const LaunchCtx& c, const __nv_bfloat16* X, const __nv_bfloat16* W1t,
                          const __nv_bfloat16* R, __nv_bfloat16* H, float* psum, int M, int K1, int d, int T,
                          const __nv_bfloat16* g, __nv_bfloat16* Hg) {
  CUtensorMap ta, tb;
  if (!make_operand_maps(&ta, &tb, X, false, W1t, false, M, d, K1, b_box_rows(c))) return cudaErrorInvalidValue;
  EpiResPrms::Params ep{};
  if (!make_tmap_store_bf16(&ep.H, H, d, M, d)) return cudaErrorInvalidValue;
  if (Hg != nullptr && !make_tmap_store_bf16(&ep.Hg, Hg, d, M, d)) return cudaErrorInvalidValue;
  ep.R = R;
  ep.ldr = d;
  ep.psum = psum;
  ep.T = T;
  ep.g = Hg != nullptr ? g : nullptr;
  return run_gemm<false, false, false, EpiResPrms>(c, ta, tb, tb, M, d, K1, (d + kBN - 1) / kBN, ep);
}

cudaError_t gemm_rowscale_swiglu(const LaunchCtx& c, const __nv_bfloat16* H, const __nv_bfloat16* W2gt,
                                 const float* rstd, __nv_bfloat16* out, __nv_bfloat16* zsave, int M, int d, int N2,
                                 bool swiglu, const float* psum, int T, float eps, float* rstd_out) {
  const float inv_d = 1.0f / static_cast<float>(d);
  CUtensorMap ta, tb, tb2;
  if (!swiglu) {
    if (!make_operand_maps(&ta, &tb, H, false, W2gt, false, M, N2, d, b_box_rows(c))) return cudaErrorInvalidValue;
    EpiStore::Params ep{};
    if (!make_tmap_store_bf16(&ep.out, out, N2, M, N2)) return cudaErrorInvalidValue;
    ep.row_scale = rstd;
    ep.psum = psum;
    ep.T = T;
    ep.inv_d = inv_d;
    ep.eps = eps;
    ep.rstd_out = rstd_out;
    return run_gemm<false, false, false, EpiStore>(c, ta, tb, tb, M, N2, d, (N2 + kBN - 1) / kBN, ep);
  }
  const int F = N2 / 2;
  if (!make_tmap_bf16(&ta, H, d, M, d, 64, BM)) return cudaErrorInvalidValue;
  // gate rows [0, F) and up rows [F, 2F) of W2gt as two separate tensors so
  // each half is zero-filled past its own end
  if (!make_tmap_bf16(&tb, W2gt, d, F, d, 64, kBN / 2)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tb2, W2gt + static_cast<int64_t>(F) * d, d, F, d, 64, kBN / 2)) return cudaErrorInvalidValue;
  EpiRowscaleSwiglu::Params ep{};
  if (!make_tmap_store_bf16(&ep.out, out, F, M, F)) return cudaErrorInvalidValue;
  if (zsave != nullptr) {
    if (!make_tmap_store_bf16(&ep.zg, zsave, F, M, N2)) return cudaErrorInvalidValue;
    if (!make_tmap_store_bf16(&ep.zu, zsave + F, F, M, N2)) return cudaErrorInvalidValue;
  }
  ep.save_z = zsave != nullptr;
  ep.rstd = rstd;
  ep.F = F;
  ep.psum = psum;
  ep.T = T;
  ep.inv_d = inv_d;
  ep.eps = eps;
  ep.rstd_out = rstd_out;
  return run_gemm<false, false, true, EpiRowscaleSwiglu>(c, ta, tb, tb2, M, F, d, (F + kBN / 2 - 1) / (kBN / 2), ep);
}

cudaError_t gemm_store(const LaunchCtx& c, const __nv_bfloat16* A, bool a_mn, const __nv_bfloat16* B, bool b_mn,
                       __nv_bfloat16* C, int M, int N, int K, const float* row_scale,
                       const __nv_bfloat16* col_scale) {
  CUtensorMap ta, tb;
  if (!make_operand_maps(&ta, &tb, A, a_mn, B, b_mn, M, N, K, b_box_rows(c))) return cudaErrorInvalidValue;
  EpiStore::Params ep{};
  if (!make_tmap_store_bf16(&ep.out, C, N, M, N)) return cudaErrorInvalidValue;
  ep.row_scale = row_scale;
  ep.col_scale = col_scale;
  const int tn = (N + kBN - 1) / kBN;
  if (!a_mn && !b_mn) return run_gemm<false, false, false, EpiStore>(c, ta, tb, tb, M, N, K, tn, ep);
  if (!a_mn && b_mn) return run_gemm<false, true, false, EpiStore>(c, ta, tb, tb, M, N, K, tn, ep);
  if (a_mn && b_mn) return run_gemm<true, true, false, EpiStore>(c, ta, tb, tb, M, N, K, tn, ep);
  return cudaErrorNotSupported;  // MN-major A with K-major B is not used on this path
}

cudaError_t gemm_store_f32(const LaunchCtx& c, const __nv_bfloat16* A, bool a_mn, const __nv_bfloat16* B, bool b_mn,
                           float* C, int M, int N, int K, bool accumulate) {
  if (a_mn || !b_mn) return cudaErrorNotSupported;  // only [M][K] x [K][N] is used
  CUtensorMap ta, tb;
  if (!make_operand_maps(&ta, &tb, A, a_mn, B, b_mn, M, N, K, b_box_rows(c))) return cudaErrorInvalidValue;
  EpiStoreF32::Params ep{};
  if (!make_tmap_store_f32(&ep.out, C, N, M, N)) return cudaErrorInvalidValue;
  ep.beta = accumulate ? 1 : 0;
  return run_gemm<false, true, false, EpiStoreF32>(c, ta, tb, tb, M, N, K, (N + kBN - 1) / kBN, ep);
}

}  // namespace coda

bool coda::wide_tiles_fit(const LaunchCtx& c, int K, int tiles_n) {
  const int nkb = (K + BK - 1) / BK;
  return c.pair && c.wide_lead > 0 && tiles_n % 2 == 0 && nkb >= 4 * c.wide_lead && nkb >= kWideMinKb;
}

int coda::split_scratch_slots(int num_sms) { return (num_sms / 2 - 1) * (kSplitMaxRanges - 1); }

// Host-side check of the split-tile schedule of the SM-pair kernel, run with
// the kernel's own iterator (coda_debug_split_schedule_violations in
// include/coda_testing.h).
extern "C" int coda_debug_split_schedule_violations(int tiles, int num_kb, int clusters) {
  using namespace coda;
  if (tiles < 1 || num_kb < 1 || clusters < 1) return -1;
  const int slots = (clusters - 1) * (kSplitMaxRanges - 1);
  const SplitPlan plan = split_plan(tiles, num_kb, clusters, slots);
  if (plan.first == tiles) return 0;  // not split: nothing to check
  GemmShape sh{};
  sh.tiles_m = tiles;
  sh.tiles_n = 1;
  sh.num_kb = num_kb;
  sh.sk_first = plan.first;
  sh.sk_ranges = plan.ranges;
  const int S = plan.ranges;
  const int rem = tiles - plan.first;
  int bad = 0;
  if (S < 2 || S > kSplitMaxRanges || rem >= clusters || rem * (S - 1) > slots) ++bad;
  std::vector<int> cover(static_cast<size_t>(tiles) * num_kb, 0);
  // which (tile, k-range) wrote each slot, and in which order each cluster met its pieces
  std::vector<int> slot_tile(static_cast<size_t>(rem) * (S - 1), -1), slot_kb0(slot_tile.size(), -1);
  std::vector<std::vector<TilePiece>> owners(clusters);
  for (int cid = 0; cid < clusters; ++cid) {
    SplitWork wk(sh, cid, clusters);
    TilePiece pc;
    bool seen_owner = false;
    while (wk.next(pc)) {
      if (pc.kb0 >= pc.kb1) ++bad;  // an empty range
      for (int k = pc.kb0; k < pc.kb1; ++k) cover[static_cast<size_t>(pc.tile) * num_kb + k]++;
      if (pc.tile < sh.sk_first) {
        if (pc.partial || pc.owner || pc.kb0 != 0 || pc.kb1 != num_kb) ++bad;
        continue;
      }
      if (pc.partial == pc.owner) ++bad;  // every split piece is exactly one of the two
      if (pc.partial) {
        if (seen_owner) ++bad;  // partial pieces come before the cluster's owner pieces
        if (pc.slot < 0 || pc.slot >= static_cast<int>(slot_tile.size()) || slot_tile[pc.slot] != -1) {
          ++bad;
        } else {
          slot_tile[pc.slot] = pc.tile;
          slot_kb0[pc.slot] = pc.kb0;
        }
      }
      if (pc.owner) {
        seen_owner = true;
        if (pc.kb1 != num_kb) ++bad;  // the owner holds the tile's last k-range
        owners[cid].push_back(pc);
      }
    }
  }
  // each owner's slots hold its tile's earlier k-ranges, in order, covering
  // k-blocks [0, owner's first k-block) without a gap
  for (int cid = 0; cid < clusters; ++cid)
    for (const TilePiece& o : owners[cid]) {
      int pos = 0;
      for (int j = 0; j < S - 1; ++j) {
        const int sl = o.slot + j;
        if (sl < 0 || sl >= static_cast<int>(slot_tile.size()) || slot_tile[sl] != o.tile || slot_kb0[sl] != pos) {
          ++bad;
          break;
        }
        SplitWork probe(sh, 0, clusters);
        pos = probe.kb_begin(j + 1);
      }
      if (pos != o.kb0) ++bad;
    }
  for (int v : cover)
    if (v != 1) ++bad;
  return bad;
}

// First tile of the split region the SM-pair launcher would choose
// (coda_debug_split_first_tile in include/coda_testing.h).
extern "C" int coda_debug_split_first_tile(int tiles, int num_kb, int clusters) {
  if (tiles < 1 || num_kb < 1 || clusters < 1) return -1;
  return coda::split_plan(tiles, num_kb, clusters, (clusters - 1) * (coda::kSplitMaxRanges - 1)).first;
}

// k-ranges per split tile the launcher would choose (1: no split).
extern "C" int coda_debug_split_ranges(int tiles, int num_kb, int clusters) {
  if (tiles < 1 || num_kb < 1 || clusters < 1) return -1;
  return coda::split_plan(tiles, num_kb, clusters, (clusters - 1) * (coda::kSplitMaxRanges - 1)).ranges;
}

// Host-side check of the wide-tile schedule of the SM-pair kernel, run with
// the kernel's own iterators (coda_debug_wide_schedule_violations in
// include/coda_testing.h).
extern "C" int coda_debug_wide_schedule_violations(int M, int N, int K, int clusters, int lead) {
  using namespace coda;
  if (M < 1 || N < 1 || K < 1 || clusters < 1 || lead < 0) return -1;
  GemmShape sh{};
  sh.M = M;
  sh.N = N;
  sh.K = K;
  sh.tiles_m = (M + BM2 - 1) / BM2;
  sh.tiles_n = (N + 255) / 256;
  if (sh.tiles_n % 2 != 0) return -1;  // the launcher takes wide tiles only for an even count
  sh.num_kb = (K + BK - 1) / BK;
  sh.group_m = 8;
  sh.w_lead = lead;
  const int tiles_w = sh.tiles_m * sh.tiles_n / 2;
  sh.w_single_from = wide_single_from(tiles_w, clusters);
  int bad = 0;
  std::vector<int> cover(static_cast<size_t>(sh.tiles_m) * sh.tiles_n, 0);
  std::vector<int> kcover(static_cast<size_t>(sh.num_kb));
  for (int cid = 0; cid < clusters; ++cid) {
    WideWork wk(sh, cid, clusters);
    WideUnit u;
    bool single_seen = false;
    while (wk.next(u)) {
      if (u.tm < 0 || u.tm >= sh.tiles_m || u.tv < 0 || u.tv + (u.wide ? 1 : 0) >= sh.tiles_n) {
        ++bad;
        continue;
      }
      // wide units first (the producer switches rings once), on even columns
      if (u.wide && (single_seen || u.tv % 2 != 0)) ++bad;
      if (!u.wide) single_seen = true;
      for (int j = 0; j < (u.wide ? 2 : 1); ++j) cover[static_cast<size_t>(u.tm) * sh.tiles_n + u.tv + j]++;
      // each half sees every k-block exactly once; its first block starts
      // the sum and its last block is where the kernel commits it
      const WidePhases ph(u, sh.num_kb, sh.w_lead);
      for (int h = 0; h < (u.wide ? 2 : 1); ++h) {
        std::fill(kcover.begin(), kcover.end(), 0);
        int first = -1, last = -1;
        for (int i = 0; i < ph.nblocks; ++i) {
          int kb;
          bool f0, f1;
          ph.block(i, kb, f0, f1);
          if (kb < 0 || kb >= sh.num_kb) {
            ++bad;
            continue;
          }
          if (!u.wide && f1) ++bad;  // a half tile feeds one half only
          if (h == 0 ? f0 : f1) {
            kcover[kb]++;
            if (first < 0) first = i;
            last = i;
          }
        }
        for (int v : kcover)
          if (v != 1) ++bad;
        if (first != (h == 0 ? 0 : ph.first_h1())) ++bad;
        if (last != (h == 0 ? ph.last_h0() : ph.last_h1())) ++bad;
      }
      if (u.wide && ph.J != (lead < sh.num_kb / 2 ? lead : sh.num_kb / 2)) ++bad;
    }
  }
  for (int v : cover)
    if (v != 1) ++bad;
  return bad;
}
