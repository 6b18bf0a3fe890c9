// SM-pair GEMM with 256 x 512 tiles ("wide" tiles) for long-K problems.
//
// Per k-block a pair of the 256 x 256 kernel (gemm_tc2.cuh) loads 128 rows
// of A and 128 rows of B into each CTA for 256 x 256 x 64 MACs.  Here each
// CTA loads 128 rows of A and two 128-row halves of B, and the leader issues
// two 256-column MMAs per K slice into the two halves of TMEM: the A bytes
// moved per MAC drop by half and the operand bytes per MAC by a quarter, and
// a wave of 76 tiles covers twice the output, so the long operand panels are
// re-read from DRAM about half as often.
//
// The accumulator of a wide tile fills all 512 TMEM columns, so there is no
// second buffer for the epilogue to drain while the next tile accumulates.
// Instead each wide tile runs its k-blocks in three phases:
//   P1  k-blocks [0, J)        into the first half only,
//   P2  k-blocks [J, nkb)      into both halves (A loaded once for both),
//   P3  k-blocks [0, J)        into the second half only.
// The first half is complete after P2 and is drained by the epilogue while
// P3 runs; the second half is complete after P3 and is drained while the
// next tile's P1 runs.  J (sh.w_lead) is sized so that J single-half
// k-blocks outlast the drain of one half.  The second half's sum runs over
// k-blocks J..nkb-1 and then 0..J-1: another fp32 summation order than the
// 256 x 256 kernel's, equally exact.
//
// Tiles are dealt round-robin.  When the last, partial wave holds at most
// half as many wide tiles as there are pairs, those tiles are instead cut
// into their two 256 x 256 halves ("single" units, one TMEM half each, the
// halves alternating so that one drains while the other accumulates): half a
// round instead of a whole one.
//
// Roles, barriers, bounded waits, abort and drain follow gemm_tc2_kernel:
// warp 0 lane 0 of each CTA loads its halves of every stage onto the
// leader's full barrier, warp 1 lane 0 of the leader issues the MMAs and
// commits to the empty barriers and the per-half accumulator barriers of
// both CTAs, warps 2.. run the epilogue program on their CTA's 128 rows of
// each 256-column half, which they see as an ordinary 256-column tile.
#pragma once

#include "gemm_tc2.cuh"

namespace coda {

constexpr int BNW = 512;  // output columns of a wide pair tile

// One unit of a cluster's work: a wide tile (both TMEM halves) or one
// 256-column half tile (a single TMEM half).
struct WideUnit {
  int tm;    // 256-row tile
  int tv;    // 256-column tile of the first (or only) half
  bool wide;
};

// The unit sequence of one cluster, the same in every role.  Wide tiles
// [0, wide_end) round-robin; then the 256-column halves of the remaining
// wide tiles, round-robin.  Tile columns count 256-column tiles (tiles_v,
// even); wide tiles are rastered like gemm_tc2_kernel's tiles.
struct WideWork {
  GemmShape shw;  // the wide-tile raster: tiles_n = tiles_v / 2
  int wide_end, n_single, P, next_wide, next_single;
  __host__ __device__ WideWork(const GemmShape& sh, int cluster, int num_clusters) {
    shw = sh;
    shw.tiles_n = sh.tiles_n / 2;
    P = num_clusters;
    const int tiles_w = shw.tiles_m * shw.tiles_n;
    wide_end = sh.w_single_from;
    n_single = 2 * (tiles_w - wide_end);
    next_wide = cluster;
    next_single = cluster;
  }
  __host__ __device__ bool next(WideUnit& u) {
    int tm, tw;
    if (next_wide < wide_end) {
      wide_coords(next_wide, tm, tw);
      u.tm = tm;
      u.tv = 2 * tw;
      u.wide = true;
      next_wide += P;
      return true;
    }
    if (next_single < n_single) {
      wide_coords(wide_end + next_single / 2, tm, tw);
      u.tm = tm;
      u.tv = 2 * tw + (next_single & 1);
      u.wide = false;
      next_single += P;
      return true;
    }
    return false;
  }
  __host__ __device__ void wide_coords(int t, int& tm, int& tw) const {
    const int group_tiles = shw.group_m * shw.tiles_n;
    const int group = t / group_tiles;
    const int first_m = group * shw.group_m;
    const int gm = shw.tiles_m - first_m < shw.group_m ? shw.tiles_m - first_m : shw.group_m;
    const int r = t - group * group_tiles;
    tm = first_m + r % gm;
    tw = r / gm;
  }
};

// The k-block phases of one unit.  ff: the TMEM half that frees first.  A
// wide unit accumulates tile column tv in half ff (P1, P2) and tv + 1 in the
// other half (P2, P3); a single unit accumulates tv in half ff over all
// k-blocks.  block(i) gives the i-th k-block and which halves it feeds.
struct WidePhases {
  int nkb, J, nblocks;
  bool wide;
  __host__ __device__ WidePhases(const WideUnit& u, int num_kb, int lead) {
    nkb = num_kb;
    wide = u.wide;
    J = wide ? (lead < num_kb / 2 ? lead : num_kb / 2) : 0;
    nblocks = wide ? num_kb + J : num_kb;
  }
  // k-block of block i, and whether it feeds the first (h0) / second (h1) half
  __host__ __device__ void block(int i, int& kb, bool& h0, bool& h1) const {
    if (!wide) {
      kb = i;
      h0 = true;
      h1 = false;
    } else if (i < J) {
      kb = i;
      h0 = true;
      h1 = false;
    } else if (i < nkb) {
      kb = i;
      h0 = h1 = true;
    } else {
      kb = i - nkb;
      h0 = false;
      h1 = true;
    }
  }
  // last block feeding the first / second half
  __host__ __device__ int last_h0() const { return wide ? nkb - 1 : nkb - 1; }
  __host__ __device__ int last_h1() const { return wide ? nblocks - 1 : -1; }
  // first block feeding the second half
  __host__ __device__ int first_h1() const { return wide ? J : -1; }
};

// First wide tile run as two half tiles: the last, partial wave's tiles
// when it holds at most half as many wide tiles as there are clusters (half
// a round of half tiles instead of a round of wide ones), else none.
__host__ __device__ inline int wide_single_from(int tiles_w, int clusters) {
  const int rem = tiles_w % clusters;
  return (rem > 0 && 2 * rem <= clusters) ? tiles_w - rem : tiles_w;
}

// A stage holds one A tile and both B halves (48 KB per CTA); a block that
// feeds one half loads only its own B half.  (A ring of 32 KB stages in which
// a two-half block took two consecutive stages kept the tensor pipe only
// 57-60 % busy against 75 % with these stages, measured.)
//
// The half-tile units at the end of a cluster's sequence use the same bytes
// as a second ring of STAGES1 stages of one A tile and one B half (32 KB per
// CTA), as gemm_tc2_kernel does: a single-half k-block in a 48 KB stage
// would leave only two thirds of the ring's bytes in flight.  The producer
// switches rings once, after every stage of the first ring has been
// consumed; each ring has its own barriers.
template <int STAGES, int EPI_BYTES>
struct Gemm2wSmem {
  static constexpr int A_BYTES = 128 * BK * 2;    // this CTA's 128 rows of A
  static constexpr int HB_BYTES = 128 * BK * 2;   // this CTA's 128 rows of one B half
  static constexpr int STAGE_BYTES = A_BYTES + 2 * HB_BYTES;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int STAGE1_BYTES = A_BYTES + HB_BYTES;  // half-tile ring
  static constexpr int STAGES1 = RING_BYTES / STAGE1_BYTES;
  static constexpr int STORE_BYTES = EPI_BYTES;
  static constexpr int BAR_BYTES = 512;
  static constexpr int BAR1_OFFSET = 256;  // the half-tile ring's barriers, in the barrier area
  static constexpr int TOTAL = RING_BYTES + STORE_BYTES + BAR_BYTES + 1024;
  static_assert(TOTAL <= MAX_DYN_SMEM, "shared memory budget");
  static constexpr int TMEM_COLS = 512;
  static_assert((2 * STAGES + 5) * 8 + 20 <= BAR1_OFFSET, "barrier area too small");
  static_assert(STAGES <= 16, "the producer's per-stage B-half counts are 2 bits each in one word");
  static_assert(BAR1_OFFSET + 2 * STAGES1 * 8 <= BAR_BYTES, "barrier area too small");
  static_assert(STAGES1 * STAGE1_BYTES == RING_BYTES, "both rings cover the same bytes");
};

template <int STAGES, bool A_MN, bool B_MN, class Epi>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(gemm_threads<Epi>(), 1)
    gemm_tc2w_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmShape sh, const KernelCtl ctl, const __grid_constant__ typename Epi::Params ep) {
  using L = Gemm2wSmem<STAGES, epi_stage_bytes<Epi>()>;
  constexpr int HBN = 256;   // columns of one TMEM half (one 256-column tile)
  constexpr int HB = 128;    // B rows one CTA holds per half
  constexpr uint32_t IDESC = idesc_bf16_f32(BM2, HBN, A_MN, B_MN);
  constexpr int MNB = 64;            // M/N elements per MN-major box
  constexpr int MN_BOX = 128 * BK;   // bytes per MN-major box
  constexpr int MN_KSTEP = 2048;     // bytes per MMA K slice, MN-major

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::RING_BYTES + L::STORE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;  // per TMEM half
  uint64_t* tempty = tfull + 2;      // per TMEM half, leader only
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // leader: the peer's fills of the wide ring + 1, of the half-tile ring, and
  // the B halves (0..2) of its last fill into each wide stage, 2 bits each
  uint32_t* fill_report = tmem_slot + 2;
  constexpr int S1 = L::STAGES1;
  uint64_t* full1 = reinterpret_cast<uint64_t*>(smem + L::RING_BYTES + L::STORE_BYTES + L::BAR1_OFFSET);
  uint64_t* empty1 = full1 + S1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster_id = blockIdx.x >> 1;
  const int num_clusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < S1; ++s) {
      mbar_init(&full1[s], 1);
      mbar_init(&empty1[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * Epi::kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fill_report[0] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  cluster_sync_all();
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, L::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_launch_dependents();
  griddep_wait();
  const float acc_scale = acc_scale_of(ctl);

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      const uint32_t leader_full = mapa_shared(smem_u32(full), 0);
      const uint32_t leader_full1 = mapa_shared(smem_u32(full1), 0);
      int stage = 0, stage1 = 0;  // wide ring / half-tile ring cursors
      uint32_t phase = 0, phase1 = 0;
      int issued = 0, issued1 = 0;  // fills of the wide / half-tile ring so far
      uint32_t halves = 0;          // B halves of the last fill into each wide stage, 2 bits each
      // test hook: one CTA of the first pair stops before its first copy
      // (1: the leader, 2: the peer)
      bool ok = !(cluster_id == 0 && ctl.skip_first_stage == (leader ? 1 : 2));
      bool ring1 = false;  // switched to the half-tile ring
      int ff = 0;          // TMEM half that frees first
      WideWork wk(sh, cluster_id, num_clusters);
      WideUnit u;
      while (ok && wk.next(u)) {
        const WidePhases ph(u, sh.num_kb, sh.w_lead);
        const int m0 = u.tm * BM2 + static_cast<int>(rank) * 128;
        // B rows of this CTA for the unit's first / second tile column
        const int n_first = u.tv * HBN + static_cast<int>(rank) * HB;
        const int n_second = n_first + HBN;
        const int hf = ff, hs = ff ^ 1;  // TMEM half (and B region) of the first / second column
        if (!u.wide && !ring1) {
          // every stage of the wide ring consumed before its bytes are reused
          for (int t = 0; t < STAGES && ok; ++t) {
            const int p = stage + t;
            const uint32_t ph_t = phase ^ (p >= STAGES ? 1u : 0u);
            if (!mbar_wait_bounded(&empty[p % STAGES], ph_t ^ 1u, abort_flag, ctl.timeout_ns)) {
              if (!*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_PRODUCER);
              ok = false;
            }
          }
          if (!ok) break;
          ring1 = true;
        }
        if (u.wide) {
          // wide unit: the 48 KB ring (this loop is kept free of the
          // half-tile ring's selects: with them the tensor pipe lost 13 %)
          for (int i = 0; i < ph.nblocks; ++i) {
            int kb;
            bool f0, f1;
            ph.block(i, kb, f0, f1);
            if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, ctl.timeout_ns)) {
              if (!*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_PRODUCER);
              ok = false;
              break;
            }
            uint8_t* sa = smem + stage * L::STAGE_BYTES;
            const uint32_t bar = leader_full + static_cast<uint32_t>(stage * 8);
            const uint32_t nh = (f0 ? 1u : 0u) + (f1 ? 1u : 0u);
            halves = (halves & ~(3u << (2 * stage))) | (nh << (2 * stage));
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * (L::A_BYTES + nh * L::HB_BYTES));
            if (!A_MN) {
              tma_load_2d_pair(sa, &tmA, bar, kb * BK, m0);
            } else {
#pragma unroll
              for (int j = 0; j < 128 / MNB; ++j) tma_load_2d_pair(sa + j * MN_BOX, &tmA, bar, m0 + j * MNB, kb * BK);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (!(h == 0 ? f0 : f1)) continue;
              uint8_t* sb = sa + L::A_BYTES + (h == 0 ? hf : hs) * L::HB_BYTES;
              const int n0 = h == 0 ? n_first : n_second;
              if (!B_MN) {
                tma_load_2d_pair(sb, &tmB, bar, kb * BK, n0);
              } else {
#pragma unroll
                for (int j = 0; j < HB / MNB; ++j)
                  tma_load_2d_pair(sb + j * MN_BOX, &tmB, bar, n0 + j * MNB, kb * BK);
              }
            }
            ++issued;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        } else {
          // half tile: the 32 KB ring, every k-block into one B region
          for (int kb = 0; kb < sh.num_kb; ++kb) {
            if (!mbar_wait_bounded(&empty1[stage1], phase1 ^ 1u, abort_flag, ctl.timeout_ns)) {
              if (!*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_PRODUCER);
              ok = false;
              break;
            }
            uint8_t* sa = smem + stage1 * L::STAGE1_BYTES;
            uint8_t* sb = sa + L::A_BYTES;
            const uint32_t bar = leader_full1 + static_cast<uint32_t>(stage1 * 8);
            if (leader) mbar_arrive_expect_tx(&full1[stage1], 2 * L::STAGE1_BYTES);
            if (!A_MN) {
              tma_load_2d_pair(sa, &tmA, bar, kb * BK, m0);
            } else {
#pragma unroll
              for (int j = 0; j < 128 / MNB; ++j) tma_load_2d_pair(sa + j * MN_BOX, &tmA, bar, m0 + j * MNB, kb * BK);
            }
            if (!B_MN) {
              tma_load_2d_pair(sb, &tmB, bar, kb * BK, n_first);
            } else {
#pragma unroll
              for (int j = 0; j < HB / MNB; ++j)
                tma_load_2d_pair(sb + j * MN_BOX, &tmB, bar, n_first + j * MNB, kb * BK);
            }
            ++issued1;
            if (++stage1 == S1) {
              stage1 = 0;
              phase1 ^= 1u;
            }
          }
        }
        if (!u.wide) ff ^= 1;
      }
      // the hand-off of gemm_tc2_kernel, over both rings: every fill of both
      // CTAs observed landed before shared memory can be released
      bool landed = true;
      if (!leader) {
        const uint32_t lead_report = mapa_shared(smem_u32(fill_report), 0);
        st_release_cluster_u32(lead_report + 4, static_cast<uint32_t>(issued1));
        st_release_cluster_u32(lead_report + 8, halves);
        st_release_cluster_u32(lead_report, static_cast<uint32_t>(issued) + 1u);
      } else {
        uint32_t r;
        landed = pair_report_wait(fill_report, ctl.timeout_ns, r);
        if (landed) {
          const int peer1 = static_cast<int>(ld_acquire_cluster_u32(fill_report + 1));
          const uint32_t peer_halves = ld_acquire_cluster_u32(fill_report + 2);
          const auto wide_bytes = [halves, peer_halves](int i, bool leader_armed) {
            const uint32_t nh = ((leader_armed ? halves : peer_halves) >> (2 * (i % STAGES))) & 3u;
            return static_cast<uint32_t>(L::A_BYTES) + nh * static_cast<uint32_t>(L::HB_BYTES);
          };
          landed = pair_ring_landed(issued, -1, static_cast<int>(r) - 1, full, STAGES, wide_bytes, ctl.timeout_ns);
          landed = pair_ring_landed(issued1, -1, peer1, full1, S1,
                                    [](int, bool) { return static_cast<uint32_t>(L::STAGE1_BYTES); },
                                    ctl.timeout_ns) && landed;
        }
      }
      if (!landed) {
        atomicOr(ctl.status, DEV_ERR_TIMEOUT_DRAIN);
        // as in gemm_tc2_kernel: a fill could not be observed, so wait out a
        // grace period far longer than any copy's latency
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // -------------------------------------------------------------- MMA
      int stage = 0, stage1 = 0;  // wide ring / half-tile ring cursors
      uint32_t phase = 0, phase1 = 0;
      int use0 = 0, use1 = 0;  // completed uses of TMEM half 0 / 1
      bool ok = true;
      bool issued_any = false;
      int ff = 0;
      WideWork wk(sh, cluster_id, num_clusters);
      WideUnit u;
      while (ok && wk.next(u)) {
        const WidePhases ph(u, sh.num_kb, sh.w_lead);
        const int hf = ff, hs = ff ^ 1;
        if (u.wide) {
          // wide unit: the 48 KB ring (kept free of the half-tile ring's
          // selects, as the producer's loop)
          for (int i = 0; i < ph.nblocks; ++i) {
            int kb;
            bool f0, f1;
            ph.block(i, kb, f0, f1);
            // a half's first block waits until the epilogue released its last
            // use (with J = 0 block 0 is the first block of both halves)
#pragma unroll
            for (int w = 0; w < 2; ++w) {
              if (!ok || !(w == 0 ? i == 0 : i == ph.first_h1())) continue;
              const int h = w == 0 ? hf : hs;
              const uint32_t uses = static_cast<uint32_t>(h == 0 ? use0 : use1);
              if (!mbar_wait_bounded_cluster(&tempty[h], (uses & 1u) ^ 1u, abort_flag, ctl.timeout_ns)) {
                if (!*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_MMA);
                ok = false;
              }
            }
            if (!ok) break;
            tc_fence_after();
            if (!mbar_wait_bounded_cluster(&full[stage], phase, abort_flag, ctl.timeout_ns)) {
              if (!*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_MMA);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * L::STAGE_BYTES);
            const uint32_t sb0 = sa + static_cast<uint32_t>(L::A_BYTES + hf * L::HB_BYTES);
            const uint32_t sb1 = sa + static_cast<uint32_t>(L::A_BYTES + hs * L::HB_BYTES);
            const uint32_t d0 = tmem_base + static_cast<uint32_t>(hf * HBN);
            const uint32_t d1 = tmem_base + static_cast<uint32_t>(hs * HBN);
            // a half's first block (k-block 0 of the first column, J of the
            // second) starts its sum.  The two halves' MMAs alternate at every
            // K slice (measured faster than all of one half's slices first)
            const uint32_t acc0 = i == 0 ? 0u : 1u;
            const uint32_t acc1 = i == ph.first_h1() ? 0u : 1u;
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k) {
              const uint64_t ad =
                  A_MN ? sdesc_sw128(sa + k * MN_KSTEP, MN_BOX, 1024) : sdesc_sw128(sa + k * 32, 16, 1024);
              const uint64_t bd0 =
                  B_MN ? sdesc_sw128(sb0 + k * MN_KSTEP, MN_BOX, 1024) : sdesc_sw128(sb0 + k * 32, 16, 1024);
              const uint64_t bd1 =
                  B_MN ? sdesc_sw128(sb1 + k * MN_KSTEP, MN_BOX, 1024) : sdesc_sw128(sb1 + k * 32, 16, 1024);
              if (f0) umma_bf16_pair(d0, ad, bd0, IDESC, k == 0 ? acc0 : 1u);
              if (f1) umma_bf16_pair(d1, ad, bd1, IDESC, k == 0 ? acc1 : 1u);
            }
            issued_any = true;
            umma_commit_pair_multicast(&empty[stage], 0x3);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            if (i == ph.last_h0()) {
              umma_commit_pair_multicast(&tfull[hf], 0x3);
              (hf == 0 ? use0 : use1) += 1;
            }
            if (i == ph.last_h1()) {
              umma_commit_pair_multicast(&tfull[hs], 0x3);
              (hs == 0 ? use0 : use1) += 1;
            }
          }
        } else {
          // half tile: the 32 KB ring, into TMEM half hf
          const uint32_t uses = static_cast<uint32_t>(hf == 0 ? use0 : use1);
          if (!mbar_wait_bounded_cluster(&tempty[hf], (uses & 1u) ^ 1u, abort_flag, ctl.timeout_ns)) {
            if (!*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_MMA);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + static_cast<uint32_t>(hf * HBN);
          for (int kb = 0; kb < sh.num_kb; ++kb) {
            if (!mbar_wait_bounded_cluster(&full1[stage1], phase1, abort_flag, ctl.timeout_ns)) {
              if (!*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_MMA);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage1 * L::STAGE1_BYTES);
            const uint32_t sb = sa + static_cast<uint32_t>(L::A_BYTES);
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k) {
              const uint64_t ad =
                  A_MN ? sdesc_sw128(sa + k * MN_KSTEP, MN_BOX, 1024) : sdesc_sw128(sa + k * 32, 16, 1024);
              const uint64_t bd =
                  B_MN ? sdesc_sw128(sb + k * MN_KSTEP, MN_BOX, 1024) : sdesc_sw128(sb + k * 32, 16, 1024);
              umma_bf16_pair(d, ad, bd, IDESC, (kb != 0 || k != 0) ? 1u : 0u);
            }
            issued_any = true;
            umma_commit_pair_multicast(&empty1[stage1], 0x3);
            if (++stage1 == S1) {
              stage1 = 0;
              phase1 ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit_pair_multicast(&tfull[hf], 0x3);
          (hf == 0 ? use0 : use1) += 1;
        }
        if (!u.wide) ff ^= 1;
      }
      if (issued_any) {
        umma_commit_pair_local(drain);
        if (!mbar_wait_timeout(drain, 0, ctl.timeout_ns)) atomicOr(ctl.status, DEV_ERR_TIMEOUT_DRAIN);
      }
    }
  } else {
    // ------------------------------------------------------------- epilogue
    constexpr int HALVES = 8 / Epi::kEpiWarps;
    const int quad = warp & 3;
    const int first_half = HALVES == 1 ? (warp - 2) >> 2 : 0;
    const int row = quad * 32 + lane;
    const uint32_t leader_tempty = mapa_shared(smem_u32(tempty), 0);
    const uint32_t stage_base = smem_u32(smem + L::RING_BYTES) +
                                static_cast<uint32_t>((warp - 2) * Epi::kStoreSlots * STORE_SLOT_BYTES);
    int use0 = 0, use1 = 0;  // consumed uses of TMEM half 0 / 1
    int ff = 0;
    bool ok = true;
    WideWork wk(sh, cluster_id, num_clusters);
    WideUnit u;
    while (ok && wk.next(u)) {
      // the unit's tile columns in the order their halves complete
      for (int j = 0; j < (u.wide ? 2 : 1); ++j) {
        const int th = j == 0 ? ff : (ff ^ 1);
        const int tv = u.tv + j;
        if constexpr (EpiHasPrefetch<Epi>::value)
          Epi::prefetch(ep, sh.M, sh.N, (u.tm * 2 + static_cast<int>(rank)) * 128 + row,
                        tv * HBN + first_half * (HBN / 2), HALVES * (HBN / 2));
        int& uses = th == 0 ? use0 : use1;
        bool got = mbar_wait_bounded(&tfull[th], static_cast<uint32_t>(uses & 1), abort_flag, ctl.timeout_ns);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
          if (lane == 0 && !*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_EPILOGUE);
          ok = false;
          break;
        }
        ++uses;
        tc_fence_after();
        EpiCtx c;
        c.M = sh.M;
        c.N = sh.N;
        c.tm = u.tm * 2 + static_cast<int>(rank);
        c.tn = tv;
        c.row = row;
        c.m = c.tm * 128 + row;
        c.m0 = c.tm * 128 + quad * 32;
        c.quad = quad;
        c.lane = lane;
        c.acc_scale = acc_scale;
        c.taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(th * HBN);
        c.stage = stage_base;
        c.nsplit = 0;
#pragma unroll 1
        for (int hh = 0; hh < HALVES; ++hh) {
          const int half = first_half + hh;
          c.c0 = half * (HBN / 2);
          c.c1 = c.c0 + HBN / 2;
          c.part = tv * 2 + half;
          Epi::template run<HBN>(ep, c);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(leader_tempty + static_cast<uint32_t>(th * 8));
      }
      if (!u.wide) ff ^= 1;
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, L::TMEM_COLS);
  }
}

}  // namespace coda
