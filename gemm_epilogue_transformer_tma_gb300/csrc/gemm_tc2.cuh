// 2-SM form of the persistent bf16 GEMM: a cluster of two CTAs (an SM pair)
// computes one 256 x BN output tile with tcgen05.mma.cta_group::2.
//
// Each CTA loads only its own half of the operands -- 128 rows of A and BN/2
// rows (columns) of B -- so per SM the shared-memory traffic per MMA is half
// of the 1-SM kernel's B traffic, which leaves room for a deeper ring (6
// stages of 32 KB).  The accumulator of each CTA holds its 128 output rows x
// BN columns in its own TMEM, so the epilogue programs of gemm_tc.cuh run
// unchanged (EpiCtx.tm is the 128-row block index).
//
// Roles, per CTA of the pair (rank 0 = leader, rank 1 = peer):
//   warp 0       TMA producer for this CTA's halves.  Both CTAs' copies of a
//                stage complete on the leader's full[s] barrier, which the
//                leader arms for the bytes of both halves.
//   warp 1       leader: MMA issuer.  It waits for full[s], issues the 2-SM
//                MMAs, and commits to empty[s] / tfull[] of both CTAs
//                (multicast).  Both CTAs' warp 1 allocate TMEM together
//                (cta_group::2).
//   warps 2..    epilogue on this CTA's 128 rows (4 or 8 warps, see
//                gemm_tc.cuh); release the accumulator by
//                arriving on the leader's tempty[].
// All waits are bounded as in the 1-SM kernel.  At the end of the producers,
// finished or stopped early, the peer reports how many stage fills it issued
// and the leader observes the last fill of every stage land, arming or
// trimming the barrier where only one CTA's copies were issued
// (pair_fills_landed); the peer's memory stays allocated until the final
// cluster barrier, which the leader's producer reaches only after that.
#pragma once

#include "gemm_tc.cuh"

namespace coda {

constexpr int BM2 = 256;  // output rows per CTA pair

// Work of one cluster.  Whole tiles first: tiles cluster, cluster + P, ...
// below sh.sk_first (every full wave).  The tiles from sk_first on, the last
// and partial wave, are each cut into sh.sk_ranges equal k-ranges.  Those
// units (k-range j of tile t) are taken range-major -- every split tile's
// first range, then every second range, ... -- and dealt round-robin, so the
// units that run at the same time cover the same k-range and read the same
// k-slices of their operand panels, as the whole tiles of one wave do.  A
// unit of a tile's last range owns the tile: its epilogue adds the fp32
// partials that the tile's earlier ranges left in their scratch slots
// (written by whichever clusters ran them) and runs the epilogue program.
// Every cluster meets all its partial units before its owner units, and
// partial units never wait, so no cluster waits on a waiting cluster.
// Producer, MMA issuer and epilogue walk the same sequence.
struct TilePiece {
  int tile, kb0, kb1;
  int slot;      // partial: its scratch slot; owner: the tile's first slot
  bool partial;  // an earlier k-range: accumulator to the slot, no epilogue program
  bool owner;    // the last k-range: the earlier ranges' partials are added before the epilogue
};

struct SplitWork {
  int next_whole, first_split, P, nkb, S, rem, u;
  __host__ __device__ SplitWork(const GemmShape& sh, int cluster, int num_clusters) {
    next_whole = cluster;
    first_split = sh.sk_first;
    P = num_clusters;
    nkb = sh.num_kb;
    S = sh.sk_ranges;
    rem = sh.tiles_m * sh.tiles_n - sh.sk_first;
    u = cluster;
  }
  // first k-block of k-range j of a split tile
  __host__ __device__ int kb_begin(int j) const {
    return static_cast<int>(static_cast<int64_t>(nkb) * j / S);
  }
  __host__ __device__ bool next(TilePiece& pc) {
    if (next_whole < first_split) {
      pc.tile = next_whole;
      pc.kb0 = 0;
      pc.kb1 = nkb;
      pc.slot = -1;
      pc.partial = pc.owner = false;
      next_whole += P;
      return true;
    }
    if (S < 2 || u >= S * rem) return false;
    const int j = u / rem;
    const int i = u - j * rem;
    pc.tile = first_split + i;
    pc.kb0 = kb_begin(j);
    pc.kb1 = kb_begin(j + 1);
    pc.partial = j < S - 1;
    pc.owner = j == S - 1;
    pc.slot = i * (S - 1) + (pc.partial ? j : 0);
    u += P;
    return true;
  }
};

// End of both producers of a CTA pair, whether their loops finished or
// stopped early.  The leader's full barriers count both CTAs' bytes and the
// peer cannot wait on them, so the peer reports how many fills it issued (a
// store into the leader's report word), and the leader makes sure that the
// last fill of every stage has landed before its producer goes on; the
// peer's shared memory stays allocated until the kernel's final cluster
// barrier, which the leader's producer reaches only after this.
//
// pair_report_wait: the leader's bounded wait for the peer's report (the
// count + 1, so that 0 means "not yet").  The limit is twice the wait limit
// plus the 10 ms a sleeping try_wait may overrun it: the peer's producer
// stops at most one expired wait after the leader's.
__device__ __forceinline__ bool pair_report_wait(const uint32_t* report, uint64_t timeout_ns, uint32_t& r) {
  r = ld_acquire_cluster_u32(report);
  if (r != 0) return true;
  const uint64_t t0 = globaltimer_ns();
  while ((r = ld_acquire_cluster_u32(report)) == 0)
    if (globaltimer_ns() - t0 > 2 * timeout_ns + 20000000ull) return false;
  return true;
}

// pair_ring_landed: the leader's walk over one ring.  Fill i goes to stage
// i % stages in lap i / stages; the leader armed fills [0, issued) except
// `skipped`, the peer issued [0, peer).  Only the last `stages` fills can be
// in flight: any older one was consumed before its stage was filled again.
// Where the leader never armed a fill that the peer issued (it stopped
// first, or the test hook skipped it), it arms the barrier for the peer's
// bytes alone; where the peer never issued a fill that the leader armed, it
// takes the peer's share off the expected bytes; then it waits for the
// phase.  peer_bytes(i, leader_armed) gives the peer's share of fill i.
template <class PeerBytes>
__device__ __forceinline__ bool pair_ring_landed(int issued, int skipped, int peer, uint64_t* full, int stages,
                                                 PeerBytes peer_bytes, uint64_t timeout_ns) {
  const int last = issued > peer ? issued : peer;
  bool ok = true;
  for (int i = last > stages ? last - stages : 0; i < last; ++i) {
    const bool armed = i < issued && i != skipped;
    const bool loaded = i < peer;
    if (!armed && !loaded) continue;
    uint64_t* bar = &full[i % stages];
    if (!armed)
      mbar_arrive_expect_tx(bar, peer_bytes(i, false));
    else if (!loaded)
      mbar_complete_tx(bar, peer_bytes(i, true));
    if (!mbar_wait_timeout(bar, static_cast<uint32_t>((i / stages) & 1), timeout_ns)) ok = false;
  }
  return ok;
}

// The hand-off for a kernel with one ring of equal fills.  Returns false
// when the report or a phase did not come in time.
__device__ __forceinline__ bool pair_fills_landed(bool leader, int issued, int skipped, uint64_t* full, int stages,
                                                  uint32_t peer_bytes, uint32_t* report, uint64_t timeout_ns) {
  if (!leader) {
    st_release_cluster_u32(mapa_shared(smem_u32(report), 0), static_cast<uint32_t>(issued) + 1u);
    return true;
  }
  uint32_t r;
  if (!pair_report_wait(report, timeout_ns, r)) return false;
  return pair_ring_landed(issued, skipped, static_cast<int>(r) - 1, full, stages,
                          [peer_bytes](int, bool) { return peer_bytes; }, timeout_ns);
}

// Wait (bounded, like the mbarrier waits) for a split partial's flag.
__device__ __forceinline__ bool split_flag_wait(const int* f, const volatile int* abort_flag, uint64_t timeout_ns) {
  if (ld_acquire_gpu(f) != 0) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    __nanosleep(200);
    if (ld_acquire_gpu(f) != 0) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

template <int BN, int STAGES, int EPI_BYTES>
struct Gemm2Smem {
  static constexpr int A_BYTES = 128 * BK * 2;        // this CTA's 128 rows of A
  static constexpr int B_BYTES = (BN / 2) * BK * 2;   // this CTA's BN/2 rows of B
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int STORE_BYTES = EPI_BYTES;       // epilogue store staging
  static constexpr int BAR_BYTES = 512;
  static constexpr int TOTAL = RING_BYTES + STORE_BYTES + BAR_BYTES + 1024;
  static_assert(TOTAL <= MAX_DYN_SMEM, "shared memory budget");
  static constexpr int TMEM_COLS = 2 * BN;
  static_assert(TMEM_COLS <= 512, "TMEM has 512 columns");
  static_assert((2 * STAGES + 5) * 8 + 12 <= BAR_BYTES, "barrier area too small");
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "1 KB aligned halves");
};

// SPLIT: the instantiation that can split tiles (launched only when the
// launch's split region is not empty); without it the partial and owner paths
// are compiled out and the epilogue reads the accumulator from TMEM alone.
template <int BN, int STAGES, bool A_MN, bool B_MN, bool B_DUAL, class Epi, bool FP8 = false, bool SPLIT = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(gemm_threads<Epi>(), 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB2, const GemmShape sh, const KernelCtl ctl,
                    const __grid_constant__ typename Epi::Params ep) {
  using L = Gemm2Smem<BN, STAGES, epi_stage_bytes<Epi>()>;
  static_assert(!(B_DUAL && B_MN), "dual-box B is K-major only");
  static_assert(BN == 256, "the pair kernel is instantiated for 256-column tiles");
  constexpr int HB = BN / 2;  // B rows held by one CTA
  constexpr uint32_t IDESC0 = FP8 ? idesc_f8_f32(BM2, BN, A_MN, B_MN) : idesc_bf16_f32(BM2, BN, A_MN, B_MN);
  constexpr int BKE = FP8 ? 128 : BK;         // K elements per 128-byte k-block row (K-major operands)
  // MN-major operands: boxes of 128 bytes along M/N (64 bf16 or 128 e4m3) by
  // BKE rows of K; one MMA's K slice is 16 (bf16) or 32 (8-bit) such rows
  constexpr int MNB = FP8 ? 128 : 64;         // M/N elements per MN-major box
  constexpr int MN_BOX = 128 * BKE;           // bytes per MN-major box
  constexpr int MN_KSTEP = FP8 ? 4096 : 2048; // bytes per MMA K slice, MN-major

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::RING_BYTES + L::STORE_BYTES);  // leader's counts both halves
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;  // leader only: both CTAs' epilogues released the buffer
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* fill_report = reinterpret_cast<uint32_t*>(tmem_slot + 2);  // leader: the peer's fills + 1

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
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * Epi::kEpiWarps);  // lane 0 of every epilogue warp of both CTAs
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *fill_report = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (B_DUAL) tma_prefetch_desc(&tmB2);
  }
  // barriers of both CTAs initialised before anyone signals across the pair
  cluster_sync_all();
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, L::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the set-up above may overlap the previous kernel; operands and outputs
  // are touched only after it has completed
  griddep_launch_dependents();
  griddep_wait();
  const float acc_scale = acc_scale_of(ctl);
  const uint32_t idesc = FP8 ? (IDESC0 | ctl.f8_fmt) : IDESC0;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      const uint32_t leader_full = mapa_shared(smem_u32(full), 0);
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0, skipped = -1;  // k-block fills so far; the one the test hook left unarmed
      bool ok = true;
      bool skip = ctl.skip_first_stage == 1 && cluster_id == 0 && leader;
      // test hook: the first pair's second CTA stops before its first copy
      if (ctl.skip_first_stage == 2 && cluster_id == 0 && !leader) ok = false;
      SplitWork wk(sh, cluster_id, num_clusters);
      TilePiece pc;
      while (ok && wk.next(pc)) {
        int tm, tn;
        tile_coords(pc.tile, sh, tm, tn);
        const int m0 = tm * BM2 + static_cast<int>(rank) * 128;  // this CTA's A rows
        for (int kb = pc.kb0; kb < pc.kb1; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, ctl.timeout_ns)) {
            if (!*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_PRODUCER);
            ok = false;
            break;
          }
          if (skip) {
            skip = false;  // test hook: the leader never arms this stage
            skipped = issued;
          } else {
            uint8_t* sa = smem + stage * L::STAGE_BYTES;
            uint8_t* sb = sa + L::A_BYTES;
            const uint32_t bar = leader_full + static_cast<uint32_t>(stage * 8);
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * L::STAGE_BYTES);
            if (!A_MN) {
              tma_load_2d_pair(sa, &tmA, bar, kb * BKE, m0);
            } else {
#pragma unroll
              for (int i = 0; i < 128 / MNB; ++i) tma_load_2d_pair(sa + i * MN_BOX, &tmA, bar, m0 + i * MNB, kb * BKE);
            }
            if (B_DUAL) {
              // leader: gate rows of the tile, peer: the matching up rows
              tma_load_2d_pair(sb, leader ? &tmB : &tmB2, bar, kb * BKE, tn * HB);
            } else if (!B_MN) {
              tma_load_2d_pair(sb, &tmB, bar, kb * BKE, tn * BN + static_cast<int>(rank) * HB);
            } else {
#pragma unroll
              for (int i = 0; i < HB / MNB; ++i)
                tma_load_2d_pair(sb + i * MN_BOX, &tmB, bar, tn * BN + static_cast<int>(rank) * HB + i * MNB, kb * BKE);
            }
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every fill of both CTAs observed landed before shared memory can be
      // released (the leader's producer holds the final cluster barrier)
      if (!pair_fills_landed(leader, issued, skipped, full, STAGES, L::STAGE_BYTES, fill_report, ctl.timeout_ns)) {
        atomicOr(ctl.status, DEV_ERR_TIMEOUT_DRAIN);
        // a fill could not be observed: wait out a grace period far longer
        // than any copy's latency (the bytes in flight on the whole GPU, at
        // most the rings of the resident CTAs, 152 SMs x 6 stages x 32 KB =
        // 29 MB, take HBM about 5 us) before the peer can exit
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      if (leader) {
        // -------------------------------------------------------------- MMA
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        bool ok = true;
        bool issued_any = false;
        SplitWork wk(sh, cluster_id, num_clusters);
        TilePiece pc;
        for (; ok && wk.next(pc); ++it) {
          const int acc = it & 1;
          const uint32_t acc_phase = (it >> 1) & 1;
          if (!mbar_wait_bounded_cluster(&tempty[acc], acc_phase ^ 1u, abort_flag, ctl.timeout_ns)) {
            if (!*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_MMA);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
          for (int kb = pc.kb0; kb < pc.kb1; ++kb) {
            if (!mbar_wait_bounded_cluster(&full[stage], phase, abort_flag, ctl.timeout_ns)) {
              if (!*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_MMA);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * L::STAGE_BYTES);
            const uint32_t sb = sa + L::A_BYTES;
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k) {
              const uint64_t ad =
                  A_MN ? sdesc_sw128(sa + k * MN_KSTEP, MN_BOX, 1024) : sdesc_sw128(sa + k * 32, 16, 1024);
              const uint64_t bd =
                  B_MN ? sdesc_sw128(sb + k * MN_KSTEP, MN_BOX, 1024) : sdesc_sw128(sb + k * 32, 16, 1024);
              const uint32_t accumulate = (kb != pc.kb0 || k != 0) ? 1u : 0u;
              if (FP8)
                umma_e4m3_pair(d_tmem, ad, bd, idesc, accumulate);
              else
                umma_bf16_pair(d_tmem, ad, bd, idesc, accumulate);
            }
            issued_any = true;
            umma_commit_pair_multicast(&empty[stage], 0x3);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit_pair_multicast(&tfull[acc], 0x3);
        }
        // every MMA this thread issued has completed before TMEM is freed
        if (issued_any) {
          umma_commit_pair_local(drain);
          if (!mbar_wait_timeout(drain, 0, ctl.timeout_ns)) atomicOr(ctl.status, DEV_ERR_TIMEOUT_DRAIN);
        }
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
    const int ew = warp - 2;  // epilogue warp index: its split flag
    int it = 0;
    SplitWork wk(sh, cluster_id, num_clusters);
    TilePiece pc;
    for (; wk.next(pc); ++it) {
      int tm, tn;
      tile_coords(pc.tile, sh, tm, tn);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      const bool partial = SPLIT && pc.partial;
      const bool owner = SPLIT && pc.owner;
      if constexpr (EpiHasPrefetch<Epi>::value)
        if (!partial)
          Epi::prefetch(ep, sh.M, sh.N, (tm * 2 + static_cast<int>(rank)) * 128 + row,
                        tn * BN + first_half * (BN / 2), HALVES * (BN / 2));
      bool ok = mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag, ctl.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0 && !*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_EPILOGUE);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if (partial) {
        // the first piece of this cluster's split range: the raw accumulator
        // of this warp's rows to the cluster's slot, then its flag
        float4* dst = reinterpret_cast<float4*>(
            ctl.sk_parts + static_cast<int64_t>((pc.slot * 2 + static_cast<int>(rank)) * 4 + quad) *
                               SPLIT_PART_FLOATS);
#pragma unroll 1
        for (int cc = first_half * (BN / 2); cc < (first_half + HALVES) * (BN / 2); cc += 32) {
          float v[32];
          tmem_ld32(taddr + static_cast<uint32_t>(cc), v);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_cg_f4(dst + split_part_f4_index(cc, lane) + j * 32,
                     make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(&ctl.sk_flags[(pc.slot * 2 + static_cast<int>(rank)) * 8 + ew], 1);
      } else {
        EpiCtx c;
        c.M = sh.M;
        c.N = sh.N;
        c.tm = tm * 2 + static_cast<int>(rank);
        c.tn = tn;
        c.row = row;
        c.m = c.tm * 128 + row;
        c.m0 = c.tm * 128 + quad * 32;
        c.quad = quad;
        c.lane = lane;
        c.acc_scale = acc_scale;
        c.taddr = taddr;
        c.stage = stage_base;
        c.nsplit = 0;
        const int n_parts = owner ? wk.S - 1 : 0;  // the tile's earlier k-ranges, one slot each
        if (owner) {
          // wait for each earlier k-range's partial of these rows
          bool got = n_parts <= kMaxSplitParts;
#pragma unroll
          for (int j = 0; j < kMaxSplitParts; ++j) {
            if (got && j < n_parts) {
              const int slot = pc.slot + j;
              const int* f = &ctl.sk_flags[(slot * 2 + static_cast<int>(rank)) * 8 + ew];
              bool seen = true;
              if (lane == 0) seen = split_flag_wait(f, abort_flag, ctl.timeout_ns);
              got = __shfl_sync(0xffffffffu, seen, 0);
              if (got) {
                (void)ld_acquire_gpu(f);  // every lane: its partial loads come after the flag
                c.split[j] = ctl.sk_parts +
                             static_cast<int64_t>((slot * 2 + static_cast<int>(rank)) * 4 + quad) * SPLIT_PART_FLOATS;
                c.nsplit = j + 1;
              }
            }
          }
          if (!got) {
            if (lane == 0 && !*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_EPILOGUE);
            break;
          }
        }
#pragma unroll 1
        for (int hh = 0; hh < HALVES; ++hh) {
          const int half = first_half + hh;
          c.c0 = half * (BN / 2);
          c.c1 = c.c0 + BN / 2;
          c.part = tn * 2 + half;
          Epi::template run<BN>(ep, c);
        }
        if (owner) {
          // every lane has read the partials: clear the flags for the next launch
          __syncwarp();
          if (lane == 0)
            for (int j = 0; j < n_parts; ++j)
              st_relaxed_gpu(&ctl.sk_flags[((pc.slot + j) * 2 + static_cast<int>(rank)) * 8 + ew], 0);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(leader_tempty + static_cast<uint32_t>(acc * 8));
    }
    // the last stores have landed before shared memory is released
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  __syncwarp();
  tc_fence_before();
  // both CTAs done with the pair's TMEM and with each other's barriers
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, L::TMEM_COLS);
  }
}

}  // namespace coda
