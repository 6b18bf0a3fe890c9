// Grouped 2-SM GEMM: two independent problems in one persistent launch.
//
// The backward pass has pairs of GEMMs that read the same operand and do not
// depend on each other: the data gradient and the weight gradient of a layer.
// Launched one after the other, each pays a partly idle last wave and a
// kernel prologue.  Here the SM pairs take the tiles of both problems from one
// schedule, so there is one tail and one prologue.  Used where it measured
// faster than two launches: the first layer (dX / dW1, 1.3 % at the 7B size)
// and the LM-head's dH / dW per vocabulary chunk (0.5 %).  The second layer's
// pair (dgrad2 / wgrad2, six times larger) measured 4-5 % slower grouped, in
// every tile order tried, and stays two launches: on a power-limited part
// the idle SMs of a partial wave let the busy ones clock higher, so filling
// them buys little.
//
// Problem 0 has A K-major or MN-major and B MN-major; problem 1 likewise
// (template flags), each with its own epilogue program.  With FP8 both
// problems take 8-bit operands of the same formats (kind::f8f6f4), each with
// its own pair of per-tensor scales.  The pipeline (TMA
// producer, 2-SM MMA issuer, epilogue warps, bounded waits, abort and drain)
// is that of gemm_tc2_kernel; only the tile sequence and the per-tile choice
// of operands, descriptors and epilogue differ.
//
// Schedule (the same arithmetic in every role, so no tile ids are passed
// between warps or CTAs).  Tiles of the two problems cost different amounts
// (about one unit per k-block).  The heavy problem's tiles are dealt
// round-robin first.  Every cluster that received one heavy tile fewer than
// the others then takes q light tiles (q = heavy cost / light cost, rounded),
// and the remaining light tiles are dealt round-robin.  Per-cluster totals
// end within about one light tile of each other.
#pragma once

#include "gemm_tc2.cuh"

namespace coda {

struct GroupSched {
  int P;       // clusters (SM pairs)
  int heavy;   // the problem whose tiles cost more (0 or 1)
  int nH, nL;  // tile counts of the heavy and the light problem
  int q;       // catch-up light tiles per cluster that holds one heavy tile fewer
};

// The k-th tile (k = 0, 1, ...) of cluster c: its problem and its index in
// that problem's raster.  False once the cluster has no tiles left.
__host__ __device__ __forceinline__ bool group_tile(const GroupSched& s, int c, int k, int& prob, int& t) {
  const int r0 = s.nH % s.P;
  const int hc = s.nH / s.P + (c < r0 ? 1 : 0);
  if (k < hc) {
    prob = s.heavy;
    t = c + k * s.P;
    return true;
  }
  k -= hc;
  const int cu_want = (s.P - r0) * s.q;
  const int cu_total = r0 > 0 ? (cu_want < s.nL ? cu_want : s.nL) : 0;
  int cu_first = 0, cu_count = 0;
  if (r0 > 0 && c >= r0) {
    cu_first = (c - r0) * s.q;
    const int left = cu_total - cu_first;
    cu_count = left <= 0 ? 0 : (left < s.q ? left : s.q);
  }
  if (k < cu_count) {
    prob = 1 - s.heavy;
    t = cu_first + k;
    return true;
  }
  k -= cu_count;
  const int j = cu_total + c + k * s.P;
  if (j < s.nL) {
    prob = 1 - s.heavy;
    t = j;
    return true;
  }
  return false;
}

template <class Epi0, class Epi1>
struct GroupArgs {
  CUtensorMap tmA0, tmB0, tmA1, tmB1;
  GemmShape sh0, sh1;
  GroupSched sched;
  typename Epi0::Params ep0;
  typename Epi1::Params ep1;
  // FP8 operands: each problem's per-tensor dequantisation scales (null = 1)
  const float* scale_a0;
  const float* scale_b0;
  const float* scale_a1;
  const float* scale_b1;
};

// This CTA's halves of one k-block of a 256 x 256 pair tile (B MN-major or
// K-major, A either), completing on the leader's barrier.  A k-block is 128
// bytes of K per row: 64 bf16 or 128 8-bit codes.  MN-major halves are 128
// (M/N) wide: two 64-wide bf16 boxes or one 128-wide box of codes.
template <bool A_MN, bool B_MN, bool FP8>
__device__ __forceinline__ void pair_load_kblock(uint8_t* sa, uint8_t* sb, const CUtensorMap* ta,
                                                 const CUtensorMap* tb, uint32_t bar, int kb, int m0, int n0) {
  constexpr int BKE = FP8 ? 128 : BK;     // K elements per k-block
  constexpr int MNB = FP8 ? 128 : 64;     // M/N elements per MN-major box
  constexpr int MN_BOX = 128 * BKE;       // bytes per MN-major box
  if (!A_MN) {
    tma_load_2d_pair(sa, ta, bar, kb * BKE, m0);
  } else {
#pragma unroll
    for (int i = 0; i < 128 / MNB; ++i) tma_load_2d_pair(sa + i * MN_BOX, ta, bar, m0 + i * MNB, kb * BKE);
  }
  if (!B_MN) {
    tma_load_2d_pair(sb, tb, bar, kb * BKE, n0);
  } else {
#pragma unroll
    for (int i = 0; i < 128 / MNB; ++i) tma_load_2d_pair(sb + i * MN_BOX, tb, bar, n0 + i * MNB, kb * BKE);
  }
}

// The four MMAs of one k-block (K = 16 bf16 or 32 8-bit codes each).
template <bool A_MN, bool B_MN, bool FP8>
__device__ __forceinline__ void pair_mma_kblock(uint32_t d_tmem, uint32_t sa, uint32_t sb, bool first,
                                                uint32_t f8_fmt) {
  constexpr uint32_t IDESC0 = FP8 ? idesc_f8_f32(BM2, 256, A_MN, B_MN) : idesc_bf16_f32(BM2, 256, A_MN, B_MN);
  constexpr int MN_BOX = FP8 ? 16384 : 8192;
  constexpr int MN_KSTEP = FP8 ? 4096 : 2048;  // bytes per MMA K slice, MN-major
  const uint32_t idesc = FP8 ? (IDESC0 | f8_fmt) : IDESC0;
#pragma unroll
  for (int k = 0; k < BK / UMMA_K; ++k) {
    const uint64_t ad = A_MN ? sdesc_sw128(sa + k * MN_KSTEP, MN_BOX, 1024) : sdesc_sw128(sa + k * 32, 16, 1024);
    const uint64_t bd = B_MN ? sdesc_sw128(sb + k * MN_KSTEP, MN_BOX, 1024) : sdesc_sw128(sb + k * 32, 16, 1024);
    if (FP8)
      umma_e4m3_pair(d_tmem, ad, bd, idesc, (first && k == 0) ? 0u : 1u);
    else
      umma_bf16_pair(d_tmem, ad, bd, idesc, (first && k == 0) ? 0u : 1u);
  }
}

template <class Epi0, class Epi1>
constexpr int group_stage_bytes() {
  return Epi0::kEpiWarps * (Epi0::kStoreSlots > Epi1::kStoreSlots ? Epi0::kStoreSlots : Epi1::kStoreSlots) *
         STORE_SLOT_BYTES;
}

template <int STAGES, bool A_MN0, bool B_MN0, bool A_MN1, bool B_MN1, class Epi0, class Epi1, bool FP8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(gemm_threads<Epi0>(), 1)
    gemm_tc2_group_kernel(const __grid_constant__ GroupArgs<Epi0, Epi1> g, const KernelCtl ctl) {
  static_assert(Epi0::kEpiWarps == Epi1::kEpiWarps, "both epilogue programs use the same warps");
  static_assert(!FP8 || (Epi0::kAccScale && Epi1::kAccScale), "8-bit operands need the accumulator scale");
  constexpr int BN = 256;
  constexpr int HB = BN / 2;
  using L = Gemm2Smem<BN, STAGES, group_stage_bytes<Epi0, Epi1>()>;
  constexpr int SLOTS = group_stage_bytes<Epi0, Epi1>() / (Epi0::kEpiWarps * STORE_SLOT_BYTES);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::RING_BYTES + L::STORE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* fill_report = reinterpret_cast<uint32_t*>(tmem_slot + 2);  // leader: the peer's fills + 1

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster_id = blockIdx.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * Epi0::kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *fill_report = 0;
    fence_mbar_init();
    tma_prefetch_desc(&g.tmA0);
    tma_prefetch_desc(&g.tmB0);
    tma_prefetch_desc(&g.tmA1);
    tma_prefetch_desc(&g.tmB1);
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
      int prob, t;
      for (int k = 0; ok && group_tile(g.sched, cluster_id, k, prob, t); ++k) {
        const GemmShape& sh = prob == 0 ? g.sh0 : g.sh1;
        int tm, tn;
        tile_coords(t, sh, tm, tn);
        const int m0 = tm * BM2 + static_cast<int>(rank) * 128;
        const int n0 = tn * BN + static_cast<int>(rank) * HB;
        for (int kb = 0; kb < sh.num_kb; ++kb) {
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
            if (prob == 0)
              pair_load_kblock<A_MN0, B_MN0, FP8>(sa, sb, &g.tmA0, &g.tmB0, bar, kb, m0, n0);
            else
              pair_load_kblock<A_MN1, B_MN1, FP8>(sa, sb, &g.tmA1, &g.tmB1, bar, kb, m0, n0);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every fill of both CTAs observed landed (as in gemm_tc2_kernel)
      if (!pair_fills_landed(leader, issued, skipped, full, STAGES, L::STAGE_BYTES, fill_report, ctl.timeout_ns)) {
        atomicOr(ctl.status, DEV_ERR_TIMEOUT_DRAIN);
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // -------------------------------------------------------------- MMA
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool issued_any = false;
      int prob, t;
      for (int it = 0; ok && group_tile(g.sched, cluster_id, it, prob, t); ++it) {
        const GemmShape& sh = prob == 0 ? g.sh0 : g.sh1;
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait_bounded_cluster(&tempty[acc], acc_phase ^ 1u, abort_flag, ctl.timeout_ns)) {
          if (!*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_MMA);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < sh.num_kb; ++kb) {
          if (!mbar_wait_bounded_cluster(&full[stage], phase, abort_flag, ctl.timeout_ns)) {
            if (!*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_MMA);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * L::STAGE_BYTES);
          const uint32_t sb = sa + L::A_BYTES;
          if (prob == 0)
            pair_mma_kblock<A_MN0, B_MN0, FP8>(d_tmem, sa, sb, kb == 0, ctl.f8_fmt);
          else
            pair_mma_kblock<A_MN1, B_MN1, FP8>(d_tmem, sa, sb, kb == 0, ctl.f8_fmt);
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
      if (issued_any) {
        umma_commit_pair_local(drain);
        if (!mbar_wait_timeout(drain, 0, ctl.timeout_ns)) atomicOr(ctl.status, DEV_ERR_TIMEOUT_DRAIN);
      }
    }
  } else {
    // ------------------------------------------------------------- epilogue
    constexpr int HALVES = 8 / Epi0::kEpiWarps;
    const int quad = warp & 3;
    const int first_half = HALVES == 1 ? (warp - 2) >> 2 : 0;
    const int row = quad * 32 + lane;
    const uint32_t leader_tempty = mapa_shared(smem_u32(tempty), 0);
    const uint32_t stage_base =
        smem_u32(smem + L::RING_BYTES) + static_cast<uint32_t>((warp - 2) * SLOTS * STORE_SLOT_BYTES);
    // each problem's accumulator scale (1 for bf16 operands): its operands'
    // scales times a host-given factor common to both problems
    float acc_scale[2] = {1.f, 1.f};
    if (FP8) {
      acc_scale[0] = ctl.scale_host * (g.scale_a0 ? *g.scale_a0 : 1.f) * (g.scale_b0 ? *g.scale_b0 : 1.f);
      acc_scale[1] = ctl.scale_host * (g.scale_a1 ? *g.scale_a1 : 1.f) * (g.scale_b1 ? *g.scale_b1 : 1.f);
    }
    int prob, t;
    for (int it = 0; group_tile(g.sched, cluster_id, it, prob, t); ++it) {
      const GemmShape& sh = prob == 0 ? g.sh0 : g.sh1;
      int tm, tn;
      tile_coords(t, sh, tm, tn);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      bool ok = mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag, ctl.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0 && !*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_EPILOGUE);
        break;
      }
      tc_fence_after();
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
      c.acc_scale = acc_scale[prob];
      c.taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN);
      c.stage = stage_base;
      c.nsplit = 0;
#pragma unroll 1
      for (int hh = 0; hh < HALVES; ++hh) {
        const int half = first_half + hh;
        c.c0 = half * (BN / 2);
        c.c1 = c.c0 + BN / 2;
        c.part = tn * 2 + half;
        if (prob == 0)
          Epi0::template run<BN>(g.ep0, c);
        else
          Epi1::template run<BN>(g.ep1, c);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(leader_tempty + static_cast<uint32_t>(acc * 8));
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
