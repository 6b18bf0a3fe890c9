// Persistent, warp-specialised bf16 GEMM for sm_103a with a programmable
// epilogue.
//
//   C[m, n] = sum_k A[m, k] * B[k, n]          (fp32 accumulate in TMEM)
//
// The mainloop is fixed; what happens to the accumulator before it leaves
// the chip is a template policy ("epilogue program").  This is the split the
// CODA write-up describes (section 尾声: a GEMM kernel = mainloop + epilogue,
// and the epilogue runs while the result is still on chip; section 五种积木:
// the epilogue exposes elementwise, vector load/store, tile load/store,
// block-reduction and stateful primitives).
//
// CTA = 2 + E warps (E = 4 or 8 epilogue warps, a trait of the epilogue program):
//   warp 0       TMA producer: fills a STAGES-deep shared-memory ring with A
//                and B tiles (128-byte swizzle), completion on mbarriers.
//   warp 1       TMEM allocator and MMA issuer: one elected thread issues
//                tcgen05.mma (M=128, N=BN, K=16) into one of two TMEM
//                accumulator buffers and commits to mbarriers.
//   warps 2..    epilogue: tcgen05.ld the accumulator (one row per thread),
//                run the epilogue program, stage its outputs in shared memory
//                and store them with TMA (32 x 32 blocks per warp), release
//                the buffer.
//                The program runs once per 128-column half of the tile: with
//                8 warps, two per TMEM lane quadrant take one half each; with
//                4 warps, each warp runs both halves in turn.  Block
//                reductions along a row (partial RMS, CE statistics,
//                SwiGLU-backward partials) are therefore per half tile
//                (PART_COLS columns).  All programs use 4 warps, which leaves
//                the producer's and MMA issuer's sub-partitions less crowded
//                (8 measured slower for GEMM2 and no faster for the
//                SwiGLU-backward epilogue once stores went through TMA).
// Two TMEM buffers let the epilogue of tile i overlap the mainloop of i+1.
//
// Operand layouts (row-major storage, element = bf16):
//   A K-major : A stored [M][K]          A MN-major : A stored [K][M]
//   B K-major : B stored [N][K]          B MN-major : B stored [K][N]
// B_DUAL (K-major only): the B tile is two half-height boxes from two tensor
// maps (used for the gate / up halves of a SwiGLU projection).
//
// Every mbarrier wait is bounded (wall-clock limit); on expiry the kernel
// records an error bit in the device status word, tells the other roles to
// stop, waits (bounded) for its own copies and MMAs in flight, frees TMEM and
// returns.
#pragma once

#include <cuda_fp8.h>

#include "ptx.cuh"

namespace coda {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int UMMA_K = 16;
// CTA size for an epilogue program with kEpiWarps epilogue warps (4 or 8)
template <class Epi>
constexpr int gemm_threads() { return 64 + 32 * Epi::kEpiWarps; }
constexpr int PART_COLS = 128;     // columns per block-reduction partial (half a tile)
constexpr int kMaxSplitParts = 5;  // earlier k-ranges (partials) a split tile may have

struct GemmShape {
  int M, N, K;        // logical problem (N = output columns the epilogue sees)
  int tiles_m, tiles_n;
  int num_kb;
  int group_m;        // tile raster: groups of group_m M-tiles sweep all N-tiles
  // SM-pair kernel only: tiles [sk_first, tiles) (the last, partial wave)
  // are each split into sk_ranges k-ranges run by different clusters;
  // sk_first = tiles_m * tiles_n (and sk_ranges = 1) means no split
  int sk_first;
  int sk_ranges;
  // wide-tile SM-pair kernel only (gemm_tc2w.cuh): tiles_n counts 256-column
  // tiles (even); w_lead = J, the single-half k-blocks before and after a
  // wide tile's shared ones; wide tiles from w_single_from on run as two
  // 256-column half tiles
  int w_lead;
  int w_single_from;
};

struct KernelCtl {
  int* status;        // device status word (atomicOr of DEV_ERR_* bits)
  uint64_t timeout_ns;
  int skip_first_stage;  // test hook: 1: CTA 0's producer never fills its first stage;
                         // 2 (SM-pair kernels): the first pair's second CTA issues no copy
  const float* scale_a;  // FP8 operands: per-tensor dequantisation scales (null = 1)
  const float* scale_b;
  uint32_t f8_fmt;       // FP8 operands: format bits of A and B (f8_format_bits)
  float scale_host;      // FP8 operands: a scale known on the host (1 otherwise)
  // split tiles (SM-pair kernel): partial-accumulator slots, one per (split
  // tile, earlier k-range) ([slot][rank][quad][32 rows x 256 columns] fp32),
  // and one flag per (slot, rank, epilogue warp); null when tiles are not split
  float* sk_parts;
  int* sk_flags;
};

// The accumulator's scale: the product of the operands' per-tensor scales
// (1 for bf16 operands).  Read after griddep_wait (a previous kernel may have
// produced the scales).
__device__ __forceinline__ float acc_scale_of(const KernelCtl& ctl) {
  float s = ctl.scale_host;
  if (ctl.scale_a != nullptr) s *= *ctl.scale_a;
  if (ctl.scale_b != nullptr) s *= *ctl.scale_b;
  return s;
}

struct EpiCtx {
  int M, N;
  int tm, tn;
  int row;            // row inside the tile, 0..127 (= TMEM lane)
  int m;              // global row
  int quad;           // TMEM lane quadrant of this warp, 0..3
  int lane;
  int c0, c1;         // this thread's columns of the tile: [c0, c1)
  int part;           // index of its half-tile partial along the row (tn * 2 + half)
  float acc_scale;    // multiply the accumulator by this (FP8 operand scales; 1 for bf16)
  uint32_t taddr;     // TMEM address of (first lane of quadrant, column 0 of this accumulator)
  int m0;             // global row of this warp's lane 0 (the warp stores rows m0 .. m0 + 31)
  uint32_t stage;     // shared address of this warp's store-staging slots
  // a split tile: fp32 partial accumulators of the tile's other K ranges,
  // added to the TMEM accumulator as it is read (acc_ld32)
  int nsplit;
  const float* split[kMaxSplitParts];
};

// Layout of one warp's partial accumulator: 32 rows x 256 columns, stored as
// [column / 4][row][4] so that a warp's 32 lanes (rows) touch 512 contiguous
// bytes per 4-column group.
__device__ __forceinline__ int split_part_f4_index(int col, int lane) { return (col >> 2) * 32 + lane; }
constexpr int SPLIT_PART_FLOATS = 32 * 256;  // per (cluster, rank, quad)

// 32 accumulator columns from `col` for this thread's row: TMEM, plus the
// partial sums of a split tile's other K ranges.
__device__ __forceinline__ void acc_ld32(const EpiCtx& c, int col, float (&v)[32]) {
  tmem_ld32(c.taddr + static_cast<uint32_t>(col), v);
  if (c.nsplit == 0) return;
#pragma unroll
  for (int q = 0; q < kMaxSplitParts; ++q) {
    if (q < c.nsplit) {
      const float4* src = reinterpret_cast<const float4*>(c.split[q]) + split_part_f4_index(col, c.lane);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 x = ld_cg_f4(src + j * 32);
        v[4 * j] += x.x;
        v[4 * j + 1] += x.y;
        v[4 * j + 2] += x.z;
        v[4 * j + 3] += x.w;
      }
    }
  }
}

// An epilogue program may declare
//   static void prefetch(const Params&, int M, int N, int m, int n0, int bn);
// the epilogue warps call it for their row m and the tile's columns
// [n0, n0 + bn) before they wait for the tile's accumulator, so the
// program's global inputs can be on their way to L2 during the mainloop.
template <class E, class = void>
struct EpiHasPrefetch {
  static constexpr bool value = false;
};
template <class E>
struct EpiHasPrefetch<E, decltype(void(&E::prefetch))> {
  static constexpr bool value = true;
};

// Store staging: every epilogue warp owns Epi::kStoreSlots slots of
// STORE_SLOT_BYTES in shared memory, after the operand ring.
constexpr int STORE_SLOT_BYTES = 2048;
template <class Epi>
constexpr int epi_stage_bytes() { return Epi::kEpiWarps * Epi::kStoreSlots * STORE_SLOT_BYTES; }
constexpr int MAX_DYN_SMEM = 232448;  // 227 KB per CTA

template <int BN, int STAGES, int EPI_BYTES>
struct GemmSmem {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int STORE_BYTES = EPI_BYTES;                 // epilogue store staging
  static constexpr int BAR_BYTES = 256;
  static constexpr int TOTAL = RING_BYTES + STORE_BYTES + BAR_BYTES + 1024;  // + alignment slack
  static_assert(TOTAL <= MAX_DYN_SMEM, "shared memory budget");
  static constexpr int TMEM_COLS = 2 * BN;                      // double-buffered accumulator
  static_assert(TMEM_COLS <= 512, "TMEM has 512 columns");
  static_assert((2 * STAGES + 5) * 8 + 8 <= BAR_BYTES, "barrier area too small");
};

__device__ __forceinline__ void tile_coords(int t, const GemmShape& s, int& tm, int& tn) {
  const int group_tiles = s.group_m * s.tiles_n;
  const int group = t / group_tiles;
  const int first_m = group * s.group_m;
  const int gm = min(s.tiles_m - first_m, s.group_m);
  const int r = t - group * group_tiles;
  tm = first_m + r % gm;
  tn = r / gm;
}

__device__ __forceinline__ void raise_error(const KernelCtl& ctl, volatile int* abort_flag, int bit) {
  atomicOr(ctl.status, bit);
  *abort_flag = 1;
}

template <int BN, int STAGES, bool A_MN, bool B_MN, bool B_DUAL, class Epi, bool FP8 = false>
__global__ void __launch_bounds__(gemm_threads<Epi>(), 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmB2, const GemmShape sh, const KernelCtl ctl,
                   const __grid_constant__ typename Epi::Params ep) {
  using L = GemmSmem<BN, STAGES, epi_stage_bytes<Epi>()>;
  static_assert(!(B_DUAL && B_MN), "dual-box B is K-major only");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  constexpr uint32_t IDESC0 = FP8 ? idesc_f8_f32(BM, BN, A_MN, B_MN) : idesc_bf16_f32(BM, BN, A_MN, B_MN);
  constexpr int BKE = FP8 ? 128 : BK;         // K elements per 128-byte k-block row (K-major operands)
  // MN-major operands: boxes of 128 bytes along M/N (64 bf16 or 128 e4m3) by
  // BKE rows of K; one MMA's K slice is 16 (bf16) or 32 (8-bit) such rows
  constexpr int MNB = FP8 ? 128 : 64;         // M/N elements per MN-major box
  constexpr int MN_BOX = 128 * BKE;           // bytes per MN-major box
  constexpr int MN_KSTEP = FP8 ? 4096 : 2048; // bytes per MMA K slice, MN-major

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::RING_BYTES + L::STORE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 32 * Epi::kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (B_DUAL) tma_prefetch_desc(&tmB2);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the set-up above may overlap the previous kernel; operands and outputs
  // are touched only after it has completed
  griddep_launch_dependents();
  griddep_wait();
  const float acc_scale = acc_scale_of(ctl);
  const uint32_t idesc = FP8 ? (IDESC0 | ctl.f8_fmt) : IDESC0;

  const int num_tiles = sh.tiles_m * sh.tiles_n;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t pending = 0;  // bit s: stage s has been filled at least once
      uint32_t parity = 0;   // bit s: phase parity of the last fill of stage s
      bool ok = true;
      bool skip = ctl.skip_first_stage != 0 && blockIdx.x == 0;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        int tm, tn;
        tile_coords(t, sh, tm, tn);
        for (int kb = 0; kb < sh.num_kb; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, ctl.timeout_ns)) {
            if (!*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_PRODUCER);
            ok = false;
            break;
          }
          if (skip) {
            // test hook: leave this stage unfilled so the MMA's wait on it expires
            skip = false;
          } else {
            uint8_t* sa = smem + stage * L::STAGE_BYTES;
            uint8_t* sb = sa + L::A_BYTES;
            mbar_arrive_expect_tx(&full[stage], L::STAGE_BYTES);
            if (!A_MN) {
              tma_load_2d(sa, &tmA, &full[stage], kb * BKE, tm * BM);
            } else {
#pragma unroll
              for (int i = 0; i < BM / MNB; ++i)
                tma_load_2d(sa + i * MN_BOX, &tmA, &full[stage], tm * BM + i * MNB, kb * BKE);
            }
            if (B_DUAL) {
              tma_load_2d(sb, &tmB, &full[stage], kb * BKE, tn * (BN / 2));
              tma_load_2d(sb + (BN / 2) * 128, &tmB2, &full[stage], kb * BKE, tn * (BN / 2));
            } else if (!B_MN) {
              tma_load_2d(sb, &tmB, &full[stage], kb * BKE, tn * BN);
            } else {
#pragma unroll
              for (int i = 0; i < BN / MNB; ++i)
                tma_load_2d(sb + i * MN_BOX, &tmB, &full[stage], tn * BN + i * MNB, kb * BKE);
            }
            pending |= 1u << stage;
            parity = (parity & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // let every copy this thread started land before shared memory is released
        for (int st = 0; st < STAGES; ++st)
          if ((pending >> st) & 1u)
            if (!mbar_wait_timeout(&full[st], (parity >> st) & 1u, ctl.timeout_ns))
              atomicOr(ctl.status, DEV_ERR_TIMEOUT_DRAIN);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, ctl.timeout_ns)) {
          if (!*abort_flag) raise_error(ctl, abort_flag, DEV_ERR_TIMEOUT_MMA);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < sh.num_kb; ++kb) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, ctl.timeout_ns)) {
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
            if (FP8)
              umma_e4m3(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            else
              umma_bf16(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
      }
      // wait for every MMA this thread issued before TMEM can be freed
      umma_commit(drain);
      if (!mbar_wait_timeout(drain, 0, ctl.timeout_ns)) atomicOr(ctl.status, DEV_ERR_TIMEOUT_DRAIN);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    constexpr int HALVES = 8 / Epi::kEpiWarps;  // halves of the tile per warp
    const int quad = warp & 3;
    const int first_half = HALVES == 1 ? (warp - 2) >> 2 : 0;
    const int row = quad * 32 + lane;
    const uint32_t stage_base = smem_u32(smem + L::RING_BYTES) +
                                static_cast<uint32_t>((warp - 2) * Epi::kStoreSlots * STORE_SLOT_BYTES);
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      int tm, tn;
      tile_coords(t, sh, tm, tn);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if constexpr (EpiHasPrefetch<Epi>::value)
        Epi::prefetch(ep, sh.M, sh.N, tm * BM + row, tn * BN + first_half * (BN / 2), HALVES * (BN / 2));
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
      c.tm = tm;
      c.tn = tn;
      c.row = row;
      c.m = tm * BM + row;
      c.m0 = tm * BM + quad * 32;
      c.quad = quad;
      c.lane = lane;
      c.acc_scale = acc_scale;
      c.taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN);
      c.stage = stage_base;
      c.nsplit = 0;
#pragma unroll 1
      for (int hh = 0; hh < HALVES; ++hh) {
        const int half = first_half + hh;
        c.c0 = half * (BN / 2);
        c.c1 = c.c0 + BN / 2;
        c.part = tn * 2 + half;
        Epi::template run<BN>(ep, c);
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
    // the last stores have landed before shared memory is released
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// epilogue helpers: 32-column row segments, groups of 8 bf16 (16 bytes);
// every extent on the boundary is a multiple of 8 so groups are all-or-none.
// ---------------------------------------------------------------------------
// 32 bf16 of a row from column n0 as raw vectors, zero past nvalid: issued
// one chunk ahead of their use, unpacked with unpack_bf16x8 when needed.
__device__ __forceinline__ void load_bf16x32_raw(const __nv_bfloat16* row, int n0, int nvalid, uint4 (&q)[4]) {
#pragma unroll
  for (int g = 0; g < 4; ++g)
    q[g] = g * 8 < nvalid ? __ldg(reinterpret_cast<const uint4*>(row + n0 + g * 8)) : make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* p, int nvalid, float (&f)[32]) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    if (g * 8 < nvalid) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(p + g * 8));
      unpack_bf16x8(q, &f[g * 8]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[g * 8 + i] = 0.f;
    }
  }
}

// ---------------------------------------------------------------------------
// Staged TMA stores.  A warp's 32 rows x 32 columns of an output are written
// row-per-lane into one of its shared-memory slots in the swizzled layout of
// the output's tensor map, and one lane stores the block with a single TMA
// copy (whole lines to L2; rows past M and columns past N are clipped by the
// tensor map).  Per step:
//   slots_acquire   lane 0 waits until the stores it issued before have read
//                   the slots, then the warp syncs;
//   stage_*         every lane writes its row;
//   slots_publish   every lane fences its writes to the async proxy, then the
//                   warp syncs; lane 0 issues the stores and commits them.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t slot_addr(const EpiCtx& c, int i) {
  return c.stage + static_cast<uint32_t>(i * STORE_SLOT_BYTES);
}

// bf16 block, 64-byte rows, 64-byte swizzle: the 16-byte chunk q of row r
// sits at chunk position q ^ ((r >> 1) & 3).
__device__ __forceinline__ void stage_bf16x32(uint32_t slot, int lane, const float (&f)[32]) {
  const uint32_t row = slot + static_cast<uint32_t>(lane) * 64u;
  const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    st_shared_v4(row + ((static_cast<uint32_t>(q) ^ sw) << 4), pack_bf16x2(f[8 * q + 0], f[8 * q + 1]),
                 pack_bf16x2(f[8 * q + 2], f[8 * q + 3]), pack_bf16x2(f[8 * q + 4], f[8 * q + 5]),
                 pack_bf16x2(f[8 * q + 6], f[8 * q + 7]));
}

// fp32 block (two slots), 128-byte rows, 128-byte swizzle: chunk q of row r
// sits at chunk position q ^ (r & 7).
__device__ __forceinline__ void stage_f32x32(uint32_t slot, int lane, const float (&f)[32]) {
  const uint32_t row = slot + static_cast<uint32_t>(lane) * 128u;
  const uint32_t sw = static_cast<uint32_t>(lane) & 7u;
#pragma unroll
  for (int q = 0; q < 8; ++q)
    st_shared_v4(row + ((static_cast<uint32_t>(q) ^ sw) << 4), __float_as_uint(f[4 * q + 0]),
                 __float_as_uint(f[4 * q + 1]), __float_as_uint(f[4 * q + 2]), __float_as_uint(f[4 * q + 3]));
}

// e5m2 block: 32 rows x 32 codes of f * inv (saturating, round to nearest
// even), 32-byte rows, 32-byte swizzle: the 16-byte chunk q of row r sits at
// chunk position q ^ ((r >> 2) & 1).
__device__ __forceinline__ void stage_e5m2x32(uint32_t slot, int lane, const float (&f)[32], float inv) {
  const uint32_t row = slot + static_cast<uint32_t>(lane) * 32u;
  const uint32_t sw = (static_cast<uint32_t>(lane) >> 2) & 1u;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = 16 * q + 4 * j;
      const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(f[i] * inv, f[i + 1] * inv), __NV_SATFINITE,
                                                   __NV_E5M2);
      const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(f[i + 2] * inv, f[i + 3] * inv), __NV_SATFINITE,
                                                   __NV_E5M2);
      w[j] = (lo & 0xFFFFu) | (hi << 16);
    }
    st_shared_v4(row + ((static_cast<uint32_t>(q) ^ sw) << 4), w[0], w[1], w[2], w[3]);
  }
}

__device__ __forceinline__ void slots_acquire(int lane) {
  if (lane == 0) bulk_wait_group_read0();
  __syncwarp();
}

// Double-buffered form for a program with one output: before chunk j of a
// run lane 0 waits until only the most recent store group (chunk j - 1, in
// the other slot) may still be reading; at the start of a run (first) it
// drains them all.  Within a run the stored chunks are a prefix of its
// chunks, so consecutive stores always alternate slots.
__device__ __forceinline__ void slots_acquire_db(int lane, bool first) {
  if (lane == 0) {
    if (first)
      bulk_wait_group_read0();
    else
      bulk_wait_group_read1();
  }
  __syncwarp();
}

__device__ __forceinline__ void slots_publish() {
  fence_proxy_async_shared();
  __syncwarp();
}

// lane l ends with sum over the 32 lanes of v[l]  (31 shuffles)
__device__ __forceinline__ float warp_transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

// ---------------------------------------------------------------------------
// Epilogue programs
// ---------------------------------------------------------------------------

// The RMSNorm row scale of row c.m taken straight from the partial sums of
// squares of the first GEMM: r = 1 / sqrt(sum_j psum[m, j] * inv_d + eps).
// The tile in column 0 also stores r (for the backward) when rstd_out is set.
__device__ __forceinline__ float rstd_from_psum(const float* psum, int T, float inv_d, float eps, float* rstd_out,
                                                const EpiCtx& c) {
  const float* p = psum + static_cast<int64_t>(c.m) * T;
  float acc = 0.f;
  for (int j = 0; j < T; ++j) acc += p[j];
  const float r = 1.0f / sqrtf(acc * inv_d + eps);
  if (rstd_out != nullptr && c.tn == 0 && c.c0 == 0) rstd_out[c.m] = r;
  return r;
}

// C = bf16(row_scale[m] * col_scale[n] * acc); both scales optional.
struct EpiStore {
  static constexpr int kEpiWarps = 4;
  static constexpr int kStoreSlots = 2;  // two slots used alternately
  static constexpr bool kAccScale = true;  // multiplies by EpiCtx::acc_scale: usable on FP8 operands
  struct Params {
    CUtensorMap out;  // [M][N] bf16
    const float* row_scale;
    const __nv_bfloat16* col_scale;
    // optional: the row scale from first-GEMM partial sums instead of row_scale
    const float* psum;
    int T;
    float inv_d;
    float eps;
    float* rstd_out;
  };
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const EpiCtx& c) {
    const bool row_ok = c.m < c.M;
    float rs = 1.f;
    if (row_ok) {
      if (p.psum != nullptr)
        rs = rstd_from_psum(p.psum, p.T, p.inv_d, p.eps, p.rstd_out, c);
      else if (p.row_scale != nullptr)
        rs = p.row_scale[c.m];
    }
    rs *= c.acc_scale;
#pragma unroll 1
    for (int cc = c.c0; cc < c.c1; cc += 32) {
      float v[32];
      acc_ld32(c, cc, v);
      const int n0 = c.tn * BN + cc;
      if (n0 < c.N && c.m0 < c.M) {
        if (p.col_scale != nullptr) {
          float s[32];
          load_bf16x32(p.col_scale + n0, c.N - n0, s);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= s[i];
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= rs;
        const int slot = ((cc - c.c0) >> 5) & 1;
        slots_acquire_db(c.lane, cc == c.c0);
        stage_bf16x32(slot_addr(c, slot), c.lane, v);
        slots_publish();
        if (c.lane == 0) {
          tma_store_2d(&p.out, slot_addr(c, slot), n0, c.m0);
          bulk_commit_group();
        }
      }
    }
  }
};

// fp32 output, overwrite (beta = 0) or accumulate (beta = 1, a TMA
// reduce-add: each element receives one add per launch).
struct EpiStoreF32 {
  static constexpr int kEpiWarps = 4;
  static constexpr int kStoreSlots = 2;  // one 4 KB fp32 block
  static constexpr bool kAccScale = true;  // multiplies by EpiCtx::acc_scale: usable on FP8 operands
  struct Params {
    CUtensorMap out;  // [M][N] fp32
    int beta;
  };
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const EpiCtx& c) {
#pragma unroll 1
    for (int cc = c.c0; cc < c.c1; cc += 32) {
      float v[32];
      acc_ld32(c, cc, v);
      const int n0 = c.tn * BN + cc;
      if (n0 < c.N && c.m0 < c.M) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= c.acc_scale;
        slots_acquire(c.lane);
        stage_f32x32(slot_addr(c, 0), c.lane, v);
        slots_publish();
        if (c.lane == 0) {
          if (p.beta)
            tma_reduce_add_2d(&p.out, slot_addr(c, 0), n0, c.m0);
          else
            tma_store_2d(&p.out, slot_addr(c, 0), n0, c.m0);
          bulk_commit_group();
        }
      }
    }
  }
};

// GEMM1 epilogue: h = bf16(acc + R); store h; psum[m, tn] = sum over the
// tile's columns of h^2 (h as stored, i.e. after rounding to bf16).
struct EpiResPrms {
  static constexpr int kEpiWarps = 4;
  static constexpr int kStoreSlots = 2;
  static constexpr bool kAccScale = true;  // multiplies by EpiCtx::acc_scale: usable on FP8 operands
  struct Params {
    CUtensorMap H;   // [M][d] bf16
    CUtensorMap Hg;  // [M][d] bf16, used when g != null
    const __nv_bfloat16* R;
    int64_t ldr;
    float* psum;
    int T;  // psum columns
    // optional: the RMSNorm weight broadcast along the row (vector load) and
    // a second output Hg = bf16(H * g), the second GEMM's A operand when g is
    // applied on the activation side instead of being folded into W2
    const __nv_bfloat16* g;
  };
  // the row's residual segment of the tile, line by line, into L2
  static __device__ __forceinline__ void prefetch(const Params& p, int M, int N, int m, int n0, int bn) {
    if (m >= M) return;
    const __nv_bfloat16* row = p.R + static_cast<int64_t>(m) * p.ldr;
    for (int n = n0; n < n0 + bn && n < N; n += 64) prefetch_l2(row + n);
  }
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const EpiCtx& c) {
    const bool row_ok = c.m < c.M;
    const bool with_g = p.g != nullptr;
    const __nv_bfloat16* rrow = p.R + static_cast<int64_t>(c.m) * p.ldr;
    const int nb = c.tn * BN;
    float ss = 0.f;
    // the residual is loaded one chunk ahead of its use
    uint4 rq[4];
    load_bf16x32_raw(rrow, nb + c.c0, row_ok ? c.N - nb - c.c0 : 0, rq);
#pragma unroll 1
    for (int cc = c.c0; cc < c.c1; cc += 32) {
      float v[32];
      acc_ld32(c, cc, v);
      const int n0 = nb + cc;
      float r[32];
#pragma unroll
      for (int g = 0; g < 4; ++g) unpack_bf16x8(rq[g], &r[g * 8]);
      if (cc + 32 < c.c1) load_bf16x32_raw(rrow, n0 + 32, row_ok ? c.N - n0 - 32 : 0, rq);
      if (n0 < c.N && c.m0 < c.M) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float hb = bf16_round(fmaf(v[i], c.acc_scale, r[i]));
          v[i] = hb;
          ss = fmaf(hb, hb, ss);
        }
        // H alone: two slots used alternately; H and Hg: one slot each
        const int slot = with_g ? 0 : ((cc - c.c0) >> 5) & 1;
        if (with_g)
          slots_acquire(c.lane);
        else
          slots_acquire_db(c.lane, cc == c.c0);
        stage_bf16x32(slot_addr(c, slot), c.lane, v);
        if (with_g) {
          load_bf16x32(p.g + n0, c.N - n0, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= r[i];
          stage_bf16x32(slot_addr(c, 1), c.lane, v);
        }
        slots_publish();
        if (c.lane == 0) {
          tma_store_2d(&p.H, slot_addr(c, slot), n0, c.m0);
          if (with_g) tma_store_2d(&p.Hg, slot_addr(c, 1), n0, c.m0);
          bulk_commit_group();
        }
      }
    }
    if (row_ok && c.tn * BN + c.c0 < c.N) p.psum[static_cast<int64_t>(c.m) * p.T + c.part] = ss;
  }
};

// GEMM2 epilogue: the accumulator holds [gate | up] halves of BN/2 columns
// (two B boxes).  z = rstd[m] * acc; out = silu(z_gate) * z_up; optionally
// save z (bf16) for the backward.
struct EpiRowscaleSwiglu {
  static constexpr int kEpiWarps = 4;
  static constexpr int kStoreSlots = 3;  // out, z gate, z up
  static constexpr bool kAccScale = true;  // multiplies by EpiCtx::acc_scale: usable on FP8 operands
  struct Params {
    CUtensorMap out;  // [M][F] bf16
    CUtensorMap zg;   // gate half of z: [M][F] with the row pitch of z
    CUtensorMap zu;   // up half of z
    int save_z;
    const float* rstd;
    int F;            // gate (= up) width; output columns
    // optional: the row scale from first-GEMM partial sums instead of rstd
    const float* psum;
    int T;
    float inv_d;
    float eps;
    float* rstd_out;
  };
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const EpiCtx& c) {
    constexpr int HB = BN / 2;
    const bool row_ok = c.m < c.M;
    float r = 0.f;
    if (row_ok) r = p.psum != nullptr ? rstd_from_psum(p.psum, p.T, p.inv_d, p.eps, p.rstd_out, c) : p.rstd[c.m];
    r *= c.acc_scale;
#pragma unroll 1
    for (int cc = c.c0 / 2; cc < c.c1 / 2; cc += 32) {
      float g[32], u[32];
      acc_ld32(c, cc, g);
      acc_ld32(c, HB + cc, u);
      const int j0 = c.tn * HB + cc;
      if (j0 < p.F && c.m0 < c.M) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          g[i] *= r;
          u[i] *= r;
        }
        slots_acquire(c.lane);
        if (p.save_z) {
          stage_bf16x32(slot_addr(c, 1), c.lane, g);
          stage_bf16x32(slot_addr(c, 2), c.lane, u);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) g[i] = silu_f(g[i]) * u[i];
        stage_bf16x32(slot_addr(c, 0), c.lane, g);
        slots_publish();
        if (c.lane == 0) {
          tma_store_2d(&p.out, slot_addr(c, 0), j0, c.m0);
          if (p.save_z) {
            tma_store_2d(&p.zg, slot_addr(c, 1), j0, c.m0);
            tma_store_2d(&p.zu, slot_addr(c, 2), j0, c.m0);
          }
          bulk_commit_group();
        }
      }
    }
  }
};

// Data gradient of GEMM2 with the RMSNorm backward in its epilogue:
//   acc = dP W2^T ; dh = g * acc - c[m] * h ; dgpart[4*tm + quad, n] =
//   sum over the warp's 32 rows of acc * h  (block reduction across lanes).
struct EpiDgradRms {
  static constexpr int kEpiWarps = 4;
  static constexpr int kStoreSlots = 2;  // dH chunks, two slots used alternately
  static constexpr bool kAccScale = true;  // multiplies by EpiCtx::acc_scale: usable on FP8 operands
  struct Params {
    CUtensorMap dH;  // [M][d] bf16
    const __nv_bfloat16* H;
    int64_t ldh;
    const __nv_bfloat16* g;
    const float* c;
    float* dgpart;  // [4 * tiles_m, N]
    // optional: c from the SwiGLU-backward epilogue's partial sums,
    // c[m] = rstd[m]^2 * inv_d * sum_j cpart[m, j], instead of the c vector
    const float* cpart;
    int Tc;
    const float* rstd;
    float inv_d;
  };
  // the row's segment of h for the tile, line by line, into L2
  static __device__ __forceinline__ void prefetch(const Params& p, int M, int N, int m, int n0, int bn) {
    if (m >= M) return;
    const __nv_bfloat16* row = p.H + static_cast<int64_t>(m) * p.ldh;
    for (int n = n0; n < n0 + bn && n < N; n += 64) prefetch_l2(row + n);
  }
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const EpiCtx& c) {
    const bool row_ok = c.m < c.M;
    const __nv_bfloat16* hrow = p.H + static_cast<int64_t>(c.m) * p.ldh;
    const int nb = c.tn * BN;
    // h is loaded one chunk ahead of its use
    uint4 hq[4];
    load_bf16x32_raw(hrow, nb + c.c0, row_ok ? c.N - nb - c.c0 : 0, hq);
    float cm = 0.f;
    if (row_ok) {
      if (p.cpart != nullptr) {
        const float* cp = p.cpart + static_cast<int64_t>(c.m) * p.Tc;
        float acc = 0.f;
        for (int j = 0; j < p.Tc; ++j) acc += cp[j];
        const float r = p.rstd[c.m];
        cm = r * r * p.inv_d * acc;
      } else {
        cm = p.c[c.m];
      }
    }
#pragma unroll 1
    for (int cc = c.c0; cc < c.c1; cc += 32) {
      float a[32];
      acc_ld32(c, cc, a);
      const int n0 = nb + cc;
      float h[32];
#pragma unroll
      for (int g = 0; g < 4; ++g) unpack_bf16x8(hq[g], &h[g * 8]);
      if (cc + 32 < c.c1) load_bf16x32_raw(hrow, n0 + 32, row_ok ? c.N - n0 - 32 : 0, hq);
      if (n0 < c.N) {
        // FP8 operands: dequantise the accumulator (acc_scale = 1 for bf16)
#pragma unroll
        for (int i = 0; i < 32; ++i) a[i] *= c.acc_scale;
        float gv[32];
        load_bf16x32(p.g + n0, c.N - n0, gv);
        if (c.m0 < c.M) {
          float dh[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) dh[i] = fmaf(gv[i], a[i], -cm * h[i]);
          const int slot = ((cc - c.c0) >> 5) & 1;
          slots_acquire_db(c.lane, cc == c.c0);
          stage_bf16x32(slot_addr(c, slot), c.lane, dh);
          slots_publish();
          if (c.lane == 0) {
            tma_store_2d(&p.dH, slot_addr(c, slot), n0, c.m0);
            bulk_commit_group();
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) a[i] *= h[i];
        const float s = warp_transpose_sum32(a, c.lane);
        // 128-row blocks wholly past M (the second half of a CTA-pair tile)
        // have no rows and no partial
        if (n0 + c.lane < c.N && c.tm * 128 < c.M)
          p.dgpart[static_cast<int64_t>(c.tm * 4 + c.quad) * c.N + n0 + c.lane] = s;
      }
    }
  }
};

// Data gradient of a down projection y = out W3 with the SwiGLU backward in
// its epilogue: the accumulator holds dY (gate-column indices j); with
// s = sigmoid(z_gate):
//   dZ_gate = dY z_up s (1 + z_gate (1 - s)),  dZ_up = dY z_gate s,
//   dP = bf16(rstd[m] dZ) into the gate / up halves,
//   cpart[m, tn] = sum over the tile's columns of dZ_gate z_gate + dZ_up z_up
// (a block reduction the RMSNorm backward later merges into c).  dY itself
// never leaves the chip.
struct EpiSwigluBwd {
  static constexpr int kEpiWarps = 4;
  static constexpr int kStoreSlots = 2;
  static constexpr bool kAccScale = false;  // ignores EpiCtx::acc_scale: bf16 operands only
  struct Params {
    CUtensorMap dPg;  // gate half of dP: [M][F] with the row pitch of dP
    CUtensorMap dPu;  // up half
    const __nv_bfloat16* z;  // [M, 2F]
    const float* rstd;
    float* cpart;            // [M, T]
    int T;
    int F;
  };
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const EpiCtx& c) {
    const bool row_ok = c.m < c.M;
    const float r = row_ok ? p.rstd[c.m] : 0.f;
    const int64_t row = static_cast<int64_t>(c.m) * 2 * p.F;
    float cp = 0.f;
#pragma unroll 1
    for (int cc = c.c0; cc < c.c1; cc += 32) {
      float dy[32];
      acc_ld32(c, cc, dy);
      const int j0 = c.tn * BN + cc;
      if (j0 < p.F && c.m0 < c.M) {
        const int nv = row_ok ? p.F - j0 : 0;
        float zg[32], zu[32];
        load_bf16x32(p.z + row + j0, nv, zg);
        load_bf16x32(p.z + row + p.F + j0, nv, zu);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float s = sigmoid_f(zg[i]);
          const float dzu = dy[i] * zg[i] * s;
          const float dzg = dy[i] * zu[i] * s * (1.0f + zg[i] * (1.0f - s));
          cp = fmaf(dzg, zg[i], fmaf(dzu, zu[i], cp));
          zg[i] = r * dzg;
          zu[i] = r * dzu;
        }
        slots_acquire(c.lane);
        stage_bf16x32(slot_addr(c, 0), c.lane, zg);
        stage_bf16x32(slot_addr(c, 1), c.lane, zu);
        slots_publish();
        if (c.lane == 0) {
          tma_store_2d(&p.dPg, slot_addr(c, 0), j0, c.m0);
          tma_store_2d(&p.dPu, slot_addr(c, 1), j0, c.m0);
          bulk_commit_group();
        }
      }
    }
    if (row_ok && c.tn * BN + c.c0 < p.F) p.cpart[static_cast<int64_t>(c.m) * p.T + c.part] = cp;
  }
};

// QKV projection with rotary position embedding in the epilogue (rotate-half
// pairing, head_dim 128 = one 128-column half tile = one head): for a q or k
// head at position p = m mod S, out_i = x_i cos - x_{i+64} sin and
// out_{i+64} = x_{i+64} cos + x_i sin with cos/sin read from [S, 64] tables
// (the vector-load primitive); v heads (columns >= rot_cols) pass through.
struct EpiRope {
  static constexpr int kEpiWarps = 4;
  static constexpr int kStoreSlots = 2;
  static constexpr bool kAccScale = false;  // ignores EpiCtx::acc_scale: bf16 operands only
  struct Params {
    CUtensorMap out;     // [M][N] bf16
    const float* cos_t;  // [S, 64]
    const float* sin_t;  // [S, 64]
    int S;
    int rot_cols;        // (heads of q + heads of k) * 128
  };
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const EpiCtx& c) {
    const int nh = c.tn * BN + c.c0;  // first column of this half tile's head
    if (nh >= c.N) return;            // the same for every lane of the warp
    const bool row_ok = c.m < c.M;
    const bool rot = nh < p.rot_cols;
    const int64_t tab = row_ok ? static_cast<int64_t>(c.m % p.S) * 64 : 0;
#pragma unroll 1
    for (int cc = 0; cc < 64; cc += 32) {
      float x1[32], x2[32];
      acc_ld32(c, c.c0 + cc, x1);
      acc_ld32(c, c.c0 + 64 + cc, x2);
      if (c.m0 >= c.M) continue;
      if (rot) {
        const float4* cs4 = reinterpret_cast<const float4*>(p.cos_t + tab + cc);
        const float4* sn4 = reinterpret_cast<const float4*>(p.sin_t + tab + cc);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 cq = __ldg(cs4 + q), sq = __ldg(sn4 + q);
          const float cv[4] = {cq.x, cq.y, cq.z, cq.w};
          const float sv[4] = {sq.x, sq.y, sq.z, sq.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int i = 4 * q + k;
            const float a = x1[i], b = x2[i];
            x1[i] = fmaf(a, cv[k], -b * sv[k]);
            x2[i] = fmaf(b, cv[k], a * sv[k]);
          }
        }
      }
      slots_acquire(c.lane);
      stage_bf16x32(slot_addr(c, 0), c.lane, x1);
      stage_bf16x32(slot_addr(c, 1), c.lane, x2);
      slots_publish();
      if (c.lane == 0) {
        if (nh + cc < c.N) tma_store_2d(&p.out, slot_addr(c, 0), nh + cc, c.m0);
        if (nh + 64 + cc < c.N) tma_store_2d(&p.out, slot_addr(c, 1), nh + 64 + cc, c.m0);
        bulk_commit_group();
      }
    }
  }
};

// LM-head forward epilogue: per (row, N-tile) running max and sum of
// exp(L - max) (online rescaling across 32-column chunks), the tile argmax
// (lowest column on ties), and the label logit when the label falls in the
// tile.  Columns >= N (vocabulary tail) are masked out.
struct EpiCeStats {
  static constexpr int kEpiWarps = 4;
  static constexpr int kStoreSlots = 0;
  static constexpr bool kAccScale = true;  // multiplies by EpiCtx::acc_scale: usable on FP8 operands
  struct Params {
    const int32_t* labels;
    float* pmax;
    float* psum;
    int32_t* parg;
    float* zy;
    int T;
    int* status;
  };
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const EpiCtx& c) {
    const bool row_ok = c.m < c.M;
    const int y = row_ok ? p.labels[c.m] : -1;
    if (row_ok && c.tn == 0 && c.c0 == 0 && (y < 0 || y >= c.N)) atomicOr(p.status, DEV_ERR_LABEL_RANGE);
    float mx = -INFINITY, se = 0.f, zy = 0.f;
    int am = -1;
    bool found = false;
#pragma unroll 1
    for (int cc = c.c0; cc < c.c1; cc += 32) {
      float v[32];
      acc_ld32(c, cc, v);
      const int n0 = c.tn * BN + cc;
      if (row_ok && n0 < c.N) {
        // one thread owns the row, so the chunk is reduced in registers: with
        // one epilogue warp per scheduler the dependency chains set the pace,
        // hence a pairwise tree for the maximum and four partial sums
        const int nv = c.N - n0;
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = i < nv ? v[i] * c.acc_scale : -INFINITY;
        // chunk maximum and its column: the left operand of every comparison
        // holds the lower columns, so a tie keeps the lower one
        float tv[16];
        int ti[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const bool right = v[2 * i + 1] > v[2 * i];
          tv[i] = right ? v[2 * i + 1] : v[2 * i];
          ti[i] = right ? 2 * i + 1 : 2 * i;
        }
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1) {
#pragma unroll
          for (int i = 0; i < w; ++i) {
            const bool right = tv[2 * i + 1] > tv[2 * i];
            tv[i] = right ? tv[2 * i + 1] : tv[2 * i];
            ti[i] = right ? ti[2 * i + 1] : ti[2 * i];
          }
        }
        const float cmax = tv[0];
        if (cmax > mx) {
          se *= __expf(mx - cmax);
          mx = cmax;
          am = n0 + ti[0];
        }
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 32; ++i) s4[i & 3] += __expf(v[i] - mx);
        se += (s4[0] + s4[1]) + (s4[2] + s4[3]);
        if (y >= n0 && y < n0 + 32) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (n0 + i == y) zy = v[i];
          found = true;
        }
      }
    }
    if (row_ok && c.tn * BN + c.c0 < c.N) {
      const int64_t o = static_cast<int64_t>(c.m) * p.T + c.part;
      p.pmax[o] = mx;
      p.psum[o] = se;
      p.parg[o] = am;
      if (found) p.zy[c.m] = zy;
    }
  }
};

// LM-head backward epilogue: dL = (exp(L - lse[m]) - [n == y_m]) / M into a
// vocabulary-chunk buffer (column n of the chunk = vocabulary v0 + n), as bf16
// or, with FP8 operands, as e5m2 codes of dL * code_inv (|dL| <= 1/M, so a
// power-of-two scale fixed in advance never saturates).
struct EpiCeGrad {
  static constexpr int kEpiWarps = 4;
  static constexpr int kStoreSlots = 1;
  static constexpr bool kAccScale = true;  // multiplies by EpiCtx::acc_scale: usable on FP8 operands
  struct Params {
    CUtensorMap dL;  // [M][Vc] bf16, or e5m2 codes when codes != 0
    const int32_t* labels;
    const float* lse;
    float inv_M;
    int v0;
    int codes;
    float code_inv;  // the inverse of the codes' power-of-two scale
  };
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const EpiCtx& c) {
    const bool row_ok = c.m < c.M;
    const float l = row_ok ? p.lse[c.m] : 0.f;
    const int y = row_ok ? p.labels[c.m] - p.v0 : -1;
#pragma unroll 1
    for (int cc = c.c0; cc < c.c1; cc += 32) {
      float v[32];
      acc_ld32(c, cc, v);
      const int n0 = c.tn * BN + cc;
      if (n0 < c.N && c.m0 < c.M) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float e = __expf(v[i] * c.acc_scale - l) - ((n0 + i == y) ? 1.f : 0.f);
          v[i] = e * p.inv_M;
        }
        slots_acquire(c.lane);
        if (p.codes)
          stage_e5m2x32(slot_addr(c, 0), c.lane, v, p.code_inv);
        else
          stage_bf16x32(slot_addr(c, 0), c.lane, v);
        slots_publish();
        if (c.lane == 0) {
          tma_store_2d(&p.dL, slot_addr(c, 0), n0, c.m0);
          bulk_commit_group();
        }
      }
    }
  }
};

}  // namespace coda
