/* Test hooks of libcoda.  These entry points exist so that the library's own
 * tests can exercise failure detection and check host-side scheduling logic
 * without a GPU fault; they are exported by libcoda.so beside the entry
 * points of coda.h but are not part of the library's interface for users,
 * and no computation of the block path depends on them. */
#pragma once

#include "coda.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Failure-detection test hook.  enable = 1: every GEMM launched through this
 * handle leaves the first shared-memory stage of its first CTA unfilled, so
 * that CTA's MMA wait cannot complete and must hit the wait limit (in the
 * 256 x 512 pair-tile kernel of coda_set_wide_tiles, the first CTA issues no
 * copy at all).  enable = 2 (SM-pair GEMMs): the second CTA of the first SM
 * pair issues no copy at all, so the pair's stages never fill; on single
 * SMs it acts as 1.  Either way the launch records
 * CODA_ERR_TIMEOUT (reported by coda_sync_status), its results are invalid,
 * every copy that was issued is still observed to land before shared memory
 * is released, and the context stays usable.  0 turns the hook off.  Pair it
 * with a short coda_set_wait_timeout_ns.  Not for production use. */
coda_status_t coda_debug_skip_first_stage(coda_handle_t h, int enable);

/* Host-side check of the tile schedule of the grouped launches (no GPU
 * needed): P clusters, the heavy problem's index (0 or 1), its tile count nH,
 * the light problem's tile count nL, q catch-up tiles.  Returns 0 when every
 * tile of both problems is assigned to exactly one cluster, the number of
 * violations otherwise, -1 for invalid arguments.  Not for production use. */
int coda_debug_group_schedule_violations(int P, int heavy, int nH, int nL, int q);

/* Host-side check of the split-tile schedule (coda_set_split_workspace) of
 * the SM-pair GEMM, run with the kernel's own work iterator (no GPU needed):
 * `tiles` output tiles of `num_kb` k-blocks on `clusters` SM pairs.  Returns
 * 0 when the launch would not split, or when every (tile, k-block) is
 * computed exactly once, every split piece is either a partial (an earlier
 * k-range, written to a slot no other piece writes) or the owner (the last
 * k-range), each cluster meets all its partial pieces before its owner
 * pieces, and each owner's slots hold its tile's earlier k-ranges in order
 * without a gap; the number of violations otherwise, -1 for invalid
 * arguments.  Not for production use. */
int coda_debug_split_schedule_violations(int tiles, int num_kb, int clusters);

/* The first tile of the split region that an SM-pair launch of `tiles` tiles
 * of `num_kb` k-blocks on `clusters` pairs would use with a split workspace
 * set (tiles when it would not split), -1 for invalid arguments.  Not for
 * production use. */
int coda_debug_split_first_tile(int tiles, int num_kb, int clusters);

/* The k-ranges per split tile of that launch (1 when it would not split),
 * -1 for invalid arguments.  Not for production use. */
int coda_debug_split_ranges(int tiles, int num_kb, int clusters);

/* Host-side check of the wide-tile schedule (coda_set_wide_tiles) of the
 * SM-pair GEMM, run with the kernel's own iterators (no GPU needed): an M x N
 * output (N with an even number of 256-column tiles) over K on `clusters` SM
 * pairs with lead `lead`.  Returns 0 when every 256 x 256 output tile is
 * computed by exactly one unit, every cluster meets its wide units before its
 * half-tile units, and each accumulator half of a unit sees every k-block
 * exactly once, starting and ending at the blocks where the kernel starts the
 * sum and commits it; the number of violations otherwise, -1 for invalid
 * arguments or an odd tile count.  Not for production use. */
int coda_debug_wide_schedule_violations(int M, int N, int K, int clusters, int lead);

/* 1 when a long-K backward GEMM (coda_gemm_dgrad_rmsbwd, or coda_gemm /
 * coda_gemm_wgrad_gscale with bf16 operands) with an M x N output over K
 * would take wide tiles on this handle now (coda_set_wide_tiles), 0 when it
 * would take 256-column tiles, -1 for invalid arguments.  Not for
 * production use. */
int coda_debug_wide_applies(coda_handle_t h, int M, int N, int K);

#ifdef __cplusplus
}
#endif
