/*
 * coda.h -- C ABI of libcoda: a Transformer block's memory-bound operations
 * run as GEMM epilogues on sm_103a (GB300).
 *
 * Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
 * (arXiv 2605.19269), as described by the Synced / KuCoin write-up:
 *   - section 尾声 / 尾聲: a GEMM is a mainloop plus an epilogue; the RMSNorm
 *     row scale r commutes with the next GEMM, so it is deferred into that
 *     GEMM's epilogue, while the first GEMM's epilogue only emits per-tile
 *     partial RMS that a very light auxiliary kernel merges; the same holds
 *     for SwiGLU, cross-entropy and the backward pass;
 *   - section 五种积木 / 五種積木: the epilogue primitives (elementwise,
 *     vector load/store, tile load/store, block reduction such as partial RMS
 *     and block log-sum-exp, stateful running max / sum-exp).
 *
 * Conventions for every call below.
 *   - Tensors are dense, row-major, with the leading dimension equal to the
 *     last extent.  "bf16" tensors are IEEE bfloat16 (passed as void*).
 *     Weights use nn.Linear layout: W1t[d][K1], W2t[N2][d], Wt[V][d].  For
 *     SwiGLU, rows [0, F) of W2t are the gate projection and rows [F, 2F) the
 *     up projection (N2 = 2F).
 *   - Every pointer is caller-owned CUDA device memory on the handle's device
 *     (except the handles, the out-parameters, and the step inputs and
 *     results of coda_block_step_host, which are host memory).  Device
 *     pointers must be 16-byte aligned.  The library allocates no device
 *     memory after coda_create and only reads or writes the buffers it is
 *     given; scratch space is passed in as a caller-owned workspace (or
 *     arena) whose size a *_workspace_bytes (*_arena_bytes) call returns.
 *   - Extents are int64_t.  Every contiguous extent (K1, d, N2, F, V) must be
 *     a positive multiple of 8 and every extent below 2^31.  M == 0 is a
 *     valid empty problem: nothing is launched and CODA_OK is returned.
 *   - Every compute call is asynchronous on `stream` (a cudaStream_t, NULL =
 *     legacy default stream).  The return value reports argument, alignment,
 *     shape and launch errors synchronously; nothing is launched when it is
 *     not CODA_OK.  Conditions detected on the device (a bounded wait that
 *     expired, a label out of range) are recorded in the handle's device
 *     status word and reported by coda_sync_status.
 *   - A handle may be used from one host thread at a time.
 */
#ifndef CODA_H_
#define CODA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum coda_status {
  CODA_OK = 0,
  CODA_ERR_INVALID_ARG = 1,        /* null pointer, non-positive or too large extent */
  CODA_ERR_ALIGNMENT = 2,          /* pointer not 16-byte aligned or extent not a multiple of 8 */
  CODA_ERR_UNSUPPORTED = 3,        /* shape or flag combination this library does not implement */
  CODA_ERR_WORKSPACE_TOO_SMALL = 4,
  CODA_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed (launch, tensor map) */
  CODA_ERR_TIMEOUT = 6,            /* device: an in-kernel wait hit its time limit */
  CODA_ERR_LABEL_RANGE = 7         /* device: a label outside [0, V) */
} coda_status_t;

typedef struct coda_handle_s* coda_handle_t;

/* flags of coda_gemm_rowscale_swiglu */
#define CODA_EPI_SWIGLU 0u /* out = silu(z[:, :F]) * z[:, F:], N2 = 2F */
#define CODA_EPI_PLAIN 1u  /* out = z (row scale only), N2 output columns */

/* ------------------------------------------------------------------------ */
/* handle, status                                                            */
/* ------------------------------------------------------------------------ */

/* Create a handle on CUDA device `device`: allocates the 4-byte device status
 * word (the only allocation the library makes).  *out receives the handle. */
coda_status_t coda_create(coda_handle_t* out, int device);

/* Free the handle and its status word.  NULL is accepted. */
coda_status_t coda_destroy(coda_handle_t h);

/* Static English description of a status code. */
const char* coda_status_string(coda_status_t s);

/* Synchronise `stream`, read and clear the device status word.  Returns
 * CODA_ERR_TIMEOUT or CODA_ERR_LABEL_RANGE if a kernel recorded that
 * condition since the last call, else CODA_OK.  If device_bits is not NULL it
 * receives the raw bit mask (bits 0-3: which wait timed out; bit 8: label
 * range). */
coda_status_t coda_sync_status(coda_handle_t h, void* stream, int32_t* device_bits);

/* Wall-clock limit, in nanoseconds, of every wait inside the library's GEMM
 * kernels (default 4e9).  On expiry the kernel records CODA_ERR_TIMEOUT, lets
 * its in-flight copies and MMAs finish, frees its tensor memory and returns.
 * 0 restores the default. */
coda_status_t coda_set_wait_timeout_ns(coda_handle_t h, uint64_t ns);

/* GEMM kernel form for every later call on this handle.  enable = 1 (the
 * default): each 256 x 256 output tile is computed by a pair of SMs with the
 * 2-SM tcgen05 MMA, each SM loading half of the operands; enable = 0: one SM
 * per 128 x 256 tile.  Results are identical up to fp32 summation order
 * inside the tensor core; the choice only affects speed. */
coda_status_t coda_set_sm_pairing(coda_handle_t h, int enable);

/* Wide tiles for the long-K GEMMs of the backward (the RMSNorm-backward
 * data gradient coda_gemm_dgrad_rmsbwd and the weight gradients of
 * coda_gemm_wgrad_gscale / coda_gemm), SM pairs only.  lead_kblocks = J > 0:
 * such a GEMM whose output has an even number of 256-column tiles and at
 * least max(4J, 256) k-blocks of 64 (K >= 16384) computes 256 x 512 tiles, two 256-column
 * halves per A tile, so each SM loads three quarters of the operand bytes
 * per MAC and the operand panels are re-read from memory less often.  The
 * tile's accumulator fills all of tensor memory; the first J k-blocks feed
 * only the first half and are repeated at the end for the second half, so
 * that the epilogue of one half runs while the other accumulates.  0 (the
 * default) turns wide tiles off.  Results equal the 256-column tiles' up to
 * fp32 summation order.  Returns CODA_ERR_INVALID_ARG outside [0, 64]. */
coda_status_t coda_set_wide_tiles(coda_handle_t h, int lead_kblocks);

/* Width of the vocabulary chunks of the LM-head backward (coda_lmhead_ce,
 * coda_lmhead_ce_fp8): the logits are recomputed and dL written for one
 * chunk of `cols` vocabulary columns at a time, then dH and that chunk's dW
 * rows are computed from it.  Narrower chunks shrink the dL buffer that
 * passes between the two launches, at the price of more and smaller launches
 * (measured slower at every width below the default).  cols: a multiple of 256 in [256, 32768]; 0
 * restores the default, 32768.  The workspace size does not depend on it.  Results equal across widths up to fp32 summation order
 * of dH.  Returns CODA_ERR_INVALID_ARG otherwise. */
coda_status_t coda_set_lmhead_chunk(coda_handle_t h, int64_t cols);

/* Scratch that lets this handle's SM-pair GEMMs keep every SM pair busy in
 * their last, partial wave.  Without it (the default) each SM pair computes
 * whole 256 x 256 tiles, and when the tile count is not a multiple of the
 * pairs the last wave leaves some pairs idle.  With it, each tile of that
 * last wave is cut into S equal k-ranges (2 <= S <= 6, the count that
 * finishes them in the fewest rounds), and the units are dealt range-major to
 * all pairs, so the units that run together cover the same k-range.  A unit
 * of an earlier range leaves its fp32 partial accumulator in this scratch;
 * the pair that runs the tile's last range adds the partials and runs the
 * epilogue.  Only launches whose ranges have at least 48 k-blocks are split,
 * and grouped launches never are.  Results differ from unsplit runs only in
 * the fp32 summation order of the split tiles, and a split launch is
 * deterministic.  Measured on the block step's long-K data gradient, it
 * neither gains nor loses beyond run-to-run noise under the power cap.
 * coda_split_workspace_bytes: bytes needed (one 256 KB partial per split
 * tile and earlier range, for the most a launch can need, plus flags; about
 * 94 MiB on a 152-SM GPU).  coda_set_split_workspace: ws (256-byte aligned,
 * at least that many bytes, caller-owned device memory) becomes the handle's
 * scratch; its flags are cleared on `stream`, so set it in stream order
 * before the GEMMs that use it; ws = NULL switches splitting off.  The
 * library allocates nothing.  While it is set, GEMMs issued through the
 * handle must not run concurrently with each other on the GPU (they share the
 * scratch): issue them on one stream, or give each stream its own handle.
 * Keep ws alive until it is replaced and the GEMMs that used it have
 * completed.  After a call reports CODA_ERR_TIMEOUT, set the workspace again
 * before the next GEMM (the aborted launch may have left flags raised). */
size_t coda_split_workspace_bytes(coda_handle_t h);
coda_status_t coda_set_split_workspace(coda_handle_t h, void* ws, size_t ws_bytes, void* stream);

/* Columns of a block-reduction partial buffer over n columns: ceil(n / 128).
 * Partial j of a row covers columns [128 j, 128 j + 128) (half of a 256-column
 * output tile).  Used for the partial RMS (n = d), the SwiGLU-backward c
 * partials (n = F) and the LM-head statistics (n = V). */
int64_t coda_prms_num_tiles(int64_t d);

/* Rows of the dg partial buffer of coda_gemm_dgrad_rmsbwd: 4 * ceil(M/128). */
int64_t coda_dgpart_rows(int64_t M);

/* ------------------------------------------------------------------------ */
/* the fixed mainloop with a plain epilogue                                  */
/* ------------------------------------------------------------------------ */

/* C[M][N] = bf16( row_scale[m] * col_scale[n] * sum_k A(m,k) B(k,n) ).
 * The mainloop of the write-up's section 尾声, epilogue = scale + store.
 * A is [M][K] (a_mn_major = 0) or stored transposed as [K][M] (a_mn_major = 1);
 * B is [N][K] (b_mn_major = 0) or [K][N] (b_mn_major = 1).  Supported
 * combinations: (0,0), (0,1), (1,1).  row_scale (fp32 [M]) and col_scale
 * (bf16 [N]) may be NULL.  M, N, K multiples of 8. */
coda_status_t coda_gemm(coda_handle_t h, const void* A, int a_mn_major, const void* B, int b_mn_major, void* C,
                        int64_t M, int64_t N, int64_t K, const float* row_scale, const void* col_scale,
                        void* stream);

/* ------------------------------------------------------------------------ */
/* forward: GEMM-Residual-PartialRMS-GEMM (+SwiGLU)                           */
/* ------------------------------------------------------------------------ */

/* W2gt[n][k] = bf16(W2t[n][k] * g[k]) -- the RMSNorm weight g (bf16 [d]) folded
 * into the second GEMM's B operand (section 尾声: r and g are per-row /
 * per-column scales that commute with the contraction; section 五种积木:
 * vector load of the RMSNorm weight).  W2t, W2gt: bf16 [N2][d]; may not
 * alias. */
coda_status_t coda_fold_rmsnorm_weight(coda_handle_t h, const void* W2t, const void* g, void* W2gt, int64_t N2,
                                       int64_t d, void* stream);

/* GEMM1 with the residual + partial-RMS epilogue (section 尾声):
 *   H[m][n] = bf16( sum_k X[m][k] W1t[n][k] + R[m][n] )
 *   psum[m][j] = sum over n in [128 j, 128 j + 128) of H[m][n]^2  (fp32, H as stored)
 * X bf16 [M][K1], W1t bf16 [d][K1], R bf16 [M][d], H bf16 [M][d],
 * psum fp32 [M][coda_prms_num_tiles(d)].  H may not alias R. */
coda_status_t coda_gemm_res_prms(coda_handle_t h, const void* X, const void* W1t, const void* R, void* H,
                                 float* psum, int64_t M, int64_t K1, int64_t d, void* stream);

/* coda_gemm_res_prms that also applies the RMSNorm weight on the activation
 * side: the epilogue broadcasts g along each row (section 五种积木: vector
 * load of the RMSNorm weight) and writes a second output
 *   Hg[m][n] = bf16( H[m][n] * g[n] )
 * which the second GEMM then takes as its A operand with the unfolded W2t
 * (coda_gemm_rowscale_swiglu(Hg, W2t, ...)).  This replaces the per-step
 * coda_fold_rmsnorm_weight pass over W2 with one extra [M][d] write.  g bf16
 * [d], Hg bf16 [M][d]; the rest as coda_gemm_res_prms. */
coda_status_t coda_gemm_res_prms_g(coda_handle_t h, const void* X, const void* W1t, const void* R, const void* g,
                                   void* H, void* Hg, float* psum, int64_t M, int64_t K1, int64_t d, void* stream);

/* The light auxiliary combine (section 尾声):
 *   rstd[m] = 1 / sqrt( sum_j psum[m][j] / d + eps )
 * psum fp32 [M][T], rstd fp32 [M]. */
coda_status_t coda_rstd_combine(coda_handle_t h, const float* psum, int64_t M, int64_t T, int64_t d, float eps,
                                float* rstd, void* stream);

/* GEMM2 with the deferred row scale and SwiGLU epilogue (section 尾声, and the
 * SwiGLU re-parameterisation it lists):
 *   z[m][n] = rstd[m] * sum_k H[m][k] W2gt[n][k]
 *   CODA_EPI_SWIGLU: out[m][j] = silu(z[m][j]) * z[m][F + j], out bf16 [M][F],
 *                    N2 = 2F; if z_save is not NULL it receives z (bf16
 *                    [M][N2], the tile store that saves activations for the
 *                    backward).
 *   CODA_EPI_PLAIN:  out[m][n] = z[m][n], out bf16 [M][N2]; z_save must be
 *                    NULL.
 * H bf16 [M][d], W2gt bf16 [N2][d] (from coda_fold_rmsnorm_weight), rstd fp32
 * [M].  N2 (and F for SwiGLU) multiples of 8. */
coda_status_t coda_gemm_rowscale_swiglu(coda_handle_t h, const void* H, const void* W2gt, const float* rstd,
                                        void* out, void* z_save, int64_t M, int64_t d, int64_t N2, uint32_t flags,
                                        void* stream);

/* The same GEMM2 with the light combine folded into its epilogue: each output
 * tile derives its rows' scale from GEMM1's partial sums,
 *   rstd[m] = 1 / sqrt( sum_j psum[m][j] / d + eps ),
 * so the separate coda_rstd_combine launch disappears (its work is T loads per
 * row per tile, read from L2).  psum fp32 [M][T] (from coda_gemm_res_prms),
 * rstd fp32 [M] receives the row scale for the backward (may be NULL); the
 * other arguments, flags and outputs are those of coda_gemm_rowscale_swiglu.
 * The row sum runs in a different order than coda_rstd_combine's, so rstd can
 * differ in the last bit. */
coda_status_t coda_gemm_prms_rowscale_swiglu(coda_handle_t h, const void* H, const void* W2gt, const float* psum,
                                             int64_t T, float eps, float* rstd, void* out, void* z_save, int64_t M,
                                             int64_t d, int64_t N2, uint32_t flags, void* stream);

/* ------------------------------------------------------------------------ */
/* backward (section 尾声: the backward of a block-local epilogue is itself    */
/* block-local)                                                              */
/* ------------------------------------------------------------------------ */

/* SwiGLU backward with the row scale folded in:
 *   dZ = d(silu(zg) * zu) applied to dY;  dP = bf16(rstd[m] * dZ)
 *   c[m] = rstd[m]^2 / d * sum_n dZ[m][n] z[m][n]
 * dY bf16 [M][F], z bf16 [M][2F] (from the forward), rstd fp32 [M],
 * dP bf16 [M][2F], c fp32 [M]; d is the hidden width. */
coda_status_t coda_swiglu_bwd(coda_handle_t h, const void* dY, const void* z, const float* rstd, void* dP,
                              float* c, int64_t M, int64_t F, int64_t d, void* stream);

/* Data gradient of GEMM2 with the RMSNorm backward in its epilogue:
 *   acc[m][k] = sum_n dP[m][n] W2t[n][k]
 *   dH[m][k]  = bf16( g[k] * acc[m][k] - c[m] * H[m][k] )
 *   dgpart[r][k] = sum over rows m of block r (32 rows) of acc[m][k] * H[m][k]
 * dP bf16 [M][N2], W2t bf16 [N2][d] (unfolded), H bf16 [M][d], g bf16 [d],
 * c fp32 [M], dH bf16 [M][d], dgpart fp32 [coda_dgpart_rows(M)][d]. */
coda_status_t coda_gemm_dgrad_rmsbwd(coda_handle_t h, const void* dP, const void* W2t, const void* H,
                                     const void* g, const float* c, void* dH, float* dgpart, int64_t M, int64_t N2,
                                     int64_t d, void* stream);

/* Allocation-free form of coda_gemm_dgrad_rmsbwd followed by coda_dg_combine:
 * the same dH and dg, but the dg partial sums live in an array compiled into
 * the library instead of a caller buffer.  The CODA write-up has no
 * counterpart to this call; it exists for callers that cannot allocate device
 * memory at all -- for example a host framework that passes a plugin only its
 * input and output tensors while its own pool owns the rest of the device, or
 * a latency-critical caller that must not pay for, or synchronise on, an
 * allocation.  It calls no cudaMalloc, cudaFree or allocating library routine.
 *   Inputs and outputs as coda_gemm_dgrad_rmsbwd; dg fp32 [d] receives the
 *   column sums directly.
 *   Limit: coda_dgpart_rows(M) * d * 4 bytes must not exceed 8 MiB (e.g. M up
 *   to 8192 at d = 8192, or 16384 at d = 4096); larger problems are rejected
 *   with CODA_ERR_WORKSPACE_TOO_SMALL before anything is launched.  The 8 MiB
 *   array is a file-scope static __device__ array: it is reserved on a device
 *   once the library's module holding it is loaded there (with the CUDA
 *   runtime's lazy loading, at the latest on the first call on that device)
 *   and held until the process exits.
 *   The first call with a given handle looks up the array's device address
 *   (with the handle's device current) and keeps it in the handle; make that
 *   first call before any stream capture.  Handles do not outlive their
 *   context: after a device reset, create a new handle, which looks the
 *   address up again.
 *   All calls share the one array per device: calls that may overlap on the
 *   GPU (different streams, or different host threads) race on it and must be
 *   serialised by the caller.  Every partial a call reads is written earlier
 *   in the same call, so what a previous call left there is never used. */
coda_status_t coda_gemm_dgrad_rmsbwd_noalloc(coda_handle_t h, const void* dP, const void* W2t, const void* H,
                                             const void* g, const float* c, void* dH, float* dg, int64_t M,
                                             int64_t N2, int64_t d, void* stream);

/* SwiGLU backward in the epilogue of the down projection's data gradient
 * (the upstream gradient dY of the SwiGLU output stays on chip and is never
 * written to HBM).  With the down projection y = out W3 (nn.Linear
 * layout W3t[d][F]) and its upstream gradient dYb:
 *   dY[m][j] = sum_k dYb[m][k] W3t[k][j]                 (mainloop, on chip)
 *   dP = bf16(rstd[m] * dZ), dZ = d(silu(z_gate) * z_up) applied to dY
 *   cpart[m][t] = sum over the gate columns j in [128 t, 128 t + 128) (and their
 *                 up columns) of dZ * z                  (block reduction)
 * so that c[m] = rstd[m]^2 / d * sum_t cpart[m][t] (coda_swiglu_bwd's c).
 * dYb bf16 [M][d], W3t bf16 [d][F], z bf16 [M][2F], rstd fp32 [M],
 * dP bf16 [M][2F], cpart fp32 [M][coda_prms_num_tiles(F)]. */
coda_status_t coda_gemm_dgrad_swiglu_bwd(coda_handle_t h, const void* dYb, const void* W3t, const void* z,
                                         const float* rstd, void* dP, float* cpart, int64_t M, int64_t d, int64_t F,
                                         void* stream);

/* coda_gemm_dgrad_rmsbwd with c formed in its epilogue from the partial sums
 * of coda_gemm_dgrad_swiglu_bwd: c[m] = rstd[m]^2 / d * sum_t cpart[m][t]
 * (Tc = coda_prms_num_tiles(F) columns); everything else as
 * coda_gemm_dgrad_rmsbwd. */
coda_status_t coda_gemm_dgrad_rmsbwd_cpart(coda_handle_t h, const void* dP, const void* W2t, const void* H,
                                           const void* g, const float* rstd, const float* cpart, int64_t Tc,
                                           void* dH, float* dgpart, int64_t M, int64_t N2, int64_t d, void* stream);

/* dg[k] = sum_r dgpart[r][k] (fixed order).  dgpart fp32 [rows][d], dg fp32 [d]. */
coda_status_t coda_dg_combine(coda_handle_t h, const float* dgpart, int64_t rows, int64_t d, float* dg,
                              void* stream);

/* Weight gradient of GEMM2 with the folded g applied per column:
 *   dW2t[n][k] = bf16( g[k] * sum_m dP[m][n] H[m][k] )
 * H bf16 [M][d], dP bf16 [M][N2], g bf16 [d], dW2t bf16 [N2][d]. */
coda_status_t coda_gemm_wgrad_gscale(coda_handle_t h, const void* H, const void* dP, const void* g, void* dW2t,
                                     int64_t M, int64_t N2, int64_t d, void* stream);

/* Workspace of coda_gemm_rowscale_swiglu_bwd: dP bf16 [M][N2], c fp32 [M],
 * dgpart fp32 [coda_dgpart_rows(M)][d], each 256-byte aligned. */
size_t coda_bwd_workspace_bytes(int64_t M, int64_t d, int64_t N2);

/* Backward of GEMM2 + deferred RMSNorm + SwiGLU, chaining coda_swiglu_bwd,
 * coda_gemm_dgrad_rmsbwd, coda_dg_combine and coda_gemm_wgrad_gscale:
 * outputs dH (bf16 [M][d], = dR = dA of the residual stream), dW2t (bf16
 * [N2][d]) and dg (fp32 [d]).  Inputs as the stage calls; SwiGLU only. */
coda_status_t coda_gemm_rowscale_swiglu_bwd(coda_handle_t h, const void* dY, const void* z, const float* rstd,
                                            const void* H, const void* W2t, const void* g, void* dH, void* dW2t,
                                            float* dg, void* ws, size_t ws_bytes, int64_t M, int64_t d, int64_t N2,
                                            void* stream);

/* Backward of GEMM1 + residual: dX = dH W1 (bf16 [M][K1]), dW1t = dH^T X
 * (bf16 [d][K1]).  With SM pairing (the default) both GEMMs run in one
 * persistent launch: the SM pairs take the tiles of both from one balanced
 * schedule, so there is one partly idle last wave and one prologue instead
 * of two (1.3 % faster than two launches at the 7B size).  dR: NULL, or == dH (aliased: nothing is written, since
 * dR = dH), or a distinct bf16 [M][d] buffer that receives a copy of dH. */
coda_status_t coda_gemm_res_prms_bwd(coda_handle_t h, const void* dH, const void* X, const void* W1t, void* dX,
                                     void* dW1t, void* dR, int64_t M, int64_t K1, int64_t d, void* stream);

/* ------------------------------------------------------------------------ */
/* block step executor: the whole step issued natively, with its inputs and  */
/* results in host memory                                                    */
/* ------------------------------------------------------------------------ */

/* One executor runs the fused step of the write-up's flagship block (section
 * 尾声: GEMM1 + residual + partial RMS with the fold of g beside it, the rstd
 * combine, GEMM2 + row scale + SwiGLU, then, with backward = 1, the SwiGLU
 * backward, dgrad2 with the RMSNorm backward, dg, wgrad2, dX and dW1) for
 * inputs that live in page-locked host memory.  Each coda_block_step_host
 * call enqueues the host-to-device copies of the step's X, R (and dY), the
 * step's kernels and the read-back of the requested results, and returns
 * without waiting.  Two device slots hold what the copies touch, so the
 * copies of step n+1 and the read-back of step n-1 overlap step n's kernels;
 * the kernels of successive steps run in submission order on one stream.
 * The executor computes exactly what the separate calls compute (same
 * kernels, same order): its results are bit-identical to theirs.  An
 * executor may be used from one host thread at a time. */
typedef struct coda_block_s* coda_block_t;

/* flags of coda_block_create */
#define CODA_BLOCK_BACKWARD 1u    /* forward + backward (else forward only) */
#define CODA_BLOCK_FP8 2u         /* 8-bit operands: e4m3 activations and weights, e5m2 gradients */
#define CODA_BLOCK_FP8_DELAYED 4u /* with FP8 and backward: dP's codes scaled by the previous step's
                                     amax (coda_swiglu_bwd_fp8_delayed) after the first step */

/* Device bytes the executor needs for a problem (its arena): H, psum, rstd
 * and z once; W2g and the backward workspace (bf16), or the weight,
 * activation and gradient codes with their scales, c and the dg partials
 * (FP8); and X, R, out (and dY, dH, dX) in each of two slots, every buffer
 * 256-byte aligned.  0 for an invalid shape. */
size_t coda_block_arena_bytes(int64_t M, int64_t K1, int64_t d, int64_t N2, uint32_t flags);

/* Create an executor on the current CUDA device, which must be the handle's.
 * Shapes as coda_gemm_res_prms / coda_gemm_rowscale_swiglu with SwiGLU
 * (N2 = 2F, F a multiple of 8; with CODA_BLOCK_FP8 K1 and d multiples of 16
 * and F of 16); eps > 0 is the RMSNorm epsilon; flags a combination of
 * CODA_BLOCK_* (CODA_ERR_INVALID_ARG for unknown bits, or for
 * CODA_BLOCK_FP8_DELAYED without FP8 and BACKWARD).
 * Weights (device, bf16, caller-owned, read by every step): W1t [d][K1], g
 * [d], W2t [N2][d].  With CODA_BLOCK_BACKWARD every step overwrites the
 * weight gradients dW1t (bf16 [d][K1]), dW2t (bf16 [N2][d]) and dg (fp32
 * [d]), device buffers the caller owns; without it they may be NULL.  arena:
 * caller-owned device memory of at least coda_block_arena_bytes bytes,
 * 16-byte aligned, used only by this executor until it is destroyed.  The
 * executor creates four CUDA streams and its events; it allocates no device
 * memory.  *out receives the executor. */
coda_status_t coda_block_create(coda_handle_t h, int64_t M, int64_t K1, int64_t d, int64_t N2, float eps,
                                uint32_t flags, const void* W1t, const void* g, const void* W2t, void* dW1t,
                                void* dW2t, float* dg, void* arena, size_t arena_bytes, coda_block_t* out);

/* FP8 executors: enqueue, on the executor's compute stream, the e4m3
 * quantisation of the weights the steps use (W1, W2 with g folded in, and
 * W2 alone for the backward), as coda_fp8_quantize does.  Call it after
 * coda_block_create and after every update of W1t, g or W2t; an FP8 step
 * before the first call is refused with CODA_ERR_INVALID_ARG.  A no-op for
 * bf16 executors. */
coda_status_t coda_block_quantize_weights(coda_block_t b);

/* Enqueue one step (bf16, or FP8 per the executor's flags: X and H quantised
 * in the step, the FP8 backward of coda_swiglu_bwd_fp8 and the 8-bit GEMMs).
 * Host pointers, each page-locked (cudaHostAlloc) or
 * registered (cudaHostRegister) memory, else CODA_ERR_INVALID_ARG:
 *   X bf16 [M][K1], R bf16 [M][d] (required), dY bf16 [M][F] (required with
 *   backward, NULL without);
 *   out bf16 [M][F] receives the SwiGLU output, dX bf16 [M][K1] the input
 *   gradient and dR bf16 [M][d] the residual gradient (= dH); each may be
 *   NULL (not read back); dX and dR must be NULL without backward.
 * The call returns once everything is enqueued.  The host inputs must stay
 * unchanged, and the results are not valid, until coda_block_wait_step for
 * this step (or coda_block_sync) has returned.  *step_id (may be NULL)
 * receives the step's index, counted from 0 per executor. */
coda_status_t coda_block_step_host(coda_block_t b, const void* X, const void* R, const void* dY, void* out, void* dX,
                                   void* dR, int64_t* step_id);

/* Block until step `step` has finished: its inputs have been read and its
 * results written to host memory.  It may also wait for the next step that
 * uses the same slot (step + 2) if that has been submitted. */
coda_status_t coda_block_wait_step(coda_block_t b, int64_t step);

/* Block until every submitted step has finished, then read and clear the
 * handle's device status word as coda_sync_status does (its return value and
 * device_bits have the same meaning). */
coda_status_t coda_block_sync(coda_block_t b, int32_t* device_bits);

/* *stream receives the executor's compute stream (a cudaStream_t): work the
 * caller enqueues there (an optimizer update of the weights, say) runs after
 * the steps submitted before it and before those submitted after it. */
coda_status_t coda_block_stream(coda_block_t b, void** stream);

/* Wait for the executor's streams, then destroy them and the executor.  NULL
 * is accepted.  The arena is the caller's to free afterwards. */
coda_status_t coda_block_destroy(coda_block_t b);

/* ------------------------------------------------------------------------ */
/* rotary position embedding on the QKV projection (section 五种积木: RoPE  */
/* among the elementwise epilogue transforms)                                */
/* ------------------------------------------------------------------------ */

/* cos_t[p][i] = cos(p * base^(-2 i / head_dim)), sin_t likewise, for
 * positions p < S and i < head_dim / 2, computed in double precision and
 * stored fp32.  cos_t, sin_t fp32 [S][head_dim / 2]; head_dim a positive
 * multiple of 16. */
coda_status_t coda_rope_table(coda_handle_t h, float* cos_t, float* sin_t, int64_t S, int64_t head_dim, float base,
                              void* stream);

/* QKV projection with RoPE in the epilogue:
 *   qkv[m][n] = sum_k X[m][k] Wqkv_t[n][k], columns [q heads | k heads | v heads]
 *   then every q and k head (columns < (n_q_heads + n_kv_heads) * head_dim)
 *   is rotated at position p = m mod S with rotate-half pairing:
 *   out_i = x_i cos - x_{i+D/2} sin, out_{i+D/2} = x_{i+D/2} cos + x_i sin.
 * X bf16 [M][d] (rows batch-major, S positions per sequence), Wqkv_t bf16
 * [(n_q_heads + 2 n_kv_heads) * head_dim][d], cos_t/sin_t from
 * coda_rope_table, qkv bf16 [M][(n_q_heads + 2 n_kv_heads) * head_dim].
 * head_dim must be 128 (one head = half an output tile): other values
 * return CODA_ERR_UNSUPPORTED. */
coda_status_t coda_gemm_qkv_rope(coda_handle_t h, const void* X, const void* Wqkv_t, const float* cos_t,
                                 const float* sin_t, void* qkv, int64_t M, int64_t d, int64_t n_q_heads,
                                 int64_t n_kv_heads, int64_t head_dim, int64_t S, void* stream);

/* The same rotation as a standalone in-place kernel on an existing qkv (the
 * unfused baseline): qkv bf16 [M][(n_q_heads + 2 n_kv_heads) * head_dim],
 * head_dim a multiple of 16. */
coda_status_t coda_rope_apply(coda_handle_t h, void* qkv, const float* cos_t, const float* sin_t, int64_t M,
                              int64_t n_q_heads, int64_t n_kv_heads, int64_t head_dim, int64_t S, void* stream);

/* ------------------------------------------------------------------------ */
/* FP8 operands (the write-up's 背景 section: FP8 speeds up the matmul, which  */
/* raises the relative cost of the memory-bound operations the epilogues     */
/* absorb): e4m3 codes with one fp32 scale per tensor                        */
/* ------------------------------------------------------------------------ */

/* Per-tensor e4m3 quantisation:
 *   amax = max |src[r][c] * g[c]|  (g = 1 when NULL; the product in fp32)
 *   scale = the smallest power of two 2^k with amax / 2^k <= 448 (k >= -126;
 *           1 when amax == 0), so the largest element lands in (224, 448]
 *   dst[r][c] = e4m3( src[r][c] * g[c] / scale ), round to nearest even,
 *               saturating at +-448 (the division by a power of two is exact:
 *               each element is rounded once, and code * scale is exact)
 * src bf16 [rows][cols], g bf16 [cols] or NULL (with g = the RMSNorm weight
 * and src = W2t this folds g into W2 while quantising), amax_scale fp32 [2]
 * receives {amax, scale}, dst e4m3 codes [rows][cols] (1 byte each).  cols a
 * multiple of 16. */
coda_status_t coda_fp8_quantize(coda_handle_t h, const void* src, const void* g, float* amax_scale, void* dst,
                                int64_t rows, int64_t cols, void* stream);

/* The same quantisation to e5m2 (5 exponent, 2 mantissa bits): scale = the
 * smallest power of two with amax / scale <= 57344, dst = e5m2( src * g /
 * scale ), saturating at +-57344.  The wider range suits gradients. */
coda_status_t coda_fp8_quantize_e5m2(coda_handle_t h, const void* src, const void* g, float* amax_scale, void* dst,
                                     int64_t rows, int64_t cols, void* stream);

/* coda_swiglu_bwd with dP delivered as per-tensor scaled 8-bit codes (the FP8
 * backward's operand of dgrad2 and wgrad2): the codes, amax and scale equal
 * those of coda_swiglu_bwd followed by coda_fp8_quantize (format 0, e4m3) or
 * coda_fp8_quantize_e5m2 (format 1) on its bf16 dP, but dP is never written.
 * Two passes over dY and z: the first writes c and the absolute maximum of
 * bf16(dP), the second recomputes bf16(dP) and writes the codes.
 * dY bf16 [M][F], z bf16 [M][2F], rstd fp32 [M]; dPq codes [M][2F] (gate
 * half, then up half); amax_scale fp32 [2] receives {amax, scale} ({0, 1}
 * when M == 0); c fp32 [M].  F and d multiples of 8. */
coda_status_t coda_swiglu_bwd_fp8(coda_handle_t h, const void* dY, const void* z, const float* rstd, int format,
                                  void* dPq, float* amax_scale, float* c, int64_t M, int64_t F, int64_t d,
                                  void* stream);

/* coda_swiglu_bwd_fp8 with delayed scaling: the scale of dP's codes comes from
 * the absolute maximum of the previous step's dP instead of this one's, so a
 * single pass over dY and z writes c, the codes and this dP's maximum.
 * amax_scale fp32 [2]: on entry amax_scale[0] holds the previous maximum (as
 * left by coda_swiglu_bwd_fp8 or by this call on the previous step); on exit
 * it holds {max |bf16(dP)| of this step, the scale used}, the scale being the
 * power of two that coda_fp8_quantize(_e5m2) derives from the entry maximum.
 * Codes of elements beyond the previous range saturate (+-448 e4m3, +-57344
 * e5m2 times the scale).  The first step of a run, with no previous maximum,
 * uses coda_swiglu_bwd_fp8.  Other arguments as coda_swiglu_bwd_fp8; M == 0
 * writes {0, 1}. */
coda_status_t coda_swiglu_bwd_fp8_delayed(coda_handle_t h, const void* dY, const void* z, const float* rstd,
                                          int format, void* dPq, float* amax_scale, float* c, int64_t M, int64_t F,
                                          int64_t d, void* stream);

/* Plain GEMM on 8-bit operands (the mainloop of the method with FP8 inputs):
 *   C[m][n] = bf16( row_scale[m] * col_scale[n] * sA * sB * sum_k A[m][k] B[k][n] )
 * A codes [M][K] (a_mn_major = 0) or [K][M] (1); B codes [N][K] (0) or [K][N]
 * (1); a_format / b_format 0 = e4m3, 1 = e5m2 (mixed allowed); sA, sB device
 * pointers to fp32 scales or NULL (1); row_scale fp32 [M], col_scale bf16 [N],
 * both optional; C bf16 [M][N].  The contiguous extent of every 8-bit operand
 * (K for K-major, M or N for MN-major) a multiple of 16, N a multiple of 8.
 * With both operands MN-major K is their row count and may take any value
 * >= 0 (a token count for a weight gradient; K = 0 writes C = 0 and A, B may
 * be NULL).  MN-major A with K-major B returns CODA_ERR_UNSUPPORTED. */
coda_status_t coda_gemm_fp8(coda_handle_t h, const void* A, int a_mn_major, int a_format, const float* sA,
                            const void* B, int b_mn_major, int b_format, const float* sB, void* C, int64_t M,
                            int64_t N, int64_t K, const float* row_scale, const void* col_scale, void* stream);

/* coda_gemm_res_prms_bwd on 8-bit operands: the first layer's data and
 * weight gradients from dH's codes,
 *   dX[m][i]   = bf16( sdH * sW1 * sum_k dHq[m][k] W1q[k][i] )
 *   dW1t[k][i] = bf16( sdH * sX  * sum_m dHq[m][k] Xq[m][i] )
 * with SM pairing in one persistent launch (the schedule of
 * coda_gemm_res_prms_bwd), otherwise two launches; the results equal those
 * of the two coda_gemm_fp8 calls bit for bit.  dHq codes [M][d] (dh_format: 0
 * = e4m3, 1 = e5m2), Xq codes [M][K1] and W1q codes [d][K1] (both w_format),
 * sdH / sX / sW1 device pointers to fp32 scales (NULL = 1); dX bf16 [M][K1],
 * dW1t bf16 [d][K1].  K1 and d multiples of 16; any M >= 0 (M == 0 writes
 * dW1t = 0). */
coda_status_t coda_gemm_res_prms_bwd_fp8(coda_handle_t h, const void* dHq, int dh_format, const float* sdH,
                                         const void* Xq, const float* sX, const void* W1q, const float* sW1,
                                         int w_format, void* dX, void* dW1t, int64_t M, int64_t K1, int64_t d,
                                         void* stream);

/* coda_gemm_dgrad_rmsbwd on 8-bit operands (the RMSNorm-backward epilogue
 * with FP8 inputs):
 *   acc = sdP * sW2 * sum_n dPq[m][n] W2q[n][k];  dH = bf16(g * acc - c * h);
 *   dgpart as coda_gemm_dgrad_rmsbwd.
 * dPq codes [M][N2] (dp_format: 0 = e4m3, 1 = e5m2, the usual choice for a
 * gradient), W2q codes of W2t [N2][d] (w_format, without g), sdP / sW2 device
 * pointers to the scales.  N2 and d multiples of 16.  The weight gradient
 * dW2t = g * dP^T H and the first layer's dX / dW1t on FP8 operands are
 * coda_gemm_fp8 calls with MN-major operands. */
coda_status_t coda_gemm_dgrad_rmsbwd_fp8(coda_handle_t h, const void* dPq, int dp_format, const float* sdP,
                                         const void* W2q, int w_format, const float* sW2, const void* H,
                                         const void* g, const float* c, void* dH, float* dgpart, int64_t M,
                                         int64_t N2, int64_t d, void* stream);

/* coda_gemm_res_prms on e4m3 operands: H = bf16( sX * sW1 * sum_k Xq[m][k]
 * W1q[n][k] + R ), psum as before.  Xq codes [M][K1], W1q codes [d][K1], sX /
 * sW1 device pointers to the tensors' scales (amax_scale + 1 of
 * coda_fp8_quantize; scalar pointers need only 4-byte alignment).  K1 and d
 * multiples of 16. */
coda_status_t coda_gemm_res_prms_fp8(coda_handle_t h, const void* Xq, const float* sX, const void* W1q,
                                     const float* sW1, const void* R, void* H, float* psum, int64_t M, int64_t K1,
                                     int64_t d, void* stream);

/* coda_gemm_rowscale_swiglu on e4m3 operands: z = rstd[m] * sH * sW2 *
 * sum_k Hq[m][k] W2gq[n][k], then the same SwiGLU / PLAIN epilogue.  Hq codes
 * [M][d], W2gq codes [N2][d] (e.g. coda_fp8_quantize of W2t with g).  d a
 * multiple of 16, and with SwiGLU N2 / 2 a multiple of 16 (CODA_ERR_ALIGNMENT
 * otherwise). */
coda_status_t coda_gemm_rowscale_swiglu_fp8(coda_handle_t h, const void* Hq, const float* sH, const void* W2gq,
                                            const float* sW2, const float* rstd, void* out, void* z_save, int64_t M,
                                            int64_t d, int64_t N2, uint32_t flags, void* stream);

/* ------------------------------------------------------------------------ */
/* LM head: blocked log-sum-exp cross-entropy epilogue (section 五种积木:     */
/* block reduction "block log-sum-exp", stateful max / sum-exp)              */
/* ------------------------------------------------------------------------ */

/* Workspace of coda_lmhead_ce (with_grads = 0: forward only): the per-tile
 * statistics partials (3 x M x ceil(V / 128) x 4 bytes), the per-row label
 * logits and losses, and with gradients the fp32 dH accumulator (M x d x 4)
 * and one vocabulary chunk of dL (M x min(V, 32768) x 2 bytes). */
size_t coda_lmhead_ce_workspace_bytes(int64_t M, int64_t d, int64_t V, int with_grads);

/* Per-row results that coda_lmhead_ce and coda_lmhead_ce_fp8 leave in their
 * workspace (the per-token losses behind the mean, e.g. for masking or
 * logging).  Writes the byte offsets, from the workspace's start, of:
 *   *label_logit_off: fp32 [M], L[m][y_m], the logit of row m's label,
 *                     gathered by the epilogue of the vocabulary tile that
 *                     holds column y_m (0 for a label outside [0, V));
 *   *row_loss_off:    fp32 [M], lse[m] - L[m][y_m] (0 for a label outside
 *                     [0, V)); the loss output is their mean.
 * Both offsets are multiples of 256.  The values are those of the last call
 * on that workspace with the same M, d, V and with_grads, once it has
 * completed on its stream.  Either output pointer may be NULL.  Returns
 * CODA_ERR_INVALID_ARG for M, d or V <= 0. */
coda_status_t coda_lmhead_ce_row_offsets(int64_t M, int64_t d, int64_t V, int with_grads, size_t* label_logit_off,
                                         size_t* row_loss_off);

/* Mean softmax cross-entropy of the logits L = Hs Wt^T against labels,
 * without ever writing an [M][V] logits tensor:
 *   per (row, 128-column vocabulary block): max, sum exp(L - max), argmax,
 *   label logit (GEMM epilogue); combine: lse[m] = log sum_v exp L[m][v];
 *   loss = mean_m (lse[m] - L[m][y_m]); argmax[m] = first maximal column.
 * If dHs is not NULL the gradients are produced too, vocabulary chunk by
 * chunk: dL = (softmax - onehot)/M recomputed in a GEMM epilogue into a
 * workspace chunk, dHs = dL Wt (fp32 accumulation across chunks), dWt =
 * dL^T Hs.
 * Hs bf16 [M][d], Wt bf16 [V][d], labels int32 [M] in [0, V) (a label outside
 * sets CODA_ERR_LABEL_RANGE in the status word and its row contributes 0 to
 * the sum), loss fp32 [1], lse fp32 [M], argmax int32 [M] or NULL,
 * dHs bf16 [M][d] or NULL, dWt bf16 [V][d] (required iff dHs != NULL). */
coda_status_t coda_lmhead_ce(coda_handle_t h, const void* Hs, const void* Wt, const int32_t* labels, float* loss,
                             float* lse, int32_t* argmax, void* dHs, void* dWt, void* ws, size_t ws_bytes, int64_t M,
                             int64_t d, int64_t V, void* stream);

/* coda_lmhead_ce on 8-bit operands (the FP8 variant of the same epilogue
 * programs): Hq e4m3 codes [M][d] with scale *sH and Wq e4m3 codes [V][d]
 * with scale *sW (coda_fp8_quantize), so L = sH * sW * Hq Wq^T; the
 * statistics, loss, lse and argmax as coda_lmhead_ce.  The backward keeps the
 * recomputed dL = (softmax - onehot)/M of each vocabulary chunk as e5m2 codes
 * with the power-of-two scale s = 2^k fixed by |dL| <= 1/M (the smallest with
 * (1/M) / s <= 57344, so no code saturates), and forms dHs = dL Wt and dWt =
 * dL^T Hs from those codes and the e4m3 codes of W and H (fp32 accumulation
 * across chunks for dHs).  Same outputs and workspace
 * (coda_lmhead_ce_workspace_bytes) as coda_lmhead_ce; d and V multiples of 16
 * (CODA_ERR_ALIGNMENT otherwise). */
coda_status_t coda_lmhead_ce_fp8(coda_handle_t h, const void* Hq, const float* sH, const void* Wq, const float* sW,
                                 const int32_t* labels, float* loss, float* lse, int32_t* argmax, void* dHs,
                                 void* dWt, void* ws, size_t ws_bytes, int64_t M, int64_t d, int64_t V,
                                 void* stream);

/* ------------------------------------------------------------------------ */
/* unfused ablation: the same GEMM kernel with standalone memory-bound       */
/* kernels in between (the "three separate operators" baseline of section    */
/* 尾声)                                                                      */
/* ------------------------------------------------------------------------ */

/* Workspace of coda_unfused_fwd / coda_unfused_bwd. */
size_t coda_unfused_workspace_bytes(int64_t M, int64_t d, int64_t N2);

/* A = X W1 (GEMM) ; H = bf16(A + R), rstd, Nrm = bf16(H rstd g) (one kernel) ;
 * z = Nrm W2 (GEMM, bf16 [M][N2]) ; out = silu(z_gate) z_up (kernel) or out = z
 * when flags == CODA_EPI_PLAIN (then `out` may equal `z`).  Nrm bf16 [M][d] is
 * kept for the backward. */
coda_status_t coda_unfused_fwd(coda_handle_t h, const void* X, const void* W1t, const void* R, const void* g,
                               const void* W2t, void* H, float* rstd, void* Nrm, void* z, void* out, void* ws,
                               size_t ws_bytes, int64_t M, int64_t K1, int64_t d, int64_t N2, float eps,
                               uint32_t flags, void* stream);

/* dZ = SwiGLU'(dY) (kernel) ; dN = dZ W2^T (GEMM) ; dH = RMSNorm'(dN) (kernel),
 * dg (kernel + combine) ; dW2t = dZ^T Nrm (GEMM) ; dX, dW1t (GEMMs).
 * SwiGLU only. */
coda_status_t coda_unfused_bwd(coda_handle_t h, const void* dY, const void* X, const void* W1t, const void* g,
                               const void* W2t, const void* H, const float* rstd, const void* Nrm, const void* z,
                               void* dH, void* dX, void* dW1t, void* dW2t, float* dg, void* ws, size_t ws_bytes,
                               int64_t M, int64_t K1, int64_t d, int64_t N2, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CODA_H_ */
