// Host-side plumbing shared by the translation units of libcoda: tensor-map
// construction, the launch context, and the internal launchers each .cu file
// provides.  Not part of the public ABI (that is include/coda.h).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace coda {

struct LaunchCtx {
  int num_sms;
  int* status;          // device status word
  uint64_t timeout_ns;  // bound on every in-kernel wait
  cudaStream_t stream;
  int skip_first_stage;  // test hook, see coda_debug_skip_first_stage
  int pair;              // 1: 2-SM GEMM kernel (CTA pairs), 0: 1-SM kernel
  const float* scale_a;  // FP8 operands: device pointers to the per-tensor scales
  const float* scale_b;
  uint32_t f8_fmt;       // FP8 operands: format bits of A and B (f8_format_bits; 0 = both e4m3)
  float scale_host;      // FP8 operands: a further accumulator scale known on the host (1 otherwise)
  float* sk_parts;       // split-tile scratch (coda_set_split_workspace), or null: no tile is split
  int* sk_flags;
  int sk_slots;          // clusters the scratch has slots for
  int wide_lead;         // > 0: long-K launches take 256 x 512 pair tiles with this lead J (coda_set_wide_tiles)
};

// Whether a bf16 GEMM over K with tiles_n 256-column output tiles takes the
// wide-tile pair kernel: the handle asks for it (a lead J > 0), the pair
// kernel is on, the column tiles pair up, and K is long: at least
// kWideMinKb k-blocks of 64 (K >= 16384), and enough that the 2J single-half
// k-blocks of a tile are at most a quarter of its 2 nkb half k-blocks.  Only
// the long-K backward programs are compiled for it.  Each tile boundary
// exposes part of an accumulator half's drain, so short-K GEMMs, with many
// tiles per SM pair, lose more there than the smaller operand traffic gains:
// measured, the 7B / 70B weight gradient (K = 8192 / 4096) ran 1-9 % slower
// on wide tiles and the data gradient (K = 28672 / 57344) 3 % faster.
constexpr int kWideMinKb = 256;
bool wide_tiles_fit(const LaunchCtx& c, int K, int tiles_n);

// 2-D bf16 tensor map with 128-byte swizzle.  The tensor is `outer` rows of
// `inner` contiguous elements with a row pitch of `ld` elements; the box is
// box_inner x box_outer elements (box_inner * 2 bytes must be <= 128).
// Returns false if the driver rejects it.
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                    uint32_t box_inner, uint32_t box_outer);
// Tensor maps for the epilogue's TMA stores: `rows` x `cols` elements with a
// row pitch of `ld` elements, 32 x 32 boxes (bf16: 64-byte swizzle; fp32:
// 128-byte swizzle), matching the staging layout of the GEMM epilogue.
bool make_tmap_store_bf16(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t ld);
bool make_tmap_store_f32(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t ld);
// 1-byte codes (32 x 32 boxes, 32-byte swizzle), matching stage_e5m2x32
bool make_tmap_store_u8_sw32(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t ld);
// The same for 1-byte elements (e4m3 codes): box_inner <= 128.
bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
                  uint32_t box_outer);

// Launch `kern` on c.stream with programmatic stream serialization: its
// prologue may overlap the tail of the previous kernel in the stream.  Every
// library kernel calls griddep_wait() before its first global-memory access,
// so the ordering of memory effects is that of a plain stream launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(const LaunchCtx& c, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Handle accessors (api.cu), for translation units that only see the
// opaque coda_handle_t.
LaunchCtx launch_ctx_of_handle(void* handle, void* stream);
int device_of_handle(void* handle);
// Partial-accumulator slots the split-tile scratch needs on a GPU with
// num_sms SMs (gemm_fwd.cu, beside the split plan it serves).
int split_scratch_slots(int num_sms);
// The handle's slot for the device address of the allocation-free call's
// scratch array (noalloc.cu); null until that call first runs on the handle.
void** noalloc_scratch_slot(void* handle);

// ---- GEMM launchers (gemm_*.cu) --------------------------------------------
// Operand majors: A K-major = [M][K], MN-major = [K][M]; B K-major = [N][K],
// MN-major = [K][N].  All row pitches equal the extents (dense tensors).

// C = bf16(row_scale[m] * col_scale[n] * sum_k A B); scales may be null.
cudaError_t gemm_store(const LaunchCtx& c, const __nv_bfloat16* A, bool a_mn, const __nv_bfloat16* B, bool b_mn,
                       __nv_bfloat16* C, int M, int N, int K, const float* row_scale,
                       const __nv_bfloat16* col_scale);

// C (fp32) = A B  or  C += A B.
cudaError_t gemm_store_f32(const LaunchCtx& c, const __nv_bfloat16* A, bool a_mn, const __nv_bfloat16* B, bool b_mn,
                           float* C, int M, int N, int K, bool accumulate);

// h = bf16(X W1 + R); psum[m, j] = sum of h^2 over column block j; with
// Hg != null also Hg = bf16(h * g).
cudaError_t gemm_res_prms(const LaunchCtx& c, const __nv_bfloat16* X, const __nv_bfloat16* W1t,
                          const __nv_bfloat16* R, __nv_bfloat16* H, float* psum, int M, int K1, int d, int T,
                          const __nv_bfloat16* g = nullptr, __nv_bfloat16* Hg = nullptr);

// z = rstd * (H W2g); out = silu(z_gate) * z_up (swiglu) or z (plain).
// With psum != null the row scale comes from the partial sums of squares
// (1 / sqrt(sum_j psum / d + eps)) instead of rstd, and is also written to
// rstd_out when that is not null.
cudaError_t gemm_rowscale_swiglu(const LaunchCtx& c, const __nv_bfloat16* H, const __nv_bfloat16* W2gt,
                                 const float* rstd, __nv_bfloat16* out, __nv_bfloat16* zsave, int M, int d, int N2,
                                 bool swiglu, const float* psum = nullptr, int T = 0, float eps = 0.f,
                                 float* rstd_out = nullptr);

// acc = dP W2^T; dH = g*acc - c*h; dgpart[4*tm+q, n] = sum_rows acc*h.
// With cpart != null, c comes from the SwiGLU-backward epilogue's partial
// sums: c[m] = rstd[m]^2 / d * sum_j cpart[m, j] (Tc columns); cvec unused.
cudaError_t gemm_dgrad_rms(const LaunchCtx& c, const __nv_bfloat16* dP, const __nv_bfloat16* W2t,
                           const __nv_bfloat16* H, const __nv_bfloat16* g, const float* cvec, __nv_bfloat16* dH,
                           float* dgpart, int M, int N2, int d, const float* cpart = nullptr, int Tc = 0,
                           const float* rstd = nullptr);

// dY = dYb W3 computed on chip, then the SwiGLU backward in the epilogue:
// dP = bf16(rstd dZ), cpart[m, j] = sum over 256-column tile j of dZ z.
cudaError_t gemm_dgrad_swiglu_bwd(const LaunchCtx& c, const __nv_bfloat16* dYb, const __nv_bfloat16* W3t,
                                  const __nv_bfloat16* z, const float* rstd, __nv_bfloat16* dP, float* cpart, int M,
                                  int d, int F, int T);

// per (row, vocab tile) max / sum-exp / argmax, label logit.
cudaError_t gemm_ce_stats(const LaunchCtx& c, const __nv_bfloat16* H, const __nv_bfloat16* Wt, const int32_t* labels,
                          float* pmax, float* psum, int32_t* parg, float* zy, int M, int d, int V, int T);

// dL chunk = (softmax - onehot) / M for vocabulary rows [v0, v0 + Vc).
cudaError_t gemm_ce_grad(const LaunchCtx& c, const __nv_bfloat16* H, const __nv_bfloat16* Wt_chunk,
                         const int32_t* labels, const float* lse, __nv_bfloat16* dL, int M, int d, int Vc, int v0,
                         float inv_M);

// qkv = X Wqkv with RoPE (head_dim 128) on the first rot_cols columns.
cudaError_t gemm_qkv_rope(const LaunchCtx& c, const __nv_bfloat16* X, const __nv_bfloat16* Wqkv_t,
                          const float* cos_t, const float* sin_t, __nv_bfloat16* qkv, int M, int d, int N,
                          int rot_cols, int S);

// FP8 (e4m3, per-tensor scales sa / sb) forms of the forward GEMMs; operands
// K-major: A [M][K] codes, B [N][K] codes.
cudaError_t gemm_res_prms_fp8(const LaunchCtx& c, const uint8_t* Xq, const float* sX, const uint8_t* W1q,
                              const float* sW1, const __nv_bfloat16* R, __nv_bfloat16* H, float* psum, int M, int K1,
                              int d, int T);
cudaError_t gemm_rowscale_swiglu_fp8(const LaunchCtx& c, const uint8_t* Hq, const float* sH, const uint8_t* W2q,
                                     const float* sW2, const float* rstd, __nv_bfloat16* out, __nv_bfloat16* zsave,
                                     int M, int d, int N2, bool swiglu);

// Independent GEMM pairs in one launch (SM-pair kernel; two launches of the
// 1-SM kernel when pairing is off):
//   dX = dH W1t (W1t [d][K1]) and dW1t = dH^T X (any such pair: A [M][d]
//   K-major with B [d][K1], and A^T with X [M][K1]);
cudaError_t gemm_group_store(const LaunchCtx& c, const __nv_bfloat16* dH, const __nv_bfloat16* W1t,
                             const __nv_bfloat16* X, __nv_bfloat16* dX, __nv_bfloat16* dW1t, int M, int K1, int d);
//   LM-head chunk: dH32 (+)= dL Wc (Wc [Vc][d]) in fp32 and dWc = dL^T H.
cudaError_t gemm_group_ce_bwd(const LaunchCtx& c, const __nv_bfloat16* dL, const __nv_bfloat16* Wc,
                              const __nv_bfloat16* H, float* dH32, bool accumulate, __nv_bfloat16* dWc, int M, int d,
                              int Vc);
//   the same first-layer pair on 8-bit codes: dX = sdH sW1 dHq W1q and
//   dW1t = sdH sX dHq^T Xq (dH format dh_fmt; W1 and X in w_fmt); two
//   launches when pairing is off.
cudaError_t gemm_group_store_fp8(const LaunchCtx& c, const uint8_t* dHq, int dh_fmt, const float* sdH,
                                 const uint8_t* W1q, const float* sW1, const uint8_t* Xq, const float* sX, int w_fmt,
                                 __nv_bfloat16* dX, __nv_bfloat16* dW1t, int M, int K1, int d);
// Host check of the grouped tile schedule (0 = every tile visited once).
int group_schedule_violations(int P, int heavy, int nH, int nL, int q);
// Tensor map of an 8-bit operand: K-major [rows][K] (boxes of 128 K x
// box_rows) or MN-major [K][mn] (boxes of 128 x 128).
bool make_f8_operand_map(CUtensorMap* m, const uint8_t* p, bool mn_major, int mn, int K, int box_rows);

// C = bf16(row_scale * col_scale * sA * sB * A B) on 8-bit operands: A
// [M][K] (K-major) or [K][M] (MN-major), B [N][K] or [K][N]; formats 0 =
// e4m3, 1 = e5m2; sA / sB device pointers to the scales (null = 1).
cudaError_t gemm_store_fp8(const LaunchCtx& c, const uint8_t* A, bool a_mn, int a_fmt, const float* sA,
                           const uint8_t* B, bool b_mn, int b_fmt, const float* sB, __nv_bfloat16* C, int M, int N,
                           int K, const float* row_scale, const __nv_bfloat16* col_scale);

// dgrad2 with the RMSNorm-backward epilogue (as gemm_dgrad_rms) on 8-bit
// operands: dP codes [M][N2] (format dp_fmt, scale sdP), W2t codes [N2][d]
// (format w_fmt, scale sW2).
cudaError_t gemm_dgrad_rms_fp8(const LaunchCtx& c, const uint8_t* dPq, int dp_fmt, const float* sdP,
                               const uint8_t* W2q, int w_fmt, const float* sW2, const __nv_bfloat16* H,
                               const __nv_bfloat16* g, const float* cvec, __nv_bfloat16* dH, float* dgpart, int M,
                               int N2, int d);

// LM-head GEMMs on 8-bit operands: the statistics GEMM on e4m3 H and W
// codes; the chunk's recomputed logits writing dL as e5m2 codes of
// dL * code_inv; the chunk's dH (+)= and dW GEMMs on those codes (scale s_dL)
cudaError_t gemm_ce_stats_fp8(const LaunchCtx& c, const uint8_t* Hq, const float* sH, const uint8_t* Wq,
                              const float* sW, const int32_t* labels, float* pmax, float* psum, int32_t* parg,
                              float* zy, int M, int d, int V, int T);
cudaError_t gemm_ce_grad_fp8(const LaunchCtx& c, const uint8_t* Hq, const float* sH, const uint8_t* Wq_chunk,
                             const float* sW, const int32_t* labels, const float* lse, uint8_t* dLq, float code_inv,
                             int M, int d, int Vc, int v0, float inv_M);
cudaError_t gemm_ce_bwd_fp8(const LaunchCtx& c, const uint8_t* dLq, float s_dL, const uint8_t* Wq_chunk,
                            const float* sW, const uint8_t* Hq, const float* sH, float* dH32, bool accumulate,
                            __nv_bfloat16* dWc, int M, int d, int Vc);
// the same two GEMMs in one grouped SM-pair launch (the two launches above
// on single SMs)
cudaError_t gemm_group_ce_bwd_fp8(const LaunchCtx& c, const uint8_t* dLq, float s_dL, const uint8_t* Wq_chunk,
                                  const float* sW, const uint8_t* Hq, const float* sH, float* dH32, bool accumulate,
                                  __nv_bfloat16* dWc, int M, int d, int Vc);

int ce_tile_cols();    // vocabulary columns per CE statistics tile
int prms_tile_cols();  // columns per partial-RMS tile of GEMM1

// ---- memory-bound kernels (mem_kernels.cu) ---------------------------------
cudaError_t launch_fold(const LaunchCtx& c, const __nv_bfloat16* W2t, const __nv_bfloat16* g, __nv_bfloat16* W2gt,
                        int64_t N2, int64_t d);
cudaError_t launch_rstd_combine(const LaunchCtx& c, const float* psum, int64_t M, int64_t T, int64_t d, float eps,
                                float* rstd);
cudaError_t launch_swiglu_bwd(const LaunchCtx& c, const __nv_bfloat16* dY, const __nv_bfloat16* z,
                              const float* rstd, __nv_bfloat16* dP, float* cvec, int64_t M, int64_t F, int64_t d);
cudaError_t launch_col_combine(const LaunchCtx& c, const float* part, int64_t rows, int64_t d, float* out);
cudaError_t launch_ce_combine(const LaunchCtx& c, const float* pmax, const float* psum, const int32_t* parg,
                              const float* zy, const int32_t* labels, int64_t M, int64_t T, int64_t V, float* lse,
                              int32_t* argmax, float* row_loss);
cudaError_t launch_mean(const LaunchCtx& c, const float* v, int64_t n, float* out);
cudaError_t launch_f32_to_bf16(const LaunchCtx& c, const float* in, __nv_bfloat16* out, int64_t n);
// cos / sin tables [S, head_dim/2] of the rotary embedding, computed in fp64
cudaError_t launch_rope_table(const LaunchCtx& c, float* cos_t, float* sin_t, int64_t S, int64_t head_dim, double base);
// RoPE in place on the first rot_cols columns of qkv [M, N] (standalone, unfused)
cudaError_t launch_rope_apply(const LaunchCtx& c, __nv_bfloat16* qkv, const float* cos_t, const float* sin_t,
                              int64_t M, int64_t N, int64_t rot_cols, int64_t head_dim, int64_t S);
// per-tensor fp8 quantisation: ws[0] = amax of src (times g[col] if g),
// ws[1] = scale = the smallest power of two with amax / scale <= fmax (1 if
// amax == 0); dst = fp8(src * g / scale), e4m3 (fmax 448) or, with
// e5m2 != 0, e5m2 (fmax 57344)
cudaError_t launch_fp8_quantize(const LaunchCtx& c, const __nv_bfloat16* src, int64_t rows, int64_t cols,
                                const __nv_bfloat16* g, float* ws, uint8_t* dst, int e5m2 = 0);
// the SwiGLU backward straight to fp8 codes of bf16(dP) (two passes over dY
// and z; ws as launch_fp8_quantize)
cudaError_t launch_swiglu_bwd_fp8(const LaunchCtx& c, const __nv_bfloat16* dY, const __nv_bfloat16* z,
                                  const float* rstd, float* ws, uint8_t* dPq, float* cvec, int64_t M, int64_t F,
                                  int64_t d, int e5m2);
// the same with delayed scaling: state = {amax, scale}; on entry state[0] is
// the previous dP's amax, on exit {this dP's amax, the scale used} (one pass)
cudaError_t launch_swiglu_bwd_fp8_delayed(const LaunchCtx& c, const __nv_bfloat16* dY, const __nv_bfloat16* z,
                                          const float* rstd, float* state, uint8_t* dPq, float* cvec, int64_t M,
                                          int64_t F, int64_t d, int e5m2);
// unfused ablation kernels
cudaError_t launch_add_rmsnorm(const LaunchCtx& c, const __nv_bfloat16* A, const __nv_bfloat16* R,
                               const __nv_bfloat16* g, __nv_bfloat16* H, float* rstd, __nv_bfloat16* Nrm, int64_t M,
                               int64_t d, float eps);
cudaError_t launch_swiglu(const LaunchCtx& c, const __nv_bfloat16* z, __nv_bfloat16* out, int64_t M, int64_t F);
cudaError_t launch_swiglu_bwd_plain(const LaunchCtx& c, const __nv_bfloat16* dY, const __nv_bfloat16* z,
                                    __nv_bfloat16* dZ, int64_t M, int64_t F);
cudaError_t launch_rmsnorm_bwd(const LaunchCtx& c, const __nv_bfloat16* dN, const __nv_bfloat16* H,
                               const float* rstd, const __nv_bfloat16* g, __nv_bfloat16* dH, int64_t M, int64_t d);
cudaError_t launch_rmsnorm_bwd_dg(const LaunchCtx& c, const __nv_bfloat16* dN, const __nv_bfloat16* H,
                                  const float* rstd, float* dgpart, int64_t M, int64_t d, int64_t rows_per_part);

}  // namespace coda
