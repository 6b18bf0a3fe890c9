// C ABI of libcoda (declared in include/coda.h): argument validation,
// workspace carving, and the launch sequences of the forward, backward,
// LM-head and unfused-ablation paths.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/coda.h"
#include "../../include/coda_testing.h"
#include "coda_internal.h"
#include "ptx.cuh"

struct coda_handle_s {
  int device;
  int num_sms;
  int* status;  // device status word
  uint64_t timeout_ns;
  int skip_first_stage;  // test hook for the bounded waits (coda_debug_skip_first_stage)
  int pair;              // GEMMs on SM pairs (coda_set_sm_pairing)
  void* noalloc_scratch;  // device address of the allocation-free call's scratch, looked up on its first use
  float* sk_parts;        // split-tile scratch (coda_set_split_workspace), or null
  int* sk_flags;
  int wide_lead;          // wide pair tiles for long-K GEMMs (coda_set_wide_tiles): lead J, 0 = off
  int64_t ce_chunk;       // vocabulary columns per LM-head backward chunk (coda_set_lmhead_chunk)
};

namespace coda {

namespace {

constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;
constexpr int64_t kMaxExtent = (int64_t(1) << 31) - 1;
// vocabulary columns per LM-head backward chunk: the default, and the widest
// chunk the workspace's dL buffer (M x this many) holds.  A quarter of a
// 128256-token vocabulary: wider chunks mean fewer launch ramps and partial
// waves (32768 ran 2.0 % faster than 16384 in bf16 and 2.8 % in FP8 at
// M = 8192, d = 2048), while the dL buffer stays a fraction of [M, V].
constexpr int64_t kCeChunk = 32768;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void resolve_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

LaunchCtx ctx_of(coda_handle_t h, void* stream) {
  LaunchCtx c;
  c.num_sms = h->num_sms;
  c.status = h->status;
  c.timeout_ns = h->timeout_ns;
  c.stream = static_cast<cudaStream_t>(stream);
  c.skip_first_stage = h->skip_first_stage;
  c.pair = h->pair;
  c.scale_a = nullptr;
  c.scale_b = nullptr;
  c.f8_fmt = 0;
  c.scale_host = 1.f;
  c.sk_parts = h->sk_parts;
  c.sk_flags = h->sk_flags;
  c.sk_slots = split_scratch_slots(h->num_sms);
  c.wide_lead = h->wide_lead;
  return c;
}

// Split-tile scratch: slots for the partials of the earlier k-ranges of a
// launch's split tiles (at most pairs - 1 split tiles, kSplitMaxRanges - 1
// partials each), a 256 x 256 fp32 accumulator per slot, then one flag per
// (slot, CTA of the pair, epilogue warp).
int split_slots(int num_sms) { return split_scratch_slots(num_sms); }
size_t split_parts_bytes(int num_sms) { return size_t(split_slots(num_sms)) * 256 * 256 * sizeof(float); }
size_t split_flags_bytes(int num_sms) { return size_t(split_slots(num_sms)) * 2 * 8 * sizeof(int); }

coda_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return CODA_OK;
  if (e == cudaErrorNotSupported) return CODA_ERR_UNSUPPORTED;
  return CODA_ERR_CUDA;
}

// argument checks ------------------------------------------------------------
struct Check {
  coda_status_t st = CODA_OK;
  Check& ptr(const void* p) {
    if (st != CODA_OK) return *this;
    if (p == nullptr)
      st = CODA_ERR_INVALID_ARG;
    else if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
      st = CODA_ERR_ALIGNMENT;
    return *this;
  }
  Check& opt_ptr(const void* p) { return p == nullptr ? *this : ptr(p); }
  Check& opt_sptr(const void* p) { return p == nullptr ? *this : sptr(p); }
  // a pointer to fp32 scalars: natural (4-byte) alignment
  Check& sptr(const void* p) {
    if (st != CODA_OK) return *this;
    if (p == nullptr)
      st = CODA_ERR_INVALID_ARG;
    else if (reinterpret_cast<uintptr_t>(p) % 4 != 0)
      st = CODA_ERR_ALIGNMENT;
    return *this;
  }
  // a tensor with a token-count (M) extent: may be empty (NULL) when M == 0
  Check& mptr(const void* p, int64_t M) { return M == 0 ? opt_ptr(p) : ptr(p); }
  // the token count M: 0 <= M < 2^31
  Check& rows(int64_t v) {
    if (st == CODA_OK && (v < 0 || v > kMaxExtent)) st = CODA_ERR_INVALID_ARG;
    return *this;
  }
  // a contiguous extent: positive multiple of 8
  Check& cols(int64_t v) {
    if (st != CODA_OK) return *this;
    if (v <= 0 || v > kMaxExtent)
      st = CODA_ERR_INVALID_ARG;
    else if (v % 8 != 0)
      st = CODA_ERR_ALIGNMENT;
    return *this;
  }
  Check& handle(coda_handle_t h) {
    if (st == CODA_OK && h == nullptr) st = CODA_ERR_INVALID_ARG;
    return *this;
  }
};

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                    uint32_t box_inner, uint32_t box_outer) {
  std::call_once(g_encode_once, resolve_encode);
  if (g_encode == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {
bool make_tmap_store(CUtensorMap* m, CUtensorMapDataType type, uint32_t esize, CUtensorMapSwizzle swz,
                     const void* base, uint64_t cols, uint64_t rows, uint64_t ld) {
  std::call_once(g_encode_once, resolve_encode);
  if (g_encode == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld * esize};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, type, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
}  // namespace

bool make_tmap_store_bf16(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t ld) {
  return make_tmap_store(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_64B, base, cols, rows, ld);
}

bool make_tmap_store_u8_sw32(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t ld) {
  return make_tmap_store(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, CU_TENSOR_MAP_SWIZZLE_32B, base, cols, rows, ld);
}

bool make_tmap_store_f32(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t ld) {
  return make_tmap_store(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, CU_TENSOR_MAP_SWIZZLE_128B, base, cols, rows, ld);
}

LaunchCtx launch_ctx_of_handle(void* handle, void* stream) {
  return ctx_of(static_cast<coda_handle_t>(handle), stream);
}

int device_of_handle(void* handle) { return static_cast<coda_handle_t>(handle)->device; }

void** noalloc_scratch_slot(void* handle) { return &static_cast<coda_handle_t>(handle)->noalloc_scratch; }

bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
                  uint32_t box_outer) {
  std::call_once(g_encode_once, resolve_encode);
  if (g_encode == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace coda

using namespace coda;
using bf16 = __nv_bfloat16;

#define CODA_TRY(expr)                        \
  do {                                        \
    const coda_status_t s_ = (expr);          \
    if (s_ != CODA_OK) return s_;             \
  } while (0)

#define CODA_CUDA(expr) CODA_TRY(from_cuda(expr))

extern "C" {

// ---------------------------------------------------------------------------
coda_status_t coda_create(coda_handle_t* out, int device) {
  if (out == nullptr) return CODA_ERR_INVALID_ARG;
  *out = nullptr;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return CODA_ERR_INVALID_ARG;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return CODA_ERR_CUDA;
  if (cudaSetDevice(device) != cudaSuccess) return CODA_ERR_CUDA;
  coda_handle_s* h = new coda_handle_s;
  h->device = device;
  h->timeout_ns = kDefaultTimeoutNs;
  h->skip_first_stage = 0;
  h->pair = 1;
  h->status = nullptr;
  h->noalloc_scratch = nullptr;
  h->sk_parts = nullptr;
  h->sk_flags = nullptr;
  h->wide_lead = 0;
  h->ce_chunk = kCeChunk;
  coda_status_t st = CODA_OK;
  if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaMalloc(&h->status, sizeof(int)) != cudaSuccess || cudaMemset(h->status, 0, sizeof(int)) != cudaSuccess)
    st = CODA_ERR_CUDA;
  cudaSetDevice(prev);
  if (st != CODA_OK) {
    if (h->status) cudaFree(h->status);
    delete h;
    return st;
  }
  *out = h;
  return CODA_OK;
}

coda_status_t coda_destroy(coda_handle_t h) {
  if (h == nullptr) return CODA_OK;
  cudaFree(h->status);
  delete h;
  return CODA_OK;
}

const char* coda_status_string(coda_status_t s) {
  switch (s) {
    case CODA_OK: return "ok";
    case CODA_ERR_INVALID_ARG: return "invalid argument (null pointer or extent out of range)";
    case CODA_ERR_ALIGNMENT: return "misaligned pointer (16 B) or extent not a multiple of 8";
    case CODA_ERR_UNSUPPORTED: return "unsupported shape or flag combination";
    case CODA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case CODA_ERR_CUDA: return "CUDA runtime or driver error";
    case CODA_ERR_TIMEOUT: return "an in-kernel wait hit its time limit";
    case CODA_ERR_LABEL_RANGE: return "a label was outside [0, V)";
  }
  return "unknown status";
}

coda_status_t coda_sync_status(coda_handle_t h, void* stream, int32_t* device_bits) {
  CODA_TRY(Check().handle(h).st);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int bits = 0;
  CODA_CUDA(cudaStreamSynchronize(s));
  CODA_CUDA(cudaMemcpyAsync(&bits, h->status, sizeof(int), cudaMemcpyDeviceToHost, s));
  CODA_CUDA(cudaMemsetAsync(h->status, 0, sizeof(int), s));
  CODA_CUDA(cudaStreamSynchronize(s));
  if (device_bits) *device_bits = bits;
  if (bits & (DEV_ERR_TIMEOUT_PRODUCER | DEV_ERR_TIMEOUT_MMA | DEV_ERR_TIMEOUT_EPILOGUE | DEV_ERR_TIMEOUT_DRAIN))
    return CODA_ERR_TIMEOUT;
  if (bits & DEV_ERR_LABEL_RANGE) return CODA_ERR_LABEL_RANGE;
  return CODA_OK;
}

coda_status_t coda_set_wait_timeout_ns(coda_handle_t h, uint64_t ns) {
  CODA_TRY(Check().handle(h).st);
  h->timeout_ns = ns == 0 ? kDefaultTimeoutNs : ns;
  return CODA_OK;
}

coda_status_t coda_set_sm_pairing(coda_handle_t h, int enable) {
  CODA_TRY(Check().handle(h).st);
  h->pair = enable != 0;
  return CODA_OK;
}

coda_status_t coda_set_wide_tiles(coda_handle_t h, int lead_kblocks) {
  CODA_TRY(Check().handle(h).st);
  if (lead_kblocks < 0 || lead_kblocks > 64) return CODA_ERR_INVALID_ARG;
  h->wide_lead = lead_kblocks;
  return CODA_OK;
}

coda_status_t coda_set_lmhead_chunk(coda_handle_t h, int64_t cols) {
  CODA_TRY(Check().handle(h).st);
  if (cols == 0) cols = kCeChunk;
  if (cols < 256 || cols > kCeChunk || cols % 256 != 0) return CODA_ERR_INVALID_ARG;
  h->ce_chunk = cols;
  return CODA_OK;
}

int coda_debug_wide_applies(coda_handle_t h, int M, int N, int K) {
  if (h == nullptr || M < 1 || N < 1 || K < 1) return -1;
  return wide_tiles_fit(ctx_of(h, nullptr), K, (N + 255) / 256) ? 1 : 0;
}

size_t coda_split_workspace_bytes(coda_handle_t h) {
  if (h == nullptr) return 0;
  return split_parts_bytes(h->num_sms) + split_flags_bytes(h->num_sms);
}

coda_status_t coda_set_split_workspace(coda_handle_t h, void* ws, size_t ws_bytes, void* stream) {
  if (h == nullptr) return CODA_ERR_INVALID_ARG;
  if (ws == nullptr) {
    h->sk_parts = nullptr;
    h->sk_flags = nullptr;
    return CODA_OK;
  }
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return CODA_ERR_ALIGNMENT;
  if (ws_bytes < coda_split_workspace_bytes(h)) return CODA_ERR_WORKSPACE_TOO_SMALL;
  float* parts = static_cast<float*>(ws);
  int* flags = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + split_parts_bytes(h->num_sms));
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return CODA_ERR_CUDA;
  if (prev != h->device && cudaSetDevice(h->device) != cudaSuccess) return CODA_ERR_CUDA;
  const cudaError_t e =
      cudaMemsetAsync(flags, 0, split_flags_bytes(h->num_sms), static_cast<cudaStream_t>(stream));
  if (prev != h->device) cudaSetDevice(prev);
  if (e != cudaSuccess) return CODA_ERR_CUDA;
  h->sk_parts = parts;
  h->sk_flags = flags;
  return CODA_OK;
}

coda_status_t coda_debug_skip_first_stage(coda_handle_t h, int enable) {
  CODA_TRY(Check().handle(h).st);
  h->skip_first_stage = enable == 2 ? 2 : (enable != 0 ? 1 : 0);
  return CODA_OK;
}

int64_t coda_prms_num_tiles(int64_t d) { return d <= 0 ? 0 : cdiv(d, prms_tile_cols()); }

int64_t coda_dgpart_rows(int64_t M) { return M <= 0 ? 0 : 4 * cdiv(M, 128); }

// ---------------------------------------------------------------------------
coda_status_t coda_gemm(coda_handle_t h, const void* A, int a_mn_major, const void* B, int b_mn_major, void* C,
                        int64_t M, int64_t N, int64_t K, const float* row_scale, const void* col_scale,
                        void* stream) {
  CODA_TRY(Check().handle(h).rows(M).mptr(A, M).ptr(B).mptr(C, M).opt_ptr(row_scale).opt_ptr(col_scale).cols(N).cols(K).st);
  if (a_mn_major && !b_mn_major) return CODA_ERR_UNSUPPORTED;
  if (a_mn_major && M % 8 != 0) return CODA_ERR_ALIGNMENT;
  if (M == 0) return CODA_OK;
  return from_cuda(gemm_store(ctx_of(h, stream), static_cast<const bf16*>(A), a_mn_major != 0,
                              static_cast<const bf16*>(B), b_mn_major != 0, static_cast<bf16*>(C), int(M), int(N),
                              int(K), row_scale, static_cast<const bf16*>(col_scale)));
}

coda_status_t coda_fold_rmsnorm_weight(coda_handle_t h, const void* W2t, const void* g, void* W2gt, int64_t N2,
                                       int64_t d, void* stream) {
  CODA_TRY(Check().handle(h).ptr(W2t).ptr(g).ptr(W2gt).cols(N2).cols(d).st);
  if (W2t == W2gt) return CODA_ERR_INVALID_ARG;
  return from_cuda(launch_fold(ctx_of(h, stream), static_cast<const bf16*>(W2t), static_cast<const bf16*>(g),
                               static_cast<bf16*>(W2gt), N2, d));
}

coda_status_t coda_gemm_res_prms(coda_handle_t h, const void* X, const void* W1t, const void* R, void* H,
                                 float* psum, int64_t M, int64_t K1, int64_t d, void* stream) {
  CODA_TRY(Check().handle(h).rows(M).mptr(X, M).ptr(W1t).mptr(R, M).mptr(H, M).mptr(psum, M).cols(K1).cols(d).st);
  if (M == 0) return CODA_OK;
  if (R == H) return CODA_ERR_INVALID_ARG;
  return from_cuda(gemm_res_prms(ctx_of(h, stream), static_cast<const bf16*>(X), static_cast<const bf16*>(W1t),
                                 static_cast<const bf16*>(R), static_cast<bf16*>(H), psum, int(M), int(K1), int(d),
                                 int(coda_prms_num_tiles(d))));
}

coda_status_t coda_gemm_res_prms_g(coda_handle_t h, const void* X, const void* W1t, const void* R, const void* g,
                                   void* H, void* Hg, float* psum, int64_t M, int64_t K1, int64_t d, void* stream) {
  CODA_TRY(Check()
               .handle(h)
               .rows(M)
               .mptr(X, M)
               .ptr(W1t)
               .mptr(R, M)
               .ptr(g)
               .mptr(H, M)
               .mptr(Hg, M)
               .mptr(psum, M)
               .cols(K1)
               .cols(d)
               .st);
  if (M == 0) return CODA_OK;
  if (R == H || R == Hg || H == Hg) return CODA_ERR_INVALID_ARG;
  return from_cuda(gemm_res_prms(ctx_of(h, stream), static_cast<const bf16*>(X), static_cast<const bf16*>(W1t),
                                 static_cast<const bf16*>(R), static_cast<bf16*>(H), psum, int(M), int(K1), int(d),
                                 int(coda_prms_num_tiles(d)), static_cast<const bf16*>(g), static_cast<bf16*>(Hg)));
}

coda_status_t coda_rstd_combine(coda_handle_t h, const float* psum, int64_t M, int64_t T, int64_t d, float eps,
                                float* rstd, void* stream) {
  CODA_TRY(Check().handle(h).rows(M).mptr(psum, M).mptr(rstd, M).st);
  if (T <= 0 || d <= 0 || !(eps >= 0.f)) return CODA_ERR_INVALID_ARG;
  if (M == 0) return CODA_OK;
  return from_cuda(launch_rstd_combine(ctx_of(h, stream), psum, M, T, d, eps, rstd));
}

coda_status_t coda_gemm_rowscale_swiglu(coda_handle_t h, const void* H, const void* W2gt, const float* rstd,
                                        void* out, void* z_save, int64_t M, int64_t d, int64_t N2, uint32_t flags,
                                        void* stream) {
  CODA_TRY(Check().handle(h).rows(M).mptr(H, M).ptr(W2gt).mptr(rstd, M).mptr(out, M).opt_ptr(z_save).cols(d).cols(N2).st);
  if (flags != CODA_EPI_SWIGLU && flags != CODA_EPI_PLAIN) return CODA_ERR_UNSUPPORTED;
  const bool swiglu = flags == CODA_EPI_SWIGLU;
  if (swiglu && (N2 / 2) % 8 != 0) return CODA_ERR_ALIGNMENT;
  if (!swiglu && z_save != nullptr) return CODA_ERR_INVALID_ARG;
  if (M == 0) return CODA_OK;
  return from_cuda(gemm_rowscale_swiglu(ctx_of(h, stream), static_cast<const bf16*>(H),
                                        static_cast<const bf16*>(W2gt), rstd, static_cast<bf16*>(out),
                                        static_cast<bf16*>(z_save), int(M), int(d), int(N2), swiglu));
}

coda_status_t coda_gemm_prms_rowscale_swiglu(coda_handle_t h, const void* H, const void* W2gt, const float* psum,
                                             int64_t T, float eps, float* rstd, void* out, void* z_save, int64_t M,
                                             int64_t d, int64_t N2, uint32_t flags, void* stream) {
  CODA_TRY(Check()
               .handle(h)
               .rows(M)
               .mptr(H, M)
               .ptr(W2gt)
               .mptr(psum, M)
               .opt_ptr(rstd)
               .mptr(out, M)
               .opt_ptr(z_save)
               .cols(d)
               .cols(N2)
               .st);
  if (flags != CODA_EPI_SWIGLU && flags != CODA_EPI_PLAIN) return CODA_ERR_UNSUPPORTED;
  const bool swiglu = flags == CODA_EPI_SWIGLU;
  if (swiglu && (N2 / 2) % 8 != 0) return CODA_ERR_ALIGNMENT;
  if (!swiglu && z_save != nullptr) return CODA_ERR_INVALID_ARG;
  if (T <= 0 || T > kMaxExtent || !(eps >= 0.f)) return CODA_ERR_INVALID_ARG;
  if (M == 0) return CODA_OK;
  return from_cuda(gemm_rowscale_swiglu(ctx_of(h, stream), static_cast<const bf16*>(H),
                                        static_cast<const bf16*>(W2gt), nullptr, static_cast<bf16*>(out),
                                        static_cast<bf16*>(z_save), int(M), int(d), int(N2), swiglu, psum, int(T), eps,
                                        rstd));
}

// ---------------------------------------------------------------------------
coda_status_t coda_swiglu_bwd(coda_handle_t h, const void* dY, const void* z, const float* rstd, void* dP,
                              float* c, int64_t M, int64_t F, int64_t d, void* stream) {
  CODA_TRY(Check().handle(h).rows(M).mptr(dY, M).mptr(z, M).mptr(rstd, M).mptr(dP, M).mptr(c, M).cols(F).cols(d).st);
  if (M == 0) return CODA_OK;
  return from_cuda(launch_swiglu_bwd(ctx_of(h, stream), static_cast<const bf16*>(dY), static_cast<const bf16*>(z),
                                     rstd, static_cast<bf16*>(dP), c, M, F, d));
}

coda_status_t coda_gemm_dgrad_rmsbwd(coda_handle_t h, const void* dP, const void* W2t, const void* H,
                                     const void* g, const float* c, void* dH, float* dgpart, int64_t M, int64_t N2,
                                     int64_t d, void* stream) {
  CODA_TRY(Check().handle(h).rows(M).mptr(dP, M).ptr(W2t).mptr(H, M).ptr(g).mptr(c, M).mptr(dH, M).mptr(dgpart, M).cols(N2).cols(d).st);
  if (M == 0) return CODA_OK;
  return from_cuda(gemm_dgrad_rms(ctx_of(h, stream), static_cast<const bf16*>(dP), static_cast<const bf16*>(W2t),
                                  static_cast<const bf16*>(H), static_cast<const bf16*>(g), c, static_cast<bf16*>(dH),
                                  dgpart, int(M), int(N2), int(d)));
}

coda_status_t coda_gemm_dgrad_swiglu_bwd(coda_handle_t h, const void* dYb, const void* W3t, const void* z,
                                         const float* rstd, void* dP, float* cpart, int64_t M, int64_t d, int64_t F,
                                         void* stream) {
  CODA_TRY(Check()
               .handle(h)
               .rows(M)
               .mptr(dYb, M)
               .ptr(W3t)
               .mptr(z, M)
               .mptr(rstd, M)
               .mptr(dP, M)
               .mptr(cpart, M)
               .cols(d)
               .cols(F)
               .st);
  if (M == 0) return CODA_OK;
  return from_cuda(gemm_dgrad_swiglu_bwd(ctx_of(h, stream), static_cast<const bf16*>(dYb),
                                         static_cast<const bf16*>(W3t), static_cast<const bf16*>(z), rstd,
                                         static_cast<bf16*>(dP), cpart, int(M), int(d), int(F),
                                         int(coda_prms_num_tiles(F))));
}

coda_status_t coda_gemm_dgrad_rmsbwd_cpart(coda_handle_t h, const void* dP, const void* W2t, const void* H,
                                           const void* g, const float* rstd, const float* cpart, int64_t Tc,
                                           void* dH, float* dgpart, int64_t M, int64_t N2, int64_t d, void* stream) {
  CODA_TRY(Check()
               .handle(h)
               .rows(M)
               .mptr(dP, M)
               .ptr(W2t)
               .mptr(H, M)
               .ptr(g)
               .mptr(rstd, M)
               .mptr(cpart, M)
               .mptr(dH, M)
               .mptr(dgpart, M)
               .cols(N2)
               .cols(d)
               .st);
  if (Tc <= 0 || Tc > kMaxExtent) return CODA_ERR_INVALID_ARG;
  if (M == 0) return CODA_OK;
  return from_cuda(gemm_dgrad_rms(ctx_of(h, stream), static_cast<const bf16*>(dP), static_cast<const bf16*>(W2t),
                                  static_cast<const bf16*>(H), static_cast<const bf16*>(g), nullptr,
                                  static_cast<bf16*>(dH), dgpart, int(M), int(N2), int(d), cpart, int(Tc), rstd));
}

coda_status_t coda_dg_combine(coda_handle_t h, const float* dgpart, int64_t rows, int64_t d, float* dg,
                              void* stream) {
  CODA_TRY(Check().handle(h).rows(rows).mptr(dgpart, rows).ptr(dg).st);
  if (d <= 0) return CODA_ERR_INVALID_ARG;
  return from_cuda(launch_col_combine(ctx_of(h, stream), dgpart, rows, d, dg));
}

coda_status_t coda_gemm_wgrad_gscale(coda_handle_t h, const void* H, const void* dP, const void* g, void* dW2t,
                                     int64_t M, int64_t N2, int64_t d, void* stream) {
  CODA_TRY(Check().handle(h).rows(M).mptr(H, M).mptr(dP, M).ptr(g).ptr(dW2t).cols(N2).cols(d).st);
  if (M == 0)  // empty batch: the gradient is zero
    return from_cuda(cudaMemsetAsync(dW2t, 0, size_t(N2) * d * 2, static_cast<cudaStream_t>(stream)));
  // dW2t[n][k] = g[k] sum_m dP[m][n] H[m][k]: GEMM with M' = N2, N' = d,
  // K' = M; A' = dP stored [K'][M'] (MN-major), B' = H stored [K'][N'].
  return from_cuda(gemm_store(ctx_of(h, stream), static_cast<const bf16*>(dP), true, static_cast<const bf16*>(H),
                              true, static_cast<bf16*>(dW2t), int(N2), int(d), int(M), nullptr,
                              static_cast<const bf16*>(g)));
}

size_t coda_bwd_workspace_bytes(int64_t M, int64_t d, int64_t N2) {
  if (M < 0 || d <= 0 || N2 <= 0) return 0;
  return align256(size_t(M) * N2 * 2) + align256(size_t(M) * 4) + align256(size_t(coda_dgpart_rows(M)) * d * 4);
}

int coda_debug_group_schedule_violations(int P, int heavy, int nH, int nL, int q) {
  if (P <= 0 || nH < 0 || nL < 0 || q < 0 || (heavy != 0 && heavy != 1)) return -1;
  return group_schedule_violations(P, heavy, nH, nL, q);
}

coda_status_t coda_gemm_rowscale_swiglu_bwd(coda_handle_t h, const void* dY, const void* z, const float* rstd,
                                            const void* H, const void* W2t, const void* g, void* dH, void* dW2t,
                                            float* dg, void* ws, size_t ws_bytes, int64_t M, int64_t d, int64_t N2,
                                            void* stream) {
  CODA_TRY(Check()
               .handle(h)
               .rows(M)
               .mptr(dY, M)
               .mptr(z, M)
               .mptr(rstd, M)
               .mptr(H, M)
               .ptr(W2t)
               .ptr(g)
               .mptr(dH, M)
               .ptr(dW2t)
               .ptr(dg)
               .opt_ptr(ws)
               .cols(d)
               .cols(N2)
               .st);
  if ((N2 / 2) % 8 != 0) return CODA_ERR_ALIGNMENT;
  if (M == 0) {  // empty batch: zero weight gradients, nothing else to write
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    CODA_CUDA(cudaMemsetAsync(dW2t, 0, size_t(N2) * d * 2, s));
    return from_cuda(cudaMemsetAsync(dg, 0, size_t(d) * 4, s));
  }
  if (ws == nullptr) return CODA_ERR_INVALID_ARG;
  if (ws_bytes < coda_bwd_workspace_bytes(M, d, N2)) return CODA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(ws);
  bf16* dP = reinterpret_cast<bf16*>(w);
  w += align256(size_t(M) * N2 * 2);
  float* c = reinterpret_cast<float*>(w);
  w += align256(size_t(M) * 4);
  float* dgpart = reinterpret_cast<float*>(w);
  const LaunchCtx cx = ctx_of(h, stream);
  CODA_CUDA(launch_swiglu_bwd(cx, static_cast<const bf16*>(dY), static_cast<const bf16*>(z), rstd, dP, c, M, N2 / 2,
                              d));
  // The data and weight gradients stay two launches here: grouped into one
  // (gemm_group.cuh) they measured 4-5 % slower at these sizes.
  CODA_CUDA(gemm_dgrad_rms(cx, dP, static_cast<const bf16*>(W2t), static_cast<const bf16*>(H),
                           static_cast<const bf16*>(g), c, static_cast<bf16*>(dH), dgpart, int(M), int(N2), int(d)));
  CODA_CUDA(launch_col_combine(cx, dgpart, coda_dgpart_rows(M), d, dg));
  CODA_CUDA(gemm_store(cx, dP, true, static_cast<const bf16*>(H), true, static_cast<bf16*>(dW2t), int(N2), int(d),
                       int(M), nullptr, static_cast<const bf16*>(g)));
  return CODA_OK;
}

coda_status_t coda_gemm_res_prms_bwd(coda_handle_t h, const void* dH, const void* X, const void* W1t, void* dX,
                                     void* dW1t, void* dR, int64_t M, int64_t K1, int64_t d, void* stream) {
  CODA_TRY(Check().handle(h).rows(M).mptr(dH, M).mptr(X, M).ptr(W1t).mptr(dX, M).ptr(dW1t).opt_ptr(dR).cols(K1).cols(d).st);
  const LaunchCtx cx = ctx_of(h, stream);
  if (M == 0) return from_cuda(cudaMemsetAsync(dW1t, 0, size_t(d) * K1 * 2, cx.stream));
  // dX[m][i] = sum_k dH[m][k] W1t[k][i] and dW1t[k][i] = sum_m dH[m][k] X[m][i],
  // one grouped launch
  CODA_CUDA(gemm_group_store(cx, static_cast<const bf16*>(dH), static_cast<const bf16*>(W1t),
                             static_cast<const bf16*>(X), static_cast<bf16*>(dX), static_cast<bf16*>(dW1t), int(M),
                             int(K1), int(d)));
  if (dR != nullptr && dR != dH)
    CODA_CUDA(cudaMemcpyAsync(dR, dH, size_t(M) * d * 2, cudaMemcpyDeviceToDevice, cx.stream));
  return CODA_OK;
}

// ---------------------------------------------------------------------------
coda_status_t coda_rope_table(coda_handle_t h, float* cos_t, float* sin_t, int64_t S, int64_t head_dim, float base,
                              void* stream) {
  CODA_TRY(Check().handle(h).ptr(cos_t).ptr(sin_t).st);
  if (S <= 0 || S > kMaxExtent || head_dim <= 0 || !(base > 1.f)) return CODA_ERR_INVALID_ARG;
  if (head_dim % 16 != 0) return CODA_ERR_ALIGNMENT;
  return from_cuda(launch_rope_table(ctx_of(h, stream), cos_t, sin_t, S, head_dim, static_cast<double>(base)));
}

namespace {
coda_status_t check_heads(int64_t n_q, int64_t n_kv, int64_t head_dim, int64_t S) {
  if (n_q <= 0 || n_kv < 0 || head_dim <= 0 || S <= 0 || S > kMaxExtent) return CODA_ERR_INVALID_ARG;
  if ((n_q + 2 * n_kv) * head_dim > kMaxExtent) return CODA_ERR_INVALID_ARG;
  if (head_dim % 16 != 0) return CODA_ERR_ALIGNMENT;
  return CODA_OK;
}
}  // namespace

coda_status_t coda_gemm_qkv_rope(coda_handle_t h, const void* X, const void* Wqkv_t, const float* cos_t,
                                 const float* sin_t, void* qkv, int64_t M, int64_t d, int64_t n_q_heads,
                                 int64_t n_kv_heads, int64_t head_dim, int64_t S, void* stream) {
  CODA_TRY(Check().handle(h).rows(M).mptr(X, M).ptr(Wqkv_t).ptr(cos_t).ptr(sin_t).mptr(qkv, M).cols(d).st);
  CODA_TRY(check_heads(n_q_heads, n_kv_heads, head_dim, S));
  if (head_dim != 128) return CODA_ERR_UNSUPPORTED;
  if (M == 0) return CODA_OK;
  const int64_t N = (n_q_heads + 2 * n_kv_heads) * head_dim;
  return from_cuda(gemm_qkv_rope(ctx_of(h, stream), static_cast<const bf16*>(X), static_cast<const bf16*>(Wqkv_t),
                                 cos_t, sin_t, static_cast<bf16*>(qkv), int(M), int(d), int(N),
                                 int((n_q_heads + n_kv_heads) * head_dim), int(S)));
}

coda_status_t coda_rope_apply(coda_handle_t h, void* qkv, const float* cos_t, const float* sin_t, int64_t M,
                              int64_t n_q_heads, int64_t n_kv_heads, int64_t head_dim, int64_t S, void* stream) {
  CODA_TRY(Check().handle(h).rows(M).mptr(qkv, M).ptr(cos_t).ptr(sin_t).st);
  CODA_TRY(check_heads(n_q_heads, n_kv_heads, head_dim, S));
  if (M == 0) return CODA_OK;
  const int64_t N = (n_q_heads + 2 * n_kv_heads) * head_dim;
  return from_cuda(launch_rope_apply(ctx_of(h, stream), static_cast<bf16*>(qkv), cos_t, sin_t, M, N,
                                     (n_q_heads + n_kv_heads) * head_dim, head_dim, S));
}

// ---------------------------------------------------------------------------
namespace {
coda_status_t fp8_quantize_impl(coda_handle_t h, const void* src, const void* g, float* amax_scale, void* dst,
                                int64_t rows, int64_t cols, void* stream, int e5m2) {
  CODA_TRY(Check().handle(h).rows(rows).mptr(src, rows).opt_ptr(g).sptr(amax_scale).mptr(dst, rows).cols(cols).st);
  if (cols % 16 != 0) return CODA_ERR_ALIGNMENT;
  if (rows == 0) {
    const float init[2] = {0.f, 1.f};
    return from_cuda(cudaMemcpyAsync(amax_scale, init, sizeof(init), cudaMemcpyHostToDevice,
                                     static_cast<cudaStream_t>(stream)));
  }
  return from_cuda(launch_fp8_quantize(ctx_of(h, stream), static_cast<const bf16*>(src), rows, cols,
                                       static_cast<const bf16*>(g), amax_scale, static_cast<uint8_t*>(dst), e5m2));
}
}  // namespace

coda_status_t coda_fp8_quantize(coda_handle_t h, const void* src, const void* g, float* amax_scale, void* dst,
                                int64_t rows, int64_t cols, void* stream) {
  return fp8_quantize_impl(h, src, g, amax_scale, dst, rows, cols, stream, 0);
}

coda_status_t coda_fp8_quantize_e5m2(coda_handle_t h, const void* src, const void* g, float* amax_scale, void* dst,
                                     int64_t rows, int64_t cols, void* stream) {
  return fp8_quantize_impl(h, src, g, amax_scale, dst, rows, cols, stream, 1);
}

coda_status_t coda_swiglu_bwd_fp8(coda_handle_t h, const void* dY, const void* z, const float* rstd, int format,
                                  void* dPq, float* amax_scale, float* c, int64_t M, int64_t F, int64_t d,
                                  void* stream) {
  CODA_TRY(Check()
               .handle(h)
               .rows(M)
               .mptr(dY, M)
               .mptr(z, M)
               .mptr(rstd, M)
               .mptr(dPq, M)
               .sptr(amax_scale)
               .mptr(c, M)
               .cols(F)
               .cols(d)
               .st);
  if (format != 0 && format != 1) return CODA_ERR_INVALID_ARG;
  if (M == 0) {
    const float init[2] = {0.f, 1.f};
    return from_cuda(cudaMemcpyAsync(amax_scale, init, sizeof(init), cudaMemcpyHostToDevice,
                                     static_cast<cudaStream_t>(stream)));
  }
  return from_cuda(launch_swiglu_bwd_fp8(ctx_of(h, stream), static_cast<const bf16*>(dY), static_cast<const bf16*>(z),
                                         rstd, amax_scale, static_cast<uint8_t*>(dPq), c, M, F, d, format));
}

coda_status_t coda_swiglu_bwd_fp8_delayed(coda_handle_t h, const void* dY, const void* z, const float* rstd,
                                          int format, void* dPq, float* amax_scale, float* c, int64_t M, int64_t F,
                                          int64_t d, void* stream) {
  CODA_TRY(Check()
               .handle(h)
               .rows(M)
               .mptr(dY, M)
               .mptr(z, M)
               .mptr(rstd, M)
               .mptr(dPq, M)
               .sptr(amax_scale)
               .mptr(c, M)
               .cols(F)
               .cols(d)
               .st);
  if (format != 0 && format != 1) return CODA_ERR_INVALID_ARG;
  if (M == 0) {
    const float init[2] = {0.f, 1.f};
    return from_cuda(cudaMemcpyAsync(amax_scale, init, sizeof(init), cudaMemcpyHostToDevice,
                                     static_cast<cudaStream_t>(stream)));
  }
  return from_cuda(launch_swiglu_bwd_fp8_delayed(ctx_of(h, stream), static_cast<const bf16*>(dY),
                                                 static_cast<const bf16*>(z), rstd, amax_scale,
                                                 static_cast<uint8_t*>(dPq), c, M, F, d, format));
}

coda_status_t coda_gemm_fp8(coda_handle_t h, const void* A, int a_mn_major, int a_format, const float* sA,
                            const void* B, int b_mn_major, int b_format, const float* sB, void* C, int64_t M,
                            int64_t N, int64_t K, const float* row_scale, const void* col_scale, void* stream) {
  if ((a_format != 0 && a_format != 1) || (b_format != 0 && b_format != 1)) return CODA_ERR_INVALID_ARG;
  if (a_mn_major && !b_mn_major) return CODA_ERR_UNSUPPORTED;
  // With both operands MN-major K is their row count (a token count for the
  // weight gradients): any K >= 0, the ragged last k-block zero-filled by TMA,
  // and K == 0 an empty sum (A and B may then be NULL).  Otherwise K is a
  // contiguous extent of 8-bit codes: a multiple of 16.
  const bool k_rows = a_mn_major && b_mn_major;
  const int64_t n_ops = k_rows && K == 0 ? 0 : M;  // operands present when M > 0 and K > 0
  CODA_TRY(Check()
               .handle(h)
               .rows(M)
               .mptr(A, n_ops)
               .opt_sptr(sA)
               .mptr(B, k_rows ? K : 1)
               .opt_sptr(sB)
               .mptr(C, M)
               .opt_ptr(row_scale)
               .opt_ptr(col_scale)
               .cols(N)
               .st);
  CODA_TRY((k_rows ? Check().rows(K) : Check().cols(K)).st);
  if (!k_rows && K % 16 != 0) return CODA_ERR_ALIGNMENT;
  if (a_mn_major && M % 16 != 0) return CODA_ERR_ALIGNMENT;
  if (b_mn_major && N % 16 != 0) return CODA_ERR_ALIGNMENT;
  if (M == 0) return CODA_OK;
  if (K == 0)
    return from_cuda(cudaMemsetAsync(C, 0, size_t(M) * N * 2, static_cast<cudaStream_t>(stream)));
  return from_cuda(gemm_store_fp8(ctx_of(h, stream), static_cast<const uint8_t*>(A), a_mn_major != 0, a_format, sA,
                                  static_cast<const uint8_t*>(B), b_mn_major != 0, b_format, sB,
                                  static_cast<bf16*>(C), int(M), int(N), int(K), row_scale,
                                  static_cast<const bf16*>(col_scale)));
}

coda_status_t coda_gemm_res_prms_bwd_fp8(coda_handle_t h, const void* dHq, int dh_format, const float* sdH,
                                         const void* Xq, const float* sX, const void* W1q, const float* sW1,
                                         int w_format, void* dX, void* dW1t, int64_t M, int64_t K1, int64_t d,
                                         void* stream) {
  CODA_TRY(Check()
               .handle(h)
               .rows(M)
               .mptr(dHq, M)
               .opt_sptr(sdH)
               .mptr(Xq, M)
               .opt_sptr(sX)
               .ptr(W1q)
               .opt_sptr(sW1)
               .mptr(dX, M)
               .ptr(dW1t)
               .cols(K1)
               .cols(d)
               .st);
  if ((dh_format != 0 && dh_format != 1) || (w_format != 0 && w_format != 1)) return CODA_ERR_INVALID_ARG;
  if (K1 % 16 != 0 || d % 16 != 0) return CODA_ERR_ALIGNMENT;
  const LaunchCtx cx = ctx_of(h, stream);
  // an empty batch: dW1t is an empty sum
  if (M == 0) return from_cuda(cudaMemsetAsync(dW1t, 0, size_t(d) * K1 * 2, cx.stream));
  return from_cuda(gemm_group_store_fp8(cx, static_cast<const uint8_t*>(dHq), dh_format, sdH,
                                        static_cast<const uint8_t*>(W1q), sW1, static_cast<const uint8_t*>(Xq), sX,
                                        w_format, static_cast<bf16*>(dX), static_cast<bf16*>(dW1t), int(M), int(K1),
                                        int(d)));
}

coda_status_t coda_gemm_dgrad_rmsbwd_fp8(coda_handle_t h, const void* dPq, int dp_format, const float* sdP,
                                         const void* W2q, int w_format, const float* sW2, const void* H,
                                         const void* g, const float* c, void* dH, float* dgpart, int64_t M,
                                         int64_t N2, int64_t d, void* stream) {
  CODA_TRY(Check()
               .handle(h)
               .rows(M)
               .mptr(dPq, M)
               .sptr(sdP)
               .ptr(W2q)
               .sptr(sW2)
               .mptr(H, M)
               .ptr(g)
               .mptr(c, M)
               .mptr(dH, M)
               .mptr(dgpart, M)
               .cols(N2)
               .cols(d)
               .st);
  if ((dp_format != 0 && dp_format != 1) || (w_format != 0 && w_format != 1)) return CODA_ERR_INVALID_ARG;
  if (N2 % 16 != 0 || d % 16 != 0) return CODA_ERR_ALIGNMENT;
  if (M == 0) return CODA_OK;
  return from_cuda(gemm_dgrad_rms_fp8(ctx_of(h, stream), static_cast<const uint8_t*>(dPq), dp_format, sdP,
                                      static_cast<const uint8_t*>(W2q), w_format, sW2, static_cast<const bf16*>(H),
                                      static_cast<const bf16*>(g), c, static_cast<bf16*>(dH), dgpart, int(M),
                                      int(N2), int(d)));
}

coda_status_t coda_gemm_res_prms_fp8(coda_handle_t h, const void* Xq, const float* sX, const void* W1q,
                                     const float* sW1, const void* R, void* H, float* psum, int64_t M, int64_t K1,
                                     int64_t d, void* stream) {
  CODA_TRY(Check()
               .handle(h)
               .rows(M)
               .mptr(Xq, M)
               .sptr(sX)
               .ptr(W1q)
               .sptr(sW1)
               .mptr(R, M)
               .mptr(H, M)
               .mptr(psum, M)
               .cols(K1)
               .cols(d)
               .st);
  if (K1 % 16 != 0) return CODA_ERR_ALIGNMENT;
  if (M == 0) return CODA_OK;
  if (R == H) return CODA_ERR_INVALID_ARG;
  return from_cuda(gemm_res_prms_fp8(ctx_of(h, stream), static_cast<const uint8_t*>(Xq), sX,
                                     static_cast<const uint8_t*>(W1q), sW1, static_cast<const bf16*>(R),
                                     static_cast<bf16*>(H), psum, int(M), int(K1), int(d),
                                     int(coda_prms_num_tiles(d))));
}

coda_status_t coda_gemm_rowscale_swiglu_fp8(coda_handle_t h, const void* Hq, const float* sH, const void* W2gq,
                                            const float* sW2, const float* rstd, void* out, void* z_save, int64_t M,
                                            int64_t d, int64_t N2, uint32_t flags, void* stream) {
  CODA_TRY(Check()
               .handle(h)
               .rows(M)
               .mptr(Hq, M)
               .sptr(sH)
               .ptr(W2gq)
               .sptr(sW2)
               .mptr(rstd, M)
               .mptr(out, M)
               .opt_ptr(z_save)
               .cols(d)
               .cols(N2)
               .st);
  if (d % 16 != 0) return CODA_ERR_ALIGNMENT;
  if (flags != CODA_EPI_SWIGLU && flags != CODA_EPI_PLAIN) return CODA_ERR_UNSUPPORTED;
  const bool swiglu = flags == CODA_EPI_SWIGLU;
  if (swiglu && (N2 / 2) % 16 != 0) return CODA_ERR_ALIGNMENT;
  if (!swiglu && z_save != nullptr) return CODA_ERR_INVALID_ARG;
  if (M == 0) return CODA_OK;
  return from_cuda(gemm_rowscale_swiglu_fp8(ctx_of(h, stream), static_cast<const uint8_t*>(Hq), sH,
                                            static_cast<const uint8_t*>(W2gq), sW2, rstd, static_cast<bf16*>(out),
                                            static_cast<bf16*>(z_save), int(M), int(d), int(N2), swiglu));
}

// ---------------------------------------------------------------------------
namespace {
struct CeWs {
  float* pmax;
  float* psum;
  int32_t* parg;
  float* zy;
  float* row_loss;
  bf16* dL;
  float* dH32;
  size_t bytes;
};

CeWs ce_layout(uint8_t* base, int64_t M, int64_t d, int64_t V, bool grads) {
  CeWs w{};
  const int64_t T = cdiv(V, ce_tile_cols());
  size_t off = 0;
  auto take = [&](size_t b) {
    uint8_t* p = base ? base + off : nullptr;
    off += align256(b);
    return p;
  };
  w.pmax = reinterpret_cast<float*>(take(size_t(M) * T * 4));
  w.psum = reinterpret_cast<float*>(take(size_t(M) * T * 4));
  w.parg = reinterpret_cast<int32_t*>(take(size_t(M) * T * 4));
  w.zy = reinterpret_cast<float*>(take(size_t(M) * 4));
  w.row_loss = reinterpret_cast<float*>(take(size_t(M) * 4));
  if (grads) {
    w.dL = reinterpret_cast<bf16*>(take(size_t(M) * std::min<int64_t>(V, kCeChunk) * 2));
    w.dH32 = reinterpret_cast<float*>(take(size_t(M) * d * 4));
  }
  w.bytes = off;
  return w;
}
}  // namespace

size_t coda_lmhead_ce_workspace_bytes(int64_t M, int64_t d, int64_t V, int with_grads) {
  if (M <= 0 || d <= 0 || V <= 0) return 0;
  return ce_layout(nullptr, M, d, V, with_grads != 0).bytes;
}

coda_status_t coda_lmhead_ce_row_offsets(int64_t M, int64_t d, int64_t V, int with_grads, size_t* label_logit_off,
                                         size_t* row_loss_off) {
  if (M <= 0 || d <= 0 || V <= 0) return CODA_ERR_INVALID_ARG;
  // carve the layout from a stand-in base (a null base gives null pointers)
  uint8_t* const base = reinterpret_cast<uint8_t*>(uintptr_t(256));
  const CeWs w = ce_layout(base, M, d, V, with_grads != 0);
  if (label_logit_off) *label_logit_off = size_t(reinterpret_cast<uint8_t*>(w.zy) - base);
  if (row_loss_off) *row_loss_off = size_t(reinterpret_cast<uint8_t*>(w.row_loss) - base);
  return CODA_OK;
}

coda_status_t coda_lmhead_ce(coda_handle_t h, const void* Hs, const void* Wt, const int32_t* labels, float* loss,
                             float* lse, int32_t* argmax, void* dHs, void* dWt, void* ws, size_t ws_bytes, int64_t M,
                             int64_t d, int64_t V, void* stream) {
  CODA_TRY(Check()
               .handle(h)
               .ptr(Hs)
               .ptr(Wt)
               .ptr(labels)
               .ptr(loss)
               .ptr(lse)
               .opt_ptr(argmax)
               .opt_ptr(dHs)
               .opt_ptr(dWt)
               .ptr(ws)
               .rows(M)
               .cols(d)
               .cols(V)
               .st);
  if (M == 0) return CODA_ERR_INVALID_ARG;  // the mean over no rows is undefined
  const bool grads = dHs != nullptr;
  if (grads != (dWt != nullptr)) return CODA_ERR_INVALID_ARG;
  if (ws_bytes < coda_lmhead_ce_workspace_bytes(M, d, V, grads)) return CODA_ERR_WORKSPACE_TOO_SMALL;
  const CeWs w = ce_layout(static_cast<uint8_t*>(ws), M, d, V, grads);
  const int64_t T = cdiv(V, ce_tile_cols());
  const LaunchCtx cx = ctx_of(h, stream);
  const bf16* Hb = static_cast<const bf16*>(Hs);
  const bf16* Wb = static_cast<const bf16*>(Wt);
  CODA_CUDA(cudaMemsetAsync(w.zy, 0, size_t(M) * 4, cx.stream));
  CODA_CUDA(gemm_ce_stats(cx, Hb, Wb, labels, w.pmax, w.psum, w.parg, w.zy, int(M), int(d), int(V), int(T)));
  CODA_CUDA(launch_ce_combine(cx, w.pmax, w.psum, w.parg, w.zy, labels, M, T, V, lse, argmax, w.row_loss));
  CODA_CUDA(launch_mean(cx, w.row_loss, M, loss));
  if (!grads) return CODA_OK;
  const float inv_M = 1.0f / static_cast<float>(M);
  const int64_t chunk = h->ce_chunk;
  for (int64_t v0 = 0; v0 < V; v0 += chunk) {
    const int64_t Vc = std::min<int64_t>(chunk, V - v0);
    const bf16* Wc = Wb + v0 * d;
    // dL[:, chunk] = (softmax - onehot) / M, recomputing the logits
    CODA_CUDA(gemm_ce_grad(cx, Hb, Wc, labels, lse, w.dL, int(M), int(d), int(Vc), int(v0), inv_M));
    // dH (+)= dL Wc (Wc stored [Vc][d]) and dWt[v0 + v][k] = sum_m dL[m][v]
    // Hs[m][k], one grouped launch
    CODA_CUDA(gemm_group_ce_bwd(cx, w.dL, Wc, Hb, w.dH32, v0 > 0, static_cast<bf16*>(dWt) + v0 * d, int(M), int(d),
                                int(Vc)));
  }
  CODA_CUDA(launch_f32_to_bf16(cx, w.dH32, static_cast<bf16*>(dHs), M * d));
  return CODA_OK;
}

coda_status_t coda_lmhead_ce_fp8(coda_handle_t h, const void* Hq, const float* sH, const void* Wq, const float* sW,
                                 const int32_t* labels, float* loss, float* lse, int32_t* argmax, void* dHs,
                                 void* dWt, void* ws, size_t ws_bytes, int64_t M, int64_t d, int64_t V,
                                 void* stream) {
  CODA_TRY(Check()
               .handle(h)
               .ptr(Hq)
               .sptr(sH)
               .ptr(Wq)
               .sptr(sW)
               .ptr(labels)
               .ptr(loss)
               .ptr(lse)
               .opt_ptr(argmax)
               .opt_ptr(dHs)
               .opt_ptr(dWt)
               .ptr(ws)
               .rows(M)
               .cols(d)
               .cols(V)
               .st);
  if (M == 0) return CODA_ERR_INVALID_ARG;  // the mean over no rows is undefined
  if (d % 16 != 0 || V % 16 != 0) return CODA_ERR_ALIGNMENT;
  const bool grads = dHs != nullptr;
  if (grads != (dWt != nullptr)) return CODA_ERR_INVALID_ARG;
  if (ws_bytes < coda_lmhead_ce_workspace_bytes(M, d, V, grads)) return CODA_ERR_WORKSPACE_TOO_SMALL;
  const CeWs w = ce_layout(static_cast<uint8_t*>(ws), M, d, V, grads);
  const int64_t T = cdiv(V, ce_tile_cols());
  const LaunchCtx cx = ctx_of(h, stream);
  const uint8_t* Hc = static_cast<const uint8_t*>(Hq);
  const uint8_t* Wc8 = static_cast<const uint8_t*>(Wq);
  CODA_CUDA(cudaMemsetAsync(w.zy, 0, size_t(M) * 4, cx.stream));
  CODA_CUDA(gemm_ce_stats_fp8(cx, Hc, sH, Wc8, sW, labels, w.pmax, w.psum, w.parg, w.zy, int(M), int(d), int(V),
                              int(T)));
  CODA_CUDA(launch_ce_combine(cx, w.pmax, w.psum, w.parg, w.zy, labels, M, T, V, lse, argmax, w.row_loss));
  CODA_CUDA(launch_mean(cx, w.row_loss, M, loss));
  if (!grads) return CODA_OK;
  const float inv_M = 1.0f / static_cast<float>(M);
  // |dL| <= 1/M: the smallest power of two s with (1/M) / s <= 57344
  // (= 0.875 * 2^16), so the e5m2 codes of dL / s never saturate
  int ea = 0;
  const float ma = std::frexp(inv_M, &ea);
  const int k = std::max(-126, ea - 16 + (ma > 0.875f ? 1 : 0));
  const float s_dL = std::ldexp(1.0f, k);
  const float code_inv = std::ldexp(1.0f, -k);
  uint8_t* dLq = reinterpret_cast<uint8_t*>(w.dL);  // the bf16 chunk buffer holds the 1-byte codes
  const int64_t chunk = h->ce_chunk;
  for (int64_t v0 = 0; v0 < V; v0 += chunk) {
    const int64_t Vc = std::min<int64_t>(chunk, V - v0);
    const uint8_t* Wqc = Wc8 + v0 * d;
    CODA_CUDA(gemm_ce_grad_fp8(cx, Hc, sH, Wqc, sW, labels, lse, dLq, code_inv, int(M), int(d), int(Vc), int(v0),
                               inv_M));
    // dH (+)= dL W and the chunk's dW rows from the codes, one grouped launch
    CODA_CUDA(gemm_group_ce_bwd_fp8(cx, dLq, s_dL, Wqc, sW, Hc, sH, w.dH32, v0 > 0,
                                    static_cast<bf16*>(dWt) + v0 * d, int(M), int(d), int(Vc)));
  }
  CODA_CUDA(launch_f32_to_bf16(cx, w.dH32, static_cast<bf16*>(dHs), M * d));
  return CODA_OK;
}

// ---------------------------------------------------------------------------
namespace {
constexpr int64_t kUnfusedDgRows = 256;  // rows per dg partial in the unfused RMSNorm backward
}

size_t coda_unfused_workspace_bytes(int64_t M, int64_t d, int64_t N2) {
  if (M < 0 || d <= 0 || N2 <= 0) return 0;
  const size_t fwd = align256(size_t(M) * d * 2);
  const size_t bwd = align256(size_t(M) * N2 * 2) + align256(size_t(M) * d * 2) +
                     align256(size_t(cdiv(M, kUnfusedDgRows)) * d * 4);
  return std::max(fwd, bwd);
}

coda_status_t coda_unfused_fwd(coda_handle_t h, const void* X, const void* W1t, const void* R, const void* g,
                               const void* W2t, void* H, float* rstd, void* Nrm, void* z, void* out, void* ws,
                               size_t ws_bytes, int64_t M, int64_t K1, int64_t d, int64_t N2, float eps,
                               uint32_t flags, void* stream) {
  CODA_TRY(Check()
               .handle(h)
               .rows(M)
               .mptr(X, M)
               .ptr(W1t)
               .mptr(R, M)
               .ptr(g)
               .ptr(W2t)
               .mptr(H, M)
               .mptr(rstd, M)
               .mptr(Nrm, M)
               .mptr(z, M)
               .mptr(out, M)
               .mptr(ws, M)
               .cols(K1)
               .cols(d)
               .cols(N2)
               .st);
  if (flags != CODA_EPI_SWIGLU && flags != CODA_EPI_PLAIN) return CODA_ERR_UNSUPPORTED;
  if (flags == CODA_EPI_SWIGLU && (N2 / 2) % 8 != 0) return CODA_ERR_ALIGNMENT;
  if (ws_bytes < coda_unfused_workspace_bytes(M, d, N2)) return CODA_ERR_WORKSPACE_TOO_SMALL;
  if (M == 0) return CODA_OK;
  const LaunchCtx cx = ctx_of(h, stream);
  bf16* A = static_cast<bf16*>(ws);
  CODA_CUDA(gemm_store(cx, static_cast<const bf16*>(X), false, static_cast<const bf16*>(W1t), false, A, int(M),
                       int(d), int(K1), nullptr, nullptr));
  CODA_CUDA(launch_add_rmsnorm(cx, A, static_cast<const bf16*>(R), static_cast<const bf16*>(g), static_cast<bf16*>(H),
                               rstd, static_cast<bf16*>(Nrm), M, d, eps));
  CODA_CUDA(gemm_store(cx, static_cast<const bf16*>(Nrm), false, static_cast<const bf16*>(W2t), false,
                       static_cast<bf16*>(z), int(M), int(N2), int(d), nullptr, nullptr));
  if (flags == CODA_EPI_SWIGLU)
    CODA_CUDA(launch_swiglu(cx, static_cast<const bf16*>(z), static_cast<bf16*>(out), M, N2 / 2));
  else if (out != z)
    CODA_CUDA(cudaMemcpyAsync(out, z, size_t(M) * N2 * 2, cudaMemcpyDeviceToDevice, cx.stream));
  return CODA_OK;
}

coda_status_t coda_unfused_bwd(coda_handle_t h, const void* dY, const void* X, const void* W1t, const void* g,
                               const void* W2t, const void* H, const float* rstd, const void* Nrm, const void* z,
                               void* dH, void* dX, void* dW1t, void* dW2t, float* dg, void* ws, size_t ws_bytes,
                               int64_t M, int64_t K1, int64_t d, int64_t N2, void* stream) {
  CODA_TRY(Check()
               .handle(h)
               .rows(M)
               .mptr(dY, M)
               .mptr(X, M)
               .ptr(W1t)
               .ptr(g)
               .ptr(W2t)
               .mptr(H, M)
               .mptr(rstd, M)
               .mptr(Nrm, M)
               .mptr(z, M)
               .mptr(dH, M)
               .mptr(dX, M)
               .ptr(dW1t)
               .ptr(dW2t)
               .ptr(dg)
               .mptr(ws, M)
               .cols(K1)
               .cols(d)
               .cols(N2)
               .st);
  if ((N2 / 2) % 8 != 0) return CODA_ERR_ALIGNMENT;
  if (ws_bytes < coda_unfused_workspace_bytes(M, d, N2)) return CODA_ERR_WORKSPACE_TOO_SMALL;
  const LaunchCtx cx = ctx_of(h, stream);
  if (M == 0) {
    CODA_CUDA(cudaMemsetAsync(dW2t, 0, size_t(N2) * d * 2, cx.stream));
    CODA_CUDA(cudaMemsetAsync(dW1t, 0, size_t(d) * K1 * 2, cx.stream));
    return from_cuda(cudaMemsetAsync(dg, 0, size_t(d) * 4, cx.stream));
  }
  uint8_t* w = static_cast<uint8_t*>(ws);
  bf16* dZ = reinterpret_cast<bf16*>(w);
  w += align256(size_t(M) * N2 * 2);
  bf16* dN = reinterpret_cast<bf16*>(w);
  w += align256(size_t(M) * d * 2);
  float* dgpart = reinterpret_cast<float*>(w);
  const int64_t parts = cdiv(M, kUnfusedDgRows);
  CODA_CUDA(launch_swiglu_bwd_plain(cx, static_cast<const bf16*>(dY), static_cast<const bf16*>(z), dZ, M, N2 / 2));
  // the GEMM launches are those of the fused path (two for the second
  // layer, one grouped launch for the first), so the comparison isolates
  // the epilogue fusion
  // dN[m][k] = sum_n dZ[m][n] W2t[n][k]
  CODA_CUDA(gemm_store(cx, dZ, false, static_cast<const bf16*>(W2t), true, dN, int(M), int(d), int(N2), nullptr,
                       nullptr));
  CODA_CUDA(launch_rmsnorm_bwd(cx, dN, static_cast<const bf16*>(H), rstd, static_cast<const bf16*>(g),
                               static_cast<bf16*>(dH), M, d));
  CODA_CUDA(launch_rmsnorm_bwd_dg(cx, dN, static_cast<const bf16*>(H), rstd, dgpart, M, d, kUnfusedDgRows));
  CODA_CUDA(launch_col_combine(cx, dgpart, parts, d, dg));
  // dW2t[n][k] = sum_m dZ[m][n] Nrm[m][k]
  CODA_CUDA(gemm_store(cx, dZ, true, static_cast<const bf16*>(Nrm), true, static_cast<bf16*>(dW2t), int(N2), int(d),
                       int(M), nullptr, nullptr));
  CODA_CUDA(gemm_group_store(cx, static_cast<const bf16*>(dH), static_cast<const bf16*>(W1t),
                             static_cast<const bf16*>(X), static_cast<bf16*>(dX), static_cast<bf16*>(dW1t), int(M),
                             int(K1), int(d)));
  return CODA_OK;
}

}  // extern "C"
