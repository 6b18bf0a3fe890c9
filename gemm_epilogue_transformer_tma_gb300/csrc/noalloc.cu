// Allocation-free variant of the second GEMM's data gradient with the RMSNorm
// backward in its epilogue (coda_gemm_dgrad_rmsbwd_noalloc in include/coda.h).
//
// Some callers cannot allocate device memory at all: a host framework that
// hands a plugin only its input and output tensors while its own pool owns
// every other byte on the device, or a latency-critical caller that must not
// pay for (or synchronise on) an allocation.  For them the per-row-block dg
// partial sums, which the allocating API keeps in a caller-provided buffer,
// live in a fixed array compiled into this library instead.
#include <mutex>

#include "../../include/coda.h"
#include "coda_internal.h"

// Scratch for the dg partial sums: 8 MiB, reserved on a device once this
// file's module is loaded there (at the latest on the first call on that
// device) and held until the process exits.  It covers coda_dgpart_rows(M)
// * d <= 2 Mi floats, e.g. M = 8192 tokens at d = 8192 or M = 16384 at
// d = 4096.
static constexpr size_t kScratchBytes = size_t(8) << 20;
static __device__ __align__(256) float g_dgpart_scratch[kScratchBytes / sizeof(float)];

namespace coda {
namespace {

std::mutex g_mu;

// Device address of g_dgpart_scratch for the handle's device and context.
// In host code the array's name is only a host-side stand-in, so the address
// is looked up with the handle's device current, on the first call with that
// handle, and kept in the handle.  A handle belongs to one context (its status
// word does too), so a handle created after a device reset looks the address
// up afresh instead of reusing one from the destroyed context.
coda_status_t scratch_of_handle(void* h, float** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  void** slot = noalloc_scratch_slot(h);
  if (*slot == nullptr) {
    const int dev = device_of_handle(h);
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return CODA_ERR_CUDA;
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) return CODA_ERR_CUDA;
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_dgpart_scratch);
    if (prev != dev) cudaSetDevice(prev);
    if (e != cudaSuccess || p == nullptr) return CODA_ERR_CUDA;
    *slot = p;
  }
  *out = static_cast<float*>(*slot);
  return CODA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace coda

extern "C" coda_status_t coda_gemm_dgrad_rmsbwd_noalloc(coda_handle_t h, const void* dP, const void* W2t,
                                                        const void* H, const void* g, const float* c, void* dH,
                                                        float* dg, int64_t M, int64_t N2, int64_t d, void* stream) {
  using namespace coda;
  using bf16 = __nv_bfloat16;
  if (h == nullptr || M < 0 || M > 0x7fffffff || N2 <= 0 || N2 > 0x7fffffff || d <= 0 || d > 0x7fffffff)
    return CODA_ERR_INVALID_ARG;
  if (N2 % 8 != 0 || d % 8 != 0) return CODA_ERR_ALIGNMENT;
  const void* always[] = {W2t, g, dg};
  const void* per_row[] = {dP, H, c, dH};
  for (const void* p : always) {
    if (p == nullptr) return CODA_ERR_INVALID_ARG;
    if (!aligned16(p)) return CODA_ERR_ALIGNMENT;
  }
  for (const void* p : per_row) {
    if (p == nullptr && M > 0) return CODA_ERR_INVALID_ARG;
    if (p != nullptr && !aligned16(p)) return CODA_ERR_ALIGNMENT;
  }
  const int64_t rows = coda_dgpart_rows(M);
  if (static_cast<size_t>(rows) * static_cast<size_t>(d) * sizeof(float) > kScratchBytes)
    return CODA_ERR_WORKSPACE_TOO_SMALL;  // beyond the built-in scratch: use coda_gemm_dgrad_rmsbwd
  const LaunchCtx cx = launch_ctx_of_handle(h, stream);
  if (M == 0) {  // empty batch: dg = 0
    return cudaMemsetAsync(dg, 0, size_t(d) * sizeof(float), cx.stream) == cudaSuccess ? CODA_OK : CODA_ERR_CUDA;
  }
  float* scratch = nullptr;
  const coda_status_t st = scratch_of_handle(h, &scratch);
  if (st != CODA_OK) return st;
  // The GEMM epilogue writes every partial the combine reads (all
  // coda_dgpart_rows(M) x d entries), so nothing left by an earlier call is
  // ever read and the scratch needs no clearing.
  cudaError_t e = gemm_dgrad_rms(cx, static_cast<const bf16*>(dP), static_cast<const bf16*>(W2t),
                                 static_cast<const bf16*>(H), static_cast<const bf16*>(g), c, static_cast<bf16*>(dH),
                                 scratch, int(M), int(N2), int(d));
  if (e == cudaSuccess) e = launch_col_combine(cx, scratch, rows, d, dg);
  if (e == cudaErrorNotSupported) return CODA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? CODA_OK : CODA_ERR_CUDA;
}
