// Block step executor: the whole fused step of the GEMM-Residual-PartialRMS-GEMM
// (+SwiGLU) block issued from native code, with its inputs and results in
// page-locked host memory.
//
// Method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
// (Synced write-up, section 尾声: GEMM1 with the residual and partial-RMS
// epilogue, a light combine, GEMM2 with the deferred row scale and SwiGLU, and
// a backward that keeps the same tile-local structure).  The executor adds no
// arithmetic: it orders the library's own calls and the host<->device copies.
//
// Streams (created here, one set per executor):
//   compute  the step's kernels, in order
//   side     the fold of g into W2 beside GEMM1 (it reads only weights); with
//            FP8 operands, the quantisation of dH beside wgrad2
//   h2d      copies of X, R (and dY) into the step's slot
//   d2h      read-back of the requested results from the step's slot
// Two slots hold everything a copy touches (X, R, dY in; out, dX, dH out), so
// the copies of step n+1 and the read-back of step n-1 run while step n
// computes.  Everything only the kernels touch (W2g, H, psum, rstd, z, the
// backward workspace; with FP8 operands the codes and scales) is single: the
// compute stream runs one step at a time.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>

#include "coda.h"

namespace {

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

constexpr int kSlots = 2;

struct Slot {
  void* X;
  void* R;
  void* dY;
  void* out;
  void* dH;
  void* dX;
  cudaEvent_t ev_in;      // X and R landed
  cudaEvent_t ev_in_bwd;  // dY landed
  cudaEvent_t ev_comp;    // the step's kernels finished with the slot's inputs
  cudaEvent_t ev_done;    // the step's results read back
  bool used;
};

// Byte offsets of every buffer of the arena, in a fixed order.
struct Layout {
  size_t W2gt, H, psum, rstd, z, ws, ws_bytes;
  // FP8: weight codes, activation and gradient codes, scales, c and dg partials
  size_t W1q, W2gq, W2q, Xq, Hq, dPq, dHq, s_w, s_a, c, dgpart;
  size_t X[kSlots], R[kSlots], dY[kSlots], out[kSlots], dH[kSlots], dX[kSlots];
  size_t total;
};

Layout layout_of(int64_t M, int64_t K1, int64_t d, int64_t N2, uint32_t flags) {
  Layout L{};
  const bool backward = (flags & CODA_BLOCK_BACKWARD) != 0, fp8 = (flags & CODA_BLOCK_FP8) != 0;
  const size_t m = size_t(M), k1 = size_t(K1), dd = size_t(d), n2 = size_t(N2), f = size_t(N2 / 2);
  const size_t T = size_t(coda_prms_num_tiles(d));
  size_t o = 0;
  auto take = [&o](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  L.H = take(m * dd * 2);
  L.psum = take(m * T * 4);
  L.rstd = take(m * 4);
  L.z = backward ? take(m * n2 * 2) : 0;
  if (!fp8) {
    L.W2gt = take(n2 * dd * 2);
    L.ws_bytes = backward ? coda_bwd_workspace_bytes(M, d, N2) : 0;
    L.ws = backward ? take(L.ws_bytes) : 0;
  } else {
    L.W1q = take(dd * k1);
    L.W2gq = take(n2 * dd);
    L.Xq = take(m * k1);
    L.Hq = take(m * dd);
    L.s_w = take(3 * 2 * 4);
    L.s_a = take(4 * 2 * 4);
    if (backward) {
      L.W2q = take(n2 * dd);
      L.dPq = take(m * n2);
      L.dHq = take(m * dd);
      L.c = take(m * 4);
      L.dgpart = take(size_t(coda_dgpart_rows(M)) * dd * 4);
    }
  }
  for (int s = 0; s < kSlots; ++s) {
    L.X[s] = take(m * k1 * 2);
    L.R[s] = take(m * dd * 2);
    L.out[s] = take(m * f * 2);
    if (backward) {
      L.dY[s] = take(m * f * 2);
      L.dH[s] = take(m * dd * 2);
      L.dX[s] = take(m * k1 * 2);
    }
  }
  L.total = o;
  return L;
}

bool shape_ok(int64_t M, int64_t K1, int64_t d, int64_t N2) {
  constexpr int64_t kMax = (int64_t(1) << 31) - 1;
  if (M < 0 || M > kMax) return false;
  for (int64_t v : {K1, d, N2})
    if (v <= 0 || v > kMax) return false;
  return true;
}

bool aligned8(int64_t K1, int64_t d, int64_t N2) { return K1 % 8 == 0 && d % 8 == 0 && N2 % 16 == 0; }

// 8-bit operands: every contiguous extent of a code tensor a multiple of 16
bool aligned16(int64_t K1, int64_t d, int64_t N2) { return K1 % 16 == 0 && d % 16 == 0 && N2 % 32 == 0; }

// A host pointer the copy engines can read or write asynchronously:
// page-locked (cudaHostAlloc) or registered (cudaHostRegister) memory.
bool pinned(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
      return;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) (void)cudaSetDevice(prev);
  }
};

}  // namespace

struct coda_block_s {
  coda_handle_t h;
  int device;
  int64_t M, K1, d, N2;
  float eps;
  int backward;
  bool fp8, delayed;
  bool weights_ready;  // FP8: weight codes written by coda_block_quantize_weights
  bool dp_amax_ready;  // FP8 delayed: the dP state holds an amax
  const void* W1t;
  const void* g;
  const void* W2t;
  void* dW1t;
  void* dW2t;
  float* dg;
  void* W2gt;
  void* H;
  float* psum;
  float* rstd;
  void* z;
  void* ws;
  size_t ws_bytes;
  uint8_t *W1q, *W2gq, *W2q, *Xq, *Hq, *dPq, *dHq;
  float *s_w, *s_a, *c, *dgpart;  // s_w: W1, W2 g, W2; s_a: X, H, dP, dH ({amax, scale} each)
  Slot slot[kSlots];
  cudaStream_t compute, side, h2d, d2h;
  cudaEvent_t ev_fork, ev_join;
  int64_t submitted;
};

namespace {

void release(coda_block_s* b) {
  for (cudaStream_t* s : {&b->compute, &b->side, &b->h2d, &b->d2h})
    if (*s) (void)cudaStreamDestroy(*s);
  for (cudaEvent_t* e : {&b->ev_fork, &b->ev_join})
    if (*e) (void)cudaEventDestroy(*e);
  for (Slot& sl : b->slot)
    for (cudaEvent_t* e : {&sl.ev_in, &sl.ev_in_bwd, &sl.ev_comp, &sl.ev_done})
      if (*e) (void)cudaEventDestroy(*e);
  delete b;
}

coda_status_t cu(cudaError_t e) { return e == cudaSuccess ? CODA_OK : CODA_ERR_CUDA; }

#define BLK_TRY(expr)                 \
  do {                                \
    const coda_status_t st_ = (expr); \
    if (st_ != CODA_OK) return st_;   \
  } while (0)

// The forward of one step on the compute stream: GEMM1 + residual + partial
// RMS with the fold beside it, the rstd combine, GEMM2 + row scale + SwiGLU.
coda_status_t forward(coda_block_s* b, Slot& sl) {
  void* cs = b->compute;
  const int64_t T = coda_prms_num_tiles(b->d);
  BLK_TRY(cu(cudaEventRecord(b->ev_fork, b->compute)));
  BLK_TRY(coda_gemm_res_prms(b->h, sl.X, b->W1t, sl.R, b->H, b->psum, b->M, b->K1, b->d, cs));
  BLK_TRY(cu(cudaStreamWaitEvent(b->side, b->ev_fork, 0)));
  BLK_TRY(coda_fold_rmsnorm_weight(b->h, b->W2t, b->g, b->W2gt, b->N2, b->d, b->side));
  BLK_TRY(cu(cudaEventRecord(b->ev_join, b->side)));
  BLK_TRY(cu(cudaStreamWaitEvent(b->compute, b->ev_join, 0)));
  BLK_TRY(coda_rstd_combine(b->h, b->psum, b->M, T, b->d, b->eps, b->rstd, cs));
  return coda_gemm_rowscale_swiglu(b->h, b->H, b->W2gt, b->rstd, sl.out, b->backward ? b->z : nullptr, b->M, b->d,
                                   b->N2, CODA_EPI_SWIGLU, cs);
}

// The backward of one step: SwiGLU backward, dgrad2 with the RMSNorm
// backward, dg, wgrad2, then dX and dW1 (dR = dH).
coda_status_t backward(coda_block_s* b, Slot& sl) {
  void* cs = b->compute;
  BLK_TRY(cu(cudaStreamWaitEvent(b->compute, sl.ev_in_bwd, 0)));
  BLK_TRY(coda_gemm_rowscale_swiglu_bwd(b->h, sl.dY, b->z, b->rstd, b->H, b->W2t, b->g, sl.dH, b->dW2t, b->dg, b->ws,
                                        b->ws_bytes, b->M, b->d, b->N2, cs));
  return coda_gemm_res_prms_bwd(b->h, sl.dH, sl.X, b->W1t, sl.dX, b->dW1t, sl.dH, b->M, b->K1, b->d, cs);
}

// The FP8 forward: X and H quantised in the step (e4m3, per-tensor
// power-of-two scales), GEMM1 and GEMM2 on the codes with the same epilogue
// programs; the weight codes come from coda_block_quantize_weights.
coda_status_t forward_fp8(coda_block_s* b, Slot& sl) {
  void* cs = b->compute;
  const int64_t T = coda_prms_num_tiles(b->d);
  BLK_TRY(coda_fp8_quantize(b->h, sl.X, nullptr, b->s_a + 0, b->Xq, b->M, b->K1, cs));
  BLK_TRY(coda_gemm_res_prms_fp8(b->h, b->Xq, b->s_a + 1, b->W1q, b->s_w + 1, sl.R, b->H, b->psum, b->M, b->K1,
                                 b->d, cs));
  BLK_TRY(coda_rstd_combine(b->h, b->psum, b->M, T, b->d, b->eps, b->rstd, cs));
  BLK_TRY(coda_fp8_quantize(b->h, b->H, nullptr, b->s_a + 2, b->Hq, b->M, b->d, cs));
  return coda_gemm_rowscale_swiglu_fp8(b->h, b->Hq, b->s_a + 3, b->W2gq, b->s_w + 3, b->rstd, sl.out,
                                       b->backward ? b->z : nullptr, b->M, b->d, b->N2, CODA_EPI_SWIGLU, cs);
}

// The FP8 backward: dP's e5m2 codes from the SwiGLU backward (delayed
// scaling after the first step if requested), dgrad2 with the RMSNorm
// backward, dg, wgrad2 with dH's e5m2 codes quantised beside it, then dX and
// dW1 in one grouped launch.
coda_status_t backward_fp8(coda_block_s* b, Slot& sl) {
  void* cs = b->compute;
  const int64_t F = b->N2 / 2;
  BLK_TRY(cu(cudaStreamWaitEvent(b->compute, sl.ev_in_bwd, 0)));
  if (b->delayed && b->dp_amax_ready)
    BLK_TRY(coda_swiglu_bwd_fp8_delayed(b->h, sl.dY, b->z, b->rstd, 1, b->dPq, b->s_a + 4, b->c, b->M, F, b->d, cs));
  else
    BLK_TRY(coda_swiglu_bwd_fp8(b->h, sl.dY, b->z, b->rstd, 1, b->dPq, b->s_a + 4, b->c, b->M, F, b->d, cs));
  b->dp_amax_ready = true;
  BLK_TRY(coda_gemm_dgrad_rmsbwd_fp8(b->h, b->dPq, 1, b->s_a + 5, b->W2q, 0, b->s_w + 5, b->H, b->g, b->c, sl.dH,
                                     b->dgpart, b->M, b->N2, b->d, cs));
  BLK_TRY(coda_dg_combine(b->h, b->dgpart, coda_dgpart_rows(b->M), b->d, b->dg, cs));
  // dW2t[n][k] = g[k] sum_m dP[m][n] H[m][k], with dH's codes (needed only by
  // the first layer's gradients) quantised beside it
  BLK_TRY(cu(cudaEventRecord(b->ev_fork, b->compute)));
  BLK_TRY(coda_gemm_fp8(b->h, b->dPq, 1, 1, b->s_a + 5, b->Hq, 1, 0, b->s_a + 3, b->dW2t, b->N2, b->d, b->M, nullptr,
                        b->g, cs));
  BLK_TRY(cu(cudaStreamWaitEvent(b->side, b->ev_fork, 0)));
  BLK_TRY(coda_fp8_quantize_e5m2(b->h, sl.dH, nullptr, b->s_a + 6, b->dHq, b->M, b->d, b->side));
  BLK_TRY(cu(cudaEventRecord(b->ev_join, b->side)));
  BLK_TRY(cu(cudaStreamWaitEvent(b->compute, b->ev_join, 0)));
  return coda_gemm_res_prms_bwd_fp8(b->h, b->dHq, 1, b->s_a + 7, b->Xq, b->s_a + 1, b->W1q, b->s_w + 1, 0, sl.dX,
                                    b->dW1t, b->M, b->K1, b->d, cs);
}

}  // namespace

extern "C" {

size_t coda_block_arena_bytes(int64_t M, int64_t K1, int64_t d, int64_t N2, uint32_t flags) {
  if (!shape_ok(M, K1, d, N2)) return 0;
  return layout_of(M, K1, d, N2, flags).total;
}

coda_status_t coda_block_create(coda_handle_t h, int64_t M, int64_t K1, int64_t d, int64_t N2, float eps,
                                uint32_t flags, const void* W1t, const void* g, const void* W2t, void* dW1t,
                                void* dW2t, float* dg, void* arena, size_t arena_bytes, coda_block_t* out) {
  if (out == nullptr) return CODA_ERR_INVALID_ARG;
  *out = nullptr;
  if (h == nullptr || !shape_ok(M, K1, d, N2) || !(eps > 0.f)) return CODA_ERR_INVALID_ARG;
  constexpr uint32_t kKnown = CODA_BLOCK_BACKWARD | CODA_BLOCK_FP8 | CODA_BLOCK_FP8_DELAYED;
  if ((flags & ~kKnown) != 0) return CODA_ERR_INVALID_ARG;
  const int backward = (flags & CODA_BLOCK_BACKWARD) ? 1 : 0;
  const bool fp8 = (flags & CODA_BLOCK_FP8) != 0;
  const bool delayed = (flags & CODA_BLOCK_FP8_DELAYED) != 0;
  if (delayed && !(fp8 && backward)) return CODA_ERR_INVALID_ARG;
  if (!aligned8(K1, d, N2)) return CODA_ERR_ALIGNMENT;
  if (fp8 && !aligned16(K1, d, N2)) return CODA_ERR_ALIGNMENT;
  for (const void* p : {W1t, g, W2t, static_cast<const void*>(arena)})
    if (p == nullptr) return CODA_ERR_INVALID_ARG;
  if (backward)
    for (const void* p : {static_cast<const void*>(dW1t), static_cast<const void*>(dW2t),
                          static_cast<const void*>(dg)})
      if (p == nullptr) return CODA_ERR_INVALID_ARG;
  for (const void* p : {W1t, g, W2t, static_cast<const void*>(arena)})
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return CODA_ERR_ALIGNMENT;
  if (backward)
    for (const void* p : {static_cast<const void*>(dW1t), static_cast<const void*>(dW2t)})
      if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return CODA_ERR_ALIGNMENT;
  const Layout L = layout_of(M, K1, d, N2, flags);
  if (arena_bytes < L.total) return CODA_ERR_WORKSPACE_TOO_SMALL;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CODA_ERR_CUDA;
  coda_block_s* b = new (std::nothrow) coda_block_s;
  if (b == nullptr) return CODA_ERR_CUDA;
  std::memset(static_cast<void*>(b), 0, sizeof(*b));
  b->h = h;
  b->device = dev;
  b->M = M;
  b->K1 = K1;
  b->d = d;
  b->N2 = N2;
  b->eps = eps;
  b->backward = backward;
  b->fp8 = fp8;
  b->delayed = delayed;
  b->W1t = W1t;
  b->g = g;
  b->W2t = W2t;
  b->dW1t = dW1t;
  b->dW2t = dW2t;
  b->dg = dg;
  uint8_t* a = static_cast<uint8_t*>(arena);
  b->H = a + L.H;
  b->psum = reinterpret_cast<float*>(a + L.psum);
  b->rstd = reinterpret_cast<float*>(a + L.rstd);
  b->z = backward ? a + L.z : nullptr;
  if (!fp8) {
    b->W2gt = a + L.W2gt;
    b->ws = backward ? a + L.ws : nullptr;
    b->ws_bytes = L.ws_bytes;
  } else {
    b->W1q = a + L.W1q;
    b->W2gq = a + L.W2gq;
    b->Xq = a + L.Xq;
    b->Hq = a + L.Hq;
    b->s_w = reinterpret_cast<float*>(a + L.s_w);
    b->s_a = reinterpret_cast<float*>(a + L.s_a);
    if (backward) {
      b->W2q = a + L.W2q;
      b->dPq = a + L.dPq;
      b->dHq = a + L.dHq;
      b->c = reinterpret_cast<float*>(a + L.c);
      b->dgpart = reinterpret_cast<float*>(a + L.dgpart);
    }
  }
  for (int s = 0; s < kSlots; ++s) {
    Slot& sl = b->slot[s];
    sl.X = a + L.X[s];
    sl.R = a + L.R[s];
    sl.out = a + L.out[s];
    sl.dY = backward ? a + L.dY[s] : nullptr;
    sl.dH = backward ? a + L.dH[s] : nullptr;
    sl.dX = backward ? a + L.dX[s] : nullptr;
  }
  bool ok = true;
  for (cudaStream_t* s : {&b->compute, &b->side, &b->h2d, &b->d2h})
    ok = ok && cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) == cudaSuccess;
  for (cudaEvent_t* e : {&b->ev_fork, &b->ev_join})
    ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
  for (Slot& sl : b->slot)
    for (cudaEvent_t* e : {&sl.ev_in, &sl.ev_in_bwd, &sl.ev_comp, &sl.ev_done})
      ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    release(b);
    return CODA_ERR_CUDA;
  }
  *out = b;
  return CODA_OK;
}

coda_status_t coda_block_step_host(coda_block_t b, const void* X, const void* R, const void* dY, void* out, void* dX,
                                   void* dR, int64_t* step_id) {
  if (b == nullptr) return CODA_ERR_INVALID_ARG;
  const bool empty = b->M == 0;
  // inputs: required (unless the batch is empty) and page-locked
  if (!b->backward && (dY != nullptr || dX != nullptr || dR != nullptr)) return CODA_ERR_INVALID_ARG;
  for (const void* p : {X, R, dY}) {
    if (p == dY && !b->backward) continue;
    if (p == nullptr) {
      if (!empty) return CODA_ERR_INVALID_ARG;
    } else if (!pinned(p)) {
      return CODA_ERR_INVALID_ARG;
    }
  }
  for (const void* p : {static_cast<const void*>(out), static_cast<const void*>(dX), static_cast<const void*>(dR)})
    if (p != nullptr && !pinned(p)) return CODA_ERR_INVALID_ARG;

  if (b->fp8 && !b->weights_ready) return CODA_ERR_INVALID_ARG;
  DeviceGuard guard(b->device);
  if (!guard.ok) return CODA_ERR_CUDA;
  const int s = int(b->submitted % kSlots);
  Slot& sl = b->slot[s];
  const size_t M = size_t(b->M), K1 = size_t(b->K1), d = size_t(b->d), F = size_t(b->N2 / 2);

  // inputs into the slot, once the kernels of the step that used it last are done with it
  if (sl.used) BLK_TRY(cu(cudaStreamWaitEvent(b->h2d, sl.ev_comp, 0)));
  if (!empty) {
    BLK_TRY(cu(cudaMemcpyAsync(sl.X, X, M * K1 * 2, cudaMemcpyHostToDevice, b->h2d)));
    BLK_TRY(cu(cudaMemcpyAsync(sl.R, R, M * d * 2, cudaMemcpyHostToDevice, b->h2d)));
  }
  BLK_TRY(cu(cudaEventRecord(sl.ev_in, b->h2d)));
  if (b->backward) {
    if (!empty) BLK_TRY(cu(cudaMemcpyAsync(sl.dY, dY, M * F * 2, cudaMemcpyHostToDevice, b->h2d)));
    BLK_TRY(cu(cudaEventRecord(sl.ev_in_bwd, b->h2d)));
  }

  // the step; its results overwrite the slot's once their last read-back is done
  BLK_TRY(cu(cudaStreamWaitEvent(b->compute, sl.ev_in, 0)));
  if (sl.used) BLK_TRY(cu(cudaStreamWaitEvent(b->compute, sl.ev_done, 0)));
  if (b->fp8) {
    BLK_TRY(forward_fp8(b, sl));
    if (b->backward) BLK_TRY(backward_fp8(b, sl));
  } else {
    BLK_TRY(forward(b, sl));
    if (b->backward) BLK_TRY(backward(b, sl));
  }
  BLK_TRY(cu(cudaEventRecord(sl.ev_comp, b->compute)));

  // results back to the host
  BLK_TRY(cu(cudaStreamWaitEvent(b->d2h, sl.ev_comp, 0)));
  if (!empty) {
    if (out) BLK_TRY(cu(cudaMemcpyAsync(out, sl.out, M * F * 2, cudaMemcpyDeviceToHost, b->d2h)));
    if (dX) BLK_TRY(cu(cudaMemcpyAsync(dX, sl.dX, M * K1 * 2, cudaMemcpyDeviceToHost, b->d2h)));
    if (dR) BLK_TRY(cu(cudaMemcpyAsync(dR, sl.dH, M * d * 2, cudaMemcpyDeviceToHost, b->d2h)));
  }
  BLK_TRY(cu(cudaEventRecord(sl.ev_done, b->d2h)));
  sl.used = true;
  if (step_id) *step_id = b->submitted;
  ++b->submitted;
  return CODA_OK;
}

coda_status_t coda_block_quantize_weights(coda_block_t b) {
  if (b == nullptr) return CODA_ERR_INVALID_ARG;
  if (!b->fp8) return CODA_OK;
  DeviceGuard guard(b->device);
  if (!guard.ok) return CODA_ERR_CUDA;
  void* cs = b->compute;
  BLK_TRY(coda_fp8_quantize(b->h, b->W1t, nullptr, b->s_w + 0, b->W1q, b->d, b->K1, cs));
  BLK_TRY(coda_fp8_quantize(b->h, b->W2t, b->g, b->s_w + 2, b->W2gq, b->N2, b->d, cs));
  if (b->backward) BLK_TRY(coda_fp8_quantize(b->h, b->W2t, nullptr, b->s_w + 4, b->W2q, b->N2, b->d, cs));
  b->weights_ready = true;
  return CODA_OK;
}

coda_status_t coda_block_wait_step(coda_block_t b, int64_t step) {
  if (b == nullptr || step < 0 || step >= b->submitted) return CODA_ERR_INVALID_ARG;
  DeviceGuard guard(b->device);
  if (!guard.ok) return CODA_ERR_CUDA;
  return cu(cudaEventSynchronize(b->slot[step % kSlots].ev_done));
}

coda_status_t coda_block_sync(coda_block_t b, int32_t* device_bits) {
  if (b == nullptr) return CODA_ERR_INVALID_ARG;
  DeviceGuard guard(b->device);
  if (!guard.ok) return CODA_ERR_CUDA;
  for (cudaStream_t s : {b->h2d, b->side, b->d2h})
    BLK_TRY(cu(cudaStreamSynchronize(s)));
  return coda_sync_status(b->h, b->compute, device_bits);
}

coda_status_t coda_block_stream(coda_block_t b, void** stream) {
  if (b == nullptr || stream == nullptr) return CODA_ERR_INVALID_ARG;
  *stream = b->compute;
  return CODA_OK;
}

coda_status_t coda_block_destroy(coda_block_t b) {
  if (b == nullptr) return CODA_OK;
  DeviceGuard guard(b->device);
  for (cudaStream_t s : {b->h2d, b->side, b->compute, b->d2h})
    if (s) (void)cudaStreamSynchronize(s);
  release(b);
  return CODA_OK;
}

}  // extern "C"
