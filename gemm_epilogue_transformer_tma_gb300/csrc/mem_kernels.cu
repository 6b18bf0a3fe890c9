// Memory-bound kernels of the path: folding the RMSNorm weight into W2, the
// light partial-RMS combine, the SwiGLU backward stream, column combines, the
// blocked log-sum-exp combine, and the unfused ablation's standalone
// add+RMSNorm / SwiGLU / SwiGLU-bwd / RMSNorm-bwd kernels.
//
// All accesses are 16-byte vectors (8 bf16 or 4 fp32) along the contiguous
// dimension; every extent on the boundary is a multiple of 8 elements.
#include <algorithm>
#include <cfloat>
#include <cuda_fp8.h>

#include "coda_internal.h"
#include "ptx.cuh"

namespace coda {

namespace {

__device__ __forceinline__ uint4 pack8(const float* f) {
  uint4 q;
  q.x = pack_bf16x2(f[0], f[1]);
  q.y = pack_bf16x2(f[2], f[3]);
  q.z = pack_bf16x2(f[4], f[5]);
  q.w = pack_bf16x2(f[6], f[7]);
  return q;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// block-wide sum for blockDim.x == 256; result valid in every thread
__device__ __forceinline__ float block_sum_256(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = (l < 8) ? red[l] : 0.f;
  return warp_sum(t);
}

// block-wide max for blockDim.x == 256; result valid in thread 0
__device__ __forceinline__ float block_max_256(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = (l < 8) ? red[l] : 0.f;
  if (w == 0) {
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
  }
  return t;
}

// Grid for the column-chunk x row-block e4m3 quantisation kernels:
// x covers the 8-column chunks in blocks of 256, y the blocks of `rows_per`
// rows.  When there are more row blocks than fit in one wave (8 CTAs of 256
// threads per SM), every CTA loops over the same number of them, so the
// launch is a single, evenly loaded wave.
dim3 chunk_rows_grid(const LaunchCtx& c, int64_t c8, int64_t rows, int rows_per) {
  const int64_t gx = (c8 + 255) / 256;
  const int64_t row_blocks = std::max<int64_t>(1, (rows + rows_per - 1) / rows_per);
  const int64_t cap_y = std::max<int64_t>(1, static_cast<int64_t>(c.num_sms) * 8 / gx);
  const int64_t iters = (row_blocks + cap_y - 1) / cap_y;
  const int64_t gy = std::min<int64_t>((row_blocks + iters - 1) / iters, 65535);
  return dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
}

int grid_for(const LaunchCtx& c, int64_t work_items, int threads) {
  const int64_t need = (work_items + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(c.num_sms) * 8;
  return static_cast<int>(need < cap ? (need > 0 ? need : 1) : cap);
}

// ---------------------------------------------------------------------------
// W2gt[n, k] = bf16(W2t[n, k] * g[k]).  A thread owns one 8-column chunk
// (its g values stay in registers) and kFoldRows rows of it: all of its row
// loads are issued before the first product, so each SM keeps enough bytes
// in flight to cover HBM latency.
constexpr int kFoldRows = 8;

__global__ void __launch_bounds__(256) fold_kernel(const uint4* __restrict__ W2t, const uint4* __restrict__ g8,
                                                   uint4* __restrict__ out, int64_t rows, int64_t d8) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t j = blockIdx.x * 256LL + threadIdx.x;
  if (j >= d8) return;
  float g[8];
  unpack_bf16x8(__ldg(&g8[j]), g);
  for (int64_t r0 = blockIdx.y * static_cast<int64_t>(kFoldRows); r0 < rows;
       r0 += static_cast<int64_t>(gridDim.y) * kFoldRows) {
    const uint4* src = W2t + r0 * d8 + j;
    uint4* dst = out + r0 * d8 + j;
    const int nr = static_cast<int>(rows - r0 < kFoldRows ? rows - r0 : kFoldRows);
    uint4 v[kFoldRows];
#pragma unroll
    for (int r = 0; r < kFoldRows; ++r)
      if (r < nr) v[r] = src[r * d8];
#pragma unroll
    for (int r = 0; r < kFoldRows; ++r) {
      if (r < nr) {
        float w[8], o[8];
        unpack_bf16x8(v[r], w);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = w[i] * g[i];
        dst[r * d8] = pack8(o);
      }
    }
  }
}

// rstd[m] = 1 / sqrt(sum_j psum[m, j] / d + eps): one warp per row
__global__ void rstd_combine_kernel(const float* __restrict__ psum, int64_t M, int64_t T, float inv_d, float eps,
                                    float* __restrict__ rstd) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  float s = 0.f;
  for (int64_t j = lane; j < T; j += 32) s += psum[row * T + j];
  s = warp_sum(s);
  if (lane == 0) rstd[row] = 1.0f / sqrtf(s * inv_d + eps);
}

// Packed fp32 pairs: one instruction performs the same IEEE round-to-nearest
// operation on both lanes of a float2 (sm_100 family).  Halves the issue slots
// of fp32 arithmetic where two independent values move in step.
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// SwiGLU backward with the deferred row scale: one CTA (256 threads) per row.
//   s = sigmoid(zg); dZg = dY*zu*s*(1 + zg*(1-s)); dZu = dY*zg*s
//   dP = bf16(r * dZ); c[m] = r^2/d * sum(dZg*zg + dZu*zu)
// Each thread loads two 8-column chunks (six 16-byte loads) before computing
// either, to keep enough bytes in flight.
__device__ __forceinline__ float swiglu_bwd_vals(const uint4& dyq, const uint4& zgq, const uint4& zuq, float r,
                                                 float* og, float* ou) {
  float dy[8], zg[8], zu[8];
  unpack_bf16x8(dyq, dy);
  unpack_bf16x8(zgq, zg);
  unpack_bf16x8(zuq, zu);
  // columns in pairs, on packed fp32 pairs; the two lanes' dot products stay
  // apart until the end
  const float2 one = make_float2(1.0f, 1.0f), neg_one = make_float2(-1.0f, -1.0f), r2 = make_float2(r, r);
  float2 dot = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const float2 y = make_float2(dy[i], dy[i + 1]);
    const float2 g = make_float2(zg[i], zg[i + 1]);
    const float2 u = make_float2(zu[i], zu[i + 1]);
    const float2 s = make_float2(sigmoid_f(g.x), sigmoid_f(g.y));
    const float2 ys = f2_mul(y, s);
    const float2 dzu = f2_mul(ys, g);                       // dY zg s
    const float2 w = f2_fma(g, f2_fma(s, neg_one, one), one);  // 1 + zg (1 - s)
    const float2 dzg = f2_mul(f2_mul(ys, u), w);            // dY zu s (1 + zg (1 - s))
    dot = f2_fma(dzg, g, f2_fma(dzu, u, dot));
    const float2 pg = f2_mul(r2, dzg), pu = f2_mul(r2, dzu);
    og[i] = pg.x;
    og[i + 1] = pg.y;
    ou[i] = pu.x;
    ou[i + 1] = pu.y;
  }
  return dot.x + dot.y;
}

__device__ __forceinline__ float swiglu_bwd_chunk(const uint4& dyq, const uint4& zgq, const uint4& zuq, float r,
                                                  uint4& pg, uint4& pu) {
  float og[8], ou[8];
  const float dot = swiglu_bwd_vals(dyq, zgq, zuq, r, og, ou);
  pg = pack8(og);
  pu = pack8(ou);
  return dot;
}

__global__ void __launch_bounds__(256) swiglu_bwd_kernel(const __nv_bfloat16* __restrict__ dY,
                                                         const __nv_bfloat16* __restrict__ z,
                                                         const float* __restrict__ rstd,
                                                         __nv_bfloat16* __restrict__ dP, float* __restrict__ cvec,
                                                         int64_t F, float inv_d) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[8];
  const int64_t m = blockIdx.x;
  const float r = rstd[m];
  const uint4* dy8 = reinterpret_cast<const uint4*>(dY + m * F);
  const uint4* zg8 = reinterpret_cast<const uint4*>(z + m * 2 * F);
  const uint4* zu8 = reinterpret_cast<const uint4*>(z + m * 2 * F + F);
  uint4* pg8 = reinterpret_cast<uint4*>(dP + m * 2 * F);
  uint4* pu8 = reinterpret_cast<uint4*>(dP + m * 2 * F + F);
  const int64_t F8 = F / 8;
  float dot = 0.f;
  for (int64_t j0 = threadIdx.x; j0 < F8; j0 += 2 * 256) {
    const int64_t j1 = j0 + 256;
    const bool two = j1 < F8;
    const uint4 a0 = dy8[j0], b0 = zg8[j0], c0 = zu8[j0];
    uint4 a1 = a0, b1 = b0, c1 = c0;
    if (two) {
      a1 = dy8[j1];
      b1 = zg8[j1];
      c1 = zu8[j1];
    }
    uint4 pg, pu;
    dot += swiglu_bwd_chunk(a0, b0, c0, r, pg, pu);
    pg8[j0] = pg;
    pu8[j0] = pu;
    if (two) {
      dot += swiglu_bwd_chunk(a1, b1, c1, r, pg, pu);
      pg8[j1] = pg;
      pu8[j1] = pu;
    }
  }
  const float tot = block_sum_256(dot, red);
  if (threadIdx.x == 0) cvec[m] = r * r * inv_d * tot;
}

// out[k] = sum_r part[r, k]; block = 32 columns x 8 row groups
__global__ void col_combine_kernel(const float* __restrict__ part, int64_t rows, int64_t d, float* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[8][33];
  const int64_t k = blockIdx.x * 32 + threadIdx.x;
  float s = 0.f;
  if (k < d)
    for (int64_t r = threadIdx.y; r < rows; r += 8) s += part[r * d + k];
  red[threadIdx.y][threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.y == 0 && k < d) {
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) t += red[i][threadIdx.x];
    out[k] = t;
  }
}

// Blocked log-sum-exp combine, one warp per row:
//   m* = max_j mx_j ; lse = m* + log(sum_j se_j * exp(mx_j - m*))
//   argmax = column of the largest tile max (lowest column on ties)
//   row_loss = lse - z_y (0 and a status bit if the label is out of range)
__global__ void ce_combine_kernel(const float* __restrict__ pmax, const float* __restrict__ psum,
                                  const int32_t* __restrict__ parg, const float* __restrict__ zy,
                                  const int32_t* __restrict__ labels, int64_t M, int64_t T, int64_t V,
                                  float* __restrict__ lse, int32_t* __restrict__ argmax, float* __restrict__ row_loss,
                                  int* status) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const float* mx = pmax + row * T;
  const float* se = psum + row * T;
  const int32_t* ag = parg + row * T;
  float best = -INFINITY;
  int bidx = 0x7fffffff;
  for (int64_t j = lane; j < T; j += 32) {
    const float v = mx[j];
    const int a = ag[j];
    if (v > best || (v == best && a < bidx)) {
      best = v;
      bidx = a;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oa = __shfl_xor_sync(0xffffffffu, bidx, o);
    if (ov > best || (ov == best && oa < bidx)) {
      best = ov;
      bidx = oa;
    }
  }
  float s = 0.f;
  for (int64_t j = lane; j < T; j += 32) s += se[j] * __expf(mx[j] - best);
  s = warp_sum(s);
  if (lane == 0) {
    const float l = best + logf(s);
    lse[row] = l;
    if (argmax != nullptr) argmax[row] = bidx;
    const int y = labels[row];
    if (y < 0 || y >= V) {
      atomicOr(status, DEV_ERR_LABEL_RANGE);
      row_loss[row] = 0.f;
    } else {
      row_loss[row] = l - zy[row];
    }
  }
}

// out = mean(v) with a fixed summation order (one CTA of 1024 threads)
__global__ void __launch_bounds__(1024) mean_kernel(const float* __restrict__ v, int64_t n, float* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[32];
  float s = 0.f;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) s += v[i];
  s = warp_sum(s);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = warp_sum(red[threadIdx.x]);
    if (threadIdx.x == 0) *out = t / static_cast<float>(n);
  }
}

__global__ void f32_to_bf16_kernel(const float4* __restrict__ in, uint2* __restrict__ out, int64_t n4) {
  griddep_wait();
  griddep_launch_dependents();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 f = in[i];
    out[i] = make_uint2(pack_bf16x2(f.x, f.y), pack_bf16x2(f.z, f.w));
  }
}

// cos / sin of theta[p, i] = p * base^(-2 i / D), in double precision
__global__ void rope_table_kernel(float* __restrict__ cos_t, float* __restrict__ sin_t, int64_t S, int half,
                                  double base) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t n = S * half;
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < n;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t pos = t / half;
    const int i = static_cast<int>(t - pos * half);
    const double th = static_cast<double>(pos) * pow(base, -2.0 * i / (2.0 * half));
    double sv, cv;
    sincos(th, &sv, &cv);
    cos_t[t] = static_cast<float>(cv);
    sin_t[t] = static_cast<float>(sv);
  }
}

// standalone RoPE (rotate-half) in place; one thread per 8 pairs of a head
__global__ void rope_apply_kernel(__nv_bfloat16* __restrict__ qkv, const float* __restrict__ cos_t,
                                  const float* __restrict__ sin_t, int64_t M, int64_t N, int64_t rot_heads,
                                  int half, int64_t S) {
  griddep_wait();
  griddep_launch_dependents();
  const int g8 = half / 8;
  const int64_t n = M * rot_heads * g8;
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < n;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t m = t / (rot_heads * g8);
    const int64_t r = t - m * rot_heads * g8;
    const int64_t head = r / g8;
    const int i0 = static_cast<int>(r - head * g8) * 8;
    __nv_bfloat16* x = qkv + m * N + head * 2 * half;
    const float* cs = cos_t + (m % S) * half + i0;
    const float* sn = sin_t + (m % S) * half + i0;
    float a[8], b[8], o1[8], o2[8];
    unpack_bf16x8(*reinterpret_cast<const uint4*>(x + i0), a);
    unpack_bf16x8(*reinterpret_cast<const uint4*>(x + half + i0), b);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      o1[k] = fmaf(a[k], cs[k], -b[k] * sn[k]);
      o2[k] = fmaf(b[k], cs[k], a[k] * sn[k]);
    }
    *reinterpret_cast<uint4*>(x + i0) = pack8(o1);
    *reinterpret_cast<uint4*>(x + half + i0) = pack8(o2);
  }
}

// Per-tensor e4m3 quantisation, two passes over src [rows][cols] (times
// g[col] when g is given): the absolute maximum, then the codes.  Like the
// fold, a thread owns one 8-column chunk (its g values in registers) and
// kQuantRows rows of it, with all row loads issued before use.  Block maxima
// are combined with atomicMax on the bit patterns (non-negative floats order
// as integers).
constexpr int kQuantRows = 8;

// Per-tensor scale s = 2^k: the smallest power of two with amax / s <= fmax
// (fmax = 448 = 0.875 * 2^9 for e4m3, 57344 = 0.875 * 2^16 for e5m2), k at
// least -126; k = 0 for an all-zero tensor.  x / s = x * 2^-k is exact, so
// every element is rounded once, by the conversion.
template <bool E5M2>
__device__ __forceinline__ int fp8_scale_exp(float amax) {
  if (!(amax > 0.f)) return 0;
  int ea;
  const float ma = frexpf(amax, &ea);  // amax = ma * 2^ea, ma in [0.5, 1)
  const int k = ea - (E5M2 ? 16 : 9) + (ma > 0.875f ? 1 : 0);
  return k < -126 ? -126 : k;
}

// 2^k for -126 <= k <= 127
__device__ __forceinline__ float pow2f(int k) { return __uint_as_float(static_cast<uint32_t>(k + 127) << 23); }

// eight codes fp8(v[k] * inv), saturating round-to-nearest-even, packed in
// column order (two conversions per instruction)
template <bool E5M2>
__device__ __forceinline__ uint2 fp8_codes8(const float* v, float inv) {
  constexpr __nv_fp8_interpretation_t kind = E5M2 ? __NV_E5M2 : __NV_E4M3;
  uint32_t w[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * h] * inv, v[4 * h + 1] * inv), __NV_SATFINITE,
                                                 kind);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * h + 2] * inv, v[4 * h + 3] * inv),
                                                 __NV_SATFINITE, kind);
    w[h] = (lo & 0xFFFFu) | (hi << 16);
  }
  return make_uint2(w[0], w[1]);
}

__global__ void __launch_bounds__(256) amax_kernel(const uint4* __restrict__ src, const uint4* __restrict__ g8,
                                                   int64_t rows, int64_t c8, unsigned int* __restrict__ amax_bits) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[8];
  const int64_t j = blockIdx.x * 256LL + threadIdx.x;
  float mx = 0.f;
  if (j < c8) {
    float gg[8];
    if (g8 != nullptr) {
      unpack_bf16x8(__ldg(&g8[j]), gg);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) gg[k] = 1.f;
    }
    for (int64_t r0 = blockIdx.y * static_cast<int64_t>(kQuantRows); r0 < rows;
         r0 += static_cast<int64_t>(gridDim.y) * kQuantRows) {
      const int nr = static_cast<int>(rows - r0 < kQuantRows ? rows - r0 : kQuantRows);
      uint4 q[kQuantRows];
#pragma unroll
      for (int r = 0; r < kQuantRows; ++r)
        if (r < nr) q[r] = src[(r0 + r) * c8 + j];
#pragma unroll
      for (int r = 0; r < kQuantRows; ++r) {
        if (r < nr) {
          float v[8];
          unpack_bf16x8(q[r], v);
#pragma unroll
          for (int k = 0; k < 8; ++k) mx = fmaxf(mx, fabsf(v[k] * gg[k]));
        }
      }
    }
  }
  const float t = block_max_256(mx, red);
  if (threadIdx.x == 0) atomicMax(amax_bits, __float_as_uint(t));
}

// dst = fp8(src * g / s), s the power-of-two scale of fp8_scale_exp (the
// product src * g in fp32), fp8 = e4m3 or e5m2; saturating round-to-
// nearest-even conversion.  ws[1] receives s.
template <bool E5M2>
__global__ void __launch_bounds__(256) fp8_quantize_kernel(const uint4* __restrict__ src,
                                                           const uint4* __restrict__ g8, int64_t rows, int64_t c8,
                                                           float* __restrict__ ws, uint2* __restrict__ dst) {
  griddep_wait();
  griddep_launch_dependents();
  const int k = fp8_scale_exp<E5M2>(ws[0]);
  const float inv = pow2f(-k);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) ws[1] = pow2f(k);
  const int64_t j = blockIdx.x * 256LL + threadIdx.x;
  if (j >= c8) return;
  float gg[8];
  if (g8 != nullptr) {
    unpack_bf16x8(__ldg(&g8[j]), gg);
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) gg[k] = 1.f;
  }
  for (int64_t r0 = blockIdx.y * static_cast<int64_t>(kQuantRows); r0 < rows;
       r0 += static_cast<int64_t>(gridDim.y) * kQuantRows) {
    const int nr = static_cast<int>(rows - r0 < kQuantRows ? rows - r0 : kQuantRows);
    uint4 q[kQuantRows];
#pragma unroll
    for (int r = 0; r < kQuantRows; ++r)
      if (r < nr) q[r] = src[(r0 + r) * c8 + j];
#pragma unroll
    for (int r = 0; r < kQuantRows; ++r) {
      if (r < nr) {
        float v[8];
        unpack_bf16x8(q[r], v);
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) v[q8] *= gg[q8];
        dst[(r0 + r) * c8 + j] = fp8_codes8<E5M2>(v, inv);
      }
    }
  }
}

// The SwiGLU backward straight to 8-bit codes of dP, in two passes over dY
// and z so that the bf16 dP never reaches HBM (one CTA per row, as
// swiglu_bwd_kernel).  Pass 1 writes c and folds max |bf16(dP)| into
// amax_bits; pass 2 recomputes bf16(dP) and writes its codes.  The chunk
// arithmetic is swiglu_bwd_vals and the conversion fp8_codes8, so the codes
// equal those of swiglu_bwd_kernel's dP quantised by fp8_quantize_kernel.
__device__ __forceinline__ float absmax8(const float* v, float mx) {
#pragma unroll
  for (int k = 0; k < 8; ++k) mx = fmaxf(mx, fabsf(v[k]));
  return mx;
}

__global__ void __launch_bounds__(256) swiglu_bwd_amax_kernel(const __nv_bfloat16* __restrict__ dY,
                                                              const __nv_bfloat16* __restrict__ z,
                                                              const float* __restrict__ rstd,
                                                              float* __restrict__ cvec, int64_t F, float inv_d,
                                                              unsigned int* __restrict__ amax_bits) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[8];
  __shared__ float red_max[8];
  const int64_t m = blockIdx.x;
  const float r = rstd[m];
  const uint4* dy8 = reinterpret_cast<const uint4*>(dY + m * F);
  const uint4* zg8 = reinterpret_cast<const uint4*>(z + m * 2 * F);
  const uint4* zu8 = reinterpret_cast<const uint4*>(z + m * 2 * F + F);
  const int64_t F8 = F / 8;
  float dot = 0.f, mx = 0.f;
  for (int64_t j0 = threadIdx.x; j0 < F8; j0 += 2 * 256) {
    const int64_t j1 = j0 + 256;
    const bool two = j1 < F8;
    const uint4 a0 = dy8[j0], b0 = zg8[j0], c0 = zu8[j0];
    uint4 a1 = a0, b1 = b0, c1 = c0;
    if (two) {
      a1 = dy8[j1];
      b1 = zg8[j1];
      c1 = zu8[j1];
    }
    float og[8], ou[8];
    dot += swiglu_bwd_vals(a0, b0, c0, r, og, ou);
    mx = absmax8(ou, absmax8(og, mx));
    if (two) {
      dot += swiglu_bwd_vals(a1, b1, c1, r, og, ou);
      mx = absmax8(ou, absmax8(og, mx));
    }
  }
  const float tot = block_sum_256(dot, red);
  if (threadIdx.x == 0) cvec[m] = r * r * inv_d * tot;
  const float t = block_max_256(mx, red_max);
  // round-to-nearest-even is monotone and odd, so the bf16 of the largest
  // fp32 magnitude is the largest magnitude of the bf16 dP
  if (threadIdx.x == 0) atomicMax(amax_bits, __float_as_uint(__bfloat162float(__float2bfloat16_rn(t))));
}

template <bool E5M2>
__global__ void __launch_bounds__(256) swiglu_bwd_fp8_kernel(const __nv_bfloat16* __restrict__ dY,
                                                             const __nv_bfloat16* __restrict__ z,
                                                             const float* __restrict__ rstd, int64_t F,
                                                             float* __restrict__ ws, uint2* __restrict__ dPq) {
  griddep_wait();
  griddep_launch_dependents();
  const int k = fp8_scale_exp<E5M2>(ws[0]);
  const float inv = pow2f(-k);
  if (blockIdx.x == 0 && threadIdx.x == 0) ws[1] = pow2f(k);
  const int64_t m = blockIdx.x;
  const float r = rstd[m];
  const uint4* dy8 = reinterpret_cast<const uint4*>(dY + m * F);
  const uint4* zg8 = reinterpret_cast<const uint4*>(z + m * 2 * F);
  const uint4* zu8 = reinterpret_cast<const uint4*>(z + m * 2 * F + F);
  const int64_t F8 = F / 8;
  uint2* qg = dPq + m * 2 * F8;  // 8 codes per uint2: gate half, then up half
  uint2* qu = qg + F8;
  for (int64_t j0 = threadIdx.x; j0 < F8; j0 += 2 * 256) {
    const int64_t j1 = j0 + 256;
    const bool two = j1 < F8;
    const uint4 a0 = dy8[j0], b0 = zg8[j0], c0 = zu8[j0];
    uint4 a1 = a0, b1 = b0, c1 = c0;
    if (two) {
      a1 = dy8[j1];
      b1 = zg8[j1];
      c1 = zu8[j1];
    }
    uint4 pg, pu;
    float v[8];
    swiglu_bwd_chunk(a0, b0, c0, r, pg, pu);
    unpack_bf16x8(pg, v);
    qg[j0] = fp8_codes8<E5M2>(v, inv);
    unpack_bf16x8(pu, v);
    qu[j0] = fp8_codes8<E5M2>(v, inv);
    if (two) {
      swiglu_bwd_chunk(a1, b1, c1, r, pg, pu);
      unpack_bf16x8(pg, v);
      qg[j1] = fp8_codes8<E5M2>(v, inv);
      unpack_bf16x8(pu, v);
      qu[j1] = fp8_codes8<E5M2>(v, inv);
    }
  }
}

// Delayed scaling of dP's codes: the scale comes from the amax of the previous
// step's dP (state[0] on entry), so a single pass over dY and z writes c, the
// codes and this dP's amax (state[0] on exit, for the next step).  The codes
// saturate where this dP exceeds the previous range.
//   rotate: state[1] = 2^fp8_scale_exp(state[0]); state[0] = 0
//   pass:   codes = fp8(bf16(dP) / state[1]); state[0] = max |bf16(dP)|
template <bool E5M2>
__global__ void fp8_delayed_rotate_kernel(float* __restrict__ state) {
  griddep_wait();
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    state[1] = pow2f(fp8_scale_exp<E5M2>(state[0]));
    state[0] = 0.f;
  }
}

template <bool E5M2>
__global__ void __launch_bounds__(256) swiglu_bwd_fp8_delayed_kernel(const __nv_bfloat16* __restrict__ dY,
                                                                     const __nv_bfloat16* __restrict__ z,
                                                                     const float* __restrict__ rstd,
                                                                     float* __restrict__ cvec, int64_t F,
                                                                     float inv_d, float* __restrict__ state,
                                                                     uint2* __restrict__ dPq) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[8];
  __shared__ float red_max[8];
  // the scale is a power of two: its exponent gives the exact inverse
  int e;
  (void)frexpf(state[1], &e);
  const float inv = pow2f(1 - e);
  const int64_t m = blockIdx.x;
  const float r = rstd[m];
  const uint4* dy8 = reinterpret_cast<const uint4*>(dY + m * F);
  const uint4* zg8 = reinterpret_cast<const uint4*>(z + m * 2 * F);
  const uint4* zu8 = reinterpret_cast<const uint4*>(z + m * 2 * F + F);
  const int64_t F8 = F / 8;
  uint2* qg = dPq + m * 2 * F8;
  uint2* qu = qg + F8;
  float dot = 0.f, mx = 0.f;
  for (int64_t j0 = threadIdx.x; j0 < F8; j0 += 2 * 256) {
    const int64_t j1 = j0 + 256;
    const bool two = j1 < F8;
    const uint4 a0 = dy8[j0], b0 = zg8[j0], c0 = zu8[j0];
    uint4 a1 = a0, b1 = b0, c1 = c0;
    if (two) {
      a1 = dy8[j1];
      b1 = zg8[j1];
      c1 = zu8[j1];
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (h == 1 && !two) break;
      const int64_t j = h == 0 ? j0 : j1;
      float og[8], ou[8], v[8];
      dot += swiglu_bwd_vals(h == 0 ? a0 : a1, h == 0 ? b0 : b1, h == 0 ? c0 : c1, r, og, ou);
      mx = absmax8(ou, absmax8(og, mx));
      unpack_bf16x8(pack8(og), v);
      qg[j] = fp8_codes8<E5M2>(v, inv);
      unpack_bf16x8(pack8(ou), v);
      qu[j] = fp8_codes8<E5M2>(v, inv);
    }
  }
  const float tot = block_sum_256(dot, red);
  if (threadIdx.x == 0) cvec[m] = r * r * inv_d * tot;
  const float t = block_max_256(mx, red_max);
  if (threadIdx.x == 0)
    atomicMax(reinterpret_cast<unsigned int*>(state), __float_as_uint(__bfloat162float(__float2bfloat16_rn(t))));
}

// ---------------------------------------------------------------------------
// unfused ablation kernels

// h = bf16(A + R); rstd = 1/sqrt(mean h^2 + eps); Nrm = bf16(h * rstd * g)
__global__ void __launch_bounds__(256) add_rmsnorm_kernel(const __nv_bfloat16* __restrict__ A,
                                                          const __nv_bfloat16* __restrict__ R,
                                                          const __nv_bfloat16* __restrict__ g,
                                                          __nv_bfloat16* __restrict__ H, float* __restrict__ rstd,
                                                          __nv_bfloat16* __restrict__ Nrm, int64_t d, float eps) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[8];
  const int64_t m = blockIdx.x;
  const uint4* a8 = reinterpret_cast<const uint4*>(A + m * d);
  const uint4* r8 = reinterpret_cast<const uint4*>(R + m * d);
  uint4* h8 = reinterpret_cast<uint4*>(H + m * d);
  float ss = 0.f;
  for (int64_t j = threadIdx.x; j < d / 8; j += blockDim.x) {
    float a[8], r[8], h[8];
    unpack_bf16x8(a8[j], a);
    unpack_bf16x8(r8[j], r);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      h[i] = bf16_round(a[i] + r[i]);
      ss = fmaf(h[i], h[i], ss);
    }
    h8[j] = pack8(h);
  }
  const float tot = block_sum_256(ss, red);
  const float rs = 1.0f / sqrtf(tot / static_cast<float>(d) + eps);
  if (threadIdx.x == 0) rstd[m] = rs;
  const uint4* g8 = reinterpret_cast<const uint4*>(g);
  uint4* n8 = reinterpret_cast<uint4*>(Nrm + m * d);
  for (int64_t j = threadIdx.x; j < d / 8; j += blockDim.x) {
    float h[8], gg[8], o[8];
    unpack_bf16x8(h8[j], h);
    unpack_bf16x8(__ldg(&g8[j]), gg);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = h[i] * rs * gg[i];
    n8[j] = pack8(o);
  }
}

__global__ void swiglu_kernel(const __nv_bfloat16* __restrict__ z, __nv_bfloat16* __restrict__ out, int64_t M,
                              int64_t F) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t f8 = F / 8;
  const int64_t n = M * f8;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t m = i / f8, j = i - m * f8;
    float zg[8], zu[8], o[8];
    unpack_bf16x8(reinterpret_cast<const uint4*>(z + m * 2 * F)[j], zg);
    unpack_bf16x8(reinterpret_cast<const uint4*>(z + m * 2 * F + F)[j], zu);
#pragma unroll
    for (int k = 0; k < 8; ++k) o[k] = silu_f(zg[k]) * zu[k];
    reinterpret_cast<uint4*>(out + m * F)[j] = pack8(o);
  }
}

__global__ void swiglu_bwd_plain_kernel(const __nv_bfloat16* __restrict__ dY, const __nv_bfloat16* __restrict__ z,
                                        __nv_bfloat16* __restrict__ dZ, int64_t M, int64_t F) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t f8 = F / 8;
  const int64_t n = M * f8;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t m = i / f8, j = i - m * f8;
    float dy[8], zg[8], zu[8], og[8], ou[8];
    unpack_bf16x8(reinterpret_cast<const uint4*>(dY + m * F)[j], dy);
    unpack_bf16x8(reinterpret_cast<const uint4*>(z + m * 2 * F)[j], zg);
    unpack_bf16x8(reinterpret_cast<const uint4*>(z + m * 2 * F + F)[j], zu);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float s = sigmoid_f(zg[k]);
      og[k] = dy[k] * zu[k] * s * (1.0f + zg[k] * (1.0f - s));
      ou[k] = dy[k] * zg[k] * s;
    }
    reinterpret_cast<uint4*>(dZ + m * 2 * F)[j] = pack8(og);
    reinterpret_cast<uint4*>(dZ + m * 2 * F + F)[j] = pack8(ou);
  }
}

// textbook RMSNorm backward for one row per CTA:
//   dn = g * dN ; dh = r*dn - (r^3/d) * h * sum(dn*h)
__global__ void __launch_bounds__(256) rmsnorm_bwd_kernel(const __nv_bfloat16* __restrict__ dN,
                                                          const __nv_bfloat16* __restrict__ H,
                                                          const float* __restrict__ rstd,
                                                          const __nv_bfloat16* __restrict__ g,
                                                          __nv_bfloat16* __restrict__ dH, int64_t d) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[8];
  const int64_t m = blockIdx.x;
  const float r = rstd[m];
  const uint4* dn8 = reinterpret_cast<const uint4*>(dN + m * d);
  const uint4* h8 = reinterpret_cast<const uint4*>(H + m * d);
  const uint4* g8 = reinterpret_cast<const uint4*>(g);
  float dot = 0.f;
  for (int64_t j = threadIdx.x; j < d / 8; j += blockDim.x) {
    float a[8], h[8], gg[8];
    unpack_bf16x8(dn8[j], a);
    unpack_bf16x8(h8[j], h);
    unpack_bf16x8(__ldg(&g8[j]), gg);
#pragma unroll
    for (int i = 0; i < 8; ++i) dot = fmaf(a[i] * gg[i], h[i], dot);
  }
  const float tot = block_sum_256(dot, red);
  const float coef = r * r * r * tot / static_cast<float>(d);
  uint4* o8 = reinterpret_cast<uint4*>(dH + m * d);
  for (int64_t j = threadIdx.x; j < d / 8; j += blockDim.x) {
    float a[8], h[8], gg[8], o[8];
    unpack_bf16x8(dn8[j], a);
    unpack_bf16x8(h8[j], h);
    unpack_bf16x8(__ldg(&g8[j]), gg);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = r * gg[i] * a[i] - coef * h[i];
    o8[j] = pack8(o);
  }
}

// dgpart[p, k] = sum over rows [p*rows_per_part, ...) of dN[m,k] * h[m,k] * r[m]
__global__ void rmsnorm_bwd_dg_kernel(const __nv_bfloat16* __restrict__ dN, const __nv_bfloat16* __restrict__ H,
                                      const float* __restrict__ rstd, float* __restrict__ dgpart, int64_t M, int64_t d,
                                      int64_t rows_per_part) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[8][33];
  const int64_t k = blockIdx.x * 32 + threadIdx.x;
  const int64_t r0 = blockIdx.y * rows_per_part;
  const int64_t r1 = min(M, r0 + rows_per_part);
  float s = 0.f;
  if (k < d)
    for (int64_t m = r0 + threadIdx.y; m < r1; m += 8)
      s += __bfloat162float(dN[m * d + k]) * __bfloat162float(H[m * d + k]) * rstd[m];
  red[threadIdx.y][threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.y == 0 && k < d) {
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) t += red[i][threadIdx.x];
    dgpart[blockIdx.y * d + k] = t;
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// launchers
cudaError_t launch_fold(const LaunchCtx& c, const __nv_bfloat16* W2t, const __nv_bfloat16* g, __nv_bfloat16* W2gt,
                        int64_t N2, int64_t d) {
  const int64_t d8 = d / 8;
  // one CTA per block of kFoldRows rows (not a single balanced wave): the
  // fold usually runs beside GEMM1, where only a few of its CTAs fit per SM,
  // and there the finer grid measured faster
  const int64_t row_blocks = (N2 + kFoldRows - 1) / kFoldRows;
  const dim3 grid(static_cast<unsigned>((d8 + 255) / 256), static_cast<unsigned>(row_blocks < 65535 ? row_blocks : 65535));
  return launch_chained(c, fold_kernel, grid, dim3(256), 0, reinterpret_cast<const uint4*>(W2t),
                        reinterpret_cast<const uint4*>(g), reinterpret_cast<uint4*>(W2gt), N2, d8);
}

cudaError_t launch_rstd_combine(const LaunchCtx& c, const float* psum, int64_t M, int64_t T, int64_t d, float eps,
                                float* rstd) {
  const int rows_per_block = 8;
  const int64_t grid = (M + rows_per_block - 1) / rows_per_block;
  return launch_chained(c, rstd_combine_kernel, dim3(static_cast<unsigned>(grid)), dim3(32 * rows_per_block), 0, psum, M, T, 1.0f / static_cast<float>(d), eps, rstd);
}

cudaError_t launch_swiglu_bwd(const LaunchCtx& c, const __nv_bfloat16* dY, const __nv_bfloat16* z,
                              const float* rstd, __nv_bfloat16* dP, float* cvec, int64_t M, int64_t F, int64_t d) {
  return launch_chained(c, swiglu_bwd_kernel, dim3(static_cast<unsigned>(M)), dim3(256), 0, dY, z, rstd, dP, cvec, F,
                                                                    1.0f / static_cast<float>(d));
}

cudaError_t launch_col_combine(const LaunchCtx& c, const float* part, int64_t rows, int64_t d, float* out) {
  return launch_chained(c, col_combine_kernel, dim3(static_cast<unsigned>((d + 31) / 32)), dim3(dim3(32, 8)), 0, part, rows, d, out);
}

cudaError_t launch_ce_combine(const LaunchCtx& c, const float* pmax, const float* psum, const int32_t* parg,
                              const float* zy, const int32_t* labels, int64_t M, int64_t T, int64_t V, float* lse,
                              int32_t* argmax, float* row_loss) {
  const int rows_per_block = 8;
  return launch_chained(c, ce_combine_kernel, dim3(static_cast<unsigned>((M + rows_per_block - 1) / rows_per_block)), dim3(32 * rows_per_block), 0, pmax, psum, parg, zy, labels, M, T, V, lse, argmax, row_loss, c.status);
}

cudaError_t launch_mean(const LaunchCtx& c, const float* v, int64_t n, float* out) {
  return launch_chained(c, mean_kernel, dim3(1), dim3(1024), 0, v, n, out);
}

cudaError_t launch_f32_to_bf16(const LaunchCtx& c, const float* in, __nv_bfloat16* out, int64_t n) {
  const int64_t n4 = n / 4;
  return launch_chained(c, f32_to_bf16_kernel, dim3(grid_for(c, n4, 256)), dim3(256), 0, reinterpret_cast<const float4*>(in),
                                                                 reinterpret_cast<uint2*>(out), n4);
}

cudaError_t launch_rope_table(const LaunchCtx& c, float* cos_t, float* sin_t, int64_t S, int64_t head_dim,
                              double base) {
  const int half = static_cast<int>(head_dim / 2);
  return launch_chained(c, rope_table_kernel, dim3(grid_for(c, S * half, 256)), dim3(256), 0, cos_t, sin_t, S, half,
                        base);
}

cudaError_t launch_rope_apply(const LaunchCtx& c, __nv_bfloat16* qkv, const float* cos_t, const float* sin_t,
                              int64_t M, int64_t N, int64_t rot_cols, int64_t head_dim, int64_t S) {
  const int half = static_cast<int>(head_dim / 2);
  const int64_t rot_heads = rot_cols / head_dim;
  return launch_chained(c, rope_apply_kernel, dim3(grid_for(c, M * rot_heads * (half / 8), 256)), dim3(256), 0, qkv,
                        cos_t, sin_t, M, N, rot_heads, half, S);
}

cudaError_t launch_fp8_quantize(const LaunchCtx& c, const __nv_bfloat16* src, int64_t rows, int64_t cols,
                                const __nv_bfloat16* g, float* ws, uint8_t* dst, int e5m2) {
  const int64_t c8 = cols / 8;
  cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(float), c.stream);
  if (e != cudaSuccess) return e;
  const uint4* g8 = reinterpret_cast<const uint4*>(g);
  const dim3 grid = chunk_rows_grid(c, c8, rows, kQuantRows);
  e = launch_chained(c, amax_kernel, grid, dim3(256), 0, reinterpret_cast<const uint4*>(src), g8, rows, c8,
                     reinterpret_cast<unsigned int*>(ws));
  if (e != cudaSuccess) return e;
  return launch_chained(c, e5m2 ? fp8_quantize_kernel<true> : fp8_quantize_kernel<false>, grid, dim3(256), 0,
                        reinterpret_cast<const uint4*>(src), g8, rows, c8, ws, reinterpret_cast<uint2*>(dst));
}

cudaError_t launch_swiglu_bwd_fp8(const LaunchCtx& c, const __nv_bfloat16* dY, const __nv_bfloat16* z,
                                  const float* rstd, float* ws, uint8_t* dPq, float* cvec, int64_t M, int64_t F,
                                  int64_t d, int e5m2) {
  cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(float), c.stream);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(M));
  e = launch_chained(c, swiglu_bwd_amax_kernel, grid, dim3(256), 0, dY, z, rstd, cvec, F,
                     1.0f / static_cast<float>(d), reinterpret_cast<unsigned int*>(ws));
  if (e != cudaSuccess) return e;
  return launch_chained(c, e5m2 ? swiglu_bwd_fp8_kernel<true> : swiglu_bwd_fp8_kernel<false>, grid, dim3(256), 0, dY,
                        z, rstd, F, ws, reinterpret_cast<uint2*>(dPq));
}

cudaError_t launch_swiglu_bwd_fp8_delayed(const LaunchCtx& c, const __nv_bfloat16* dY, const __nv_bfloat16* z,
                                          const float* rstd, float* state, uint8_t* dPq, float* cvec, int64_t M,
                                          int64_t F, int64_t d, int e5m2) {
  cudaError_t e = launch_chained(c, e5m2 ? fp8_delayed_rotate_kernel<true> : fp8_delayed_rotate_kernel<false>,
                                 dim3(1), dim3(32), 0, state);
  if (e != cudaSuccess) return e;
  return launch_chained(c, e5m2 ? swiglu_bwd_fp8_delayed_kernel<true> : swiglu_bwd_fp8_delayed_kernel<false>,
                        dim3(static_cast<unsigned>(M)), dim3(256), 0, dY, z, rstd, cvec, F,
                        1.0f / static_cast<float>(d), state, reinterpret_cast<uint2*>(dPq));
}

cudaError_t launch_add_rmsnorm(const LaunchCtx& c, const __nv_bfloat16* A, const __nv_bfloat16* R,
                               const __nv_bfloat16* g, __nv_bfloat16* H, float* rstd, __nv_bfloat16* Nrm, int64_t M,
                               int64_t d, float eps) {
  return launch_chained(c, add_rmsnorm_kernel, dim3(static_cast<unsigned>(M)), dim3(256), 0, A, R, g, H, rstd, Nrm, d, eps);
}

cudaError_t launch_swiglu(const LaunchCtx& c, const __nv_bfloat16* z, __nv_bfloat16* out, int64_t M, int64_t F) {
  return launch_chained(c, swiglu_kernel, dim3(grid_for(c, M * F / 8, 256)), dim3(256), 0, z, out, M, F);
}

cudaError_t launch_swiglu_bwd_plain(const LaunchCtx& c, const __nv_bfloat16* dY, const __nv_bfloat16* z,
                                    __nv_bfloat16* dZ, int64_t M, int64_t F) {
  return launch_chained(c, swiglu_bwd_plain_kernel, dim3(grid_for(c, M * F / 8, 256)), dim3(256), 0, dY, z, dZ, M, F);
}

cudaError_t launch_rmsnorm_bwd(const LaunchCtx& c, const __nv_bfloat16* dN, const __nv_bfloat16* H,
                               const float* rstd, const __nv_bfloat16* g, __nv_bfloat16* dH, int64_t M, int64_t d) {
  return launch_chained(c, rmsnorm_bwd_kernel, dim3(static_cast<unsigned>(M)), dim3(256), 0, dN, H, rstd, g, dH, d);
}

cudaError_t launch_rmsnorm_bwd_dg(const LaunchCtx& c, const __nv_bfloat16* dN, const __nv_bfloat16* H,
                                  const float* rstd, float* dgpart, int64_t M, int64_t d, int64_t rows_per_part) {
  const dim3 grid(static_cast<unsigned>((d + 31) / 32),
                  static_cast<unsigned>((M + rows_per_part - 1) / rows_per_part));
  return launch_chained(c, rmsnorm_bwd_dg_kernel, dim3(grid), dim3(dim3(32, 8)), 0, dN, H, rstd, dgpart, M, d, rows_per_part);
}

}  // namespace coda
