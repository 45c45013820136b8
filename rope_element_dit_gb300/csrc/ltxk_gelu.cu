// ltxk_gelu.cu -- tanh-approximated GELU and GEGLU, bf16 in and out.
//
// "cuda-kernels" skill page (Hugging Face), "Kernel-Specific Guidelines /
// GEGLU vs GELU": LTX-Video uses the tanh approximation ("gelu-approximate");
// GEGLU maps [.., 2h] -> [.., h].  Definition implemented:
//   gelu(x) = x/2 (1 + tanh(z)),  z = sqrt(2/pi) (x + 0.044715 x^3),
//   geglu(x)[j] = x[j] * gelu(x[h + j])   (value first, gate second).
// Evaluated in fp32 as the logistic form of the same function:
//   (1 + tanh z)/2 = 2^q / (1 + 2^q),   q = (2/ln 2) z = x (c0 + c1 x^2),
//   c0 = (2/ln 2) sqrt(2/pi),  c1 = 0.044715 c0,
// so gelu(x) = x * s / (1 + s) with s = 2^q.  1 + s adds two positive terms
// (no cancellation).  s is formed as 2^(min(q, 63) + 64) * 2^-64: the PTX
// ex2.approx instruction (relative error ~2^-22) then never flushes a result
// that fp32 can hold, the exact power-of-two product rounds it once into the
// subnormal range, and q > 63 (where s/(1+s) rounds to 1) cannot overflow.
// rcp.approx (1 ulp) gives 1/(1+s).  The fp32 value stays within ~2e-5
// relative of the exact one, far inside half a bf16 spacing (2^-9), for
// every bf16 input: no branch, no select.
//
// GEGLU multiplies by the value v.  Only where s < 2^-139 (q < -139) does s
// keep fewer than 10 significant bits, which a |v| >= 2 could lift into the
// bf16 range; those elements take an exact path that forms v * x * 2^q from
// frexp(v), the fractional power of two of the exponent sum and one exact
// ldexp.  Whether an element takes it depends only on the element, so every
// kernel gives the same bits.
//
// Memory-bound streams: every 16-byte vector is read once and written once,
// two vectors per thread in flight; a scalar kernel covers ragged tails and
// pointers that are not 16-byte aligned.  The vector path runs on packed
// f32x2 arithmetic.
#include <cuda_runtime.h>

#include <cstdint>

#include "ltxk.h"
#include "ltxk_kernels.cuh"
#include "ltxk_launch.h"

namespace {

#ifndef LTXK_GELU_VEC_PER_THREAD
#define LTXK_GELU_VEC_PER_THREAD 2
#endif
constexpr int kBlock = 256;
constexpr int kVecPerThread = LTXK_GELU_VEC_PER_THREAD;
constexpr int64_t kMaxElements = int64_t{1} << 40;   // keeps every grid below 2^31 blocks

constexpr float kQ0 = 2.3022082f;                    // (2 / ln 2) * sqrt(2 / pi)
constexpr float kQ1 = 2.3022082f * 0.044715f;
constexpr float kShift = 64.f;                       // s = 2^(q + 64) * 2^-64
constexpr float kUnshift = 5.42101086242752217e-20f; // 2^-64
constexpr float kMaxQ64 = 127.f;                     // q + 64 clamped: 2^127 is finite
constexpr float kDeepQ64 = -139.f + kShift;          // s < 2^-139: fewer than 10 bits

__device__ __forceinline__ float ex2_approx(float a) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
  return r;
}

__device__ __forceinline__ float rcp_approx(float a) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
  return r;
}

// q = (2 / ln 2) z, so that e^{2z} = 2^q (q has the sign of x); q + 64.
__device__ __forceinline__ float q_of(float x) { return x * __fmaf_rn(kQ1, x * x, kQ0); }
__device__ __forceinline__ float q64_of(float x) {
  return __fmaf_rn(x, __fmaf_rn(kQ1, x * x, kQ0), kShift);
}

__device__ __forceinline__ float2 q64_of2(float2 x) {
  const float2 p = __ffma2_rn(__fmul2_rn(x, x), make_float2(kQ1, kQ1), make_float2(kQ0, kQ0));
  return __ffma2_rn(x, p, make_float2(kShift, kShift));
}

// x * s / (1 + s), s = 2^q.
__device__ __forceinline__ float gelu_fast(float x, float q64) {
  const float e = ex2_approx(fminf(q64, kMaxQ64));
  const float r = rcp_approx(__fmaf_rn(e, kUnshift, 1.f));
  return (x * r) * (e * kUnshift);
}

__device__ __forceinline__ float2 gelu_fast2(float2 x, float2 q64) {
  const float2 e = make_float2(ex2_approx(fminf(q64.x, kMaxQ64)), ex2_approx(fminf(q64.y, kMaxQ64)));
  const float2 d = __ffma2_rn(e, make_float2(kUnshift, kUnshift), make_float2(1.f, 1.f));
  const float2 r = make_float2(rcp_approx(d.x), rcp_approx(d.y));
  return __fmul2_rn(__fmul2_rn(x, r), __fmul2_rn(e, make_float2(kUnshift, kUnshift)));
}

// v * gelu(x) exactly scaled, for q < -139 (there 1 + 2^q == 1 in fp32).
__device__ __noinline__ float gelu_deep(float x, float v) {
  const float q = q_of(x);
  if (q == -INFINITY) return v * (x * 0.f);   // x = -inf gives NaN, as -inf*0 does
  int ev;
  const float mv = frexpf(v, &ev);            // v = mv * 2^ev
  const float u = fmaxf(static_cast<float>(ev) + q, -320.f);
  const float n = floorf(u);
  return ldexpf(mv * x * exp2f(u - n), static_cast<int>(n));
}

__device__ __forceinline__ bool needs_deep(float q64, float v) {
  return q64 < kDeepQ64 && fabsf(v) >= 2.f;
}

// v * gelu(x), one element (v == 1: the plain activation, never deep).
__device__ __forceinline__ float gelu_pick(float x, float v) {
  const float q64 = q64_of(x);
  return needs_deep(q64, v) ? gelu_deep(x, v) : v * gelu_fast(x, q64);
}

// Eight elements: x and (GEGLU) the values v, as bf16 vectors.
template <bool kGated>
__device__ __forceinline__ uint4 gelu8(uint4 xv, uint4 vv) {
  const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
  const uint32_t vs[4] = {vv.x, vv.y, vv.z, vv.w};
  float2 x[4], q64[4], v[4];
  bool deep = false;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[k] = ltxk::bf2_of(xs[k]);
    q64[k] = q64_of2(x[k]);
    if (kGated) {
      v[k] = ltxk::bf2_of(vs[k]);
      deep |= needs_deep(q64[k].x, v[k].x) | needs_deep(q64[k].y, v[k].y);
    }
  }
  uint32_t o[4];
  if (kGated && deep) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      o[k] = ltxk::pack_bf2(gelu_pick(x[k].x, v[k].x), gelu_pick(x[k].y, v[k].y));
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 y = gelu_fast2(x[k], q64[k]);
      if (kGated) y = __fmul2_rn(v[k], y);
      o[k] = ltxk::pack_f2(y);
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// n_vec 16-byte vectors of x -> y.
__global__ void __launch_bounds__(kBlock) gelu_vec_kernel(uint16_t* y, const uint16_t* x,
                                                          int64_t n_vec) {
  const int64_t base = (static_cast<int64_t>(blockIdx.x) * kBlock * kVecPerThread) + threadIdx.x;
  uint4 v[kVecPerThread];
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const int64_t i = base + k * kBlock;
    v[k] = i < n_vec ? ltxk::ld_stream16(x + i * 8) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const int64_t i = base + k * kBlock;
    if (i < n_vec)
      ltxk::st16(y + i * 8, gelu8<false>(v[k], v[k]));
  }
}

__global__ void __launch_bounds__(kBlock) gelu_elem_kernel(uint16_t* y, const uint16_t* x,
                                                           int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; i < n; i += stride) {
    const float xf = ltxk::bf_to_f(x[i]);
    y[i] = ltxk::f_to_bf(gelu_pick(xf, 1.f));
  }
}

// x [rows, 2h], y [rows, h]; hv = h / 8 vectors per output row.  Index is
// uint32_t whenever rows * hv fits, which keeps the row division short.
template <typename Index>
__global__ void __launch_bounds__(kBlock) geglu_vec_kernel(uint16_t* y, const uint16_t* x,
                                                           Index n_vec, Index hv) {
  const Index base = static_cast<Index>(blockIdx.x) * (kBlock * kVecPerThread) + threadIdx.x;
  uint4 val[kVecPerThread], gate[kVecPerThread];
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const Index i = base + k * kBlock;
    if (i < n_vec) {
      const Index r = i / hv;
      const uint16_t* xv = x + (static_cast<int64_t>(i) + static_cast<int64_t>(r) * hv) * 8;
      val[k] = ltxk::ld_stream16(xv);
      gate[k] = ltxk::ld_stream16(xv + static_cast<int64_t>(hv) * 8);
    } else {
      val[k] = gate[k] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const Index i = base + k * kBlock;
    if (i < n_vec)
      ltxk::st16(y + static_cast<int64_t>(i) * 8, gelu8<true>(gate[k], val[k]));
  }
}

__global__ void __launch_bounds__(kBlock) geglu_elem_kernel(uint16_t* y, const uint16_t* x,
                                                            int64_t rows, int64_t h) {
  const int64_t n = rows * h;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; i < n; i += stride) {
    const int64_t r = i / h, j = i - r * h;
    const float v = ltxk::bf_to_f(x[r * 2 * h + j]);
    const float g = ltxk::bf_to_f(x[r * 2 * h + h + j]);
    y[i] = ltxk::f_to_bf(gelu_pick(g, v));
  }
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlaps(const void* a, uint64_t na, const void* b, uint64_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return na && nb && a0 < b0 + nb && b0 < a0 + na;
}

int fail(cudaError_t e) {
  ltxk::record_cuda_error(static_cast<int>(e));
  return LTXK_ERR_CUDA;
}

unsigned vec_grid(int64_t n_vec) {
  return static_cast<unsigned>((n_vec + kBlock * kVecPerThread - 1) / (kBlock * kVecPerThread));
}

unsigned elem_grid(int64_t n) {
  const int64_t g = (n + kBlock - 1) / kBlock;
  return static_cast<unsigned>(g < 65536 ? g : 65536);   // grid-stride beyond
}

}  // namespace

extern "C" int ltxk_gelu_tanh(void* out, const void* x, int64_t n, ltxk_stream_t stream) {
  if (out == nullptr || x == nullptr) return LTXK_ERR_NULL;
  if (n < 0 || n > kMaxElements) return LTXK_ERR_SHAPE;
  if (!aligned_to(out, 2) || !aligned_to(x, 2)) return LTXK_ERR_ALIGN;
  const uint64_t bytes = static_cast<uint64_t>(n) * 2;
  if (out != x && overlaps(out, bytes, x, bytes)) return LTXK_ERR_OVERLAP;
  if (n == 0) return LTXK_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint16_t* y = static_cast<uint16_t*>(out);
  const uint16_t* xi = static_cast<const uint16_t*>(x);
  int64_t done = 0;
  if (aligned_to(out, 16) && aligned_to(x, 16)) {
    const int64_t n_vec = n / 8;
    if (n_vec > 0) {
      gelu_vec_kernel<<<vec_grid(n_vec), kBlock, 0, s>>>(y, xi, n_vec);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return fail(e);
    }
    done = n_vec * 8;
  }
  if (done < n) {
    gelu_elem_kernel<<<elem_grid(n - done), kBlock, 0, s>>>(y + done, xi + done, n - done);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(e);
  }
  return LTXK_OK;
}

extern "C" int ltxk_geglu(void* out, const void* x, int64_t rows, int64_t hidden,
                          ltxk_stream_t stream) {
  if (out == nullptr || x == nullptr) return LTXK_ERR_NULL;
  if (rows < 0 || hidden <= 0 || hidden > LTXK_MAX_HIDDEN) return LTXK_ERR_SHAPE;
  if (rows > kMaxElements / hidden) return LTXK_ERR_SHAPE;
  if (!aligned_to(out, 2) || !aligned_to(x, 2)) return LTXK_ERR_ALIGN;
  if (overlaps(out, static_cast<uint64_t>(rows) * hidden * 2, x,
               static_cast<uint64_t>(rows) * hidden * 4))
    return LTXK_ERR_OVERLAP;
  if (rows == 0) return LTXK_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint16_t* y = static_cast<uint16_t*>(out);
  const uint16_t* xi = static_cast<const uint16_t*>(x);
  if (hidden % 8 == 0 && aligned_to(out, 16) && aligned_to(x, 16)) {
    const int64_t hv = hidden / 8, n_vec = rows * hv;
    if (n_vec + kBlock * kVecPerThread < (int64_t{1} << 32))
      geglu_vec_kernel<uint32_t><<<vec_grid(n_vec), kBlock, 0, s>>>(
          y, xi, static_cast<uint32_t>(n_vec), static_cast<uint32_t>(hv));
    else
      geglu_vec_kernel<int64_t><<<vec_grid(n_vec), kBlock, 0, s>>>(y, xi, n_vec, hv);
  } else {
    geglu_elem_kernel<<<elem_grid(rows * hidden), kBlock, 0, s>>>(y, xi, rows, hidden);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(e);
  return LTXK_OK;
}
