// ltxk_gelu.cu -- tanh-approximated GELU and GEGLU, bf16 in and out.
//
// "cuda-kernels" skill page (Hugging Face), "Kernel-Specific Guidelines /
// GEGLU vs GELU": LTX-Video uses the tanh approximation ("gelu-approximate");
// GEGLU maps [.., 2h] -> [.., h].  Definition implemented:
//   gelu(x) = x/2 (1 + tanh(z)),  z = sqrt(2/pi) (x + 0.044715 x^3),
//   geglu(x)[j] = x[j] * gelu(x[h + j])   (value first, gate second).
// Evaluated in fp32 through (1 + tanh z)/2 = sigma(2z) = 1/(1 + e^{-2z}),
// written with e = exp(-2|z|) so that it never overflows and never cancels:
//   sigma(2z) = 1/(1+e) for z >= 0,  e/(1+e) for z < 0.
// __expf (ex2-based, relative error a few 1e-6 at |2z| <= 45) and
// __fdividef (2 ulp) keep the fp32 value within ~1e-5 relative of the exact
// one, far inside half a bf16 spacing (2^-9).
//
// Far negative tail (z < -22.18, i.e. e^{2z} < 2^-64): there e^{2z} leaves
// the fp32 normal range long before v * x * e^{2z} leaves bf16's, so the
// product is formed from frexp(v), the fractional power of two of its
// exponent sum and one exact ldexp: no flush to zero, no early overflow.
//
// Memory-bound streams: every 16-byte vector is read once and written once,
// two vectors per thread in flight; a scalar kernel covers ragged tails and
// pointers that are not 16-byte aligned.
#include <cuda_runtime.h>

#include <cstdint>

#include "ltxk.h"
#include "ltxk_kernels.cuh"
#include "ltxk_launch.h"

namespace {

constexpr int kBlock = 256;
constexpr int kVecPerThread = 2;

constexpr int64_t kMaxElements = int64_t{1} << 40;   // keeps every grid below 2^31 blocks

constexpr float kSqrt2OverPi = 0.7978845608028654f;
constexpr float kCubic = 0.044715f;
constexpr float kTwoLog2e = 2.8853900817779268f;   // 2 / ln 2
constexpr float kTailZ = -22.180709777918249f;     // e^{2z} = 2^-64

// v * gelu(x) in fp32 (v = 1 for the plain activation).
__device__ __forceinline__ float gelu_times(float x, float v) {
  const float z = kSqrt2OverPi * __fmaf_rn(kCubic * x * x, x, x);
  if (!(z < kTailZ)) {                      // also NaN
    const float e = __expf(-2.f * fabsf(z));
    const float r = __fdividef(1.f, 1.f + e);
    const float s = z >= 0.f ? r : e * r;
    return v * (x * s);
  }
  // z < -22.18: 1 + e^{2z} == 1 in fp32, so v*gelu(x) = v * x * 2^{-t}.
  const float t = -kTwoLog2e * z;
  if (t == INFINITY) return v * (x * 0.f);  // x = -inf gives NaN, as -inf*0 does
  int ev;
  const float mv = frexpf(v, &ev);          // v = mv * 2^ev
  const float u = fmaxf(static_cast<float>(ev) - t, -320.f);
  const float n = floorf(u);
  return ldexpf(mv * x * exp2f(u - n), static_cast<int>(n));
}

__device__ __forceinline__ uint32_t gelu_word(uint32_t u) {
  return ltxk::pack_bf2(gelu_times(ltxk::bf_lo(u), 1.f), gelu_times(ltxk::bf_hi(u), 1.f));
}

__device__ __forceinline__ uint32_t geglu_word(uint32_t val, uint32_t gate) {
  return ltxk::pack_bf2(gelu_times(ltxk::bf_lo(gate), ltxk::bf_lo(val)),
                        gelu_times(ltxk::bf_hi(gate), ltxk::bf_hi(val)));
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
      ltxk::st16(y + i * 8, make_uint4(gelu_word(v[k].x), gelu_word(v[k].y),
                                       gelu_word(v[k].z), gelu_word(v[k].w)));
  }
}

__global__ void __launch_bounds__(kBlock) gelu_elem_kernel(uint16_t* y, const uint16_t* x,
                                                           int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; i < n; i += stride)
    y[i] = ltxk::f_to_bf(gelu_times(ltxk::bf_to_f(x[i]), 1.f));
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
      ltxk::st16(y + static_cast<int64_t>(i) * 8,
                 make_uint4(geglu_word(val[k].x, gate[k].x), geglu_word(val[k].y, gate[k].y),
                            geglu_word(val[k].z, gate[k].z), geglu_word(val[k].w, gate[k].w)));
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
    y[i] = ltxk::f_to_bf(gelu_times(g, v));
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
