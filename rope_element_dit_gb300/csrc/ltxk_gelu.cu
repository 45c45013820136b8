// ltxk_gelu.cu -- tanh-approximated GELU and GEGLU; bf16, fp16 or fp32 in
// and out (the element format is a template argument of every kernel).
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
// fp16 uses the same form (its outputs are far coarser; v * x * 2^q below
// 2^-119 rounds to zero there, so no element needs the exact path).  fp32
// avoids the offset where it costs accuracy: q + 64 carries a rounding error
// of up to 2^-18 for small |q|, a relative error of ~2^-18 that fp32 output
// would show.  There s is
// 2^q itself while q >= -64, and 2^(q + 64) with a final exact scaling by
// 2^-64 below (q + 64 is exact for q in [-128, -64]), the last product
// rounding once into the subnormal range; q is clamped to 126 so that
// 1/(1 + s) stays normal.  The fp32 GEGLU multiplies v * x before the
// normal-range factor s / (1 + s), so that a subnormal gate under a large
// value keeps its bits, and takes the exact path where gelu(x) is below the
// smallest normal (q < -126) and |v| >= 2.
//
// Memory-bound streams: every 16-byte slot (8 bf16/fp16 values, or a chunk
// of 4 fp32 values) is read once and written once, 16-byte accesses of
// consecutive lanes adjacent in every instruction; a scalar kernel covers ragged tails and
// pointers that are not 16-byte aligned.  The vector path runs on packed
// f32x2 arithmetic.
#include <cuda_runtime.h>

#include <cstdint>

#include "ltxk.h"
#include "ltxk_kernels.cuh"
#include "ltxk_launch.h"

namespace {

using ltxk::Io;
using ltxk::kBf16;
using ltxk::kF16;
using ltxk::kF32;

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
constexpr float kMaxQ32 = 126.f;                     // fp32: 1 / (1 + 2^126) is normal
constexpr float kDeepQ32 = -126.f;                   // fp32: gelu(x) below the normals

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

// The argument each format's fast form starts from: q + 64 (bf16, fp16) or
// q (fp32).
template <int FMT>
__device__ __forceinline__ float qarg(float x) {
  if constexpr (FMT == kF32) return q_of(x);
  else return q64_of(x);
}

template <int FMT>
__device__ __forceinline__ float2 qarg2(float2 x) {
  const float2 p = __ffma2_rn(__fmul2_rn(x, x), make_float2(kQ1, kQ1), make_float2(kQ0, kQ0));
  if constexpr (FMT == kF32) return __fmul2_rn(x, p);
  else return __ffma2_rn(x, p, make_float2(kShift, kShift));
}

// fp32: v * x * s / (1 + s), s = 2^q.  sigma' = s / (1 + s) is formed in
// the normal range: as itself for q >= -64, else as 2^64 s / (1 + s) with
// sc = 2^-64 applied last, so that a subnormal result is rounded once.  v * x
// comes first, so that a tiny (subnormal) x is not rounded before a large v
// scales it up; when v * x overflows, v is large, v * sc is exact and
// x * sigma' normal, and the product is taken in that order.
__device__ __forceinline__ float gelu_f32(float x, float q, float v) {
  const bool lo = q < -kShift;
  const float e = ex2_approx(fminf(lo ? q + kShift : q, kMaxQ32));
  const float sc = lo ? kUnshift : 1.f;
  const float sig = e * rcp_approx(__fmaf_rn(e, sc, 1.f));
  const float vx = v * x;
  return fabsf(vx) <= 3.40282347e38f ? (vx * sig) * sc : (v * sc) * (x * sig);
}

// x * s / (1 + s), s = 2^q, from qa = q + 64 (bf16, fp16).
__device__ __forceinline__ float gelu_fast(float x, float qa) {
  const float e = ex2_approx(fminf(qa, kMaxQ64));
  const float r = rcp_approx(__fmaf_rn(e, kUnshift, 1.f));
  return (x * r) * (e * kUnshift);
}

// v * gelu(x) by each format's fast form, from qa = qarg<FMT>(x).
template <int FMT>
__device__ __forceinline__ float gelu_val(float x, float qa, float v) {
  if constexpr (FMT == kF32) return gelu_f32(x, qa, v);
  else return v * gelu_fast(x, qa);
}

// Two elements of the bf16 / fp16 fast form on packed f32x2 arithmetic.
__device__ __forceinline__ float2 gelu_fast2(float2 x, float2 qa) {
  {
    const float2 e = make_float2(ex2_approx(fminf(qa.x, kMaxQ64)), ex2_approx(fminf(qa.y, kMaxQ64)));
    const float2 d = __ffma2_rn(e, make_float2(kUnshift, kUnshift), make_float2(1.f, 1.f));
    const float2 r = make_float2(rcp_approx(d.x), rcp_approx(d.y));
    return __fmul2_rn(__fmul2_rn(x, r), __fmul2_rn(e, make_float2(kUnshift, kUnshift)));
  }
}

// v * gelu(x) exactly scaled, for q below the fast form's range (there
// 1 + 2^q == 1 in fp32).
__device__ __noinline__ float gelu_deep(float x, float v) {
  const float q = q_of(x);
  if (q == -INFINITY) return v * (x * 0.f);   // x = -inf gives NaN, as -inf*0 does
  int ev;
  const float mv = frexpf(v, &ev);            // v = mv * 2^ev
  const float u = fmaxf(static_cast<float>(ev) + q, -320.f);
  const float n = floorf(u);
  return ldexpf(mv * x * exp2f(u - n), static_cast<int>(n));
}

// Whether v * gelu(x) needs the exact path.  fp16: never (v * x * 2^q is
// below 2^-119 wherever s has lost bits, and rounds to zero in fp16).
template <int FMT>
__device__ __forceinline__ bool needs_deep(float qa, float v) {
  if constexpr (FMT == kF16) return false;
  else if constexpr (FMT == kF32) return qa < kDeepQ32 && fabsf(v) >= 2.f;
  else return qa < kDeepQ64 && fabsf(v) >= 2.f;
}

// v * gelu(x), one element (v == 1: the plain activation, never deep).
template <int FMT>
__device__ __forceinline__ float gelu_pick(float x, float v) {
  const float qa = qarg<FMT>(x);
  return needs_deep<FMT>(qa, v) ? gelu_deep(x, v) : gelu_val<FMT>(x, qa, v);
}

// Eight elements: x and (GEGLU) the values v, as 16-byte slots of a 16-bit
// format.
template <int FMT, bool kGated>
__device__ __forceinline__ typename Io<FMT>::Vec gelu8(const typename Io<FMT>::Vec& xv,
                                                       const typename Io<FMT>::Vec& vv) {
  static_assert(FMT != kF32, "fp32 runs on 4-element chunks");
  using I = Io<FMT>;
  float2 x[4], qa[4], v[4];
  bool deep = false;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[k] = I::pair(xv, k);
    qa[k] = qarg2<FMT>(x[k]);
    if (kGated) {
      v[k] = I::pair(vv, k);
      deep |= needs_deep<FMT>(qa[k].x, v[k].x) | needs_deep<FMT>(qa[k].y, v[k].y);
    }
  }
  float2 o[4];
  if (kGated && deep) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      o[k] = make_float2(gelu_pick<FMT>(x[k].x, v[k].x), gelu_pick<FMT>(x[k].y, v[k].y));
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      o[k] = gelu_fast2(x[k], qa[k]);
      if (kGated) o[k] = __fmul2_rn(v[k], o[k]);
    }
  }
  return I::pack(o[0], o[1], o[2], o[3]);
}

// n_vec 8-element slots of x -> y.
template <int FMT>
__global__ void __launch_bounds__(kBlock) gelu_vec_kernel(void* y, const void* x, int64_t n_vec) {
  using I = Io<FMT>;
  const int64_t base = (static_cast<int64_t>(blockIdx.x) * kBlock * kVecPerThread) + threadIdx.x;
  typename I::Vec v[kVecPerThread];
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const int64_t i = base + k * kBlock;
    v[k] = i < n_vec ? I::load(x, i * 8) : typename I::Vec{};
  }
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const int64_t i = base + k * kBlock;
    if (i < n_vec) I::store(y, i * 8, gelu8<FMT, false>(v[k], v[k]));
  }
}

template <int FMT>
__global__ void __launch_bounds__(kBlock) gelu_elem_kernel(void* y, const void* x, int64_t n) {
  using I = Io<FMT>;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; i < n; i += stride)
    I::put(y, i, gelu_pick<FMT>(I::get(x, i), 1.f));
}

// x [rows, 2h], y [rows, h]; hv = h / 8 slots per output row.  Index is
// uint32_t whenever rows * hv fits, which keeps the row division short.
template <typename Index, int FMT>
__global__ void __launch_bounds__(kBlock) geglu_vec_kernel(void* y, const void* x, Index n_vec,
                                                           Index hv) {
  using I = Io<FMT>;
  const Index base = static_cast<Index>(blockIdx.x) * (kBlock * kVecPerThread) + threadIdx.x;
  typename I::Vec val[kVecPerThread], gate[kVecPerThread];
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const Index i = base + k * kBlock;
    if (i < n_vec) {
      const Index r = i / hv;
      const int64_t e = (static_cast<int64_t>(i) + static_cast<int64_t>(r) * hv) * 8;
      val[k] = I::load(x, e);
      gate[k] = I::load(x, e + static_cast<int64_t>(hv) * 8);
    } else {
      val[k] = gate[k] = typename I::Vec{};
    }
  }
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const Index i = base + k * kBlock;
    if (i < n_vec) I::store(y, static_cast<int64_t>(i) * 8, gelu8<FMT, true>(gate[k], val[k]));
  }
}

template <int FMT>
__global__ void __launch_bounds__(kBlock) geglu_elem_kernel(void* y, const void* x, int64_t rows,
                                                            int64_t h) {
  using I = Io<FMT>;
  const int64_t n = rows * h;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; i < n; i += stride) {
    const int64_t r = i / h, j = i - r * h;
    I::put(y, i, gelu_pick<FMT>(I::get(x, r * 2 * h + h + j), I::get(x, r * 2 * h + j)));
  }
}

// fp32: 16-byte chunks of 4 floats, consecutive lanes on consecutive chunks
// in every load and store (a 32-byte slot per lane would leave each
// instruction half of every 32-byte sector it touches, which costs nothing
// in HBM behind L2 but halves the rate across the host link).
constexpr int kChunksPerThread = 2 * kVecPerThread;

template <bool kGated>
__device__ __forceinline__ uint4 gelu4_f32(uint4 xc, uint4 vc) {
  const float x[4] = {__uint_as_float(xc.x), __uint_as_float(xc.y), __uint_as_float(xc.z),
                      __uint_as_float(xc.w)};
  const float v[4] = {kGated ? __uint_as_float(vc.x) : 1.f, kGated ? __uint_as_float(vc.y) : 1.f,
                      kGated ? __uint_as_float(vc.z) : 1.f, kGated ? __uint_as_float(vc.w) : 1.f};
  return make_uint4(__float_as_uint(gelu_pick<kF32>(x[0], v[0])),
                    __float_as_uint(gelu_pick<kF32>(x[1], v[1])),
                    __float_as_uint(gelu_pick<kF32>(x[2], v[2])),
                    __float_as_uint(gelu_pick<kF32>(x[3], v[3])));
}

// n_chunk 4-float chunks of x -> y.
__global__ void __launch_bounds__(kBlock) gelu_chunk_kernel(float* y, const float* x,
                                                            int64_t n_chunk) {
  const int64_t base = static_cast<int64_t>(blockIdx.x) * (kBlock * kChunksPerThread) + threadIdx.x;
  uint4 c[kChunksPerThread];
#pragma unroll
  for (int k = 0; k < kChunksPerThread; ++k) {
    const int64_t i = base + k * kBlock;
    c[k] = i < n_chunk ? ltxk::ld_stream16(x + i * 4) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int k = 0; k < kChunksPerThread; ++k) {
    const int64_t i = base + k * kBlock;
    if (i < n_chunk) ltxk::st16(y + i * 4, gelu4_f32<false>(c[k], c[k]));
  }
}

// x [rows, 2h], y [rows, h] fp32; hc = h / 4 chunks per output row.
template <typename Index>
__global__ void __launch_bounds__(kBlock) geglu_chunk_kernel(float* y, const float* x,
                                                             Index n_chunk, Index hc) {
  const Index base = static_cast<Index>(blockIdx.x) * (kBlock * kChunksPerThread) + threadIdx.x;
  uint4 val[kChunksPerThread], gate[kChunksPerThread];
#pragma unroll
  for (int k = 0; k < kChunksPerThread; ++k) {
    const Index i = base + k * kBlock;
    if (i < n_chunk) {
      const Index r = i / hc;
      const float* xv = x + (static_cast<int64_t>(i) + static_cast<int64_t>(r) * hc) * 4;
      val[k] = ltxk::ld_stream16(xv);
      gate[k] = ltxk::ld_stream16(xv + static_cast<int64_t>(hc) * 4);
    } else {
      val[k] = gate[k] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int k = 0; k < kChunksPerThread; ++k) {
    const Index i = base + k * kBlock;
    if (i < n_chunk) ltxk::st16(y + static_cast<int64_t>(i) * 4, gelu4_f32<true>(gate[k], val[k]));
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

unsigned chunk_grid(int64_t n_chunk) {
  return static_cast<unsigned>((n_chunk + kBlock * kChunksPerThread - 1) /
                               (kBlock * kChunksPerThread));
}

unsigned elem_grid(int64_t n) {
  const int64_t g = (n + kBlock - 1) / kBlock;
  return static_cast<unsigned>(g < 65536 ? g : 65536);   // grid-stride beyond
}

int fmt_of_dtype(int dtype) {
  return dtype == LTXK_DTYPE_BF16 ? kBf16
         : dtype == LTXK_DTYPE_F16 ? kF16
         : dtype == LTXK_DTYPE_F32 ? kF32 : -1;
}

template <int FMT>
int gelu_launch(void* out, const void* x, int64_t n, cudaStream_t s) {
  constexpr int64_t esz = Io<FMT>::kBytes;
  int64_t done = 0;
  if (aligned_to(out, 16) && aligned_to(x, 16)) {
    if constexpr (FMT == kF32) {
      const int64_t n_chunk = n / 4;
      if (n_chunk > 0) {
        gelu_chunk_kernel<<<chunk_grid(n_chunk), kBlock, 0, s>>>(
            static_cast<float*>(out), static_cast<const float*>(x), n_chunk);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail(e);
      }
      done = n_chunk * 4;
    } else {
      const int64_t n_vec = n / 8;
      if (n_vec > 0) {
        gelu_vec_kernel<FMT><<<vec_grid(n_vec), kBlock, 0, s>>>(out, x, n_vec);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail(e);
      }
      done = n_vec * 8;
    }
  }
  if (done < n) {
    gelu_elem_kernel<FMT><<<elem_grid(n - done), kBlock, 0, s>>>(
        static_cast<char*>(out) + done * esz, static_cast<const char*>(x) + done * esz, n - done);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(e);
  }
  return LTXK_OK;
}

template <int FMT>
int geglu_launch(void* out, const void* x, int64_t rows, int64_t hidden, cudaStream_t s) {
  const bool aligned = aligned_to(out, 16) && aligned_to(x, 16);
  if constexpr (FMT == kF32) {
    if (hidden % 4 == 0 && aligned) {
      const int64_t hc = hidden / 4, n_chunk = rows * hc;
      float* y = static_cast<float*>(out);
      const float* xf = static_cast<const float*>(x);
      if (n_chunk + kBlock * kChunksPerThread < (int64_t{1} << 32))
        geglu_chunk_kernel<uint32_t><<<chunk_grid(n_chunk), kBlock, 0, s>>>(
            y, xf, static_cast<uint32_t>(n_chunk), static_cast<uint32_t>(hc));
      else
        geglu_chunk_kernel<int64_t><<<chunk_grid(n_chunk), kBlock, 0, s>>>(y, xf, n_chunk, hc);
    } else {
      geglu_elem_kernel<FMT><<<elem_grid(rows * hidden), kBlock, 0, s>>>(out, x, rows, hidden);
    }
  } else {
    if (hidden % 8 == 0 && aligned) {
      const int64_t hv = hidden / 8, n_vec = rows * hv;
      if (n_vec + kBlock * kVecPerThread < (int64_t{1} << 32))
        geglu_vec_kernel<uint32_t, FMT><<<vec_grid(n_vec), kBlock, 0, s>>>(
            out, x, static_cast<uint32_t>(n_vec), static_cast<uint32_t>(hv));
      else
        geglu_vec_kernel<int64_t, FMT><<<vec_grid(n_vec), kBlock, 0, s>>>(out, x, n_vec, hv);
    } else {
      geglu_elem_kernel<FMT><<<elem_grid(rows * hidden), kBlock, 0, s>>>(out, x, rows, hidden);
    }
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(e);
  return LTXK_OK;
}

}  // namespace

extern "C" int ltxk_gelu_tanh_dt(void* out, const void* x, int64_t n, int dtype,
                                 ltxk_stream_t stream) {
  const int fmt = fmt_of_dtype(dtype);
  if (fmt < 0) return LTXK_ERR_DTYPE;
  if (out == nullptr || x == nullptr) return LTXK_ERR_NULL;
  if (n < 0 || n > kMaxElements) return LTXK_ERR_SHAPE;
  const int esz = fmt == kF32 ? 4 : 2;
  if (!aligned_to(out, esz) || !aligned_to(x, esz)) return LTXK_ERR_ALIGN;
  const uint64_t bytes = static_cast<uint64_t>(n) * esz;
  if (out != x && overlaps(out, bytes, x, bytes)) return LTXK_ERR_OVERLAP;
  if (n == 0) return LTXK_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (fmt == kF16) return gelu_launch<kF16>(out, x, n, s);
  if (fmt == kF32) return gelu_launch<kF32>(out, x, n, s);
  return gelu_launch<kBf16>(out, x, n, s);
}

extern "C" int ltxk_gelu_tanh(void* out, const void* x, int64_t n, ltxk_stream_t stream) {
  return ltxk_gelu_tanh_dt(out, x, n, LTXK_DTYPE_BF16, stream);
}

extern "C" int ltxk_geglu_dt(void* out, const void* x, int64_t rows, int64_t hidden, int dtype,
                             ltxk_stream_t stream) {
  const int fmt = fmt_of_dtype(dtype);
  if (fmt < 0) return LTXK_ERR_DTYPE;
  if (out == nullptr || x == nullptr) return LTXK_ERR_NULL;
  if (rows < 0 || hidden <= 0 || hidden > LTXK_MAX_HIDDEN) return LTXK_ERR_SHAPE;
  if (rows > kMaxElements / hidden) return LTXK_ERR_SHAPE;
  const int esz = fmt == kF32 ? 4 : 2;
  if (!aligned_to(out, esz) || !aligned_to(x, esz)) return LTXK_ERR_ALIGN;
  if (overlaps(out, static_cast<uint64_t>(rows) * hidden * esz, x,
               static_cast<uint64_t>(rows) * hidden * 2 * esz))
    return LTXK_ERR_OVERLAP;
  if (rows == 0) return LTXK_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (fmt == kF16) return geglu_launch<kF16>(out, x, rows, hidden, s);
  if (fmt == kF32) return geglu_launch<kF32>(out, x, rows, hidden, s);
  return geglu_launch<kBf16>(out, x, rows, hidden, s);
}

extern "C" int ltxk_geglu(void* out, const void* x, int64_t rows, int64_t hidden,
                          ltxk_stream_t stream) {
  return ltxk_geglu_dt(out, x, rows, hidden, LTXK_DTYPE_BF16, stream);
}
