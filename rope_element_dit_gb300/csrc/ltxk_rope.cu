// ltxk_rope.cu -- standalone rotary position embedding with the angles
// computed on the device from token positions (no cos/sin tables in HBM).
//
// "cuda-kernels" skill page (Hugging Face), "Kernel-Specific Guidelines /
// RoPE": x is [batch, seq, heads, head_dim] for text (1D positions) or
// [batch, t*h*w, heads, head_dim] for video (3D positions), and LTX-Video
// computes its own rotary angles.  Definition implemented (the pages print no
// frequency formula; this is the recipe the fused form's tables follow):
//   token s = r mod (T*H*W) of row r has coordinates
//     (ct, ch, cw) = (s / (H*W), (s / W) mod H, s mod W);
//   the head_dim/2 pairs split into consecutive groups of nt, nh, nw pairs
//   (axis t, then h, then w; 1D text: nt = head_dim/2, H = W = 1);
//   pair k of an axis with n pairs turns by coordinate * theta^(-k/n);
//   a' = a cos - b sin, b' = a sin + b cos, pairs (2p, 2p+1) (interleaved)
//   or (p, p + head_dim/2) (split-half) of every head; one rounding.
//
// Design.  The angles of a token are shared by all heads of its row, so
// each CTA computes them once per row into shared memory and every head
// reuses them (heads-fold reuse).  Persistent CTAs of 128 threads (64 when a
// row is at most 64 threads' units, so that small rows fill every unit slot
// and twice the rows are in flight per SM):
//   * the per-pair frequencies theta^(-k/n) are launch constants: the host
//     evaluates them in fp64, as turns per coordinate unit theta^(-k/n)/(2 pi)
//     split into two floats th + tl (exact to ~2^-48), and passes them in the
//     kernel parameters;
//   * a row's angles are formed in fp32 double-float arithmetic: the product
//     with the coordinate is split exactly (an FMA two-product), the whole
//     turns are dropped exactly, the fractional turn is summed without loss
//     (two-sum), sincospif takes the leading part and a first-order term the
//     remainder.  No fp64 per row (GB300's FP64 rate is 1/64 of FP32);
//     coordinates of 2^24 and beyond take an fp64 reduction;
//   * the angle table is double-buffered and computed one row ahead: after
//     the barrier of row i, the threads k < P fill the other buffer for the
//     CTA's next row while everyone rotates row i, so the barrier never waits
//     on sincospif; cos and sin are separate arrays read as float4 (no bank
//     conflicts);
//   * a row's x loads are issued before its barrier;
//   * the rotation runs on the widened pairs with Kahan's 2x2-determinant
//     algorithm (as in the fused kernels), then one rounding per element.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>

#include "ltxk.h"
#include "ltxk_kernels.cuh"
#include "ltxk_launch.h"

namespace ltxk {

// Threads per CTA: 128, or 64 when a row is at most 64 threads' units (one
// pass either way): a small row then fills every unit slot of a thread, and
// twice the CTAs -- rows in flight -- fit on an SM.
constexpr int kRopeBlock = 128;
constexpr int kRopeSmallBlock = 64;
constexpr int kRopeThreadsPerSm = 1024;
// 16-byte units per thread per pass over a row: 16 registers of row data
// (split-half units are two vectors, fp32 vectors two registers wide).
template <int MODE, int FMT>
struct RopeUnits {
  static constexpr int value = (MODE == kSplitHalf ? 2 : 4) / (FMT == kF32 ? 2 : 1);
};
constexpr int kRopeMaxPairs = 256;    // head_dim <= 512 (frequencies travel as kernel parameters)

struct RopeArgs {
  void* out;
  const void* x;
  int64_t rows;
  int heads;
  int head_dim;
  int64_t thw, hw, w;                 // T*H*W, H*W, W
  uint64_t thw_mul, hw_mul, w_mul;    // div_fast multipliers of the three
  int nt, nh, nw;                     // pairs per axis
  float2 turns[kRopeMaxPairs];        // theta^(-k/n) / (2 pi) of pair k as hi + lo
};

// pair k's axis, index in the axis and pair count of the axis
__device__ __forceinline__ void pair_axis(const RopeArgs& a, int k, int* axis, int* kk, int* n) {
  if (k < a.nt) {
    *axis = 0; *kk = k; *n = a.nt;
  } else if (k < a.nt + a.nh) {
    *axis = 1; *kk = k - a.nt; *n = a.nh;
  } else {
    *axis = 2; *kk = k - a.nt - a.nh; *n = a.nw;
  }
}

// (cos, sin) of coord * inv, inv in fp64.  The product and its reduction by
// a whole number of turns are fp64 (coord * inv carries a relative error of
// 2^-52, ~2^-28 absolute at 2^24 radians); the reduced angle is split into
// an fp32 value and its fp32 remainder, and the remainder enters through the
// first-order terms cos(r + e) = cos r - e sin r, sin(r + e) = sin r + e cos r.
__device__ __noinline__ float2 angle_cs(int64_t coord, double inv) {
  const double kInvTwoPi = 0.15915494309189535;   // 1 / (2 pi)
  const double kTwoPi = 6.283185307179586;
  const double ang = static_cast<double>(coord) * inv;
  const double turns = rint(ang * kInvTwoPi);
  const double r = fma(-turns, kTwoPi, ang);       // |r| <= pi (+ rounding)
  const float rh = static_cast<float>(r);
  const float rl = static_cast<float>(r - static_cast<double>(rh));
  float s, c;
  sincosf(rh, &s, &c);
  return make_float2(__fmaf_rn(-s, rl, c), __fmaf_rn(c, rl, s));
}

// (cos, sin) of 2 pi * c * (th + tl) for an integer c < 2^24 (exact in fp32):
//   c*th = P + E exactly (FMA two-product); N = rint(P); F = P - N is exact
//   (Sterbenz: P and N are within a factor of two once N >= 1); G = E + c*tl
//   in one FMA (|G| < 0.3 turns, one rounding of at most 2^-27 turns); and
//   F + G = S + e exactly (Knuth's two-sum).  sincospif(2S) gives cos and sin
//   of 2 pi S to about an ulp, and d = 2 pi e (below 2^-24) enters as
//   cos(x + d) = cos x - d sin x, sin(x + d) = sin x + d cos x.  Emulated on
//   the CPU over c < 2^24 and theta^(-k/n): within 2 * 2^-24 of fp64 cos/sin.
__device__ __forceinline__ float2 angle_cs_turns(float c, float2 t) {
  const float p = c * t.x;
  const float e1 = __fmaf_rn(c, t.x, -p);
  const float f = p - rintf(p);
  const float g = __fmaf_rn(c, t.y, e1);
  const float sum = f + g;
  const float bb = sum - f;
  const float e2 = (f - (sum - bb)) + (g - bb);
  const float d = 6.2831853071795865f * e2;
  float sn, cs;
  sincospif(2.f * sum, &sn, &cs);
  return make_float2(__fmaf_rn(-sn, d, cs), __fmaf_rn(cs, d, sn));
}

// The coordinates (t, h, w) of token s (taken mod T*H*W).
__device__ __forceinline__ void token_coords(const RopeArgs& a, int64_t r, int64_t coord[3]) {
  const int64_t s = r - div_fast(r, a.thw, a.thw_mul) * a.thw;
  const int64_t ct = div_fast(s, a.hw, a.hw_mul);
  const int64_t rem = s - ct * a.hw;
  const int64_t ch = div_fast(rem, a.w, a.w_mul);
  coord[0] = ct;
  coord[1] = ch;
  coord[2] = rem - ch * a.w;
}

// (cos, sin) of pair k of a token with coordinates coord.
__device__ __forceinline__ float2 pair_angle(const RopeArgs& a, const int64_t coord[3], int k) {
  int axis, kk, n;
  pair_axis(a, k, &axis, &kk, &n);
  const int64_t c = coord[axis];
  const float2 t = a.turns[k];
  return c < (int64_t{1} << 24)
             ? angle_cs_turns(static_cast<float>(c), t)
             : angle_cs(c, 6.283185307179586 * (static_cast<double>(t.x) + t.y));
}

// cos and sin tables [tokens, head_dim/2] (fp32) of tokens 0 .. tokens-1,
// token s at position s mod T*H*W: the inputs of the fused RMSNorm + RoPE,
// with the angles of the standalone kernel.  One thread per (token, pair).
__global__ void __launch_bounds__(256) rope_tables_kernel(float* cos_out, float* sin_out,
                                                          int64_t tokens, const RopeArgs a) {
  const int P = a.head_dim >> 1;
  const int64_t n = tokens * P;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const int64_t s = i / P;
    int64_t coord[3];
    token_coords(a, s, coord);
    const float2 v = pair_angle(a, coord, static_cast<int>(i - s * P));
    cos_out[i] = v.x;
    sin_out[i] = v.y;
  }
}

// VEC: 16-byte slots (interleaved: head_dim % 8 == 0, split-half: % 16 == 0,
// 16-byte aligned pointers); otherwise one thread per rotation pair.
template <int MODE, int FMT, bool VEC, int BLOCK>
__global__ void __launch_bounds__(BLOCK, kRopeThreadsPerSm / BLOCK) rope_kernel(const RopeArgs a) {
  using I = Io<FMT>;
  using Vec = typename I::Vec;
  constexpr int kU = RopeUnits<MODE, FMT>::value;
  __shared__ __align__(16) float cosv[2][kRopeMaxPairs];
  __shared__ __align__(16) float sinv[2][kRopeMaxPairs];
  const int P = a.head_dim >> 1;
  const int D = a.head_dim;
  const int tid = threadIdx.x;

  // the angles of row r's token into buffer b
  auto fill_table = [&](int64_t r, int b) {
    int64_t coord[3];
    token_coords(a, r, coord);
    for (int k = tid; k < P; k += BLOCK) {
      const float2 v = pair_angle(a, coord, k);
      cosv[b][k] = v.x;
      sinv[b][k] = v.y;
    }
  };

  const int64_t HD = static_cast<int64_t>(a.heads) * D;
  // Units of a row: 16-byte vectors (interleaved), (lo, hi) vector pairs of a
  // head (split-half), or single rotation pairs (element-wise).  Unit u of a
  // pass is u0 + i * BLOCK; its column in the head (interleaved) or its
  // (head, vector pair) (split-half) advance by fixed steps, no division.
  const int qph = D >> 4;   // split-half: vector pairs per head
  const int units = VEC ? (MODE == kInterleaved ? static_cast<int>(HD >> 3) : a.heads * qph)
                        : a.heads * P;
  const int step_col = (BLOCK * 8) % D;
  const int step_head = qph > 0 ? BLOCK / qph : 0;
  const int step_jv = qph > 0 ? BLOCK % qph : 0;

  int buf = 0;
  if (static_cast<int64_t>(blockIdx.x) < a.rows) fill_table(blockIdx.x, 0);
  for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x, buf ^= 1) {
    const int64_t rb = row * HD;
    Vec lo[kU], hi[MODE == kSplitHalf && VEC ? kU : 1];
    auto load_pass = [&](int base) {
      if constexpr (VEC) {
        if constexpr (MODE == kInterleaved) {
#pragma unroll
          for (int i = 0; i < kU; ++i) {
            const int u = base + tid + i * BLOCK;
            if (u < units) lo[i] = I::load(a.x, rb + static_cast<int64_t>(u) * 8);
          }
        } else {
          int head = (base + tid) / qph, jv = (base + tid) - head * qph;
#pragma unroll
          for (int i = 0; i < kU; ++i) {
            const int u = base + tid + i * BLOCK;
            if (u < units) {
              const int64_t off = static_cast<int64_t>(head) * D + jv * 8;
              lo[i] = I::load(a.x, rb + off);
              hi[i] = I::load(a.x, rb + off + P);
            }
            head += step_head;
            jv += step_jv;
            if (jv >= qph) {
              jv -= qph;
              ++head;
            }
          }
        }
      }
    };
    load_pass(0);
    // this row's table (buf) is complete, and the other buffer's last reader
    // (the previous row) is done: fill it for the next row while rotating
    __syncthreads();
    const int64_t next = row + gridDim.x;
    if (next < a.rows) fill_table(next, buf ^ 1);
    const float* ct = cosv[buf];
    const float* st = sinv[buf];
    if constexpr (VEC) {
      for (int base = 0; base < units; base += BLOCK * kU) {
        if (base > 0) load_pass(base);
        if constexpr (MODE == kInterleaved) {
          int col = ((base + tid) * 8) % D;   // element column of unit i in its head
#pragma unroll
          for (int i = 0; i < kU; ++i) {
            const int u = base + tid + i * BLOCK;
            if (u < units) {
              const int p0 = col >> 1;   // rotation pairs p0 .. p0 + 3 (p0 % 4 == 0)
              const float4 c4 = *reinterpret_cast<const float4*>(ct + p0);
              const float4 s4 = *reinterpret_cast<const float4*>(st + p0);
              const float2 c[2] = {make_float2(c4.x, c4.y), make_float2(c4.z, c4.w)};
              const float2 sn[2] = {make_float2(s4.x, s4.y), make_float2(s4.z, s4.w)};
              float2 o[4];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const float2 x0 = I::pair(lo[i], 2 * h), x1 = I::pair(lo[i], 2 * h + 1);
                const float2 av = make_float2(x0.x, x1.x), bv = make_float2(x0.y, x1.y);
                const float2 ra = diff_of_products2(av, c[h], bv, sn[h]);
                const float2 rb2 = diff_of_products2(av, sn[h], neg2(bv), c[h]);
                o[2 * h] = make_float2(ra.x, rb2.x);
                o[2 * h + 1] = make_float2(ra.y, rb2.y);
              }
              I::store(a.out, rb + static_cast<int64_t>(u) * 8, I::pack(o[0], o[1], o[2], o[3]));
            }
            col += step_col;
            if (col >= D) col -= D;
          }
        } else {
          int head = (base + tid) / qph, jv = (base + tid) - head * qph;
#pragma unroll
          for (int i = 0; i < kU; ++i) {
            const int u = base + tid + i * BLOCK;
            if (u < units) {
              const int64_t off = static_cast<int64_t>(head) * D + jv * 8;
              const float4 c0 = *reinterpret_cast<const float4*>(ct + jv * 8);
              const float4 c1 = *reinterpret_cast<const float4*>(ct + jv * 8 + 4);
              const float4 s0 = *reinterpret_cast<const float4*>(st + jv * 8);
              const float4 s1 = *reinterpret_cast<const float4*>(st + jv * 8 + 4);
              const float2 c[4] = {make_float2(c0.x, c0.y), make_float2(c0.z, c0.w),
                                   make_float2(c1.x, c1.y), make_float2(c1.z, c1.w)};
              const float2 sn[4] = {make_float2(s0.x, s0.y), make_float2(s0.z, s0.w),
                                    make_float2(s1.x, s1.y), make_float2(s1.z, s1.w)};
              float2 ol[4], oh[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {   // pairs jv*8 + 2j, +1: (lo pair j, hi pair j)
                const float2 av = I::pair(lo[i], j), bv = I::pair(hi[i], j);
                ol[j] = diff_of_products2(av, c[j], bv, sn[j]);
                oh[j] = diff_of_products2(av, sn[j], neg2(bv), c[j]);
              }
              I::store(a.out, rb + off, I::pack(ol[0], ol[1], ol[2], ol[3]));
              I::store(a.out, rb + off + P, I::pack(oh[0], oh[1], oh[2], oh[3]));
            }
            head += step_head;
            jv += step_jv;
            if (jv >= qph) {
              jv -= qph;
              ++head;
            }
          }
        }
      }
    } else {
      for (int q = tid; q < units; q += BLOCK) {
        const int head = q / P, p = q - head * P;
        const int64_t ia = MODE == kInterleaved ? static_cast<int64_t>(head) * D + 2 * p
                                                : static_cast<int64_t>(head) * D + p;
        const int64_t ib = MODE == kInterleaved ? ia + 1 : ia + P;
        const float av = I::get(a.x, rb + ia), bv = I::get(a.x, rb + ib);
        const float c = ct[p], sn = st[p];
        I::put(a.out, rb + ia, diff_of_products(av, c, bv, sn));
        I::put(a.out, rb + ib, sum_of_products(av, sn, bv, c));
      }
    }
  }
}

}  // namespace ltxk

namespace {

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlaps(const void* a, uint64_t na, const void* b, uint64_t nb) {
  if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

uint64_t div_mul(int64_t d) {
  return (d < 2 || d >= (int64_t{1} << 32)) ? 0 : UINT64_MAX / static_cast<uint64_t>(d) + 1;
}

int fail(cudaError_t e) {
  ltxk::record_cuda_error(static_cast<int>(e));
  return LTXK_ERR_CUDA;
}

// SM count of the current device, queried once per device.
cudaError_t sm_count(int* sms) {
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it == cache.end()) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    it = cache.emplace(dev, n).first;
  }
  *sms = it->second;
  return cudaSuccess;
}

template <int MODE, int FMT>
const void* rope_fn(bool vec, bool small) {
  if (!vec) return reinterpret_cast<const void*>(&ltxk::rope_kernel<MODE, FMT, false, ltxk::kRopeBlock>);
  return small ? reinterpret_cast<const void*>(&ltxk::rope_kernel<MODE, FMT, true, ltxk::kRopeSmallBlock>)
               : reinterpret_cast<const void*>(&ltxk::rope_kernel<MODE, FMT, true, ltxk::kRopeBlock>);
}

template <int MODE>
const void* rope_fn_fmt(int fmt, bool vec, bool small) {
  if (fmt == ltxk::kF16) return rope_fn<MODE, ltxk::kF16>(vec, small);
  if (fmt == ltxk::kF32) return rope_fn<MODE, ltxk::kF32>(vec, small);
  return rope_fn<MODE, ltxk::kBf16>(vec, small);
}

// Units of a row of the vector kernel (16-byte vectors, or lo/hi vector
// pairs for split-half), and units per thread per pass.
int64_t row_units(int mode, int heads, int head_dim) {
  return mode == LTXK_ROPE_INTERLEAVED ? static_cast<int64_t>(heads) * head_dim / 8
                                       : static_cast<int64_t>(heads) * (head_dim / 16);
}
int units_per_thread(int mode, int fmt) {
  using ltxk::RopeUnits;
  if (mode == LTXK_ROPE_INTERLEAVED)
    return fmt == ltxk::kF32 ? RopeUnits<ltxk::kInterleaved, ltxk::kF32>::value
                             : RopeUnits<ltxk::kInterleaved, ltxk::kBf16>::value;
  return fmt == ltxk::kF32 ? RopeUnits<ltxk::kSplitHalf, ltxk::kF32>::value
                           : RopeUnits<ltxk::kSplitHalf, ltxk::kBf16>::value;
}

// Validates the position grid, the pair split and theta, and fills the
// position fields of a: T*H*W, H*W, W and their division multipliers, the
// pairs per axis, and the frequencies as turns per coordinate unit.
int position_args(ltxk::RopeArgs* a, int head_dim, int64_t grid_t, int64_t grid_h,
                  int64_t grid_w, int pairs_t, int pairs_h, int pairs_w, double theta) {
  if (grid_t < 1 || grid_h < 1 || grid_w < 1 || grid_t > (int64_t{1} << 31) ||
      grid_h > (int64_t{1} << 31) || grid_w > (int64_t{1} << 31) ||
      grid_t * grid_h > (int64_t{1} << 62) / grid_w)
    return LTXK_ERR_SHAPE;
  if (pairs_t < 0 || pairs_h < 0 || pairs_w < 0 ||
      static_cast<int64_t>(pairs_t) + pairs_h + pairs_w != head_dim / 2)
    return LTXK_ERR_SHAPE;
  if (!(theta > 0.0) || !(theta < 1e300)) return LTXK_ERR_SHAPE;
  a->head_dim = head_dim;
  a->thw = grid_t * grid_h * grid_w;
  a->hw = grid_h * grid_w;
  a->w = grid_w;
  a->thw_mul = div_mul(a->thw);
  a->hw_mul = div_mul(a->hw);
  a->w_mul = div_mul(grid_w);
  a->nt = pairs_t;
  a->nh = pairs_h;
  a->nw = pairs_w;
  // pair k of an axis with n pairs: theta^(-k/n), in fp64
  const int per_axis[3] = {pairs_t, pairs_h, pairs_w};
  for (int axis = 0, k = 0; axis < 3; ++axis)
    for (int j = 0; j < per_axis[axis]; ++j, ++k) {
      const double tpu = pow(theta, -static_cast<double>(j) / per_axis[axis]) *
                         0.15915494309189535;   // turns per coordinate unit
      const float th = static_cast<float>(tpu);
      a->turns[k] = make_float2(th, static_cast<float>(tpu - static_cast<double>(th)));
    }
  return LTXK_OK;
}

}  // namespace

extern "C" int ltxk_rope(void* out, const void* x, int64_t rows, int heads, int head_dim,
                         int mode, int64_t grid_t, int64_t grid_h, int64_t grid_w, int pairs_t,
                         int pairs_h, int pairs_w, double theta, int dtype,
                         ltxk_stream_t stream) {
  const int fmt = dtype == LTXK_DTYPE_BF16 ? ltxk::kBf16
                  : dtype == LTXK_DTYPE_F16 ? ltxk::kF16
                  : dtype == LTXK_DTYPE_F32 ? ltxk::kF32 : -1;
  if (fmt < 0) return LTXK_ERR_DTYPE;
  if (out == nullptr || x == nullptr) return LTXK_ERR_NULL;
  if (mode != LTXK_ROPE_INTERLEAVED && mode != LTXK_ROPE_SPLIT_HALF) return LTXK_ERR_MODE;
  if (rows < 0 || heads < 1 || head_dim < 2 || head_dim % 2 != 0 ||
      head_dim / 2 > ltxk::kRopeMaxPairs)
    return LTXK_ERR_SHAPE;
  const int64_t hd = static_cast<int64_t>(heads) * head_dim;
  if (hd > LTXK_MAX_HIDDEN || (rows > 0 && rows > INT64_MAX / 8 / hd)) return LTXK_ERR_SHAPE;
  ltxk::RopeArgs a{};
  const int st = position_args(&a, head_dim, grid_t, grid_h, grid_w, pairs_t, pairs_h, pairs_w,
                               theta);
  if (st != LTXK_OK) return st;
  const int esz = fmt == ltxk::kF32 ? 4 : 2;
  if (!aligned_to(out, esz) || !aligned_to(x, esz)) return LTXK_ERR_ALIGN;
  const uint64_t bytes = static_cast<uint64_t>(rows) * hd * esz;
  if (out != x && overlaps(out, bytes, x, bytes)) return LTXK_ERR_OVERLAP;
  if (rows == 0) return LTXK_OK;

  const bool vec = aligned_to(out, 16) && aligned_to(x, 16) &&
                   head_dim % (mode == LTXK_ROPE_INTERLEAVED ? 8 : 16) == 0 &&
                   hd / 8 <= static_cast<int64_t>(1) << 30;
  a.out = out;
  a.x = x;
  a.rows = rows;
  a.heads = heads;
  int sms = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return fail(e);
  const bool small = vec && row_units(mode, heads, head_dim) <=
                               static_cast<int64_t>(ltxk::kRopeSmallBlock) *
                                   units_per_thread(mode, fmt);
  const int block = small ? ltxk::kRopeSmallBlock : ltxk::kRopeBlock;
  const int64_t cap = static_cast<int64_t>(sms) * (ltxk::kRopeThreadsPerSm / block);
  const unsigned grid = static_cast<unsigned>(rows < cap ? rows : cap);
  const void* fn = mode == LTXK_ROPE_INTERLEAVED
                       ? rope_fn_fmt<ltxk::kInterleaved>(fmt, vec, small)
                       : rope_fn_fmt<ltxk::kSplitHalf>(fmt, vec, small);
  void* params[] = {&a};
  e = cudaLaunchKernel(fn, dim3(grid), dim3(block), params, 0,
                       reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(e);
  return LTXK_OK;
}

extern "C" int ltxk_rope_tables(float* cos_out, float* sin_out, int64_t tokens, int head_dim,
                                int64_t grid_t, int64_t grid_h, int64_t grid_w, int pairs_t,
                                int pairs_h, int pairs_w, double theta, ltxk_stream_t stream) {
  if (cos_out == nullptr || sin_out == nullptr) return LTXK_ERR_NULL;
  if (tokens < 0 || head_dim < 2 || head_dim % 2 != 0 || head_dim / 2 > ltxk::kRopeMaxPairs ||
      (tokens > 0 && tokens > (int64_t{1} << 40) / head_dim))
    return LTXK_ERR_SHAPE;
  ltxk::RopeArgs a{};
  const int st = position_args(&a, head_dim, grid_t, grid_h, grid_w, pairs_t, pairs_h, pairs_w,
                               theta);
  if (st != LTXK_OK) return st;
  if (!aligned_to(cos_out, 4) || !aligned_to(sin_out, 4)) return LTXK_ERR_ALIGN;
  const int64_t n = tokens * (head_dim / 2);
  if (overlaps(cos_out, static_cast<uint64_t>(n) * 4, sin_out, static_cast<uint64_t>(n) * 4))
    return LTXK_ERR_OVERLAP;
  if (tokens == 0) return LTXK_OK;
  int sms = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return fail(e);
  const int64_t blocks = (n + 255) / 256, cap = static_cast<int64_t>(sms) * 8;
  ltxk::rope_tables_kernel<<<static_cast<unsigned>(blocks < cap ? blocks : cap), 256, 0,
                             reinterpret_cast<cudaStream_t>(stream)>>>(cos_out, sin_out, tokens, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(e);
  return LTXK_OK;
}
