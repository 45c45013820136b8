// ltxk_kernels.cuh -- device code for RMSNorm, fused RMSNorm + RoPE, the
// AdaLN-modulated norm and the fused residual add + RMSNorm on sm_103a
// (GB300), for bf16, fp16 and fp32 rows.
//
// The operation (no formula is printed on the pages; this is the definition
// the library implements):
//   per row r:  ms = (1/H) sum_j x_j^2,  n_j = x_j * w_j / sqrt(ms + eps)
//   fused:      per head and pair (a, b):  a' = a c - b s,  b' = a s + b c
//   one round-to-nearest-even to the row format (bf16, fp16 or fp32) at the
//   end ("cuda-kernels" page, "Supported Data Types": the three precision
//   modes).
// Sources: "cuda-kernels" skill page (Hugging Face), "Kernel-Specific
// Guidelines / RMSNorm" and "/ RoPE", "Core Kernel Patterns / Vectorized
// Memory Access" and "/ Warp Shuffle Reductions"; "ltx-kernels" README,
// opening list (`ops_cpp`: rms_norm_rope, rms_norm_split_rope).
//
// The path is bound by HBM bandwidth (4 bytes moved per element against a
// handful of fp32 operations), so it uses no tensor cores.  Design:
//   * Each row is read from HBM exactly once, as 16-byte vectors, into
//     registers; a group of G warps owns one row, with G and the slots per
//     lane chosen by the host planner (e.g. G = 4 for hidden 3072 and 4096).
//     fp32 rows without rotation use a chunk map (two 4-float chunks per
//     slot) so that every warp access is one contiguous span.
//   * fp32 sum of squares: per-lane partials, an xor-butterfly over the
//     warp, then (G > 1) a fixed-order sum of the G warp totals through
//     shared memory.  Every thread ends with the same bit-identical total.
//   * inv_rms = rsqrtf(ss / H + eps); y = (x * w) * inv_rms, where x * w is
//     exact in fp32 for bf16 and fp16 rows (two significands of at most 11
//     bits), so each output is one fp32 rounding away from (x w) * inv_rms
//     before the final rounding; fp32 rows add one rounding of x * w.
//   * For bf16 and fp16 rows the squares and the products x * w come from
//     the mixed-precision FMA of sm_100 and later (fma.rn.f32.bf16 / .f16),
//     which reads the 16-bit halves of a register in place: no widening
//     instructions, the same bits.  The epilogue is compiled with and
//     without a weight and chosen once per launch.
//   * RoPE rotates (u, v) = (x_a w_a, x_b w_b) (both exact) and scales by
//     inv_rms afterwards; u c - v s and u s + v c are evaluated with Kahan's
//     2x2-determinant algorithm (W. Kahan; error bound in Jeannerod, Louvet &
//     Muller, "Further analysis of Kahan's algorithm for the accurate
//     computation of 2x2 determinants", Math. Comp. 82, 2013), which keeps
//     the relative error of a rotated value at a few fp32 ulps even when the
//     two products nearly cancel.
//   * CTAs stride over rows, so any grid covers any row count: the host
//     launches one CTA per row group for the row-only forms and persistent
//     grids for the fused ones; split-half rows of the 16-bit formats are
//     software-pipelined (a warp loads its next row, and that row's cos/sin
//     vectors, before this row's epilogue) and keep the thread's weight
//     vectors in registers for all their rows.
//   * Read-only rows a CTA uses for many of its rows are staged once: AdaLN's
//     conditioning row (scale, shift) goes to shared memory.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ltxk {

enum Mode : int { kPlain = 0, kInterleaved = 1, kSplitHalf = 2, kAdaLN = 3, kAddNorm = 4 };

// Element formats of the rows, weight and conditioning (tables are fp32).
enum Fmt : int { kBf16 = 0, kF16 = 1, kF32 = 2 };

struct RowArgs {
  void* out;                // [rows, hidden] in the row format
  const void* x;            // [rows, hidden]
  const void* w;            // [hidden] or nullptr (ones)
  const float* cos_t;       // [table_rows, head_dim/2] fp32 (fused only)
  const float* sin_t;
  int64_t rows;
  int64_t table_rows;       // row r uses table row r % table_rows
  int hidden;
  int head_dim;
  float eps;
  int stage_cond;           // 1: AdaLN's conditioning row (scale, then shift)
                            //    is staged in dynamic shared memory (this
                            //    fills the padding before the next pointer)
  const void* scale;        // AdaLN: [n_cond, hidden]
  const void* shift;        // AdaLN: [n_cond, hidden]
  int64_t rows_per_cond;    // AdaLN: row r uses conditioning row r / rows_per_cond
  const void* res;          // residual add: [rows, hidden] residual in
  void* h_out;              // residual add: [rows, hidden] h = x + res out
  uint64_t table_mul;       // div_fast multiplier of table_rows (0: divide)
  uint64_t cond_mul;        // div_fast multiplier of rows_per_cond (0: divide)
};

// n / d for n >= 0, d >= 1, given m = floor((2^64 - 1) / d) + 1 for
// 2 <= d < 2^32 and m = 0 otherwise (W. Granlund and P. Montgomery, "Division
// by invariant integers using multiplication", PLDI 1994: a rounded-up
// reciprocal and a high product).  For n < 2^32, n*m / 2^64 exceeds n/d by
// less than n / 2^64 < 1/d, which cannot carry past the next integer, so
// the high 64 bits of n*m are the quotient: one 64-bit multiply-high instead
// of a 64-bit division.
__device__ __forceinline__ int64_t div_fast(int64_t n, int64_t d, uint64_t m) {
  if (m != 0 && n < (int64_t{1} << 32))
    return static_cast<int64_t>(__umul64hi(static_cast<uint64_t>(n), m));
  return d == 1 ? n : n / d;
}

// ---- element helpers -----------------------------------------------------

// The two bf16 halves of a 32-bit word, widened exactly to fp32.
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Round two fp32 values to bf16 (RNE) and pack them, lo in the low half.
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float bf_to_f(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t f_to_bf(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// a*b - c*d with Kahan's algorithm: the rounding error of c*d is recovered
// exactly by an FMA and added back.
__device__ __forceinline__ float diff_of_products(float a, float b, float c, float d) {
  const float cd = __fmul_rn(c, d);
  const float err = __fmaf_rn(-c, d, cd);     // cd - c*d, exact
  const float dop = __fmaf_rn(a, b, -cd);     // a*b - cd, one rounding
  return __fadd_rn(dop, err);
}

__device__ __forceinline__ float sum_of_products(float a, float b, float c, float d) {
  return diff_of_products(a, b, -c, d);
}

// ---- two-wide fp32 (Blackwell f32x2: two independently rounded IEEE
// operations per instruction, bit-identical to the scalar forms) -----------

__device__ __forceinline__ float2 neg2(float2 v) { return make_float2(-v.x, -v.y); }

// The two bf16 halves of a word as (lo, hi), exactly.
__device__ __forceinline__ float2 bf2_of(uint32_t u) { return make_float2(bf_lo(u), bf_hi(u)); }

__device__ __forceinline__ uint32_t pack_f2(float2 v) { return pack_bf2(v.x, v.y); }

// Kahan's a*b - c*d on both lanes.
__device__ __forceinline__ float2 diff_of_products2(float2 a, float2 b, float2 c, float2 d) {
  const float2 cd = __fmul2_rn(c, d);
  const float2 err = __ffma2_rn(neg2(c), d, cd);
  const float2 dop = __ffma2_rn(a, b, neg2(cd));
  return __fadd2_rn(dop, err);
}

// ---- memory helpers ------------------------------------------------------

// Streaming 16-byte load: x is read once, so it should not displace L1 lines.
// A plain (coherent) load, because out may alias x in place.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ void st16(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Bring `bytes` at p (16-byte aligned, a multiple of 16) into L2 with one
// bulk-copy-engine request; nothing is written to shared memory or registers.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// Bring the line holding p toward the SM (1: into L1, 2: into L2) without
// holding a register.
template <int LEVEL>
__device__ __forceinline__ void prefetch_line(const void* p) {
  if constexpr (LEVEL == 1) asm volatile("prefetch.global.L1 [%0];" :: "l"(p));
  else asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

// Fused kernels: prefetch the row's cos/sin columns right after the row's
// loads are issued, so that their first touch (cold after the row's start)
// overlaps the wait for x instead of following it (0 = off, 1 = L1, 2 = L2).
#ifndef LTXK_TABLE_PREFETCH
#define LTXK_TABLE_PREFETCH 0
#endif

// AdaLN rows of 16-bit formats: each CTA stages the conditioning row of
// its first row in shared memory (1), or every slot reads scale and shift
// through L1/L2 (0).
#ifndef LTXK_ADALN_STAGE
#define LTXK_ADALN_STAGE 1
#endif
// Split-half rotation, 16-bit rows: each thread keeps the weight of its own
// slots in registers for all the rows it serves (1), or loads it in every
// row's epilogue (0).
#ifndef LTXK_W_REGS
#define LTXK_W_REGS 1
#endif
// Software-pipelined rotation rows: the next row's shared cos/sin vectors
// are loaded together with its x (1), instead of in its epilogue after the
// reduction (0), where each row's cold table row was a DRAM round trip the
// warp waited on.  They cost 16 registers per thread (LTXK_TABLE_NEXT_REGS):
// split-half [6144, 32x64] runs at 198 registers, 2 instead of 3 CTAs of 128
// threads per SM, and still gains on most boxes: 14.58 -> 14.26 us,
// 14.77 -> 14.26 us, 14.37 -> 14.38 us (GB300, event means, 3-4 x 300
// launches, three boxes).  Held within the old budget instead (3 CTAs per
// SM, 44 bytes spilled) it gave 14.50 us; two warps per row with it, 14.19
// and 14.32 us against 14.62 and 14.38 us (not adopted: within the spread).
#ifndef LTXK_TABLE_NEXT
#define LTXK_TABLE_NEXT 1
#endif

// Rows ahead that the register kernel asks the bulk-copy engine to bring
// into L2 (0 = off).  Measured on GB300 with the persistent RoPE grids
// (event means): one row ahead, interleaved [2x4096, 32x128] 23.8 -> 25.0 us
// and split-half [6144, 32x64] 14.8 -> 14.9 us; two rows ahead 25.8 and
// 16.0 us.
#ifndef LTXK_L2_PREFETCH_ROWS
#define LTXK_L2_PREFETCH_ROWS 0
#endif

// Read-only 16-byte loads for the weight and the tables (reused by every
// row, so they stay in L1/L2).  They are volatile so that they stay in
// program order between the stores: hoisting all of them ahead of the
// epilogue would hold 4 more registers per slot for data that hits in L1.
__device__ __forceinline__ uint4 ld_ro16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ float4 ld_ro16f(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// Make the compiler treat a packed vector as freshly defined, so that the
// widened halves computed for the sum of squares are not kept alive into
// the epilogue (that would double the registers a row needs).
__device__ __forceinline__ void launder(uint4& v) {
  asm volatile("" : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void group_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

constexpr uint32_t kOnes2 = 0x3F803F80u;   // two bf16 1.0 values

// ---- element formats -------------------------------------------------------
//
// A slot always holds 8 consecutive elements: one 16-byte vector of bf16 or
// fp16, two of fp32.  Pair i (0..3) of a slot is its elements 2i and 2i+1,
// widened exactly to fp32; pack() rounds four pairs once (RNE) into a slot.

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <int FMT>
struct Io;

template <>
struct Io<kBf16> {
  using Vec = uint4;
  static constexpr int kWords = 4;   // registers per slot
  static constexpr int kBytes = 2;
  __device__ static Vec load(const void* p, int64_t e) {
    return ld_stream16(static_cast<const uint16_t*>(p) + e);
  }
  __device__ static Vec load_ro(const void* p, int64_t e) {
    return ld_ro16(static_cast<const uint16_t*>(p) + e);
  }
  __device__ static void store(void* p, int64_t e, const Vec& v) {
    st16(static_cast<uint16_t*>(p) + e, v);
  }
  __device__ static float2 pair(const Vec& v, int i) { return bf2_of(word_of(v, i)); }
  __device__ static Vec pack(float2 a, float2 b, float2 c, float2 d) {
    return make_uint4(pack_f2(a), pack_f2(b), pack_f2(c), pack_f2(d));
  }
  __device__ static Vec ones() { return make_uint4(kOnes2, kOnes2, kOnes2, kOnes2); }
  __device__ static void launder_vec(Vec& v) { launder(v); }
  __device__ static float get(const void* p, int64_t e) {
    return bf_to_f(static_cast<const uint16_t*>(p)[e]);
  }
  __device__ static void put(void* p, int64_t e, float f) {
    static_cast<uint16_t*>(p)[e] = f_to_bf(f);
  }
};

template <>
struct Io<kF16> {
  using Vec = uint4;
  static constexpr int kWords = 4;
  static constexpr int kBytes = 2;
  __device__ static Vec load(const void* p, int64_t e) {
    return ld_stream16(static_cast<const uint16_t*>(p) + e);
  }
  __device__ static Vec load_ro(const void* p, int64_t e) {
    return ld_ro16(static_cast<const uint16_t*>(p) + e);
  }
  __device__ static void store(void* p, int64_t e, const Vec& v) {
    st16(static_cast<uint16_t*>(p) + e, v);
  }
  __device__ static float2 pair(const Vec& v, int i) {
    const uint32_t u = word_of(v, i);
    return __half22float2(*reinterpret_cast<const __half2*>(&u));
  }
  __device__ static uint32_t pack2(float2 f) {
    const __half2 h = __floats2half2_rn(f.x, f.y);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  __device__ static Vec pack(float2 a, float2 b, float2 c, float2 d) {
    return make_uint4(pack2(a), pack2(b), pack2(c), pack2(d));
  }
  __device__ static Vec ones() {
    constexpr uint32_t k = 0x3C003C00u;   // two fp16 1.0 values
    return make_uint4(k, k, k, k);
  }
  __device__ static void launder_vec(Vec& v) { launder(v); }
  __device__ static float get(const void* p, int64_t e) {
    return __half2float(__ushort_as_half(static_cast<const uint16_t*>(p)[e]));
  }
  __device__ static void put(void* p, int64_t e, float f) {
    static_cast<uint16_t*>(p)[e] = __half_as_ushort(__float2half_rn(f));
  }
};

struct V32 {
  uint4 lo, hi;   // elements 0-3 and 4-7 as fp32 bit patterns
};

template <>
struct Io<kF32> {
  using Vec = V32;
  static constexpr int kWords = 8;
  static constexpr int kBytes = 4;
  __device__ static Vec load(const void* p, int64_t e) {
    const float* f = static_cast<const float*>(p) + e;
    return V32{ld_stream16(f), ld_stream16(f + 4)};
  }
  __device__ static Vec load_ro(const void* p, int64_t e) {
    const float* f = static_cast<const float*>(p) + e;
    return V32{ld_ro16(f), ld_ro16(f + 4)};
  }
  __device__ static void store(void* p, int64_t e, const Vec& v) {
    float* f = static_cast<float*>(p) + e;
    st16(f, v.lo);
    st16(f + 4, v.hi);
  }
  __device__ static float2 pair(const Vec& v, int i) {
    const uint4& h = i < 2 ? v.lo : v.hi;
    return (i & 1) ? make_float2(__uint_as_float(h.z), __uint_as_float(h.w))
                   : make_float2(__uint_as_float(h.x), __uint_as_float(h.y));
  }
  __device__ static Vec pack(float2 a, float2 b, float2 c, float2 d) {
    return V32{make_uint4(__float_as_uint(a.x), __float_as_uint(a.y), __float_as_uint(b.x),
                          __float_as_uint(b.y)),
               make_uint4(__float_as_uint(c.x), __float_as_uint(c.y), __float_as_uint(d.x),
                          __float_as_uint(d.y))};
  }
  __device__ static Vec ones() {
    constexpr uint32_t k = 0x3F800000u;
    return V32{make_uint4(k, k, k, k), make_uint4(k, k, k, k)};
  }
  __device__ static void launder_vec(Vec& v) {
    launder(v.lo);
    launder(v.hi);
  }
  __device__ static float get(const void* p, int64_t e) { return static_cast<const float*>(p)[e]; }
  __device__ static void put(void* p, int64_t e, float f) { static_cast<float*>(p)[e] = f; }
};

// Mixed-precision FMA (sm_100 and later): a*b + c with a and b the 16-bit
// halves of 32-bit words (bf16 for FMT 0, fp16 for FMT 1), widened exactly,
// c and the result fp32, one rounding.  It reads the halves where they are,
// so no widening instruction is needed.  `LTXK_MIXED_FMA` 0 keeps the
// widen-then-f32x2 forms; both give the same bits.  Measured on GB300 (event
// means, 3 x 200 launches): interleaved RoPE [2 x 4096 x 32x128]
// 26.52 -> 24.95 us, RMSNorm [2x4096x3072] 18.03 -> 17.70 us; the
// bandwidth-bound shapes unchanged.
#ifndef LTXK_MIXED_FMA
#define LTXK_MIXED_FMA 1
#endif

// (lo(a)*lo(b) + c.x, hi(a)*hi(b) + c.y)
template <int FMT>
__device__ __forceinline__ float2 fma_halves(uint32_t a, uint32_t b, float2 c) {
  float2 d;
  if constexpr (FMT == kBf16) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %4;\n\tfma.rn.f32.bf16 %1, ah, bh, %5;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "r"(a), "r"(b), "f"(c.x), "f"(c.y));
  } else {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %4;\n\tfma.rn.f32.f16 %1, ah, bh, %5;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "r"(a), "r"(b), "f"(c.x), "f"(c.y));
  }
  return d;
}

// Exact products of same halves, (lo(a)*lo(b), hi(a)*hi(b)): two 16-bit
// significands fit fp32, and adding -0 keeps every product, signed zeros
// included, unchanged.
template <int FMT>
__device__ __forceinline__ float2 mul_halves(uint32_t a, uint32_t b) {
  return fma_halves<FMT>(a, b, make_float2(-0.f, -0.f));
}

// Sum of squares of a slot's 8 values, as two fp32 partial sums (even, odd).
template <int FMT>
__device__ __forceinline__ float2 sumsq8(const typename Io<FMT>::Vec& v, float2 s) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (FMT != kF32 && LTXK_MIXED_FMA != 0) {
      const uint32_t u = word_of(v, i);
      s = fma_halves<FMT>(u, u, s);
    } else {
      const float2 p = Io<FMT>::pair(v, i);
      s = __ffma2_rn(p, p, s);
    }
  }
  return s;
}

// round(a + b) for the 8 lanes of two slots.  For bf16 and fp16 the fp32 sum
// of two values is exact unless their exponents differ by more than 12, and
// then the smaller is far below half a spacing of the larger, so the one RNE
// conversion gives the correctly rounded sum; for fp32 it is one rounding.
template <int FMT>
__device__ __forceinline__ typename Io<FMT>::Vec add8(const typename Io<FMT>::Vec& a,
                                                      const typename Io<FMT>::Vec& b) {
  using I = Io<FMT>;
  return I::pack(__fadd2_rn(I::pair(a, 0), I::pair(b, 0)), __fadd2_rn(I::pair(a, 1), I::pair(b, 1)),
                 __fadd2_rn(I::pair(a, 2), I::pair(b, 2)), __fadd2_rn(I::pair(a, 3), I::pair(b, 3)));
}

// ---- slot map, reduction and epilogue shared by the vectorised kernels ----
//
// Thread-to-data map.  A row has NV = hidden/8 16-byte vectors.  The GT
// threads that share a row own VPL vector slots each:
//   plain / interleaved: slot k of thread t holds vector k*GT + t, so each
//     warp-wide access is one contiguous 512-byte span;
//   split-half: slots come in (lo, hi) pairs; pair j of thread t is the
//     pair-vector q = j*GT + t, i.e. vector jv = q % QPH of head q / QPH in
//     the first half (lo) and the same vector in the second half (hi), with
//     QPH = head_dim/16 pair-vectors per head.  Both elements of every
//     rotation pair are then in one thread.

template <int MODE, int VPL, int GT>
struct SlotMap {
  // Offsets are generated slot by slot: plain / interleaved slot k is vector
  // k*GT + t; the rotation-pair column (interleaved) and the (head, vector in
  // head) position (split-half) advance by fixed steps with one conditional
  // subtraction, so no division happens inside the row loop and no per-slot
  // registers are kept.
  int t, nv, D, P, QPH;
  int a0, a1, b0, b1;   // interleaved: (t*8)%D, (GT*8)%D; split: t/QPH, GT/QPH, t%QPH, GT%QPH

  __device__ __forceinline__ SlotMap(const RowArgs& a, int t_)
      : t(t_), nv(a.hidden >> 3), D(a.head_dim), P(a.head_dim >> 1), QPH(a.head_dim >> 4),
        a0(0), a1(0), b0(0), b1(0) {
    if constexpr (MODE == kInterleaved) {
      a0 = (t * 8) % D;
      a1 = (GT * 8) % D;
    } else if constexpr (MODE == kSplitHalf) {
      a0 = t / QPH;
      a1 = GT / QPH;
      b0 = t - a0 * QPH;
      b1 = GT - a1 * QPH;
    }
  }

  // f(k, element offset, first pair column, slot exists) for every slot k.
  template <class F>
  __device__ __forceinline__ void each_slot(F&& f) const {
    static_assert(MODE != kSplitHalf, "split-half slots come in pairs");
    int r = a0;
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const int v = k * GT + t;
      f(k, v * 8, r >> 1, v < nv);
      if constexpr (MODE == kInterleaved) {
        r += a1;
        if (r >= D) r -= D;
      }
    }
  }

  // Split-half: f(j, offset of the lo vector, offset of the hi vector,
  // first pair column, pair exists) for every slot pair j (slots 2j, 2j+1).
  template <class F>
  __device__ __forceinline__ void each_pair(F&& f) const {
    int head = a0, jv = b0;
#pragma unroll
    for (int j = 0; j < VPL / 2; ++j) {
      const int lo = head * D + jv * 8;
      f(j, lo, lo + P, jv * 8, j * GT + t < (nv >> 1));
      head += a1;
      jv += b1;
      if (jv >= QPH) {
        jv -= QPH;
        ++head;
      }
    }
  }

  // fp32 rows without rotation: slot k of thread t is the two 4-float chunks
  // c = 2k*GT + t and c + GT, so that every 16-byte access of a warp is one
  // contiguous 512-byte span (an 8-float slot per lane would leave each
  // access half of every 32-byte sector).  f(k, element offset of the first
  // chunk, of the second, first exists, second exists).
  template <class F>
  __device__ __forceinline__ void each_chunk_slot(F&& f) const {
    const int nc = nv * 2;
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const int c = 2 * k * GT + t;
      f(k, c * 4, (c + GT) * 4, c < nc, c + GT < nc);
    }
  }

  // Load this thread's slots of one row (fetch(off) returns one slot).
  template <class Vec, class Fetch>
  __device__ __forceinline__ void load(Vec (&v)[VPL], Fetch&& fetch) const {
    if constexpr (MODE == kSplitHalf) {
      each_pair([&](int j, int lo, int hi, int, bool ok) {
        v[2 * j] = ok ? fetch(lo) : Vec{};
        v[2 * j + 1] = ok ? fetch(hi) : Vec{};
      });
    } else {
      each_slot([&](int k, int off, int, bool ok) { v[k] = ok ? fetch(off) : Vec{}; });
    }
  }
};

// Whether a row mode and format run on the chunk map above.
template <int MODE, int FMT>
struct ChunkMap {
  static constexpr bool value =
      FMT == kF32 && (MODE == kPlain || MODE == kAdaLN || MODE == kAddNorm);
};

// One fp32 slot from two chunks (absent chunks read as zeros), and back.
__device__ __forceinline__ V32 load_chunks(const void* p, int64_t base, int lo, int hi, bool ok_lo,
                                           bool ok_hi) {
  const float* f = static_cast<const float*>(p) + base;
  return V32{ok_lo ? ld_stream16(f + lo) : make_uint4(0u, 0u, 0u, 0u),
             ok_hi ? ld_stream16(f + hi) : make_uint4(0u, 0u, 0u, 0u)};
}
__device__ __forceinline__ V32 load_chunks_ro(const void* p, int64_t base, int lo, int hi,
                                              bool ok_lo, bool ok_hi) {
  const float* f = static_cast<const float*>(p) + base;
  return V32{ok_lo ? ld_ro16(f + lo) : make_uint4(0u, 0u, 0u, 0u),
             ok_hi ? ld_ro16(f + hi) : make_uint4(0u, 0u, 0u, 0u)};
}
__device__ __forceinline__ void store_chunks(void* p, int64_t base, int lo, int hi, bool ok_lo,
                                             bool ok_hi, const V32& v) {
  float* f = static_cast<float*>(p) + base;
  if (ok_lo) st16(f + lo, v.lo);
  if (ok_hi) st16(f + hi, v.hi);
}

template <int FMT, int VPL>
__device__ __forceinline__ float slots_sumsq(const typename Io<FMT>::Vec (&v)[VPL]) {
  float2 ss = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < VPL; ++k) ss = sumsq8<FMT>(v[k], ss);
  return ss.x + ss.y;
}

__device__ __forceinline__ float inv_rms_of(float ss, const RowArgs& a) {
  return rsqrtf(__fdiv_rn(ss, static_cast<float>(a.hidden)) + a.eps);
}

// Epilogues of the row-only forms: load the next slot's read-only vectors
// (weight; AdaLN's scale and shift) before this slot is stored (1), or each
// slot's right before its use (0).  The loads are kept in program order with
// the stores, so one slot's loads are in flight while the previous slot is
// finished, for the registers of one more slot.  Measured on GB300 (event
// means, 3 x 200 launches): [4x1024x2048] 11.33 -> 10.65 us, [1x1024x2048]
// 8.25 -> 7.90 us, AdaLN [2x6144x2048] 23.88 -> 23.62 us, the other shapes
// unchanged.  (On the interleaved rotation the same lookahead of the weight
// was slower: 24.0 -> 24.85 us.)
#ifndef LTXK_EPI_LOOKAHEAD
#define LTXK_EPI_LOOKAHEAD 1
#endif

// x * w for pair i of a slot, exact for 16-bit formats (two significands of
// at most 11 bits); without a weight (W false: w == NULL, a weight of ones)
// it is x itself, so nothing is loaded, widened or multiplied.
template <bool W, int FMT>
__device__ __forceinline__ float2 times_w(const typename Io<FMT>::Vec& x,
                                          const typename Io<FMT>::Vec& w, int i) {
  if constexpr (W && FMT != kF32 && LTXK_MIXED_FMA != 0)
    return mul_halves<FMT>(word_of(x, i), word_of(w, i));
  else if constexpr (W) return __fmul2_rn(Io<FMT>::pair(x, i), Io<FMT>::pair(w, i));
  else return Io<FMT>::pair(x, i);
}

// Issue a rotation row's shared cos/sin loads together with the row's x
// loads (1), or in the epilogue after the reduction (0).  Rows that are
// software-pipelined keep them in the epilogue.  Measured on GB300 with the
// mixed-precision FMA forms (event means, 3 x 200 launches): interleaved
// [2 x 4096 x 32x128] 24.95 -> 24.01 us.
#ifndef LTXK_TABLE_EARLY
#define LTXK_TABLE_EARLY 1
#endif

// The cos/sin vectors a thread uses for every slot of a row, when its slot
// stride keeps it on the same rotation columns.
struct RowTables {
  float4 c[2], s[2];
};

template <int MODE, int VPL, int GT>
__device__ __forceinline__ bool shares_columns(const SlotMap<MODE, VPL, GT>& m) {
  return MODE == kInterleaved ? m.a1 == 0 : m.b1 == 0;
}

template <int MODE, int VPL, int GT>
__device__ __forceinline__ void load_row_tables(const RowArgs& a, int64_t row,
                                                const SlotMap<MODE, VPL, GT>& m, RowTables& tb) {
  const int64_t pos = row - div_fast(row, a.table_rows, a.table_mul) * a.table_rows;
  const float* ct = a.cos_t + pos * m.P;
  const float* st = a.sin_t + pos * m.P;
  if constexpr (MODE == kInterleaved) {
    tb.c[0] = ld_ro16f(ct + (m.a0 >> 1));
    tb.s[0] = ld_ro16f(st + (m.a0 >> 1));
  } else {
    tb.c[0] = ld_ro16f(ct + m.b0 * 8);
    tb.c[1] = ld_ro16f(ct + m.b0 * 8 + 4);
    tb.s[0] = ld_ro16f(st + m.b0 * 8);
    tb.s[1] = ld_ro16f(st + m.b0 * 8 + 4);
  }
}

// Split-half rows of 16-bit formats, of at most 8 warps and 8 slots per
// lane, keep the thread's weight in registers within the same budget (fp32
// rows, wider slot sets and the 512- and 1024-thread row groups would spill).
// The interleaved rows keep loading theirs: in registers (16 more per
// thread, 6 instead of 8 CTAs per SM) [2x4096, 32x128] measured 24.1 ->
// 24.8 us on GB300 (event means).
#ifndef LTXK_W_REGS_INTERLEAVED
#define LTXK_W_REGS_INTERLEAVED 0
#endif
template <int MODE, int G, int VPL, int FMT>
struct WeightInRegs {
  static constexpr bool value =
      FMT != kF32 && G <= 8 && VPL <= 8 &&
      ((MODE == kSplitHalf && LTXK_W_REGS != 0) ||
       (MODE == kInterleaved && LTXK_W_REGS_INTERLEAVED != 0));
};

// Scale (and rotate) the thread's slots of one row and store them.  W says
// whether the row has a weight (a.w != NULL); the kernels dispatch on it once
// per launch, so a weightless norm skips the weight entirely.  WR: the
// rotation forms take the thread's weight vectors from wr[] (registers the
// caller loaded once) instead of loading them.
template <int MODE, int VPL, int GT, int FMT, bool W, bool WR = false>
__device__ __forceinline__ void row_epilogue(const RowArgs& a, int64_t row,
                                             typename Io<FMT>::Vec (&v)[VPL],
                                             const SlotMap<MODE, VPL, GT>& m, float inv_rms,
                                             const RowTables* early = nullptr,
                                             const unsigned char* cond_s = nullptr,
                                             const typename Io<FMT>::Vec* wr = nullptr) {
  using I = Io<FMT>;
  using Vec = typename I::Vec;
#pragma unroll
  for (int k = 0; k < VPL; ++k) I::launder_vec(v[k]);
  const int64_t rb = row * a.hidden;
  const float2 inv2 = make_float2(inv_rms, inv_rms);
  if constexpr (ChunkMap<MODE, FMT>::value) {
    // the same arithmetic as below, on the chunk map
    const int64_t cb = MODE == kAdaLN ? div_fast(row, a.rows_per_cond, a.cond_mul) * a.hidden : 0;
    const float2 one2 = make_float2(1.f, 1.f);
    m.each_chunk_slot([&](int k, int lo, int hi, bool ok_lo, bool ok_hi) {
      Vec wv{};
      if constexpr (W) wv = load_chunks_ro(a.w, 0, lo, hi, ok_lo, ok_hi);
      float2 o[4];
      if constexpr (MODE == kAdaLN) {
        const Vec sv = load_chunks_ro(a.scale, cb, lo, hi, ok_lo, ok_hi);
        const Vec tv = load_chunks_ro(a.shift, cb, lo, hi, ok_lo, ok_hi);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 n = __fmul2_rn(times_w<W, FMT>(v[k], wv, i), inv2);
          o[i] = __ffma2_rn(n, __fadd2_rn(one2, I::pair(sv, i)), I::pair(tv, i));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = __fmul2_rn(times_w<W, FMT>(v[k], wv, i), inv2);
      }
      store_chunks(a.out, rb, lo, hi, ok_lo, ok_hi, I::pack(o[0], o[1], o[2], o[3]));
    });
    return;
  } else if constexpr ((MODE == kPlain || MODE == kAddNorm || MODE == kAdaLN) &&
                       LTXK_EPI_LOOKAHEAD != 0) {
    // The same arithmetic as below, with slot k+1's read-only vectors (w,
    // scale, shift) loaded before slot k is computed and stored, so that one
    // slot's loads are in flight while the previous one is finished.
    const int64_t cb = MODE == kAdaLN ? div_fast(row, a.rows_per_cond, a.cond_mul) * a.hidden : 0;
    const float2 one2 = make_float2(1.f, 1.f);
    Vec wn{}, sn{}, tn{};
    auto fetch = [&](int k, Vec& wv, Vec& sv, Vec& tv) {
      const int vec = k * GT + m.t;
      if (vec >= m.nv) return;
      if constexpr (W) wv = I::load_ro(a.w, vec * 8);
      if constexpr (MODE == kAdaLN) {
        if (cond_s != nullptr) {   // this row's conditioning row, staged
          sv = *reinterpret_cast<const Vec*>(cond_s + vec * 8 * I::kBytes);
          tv = *reinterpret_cast<const Vec*>(cond_s + (a.hidden + vec * 8) * I::kBytes);
        } else {
          sv = I::load_ro(a.scale, cb + vec * 8);
          tv = I::load_ro(a.shift, cb + vec * 8);
        }
      }
    };
    fetch(0, wn, sn, tn);
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const Vec wv = wn, sv = sn, tv = tn;
      if (k + 1 < VPL) fetch(k + 1, wn, sn, tn);
      const int vec = k * GT + m.t;
      if (vec >= m.nv) continue;
      float2 o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 n = __fmul2_rn(times_w<W, FMT>(v[k], wv, i), inv2);
        if constexpr (MODE == kAdaLN)
          o[i] = __ffma2_rn(n, __fadd2_rn(one2, I::pair(sv, i)), I::pair(tv, i));
        else
          o[i] = n;
      }
      I::store(a.out, rb + vec * 8, I::pack(o[0], o[1], o[2], o[3]));
    }
    return;
  } else if constexpr (MODE == kPlain || MODE == kAddNorm) {
    m.each_slot([&](int k, int off, int, bool ok) {
      if (!ok) return;
      Vec wv{};
      if constexpr (W) wv = I::load_ro(a.w, off);
      float2 o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)   // (x * w) exact for 16-bit formats; one rounding by inv_rms
        o[i] = __fmul2_rn(times_w<W, FMT>(v[k], wv, i), inv2);
      I::store(a.out, rb + off, I::pack(o[0], o[1], o[2], o[3]));
    });
    return;
  } else if constexpr (MODE == kAdaLN) {
    // y = n * (1 + scale) + shift with n = (x * w) * inv_rms; one conditioning
    // row serves rows_per_cond rows, so its vectors come from L1/L2
    const int64_t cb = div_fast(row, a.rows_per_cond, a.cond_mul) * a.hidden;
    const float2 one2 = make_float2(1.f, 1.f);
    m.each_slot([&](int k, int off, int, bool ok) {
      if (!ok) return;
      Vec wv{};
      if constexpr (W) wv = I::load_ro(a.w, off);
      const Vec sv = I::load_ro(a.scale, cb + off);
      const Vec tv = I::load_ro(a.shift, cb + off);
      float2 o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 n = __fmul2_rn(times_w<W, FMT>(v[k], wv, i), inv2);
        o[i] = __ffma2_rn(n, __fadd2_rn(one2, I::pair(sv, i)), I::pair(tv, i));
      }
      I::store(a.out, rb + off, I::pack(o[0], o[1], o[2], o[3]));
    });
    return;
  } else {
    const int64_t pos = row - div_fast(row, a.table_rows, a.table_mul) * a.table_rows;
    const float* ct = a.cos_t + pos * m.P;
    const float* st = a.sin_t + pos * m.P;
    if constexpr (MODE == kInterleaved) {
      // When the slot stride is a multiple of head_dim (a1 == 0), every slot
      // of this thread uses the same four rotation columns: load them once.
      const bool same_cols = m.a1 == 0;
      float4 c4h = make_float4(0.f, 0.f, 0.f, 0.f), s4h = c4h;
      if (same_cols && early != nullptr) {
        c4h = early->c[0];
        s4h = early->s[0];
      } else if (same_cols) {
        c4h = ld_ro16f(ct + (m.a0 >> 1));
        s4h = ld_ro16f(st + (m.a0 >> 1));
      }
      m.each_slot([&](int k, int off, int pair0, bool ok) {
        if (!ok) return;
        Vec wv{};
        if constexpr (W && WR) wv = wr[k];
        else if constexpr (W) wv = I::load_ro(a.w, off);
        const float4 c4 = same_cols ? c4h : ld_ro16f(ct + pair0);
        const float4 s4 = same_cols ? s4h : ld_ro16f(st + pair0);
        const float2 c[2] = {make_float2(c4.x, c4.y), make_float2(c4.z, c4.w)};
        const float2 s[2] = {make_float2(s4.x, s4.y), make_float2(s4.z, s4.w)};
        float2 o[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // pairs 2h and 2h+1 of the slot are rotation pairs 2h and 2h+1:
          // lane x of each float2 is the first of them, lane y the second
          float2 u, q;
          if constexpr (W && FMT != kF32 && LTXK_MIXED_FMA != 0) {
            const float2 p0 = mul_halves<FMT>(word_of(v[k], 2 * h), word_of(wv, 2 * h));
            const float2 p1 = mul_halves<FMT>(word_of(v[k], 2 * h + 1), word_of(wv, 2 * h + 1));
            u = make_float2(p0.x, p1.x);   // a * w
            q = make_float2(p0.y, p1.y);   // b * w
          } else {
            const float2 x0 = I::pair(v[k], 2 * h), x1 = I::pair(v[k], 2 * h + 1);
            u = make_float2(x0.x, x1.x);
            q = make_float2(x0.y, x1.y);
            if constexpr (W) {
              const float2 w0 = I::pair(wv, 2 * h), w1 = I::pair(wv, 2 * h + 1);
              u = __fmul2_rn(u, make_float2(w0.x, w1.x));   // a * w
              q = __fmul2_rn(q, make_float2(w0.y, w1.y));   // b * w
            }
          }
          const float2 ra = __fmul2_rn(diff_of_products2(u, c[h], q, s[h]), inv2);
          const float2 rb2 = __fmul2_rn(diff_of_products2(u, s[h], neg2(q), c[h]), inv2);
          o[2 * h] = make_float2(ra.x, rb2.x);
          o[2 * h + 1] = make_float2(ra.y, rb2.y);
        }
        I::store(a.out, rb + off, I::pack(o[0], o[1], o[2], o[3]));
      });
    } else {
      // Same idea: when the pair-vector stride is a multiple of the vectors
      // per half-head (b1 == 0), the columns are the same for every pair.
      const bool same_cols = m.b1 == 0;
      float4 c0h = make_float4(0.f, 0.f, 0.f, 0.f), c1h = c0h, s0h = c0h, s1h = c0h;
      if (same_cols && early != nullptr) {
        c0h = early->c[0];
        c1h = early->c[1];
        s0h = early->s[0];
        s1h = early->s[1];
      } else if (same_cols) {
        c0h = ld_ro16f(ct + m.b0 * 8);
        c1h = ld_ro16f(ct + m.b0 * 8 + 4);
        s0h = ld_ro16f(st + m.b0 * 8);
        s1h = ld_ro16f(st + m.b0 * 8 + 4);
      }
      m.each_pair([&](int j, int lo_off, int hi_off, int pair0, bool ok) {
        if (!ok) return;
        const int kl = 2 * j, kh = 2 * j + 1;
        Vec wl{}, wh{};
        if constexpr (W && WR) {   // kept in registers by the caller
          wl = wr[kl];
          wh = wr[kh];
        } else if constexpr (W) {
          wl = I::load_ro(a.w, lo_off);
          wh = I::load_ro(a.w, hi_off);
        }
        const float4 c0 = same_cols ? c0h : ld_ro16f(ct + pair0);
        const float4 c1 = same_cols ? c1h : ld_ro16f(ct + pair0 + 4);
        const float4 s0 = same_cols ? s0h : ld_ro16f(st + pair0);
        const float4 s1 = same_cols ? s1h : ld_ro16f(st + pair0 + 4);
        const float2 c[4] = {make_float2(c0.x, c0.y), make_float2(c0.z, c0.w),
                             make_float2(c1.x, c1.y), make_float2(c1.z, c1.w)};
        const float2 s[4] = {make_float2(s0.x, s0.y), make_float2(s0.z, s0.w),
                             make_float2(s1.x, s1.y), make_float2(s1.z, s1.w)};
        float2 ol[4], oh[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {   // rotation pairs 2i, 2i+1: (lo pair i, hi pair i)
          const float2 u = times_w<W, FMT>(v[kl], wl, i);
          const float2 q = times_w<W, FMT>(v[kh], wh, i);
          ol[i] = __fmul2_rn(diff_of_products2(u, c[i], q, s[i]), inv2);
          oh[i] = __fmul2_rn(diff_of_products2(u, s[i], neg2(q), c[i]), inv2);
        }
        I::store(a.out, rb + lo_off, I::pack(ol[0], ol[1], ol[2], ol[3]));
        I::store(a.out, rb + hi_off, I::pack(oh[0], oh[1], oh[2], oh[3]));
      });
    }
  }
}

// ---- register kernel: G warps per row, row loaded straight into registers -

// Threads per CTA of the register kernel when a row group is smaller.  Plain
// and AdaLN rows of one or two warps use LTXK_VEC_BLOCK_SMALL_ROWS: eight or
// four rows per CTA, which halves the per-row share of a CTA's set-up
// (AdaLN's staged conditioning row above all).  Measured on GB300 (event
// means): AdaLN [2x6144x2048] 21.05 -> 20.77 us, [2x1024x2048] 9.65 -> 8.55 us,
// the stress rows unchanged; four-warp rows keep 128 threads (with 256 they
// were slower: [4x4096x3072] 30.5 -> 33.1 us), and so do the residual-add
// rows (two rows of inputs in registers: at 256 threads only one CTA fits
// on an SM).
#ifndef LTXK_VEC_BLOCK
#define LTXK_VEC_BLOCK 128
#endif
#ifndef LTXK_VEC_BLOCK_SMALL_ROWS
#define LTXK_VEC_BLOCK_SMALL_ROWS 256
#endif

__host__ __device__ constexpr int vec_block(int mode, int g) {
  return (mode == kPlain || mode == kAdaLN) && g <= 2
             ? LTXK_VEC_BLOCK_SMALL_ROWS
             : (32 * g >= LTXK_VEC_BLOCK ? 32 * g : LTXK_VEC_BLOCK);
}

template <int MODE, int G>
struct GroupShape {
  static constexpr int kThreadsPerGroup = 32 * G;
  static constexpr int kBlock = vec_block(MODE, G);
  static constexpr int kGroupsPerCta = kBlock / kThreadsPerGroup;
};

// Register budget per thread of the register kernel: the row's kWords*VPL
// words plus what the epilogue needs (weights, and for RoPE the cos/sin
// vectors).
// Capping it lets more warps, hence more bytes of x, be in flight per SM.
#ifndef LTXK_REG_EXTRA_PLAIN
#define LTXK_REG_EXTRA_PLAIN 32
#endif
#ifndef LTXK_REG_EXTRA_INTERLEAVED
#define LTXK_REG_EXTRA_INTERLEAVED 48
#endif
#ifndef LTXK_REG_EXTRA_SPLIT
#define LTXK_REG_EXTRA_SPLIT 96
#endif
#ifndef LTXK_REG_EXTRA_ADALN
#define LTXK_REG_EXTRA_ADALN (LTXK_REG_EXTRA_PLAIN + 16)
#endif
// Software pipelining of the register kernel: a warp issues the loads of
// its next row before the epilogue of the current one, so HBM reads keep
// flowing while rows are scaled and stored (costs one more row of slots in
// registers).  Not for the residual-add form (two rows of inputs already).
// Measured on GB300 under the bench protocol: split-half RoPE
// [6144 x 32x64] 16.1 -> 15.4 us, so it is on there for the 16-bit formats
// and rows of at most 8 warps (LTXK_PIPELINE_SPLIT; fp32 rows, and the
// 512- and 1024-thread row groups, would spill the second row of slots);
// interleaved RoPE unchanged, AdaLN +7 %, plain RMSNorm +1-2 %, so it is
// off for them (LTXK_PIPELINE turns it on for every mode and format).
#ifndef LTXK_PIPELINE
#define LTXK_PIPELINE 0
#endif
#ifndef LTXK_PIPELINE_SPLIT
#define LTXK_PIPELINE_SPLIT 1
#endif
#ifndef LTXK_TABLE_NEXT_REGS
#define LTXK_TABLE_NEXT_REGS (LTXK_TABLE_NEXT != 0 ? 16 : 0)
#endif
template <int MODE, int G, int FMT>
struct Pipelined {
  static constexpr bool value =
      LTXK_PIPELINE != 0
          ? MODE != kAddNorm
          : (MODE == kSplitHalf && FMT != kF32 && G <= 8 && LTXK_PIPELINE_SPLIT != 0);
};


template <int MODE, int G, int VPL, int FMT>
struct RegBudget {
  static constexpr int kW = Io<FMT>::kWords;
  static constexpr int kRegs =
      kW * VPL * (Pipelined<MODE, G, FMT>::value ? 2 : 1) +
      (Pipelined<MODE, G, FMT>::value && (MODE == kInterleaved || MODE == kSplitHalf)
           ? LTXK_TABLE_NEXT_REGS   // the next row's cos/sin vectors
           : 0) +
                 (MODE == kPlain          ? LTXK_REG_EXTRA_PLAIN
                  : MODE == kInterleaved  ? LTXK_REG_EXTRA_INTERLEAVED
                  : MODE == kSplitHalf    ? LTXK_REG_EXTRA_SPLIT
                  : MODE == kAddNorm      ? kW * VPL + LTXK_REG_EXTRA_PLAIN  // x and res in flight
                                          : LTXK_REG_EXTRA_ADALN);
};
template <int MODE, int G, int VPL, int FMT>
struct VecLaunch {
  static constexpr int kBlock = GroupShape<MODE, G>::kBlock;
  static constexpr int kMin = 65536 / (kBlock * RegBudget<MODE, G, VPL, FMT>::kRegs);
  static constexpr int kMinBlocks = kMin < 1 ? 1 : kMin;
};

template <int MODE, int G, int VPL, int FMT>
__global__ void __launch_bounds__(VecLaunch<MODE, G, VPL, FMT>::kBlock,
                                  VecLaunch<MODE, G, VPL, FMT>::kMinBlocks)
rows_vec_kernel(const RowArgs a) {
  using I = Io<FMT>;
  using Vec = typename I::Vec;
  using S = GroupShape<MODE, G>;
  constexpr int GT = S::kThreadsPerGroup;
  static_assert(MODE != kSplitHalf || VPL % 2 == 0, "split-half slots come in pairs");
  __shared__ float red[2][S::kGroupsPerCta][G];

  const int tid = threadIdx.x;
  const int group = tid / GT;
  const int t = tid % GT;
  const int warp_in_group = t >> 5;
  const int lane = tid & 31;
  const SlotMap<MODE, VPL, GT> m(a, t);

  const int64_t row_step = static_cast<int64_t>(gridDim.x) * S::kGroupsPerCta;
  constexpr bool kPipe = Pipelined<MODE, G, FMT>::value;
  int parity = 0;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * S::kGroupsPerCta + group;
  Vec v[VPL];
  // one row of slots of src at element base (the chunk map for fp32 rows
  // without rotation, the vector map otherwise)
  auto load_row = [&](Vec (&dst)[VPL], const void* src, int64_t base) {
    if constexpr (ChunkMap<MODE, FMT>::value) {
      m.each_chunk_slot([&](int k, int lo, int hi, bool ok_lo, bool ok_hi) {
        dst[k] = load_chunks(src, base, lo, hi, ok_lo, ok_hi);
      });
    } else {
      m.load(dst, [&](int off) { return I::load(src, base + off); });
    }
  };
  if (kPipe && first < a.rows) load_row(v, a.x, first * a.hidden);
  // AdaLN, 16-bit rows: the CTA stages the conditioning row of its first row
  // (scale, then shift) in shared memory once, after that row's x loads are
  // out; its rows of that conditioning row read it there, the others from
  // memory.  Every slot would otherwise wait on two L1/L2 loads.
  constexpr bool kStageCond = MODE == kAdaLN && FMT != kF32 && LTXK_ADALN_STAGE != 0;
  extern __shared__ __align__(16) unsigned char stage_smem[];
  const unsigned char* cond_base = nullptr;
  int64_t staged_cond = -1;
  bool preloaded = false;
  if constexpr (kStageCond) {
    if (a.stage_cond != 0) {   // the same for the whole CTA
      if (!kPipe && first < a.rows) {
        load_row(v, a.x, first * a.hidden);
        preloaded = true;
      }
      const int64_t r0 = static_cast<int64_t>(blockIdx.x) * S::kGroupsPerCta;
      if (r0 < a.rows) {
        const int nvec = a.hidden * I::kBytes / 16;   // 16-byte vectors per row
        staged_cond = div_fast(r0, a.rows_per_cond, a.cond_mul);
        const unsigned char* scp =
            static_cast<const unsigned char*>(a.scale) + staged_cond * nvec * 16;
        const unsigned char* shp =
            static_cast<const unsigned char*>(a.shift) + staged_cond * nvec * 16;
        uint4* d = reinterpret_cast<uint4*>(stage_smem);
        for (int i = tid; i < nvec; i += static_cast<int>(blockDim.x)) {
          d[i] = ld_ro16(scp + i * 16);
          d[nvec + i] = ld_ro16(shp + i * 16);
        }
        cond_base = stage_smem;
      }
      __syncthreads();
    }
  }
  // Split-half rotation: the thread's weight vectors, loaded once (after the
  // first row's x loads) for all the rows the persistent CTA serves.
  constexpr bool kWRegs = WeightInRegs<MODE, G, VPL, FMT>::value;
  Vec wreg[kWRegs ? VPL : 1];
  if constexpr (kWRegs) {
    if (a.w != nullptr) {
      if (!kPipe && first < a.rows) {
        load_row(v, a.x, first * a.hidden);
        preloaded = true;
      }
      if constexpr (MODE == kInterleaved) {
        m.each_slot([&](int k, int off, int, bool ok) {
          if (ok) wreg[k] = I::load_ro(a.w, off);
        });
      } else {
        m.each_pair([&](int j, int lo_off, int hi_off, int, bool ok) {
          if (!ok) return;
          wreg[2 * j] = I::load_ro(a.w, lo_off);
          wreg[2 * j + 1] = I::load_ro(a.w, hi_off);
        });
      }
    }
  }
  // Pipelined rotation rows: the next row's shared cos/sin vectors go out
  // with its x loads (LTXK_TABLE_NEXT), held in registers until its epilogue;
  // tbc holds the current row's.
  constexpr bool kTableNext = kPipe && (MODE == kInterleaved || MODE == kSplitHalf) &&
                              LTXK_TABLE_NEXT != 0;
  RowTables tbc, tbn;
  if constexpr (kTableNext) {
    if (first < a.rows && shares_columns(m)) load_row_tables(a, first, m, tbc);
  }
  for (int64_t row = first; row < a.rows; row += row_step) {
    const int64_t rb = row * a.hidden;
    if (LTXK_L2_PREFETCH_ROWS > 0 && t == 0 && (a.hidden & 7) == 0) {
      const int64_t ahead = row + LTXK_L2_PREFETCH_ROWS * row_step;
      if (ahead < a.rows)
        prefetch_l2(static_cast<const char*>(a.x) + ahead * a.hidden * I::kBytes,
                    static_cast<uint32_t>(a.hidden) * I::kBytes);
    }
    Vec nv[kPipe ? VPL : 1];
    constexpr bool kEarly = (MODE == kInterleaved || MODE == kSplitHalf) && !kPipe &&
                            LTXK_TABLE_EARLY != 0;
    RowTables tb;
    if constexpr (kPipe) {
      const int64_t next = row + row_step;
      if (next < a.rows) {
        load_row(nv, a.x, next * a.hidden);
        if constexpr (kTableNext) {
          if (shares_columns(m)) load_row_tables(a, next, m, tbn);
        }
      }
    } else {
      if constexpr (kStageCond || kWRegs) {
        if (preloaded) preloaded = false;   // the first row went out before the set-up
        else load_row(v, a.x, rb);
      } else {
        load_row(v, a.x, rb);
      }
      if constexpr (kEarly) {
        if (shares_columns(m)) load_row_tables(a, row, m, tb);
      }
    }
    if constexpr ((MODE == kInterleaved || MODE == kSplitHalf) && LTXK_TABLE_PREFETCH > 0) {
      const int64_t pos = row - div_fast(row, a.table_rows, a.table_mul) * a.table_rows;
      const int col = MODE == kInterleaved ? (m.a0 >> 1) : m.b0 * 8;
      prefetch_line<LTXK_TABLE_PREFETCH>(a.cos_t + pos * m.P + col);
      prefetch_line<LTXK_TABLE_PREFETCH>(a.sin_t + pos * m.P + col);
    }
    if constexpr (MODE == kAddNorm) {
      // h = round(x + res): stored as the new residual stream, then normalised
      Vec rv[VPL];
      load_row(rv, a.res, rb);
#pragma unroll
      for (int k = 0; k < VPL; ++k) v[k] = add8<FMT>(v[k], rv[k]);
      if constexpr (ChunkMap<MODE, FMT>::value) {
        m.each_chunk_slot([&](int k, int lo, int hi, bool ok_lo, bool ok_hi) {
          store_chunks(a.h_out, rb, lo, hi, ok_lo, ok_hi, v[k]);
        });
      } else {
        m.each_slot([&](int k, int off, int, bool ok) {
          if (ok) I::store(a.h_out, rb + off, v[k]);
        });
      }
    }

    float ss = warp_sum(slots_sumsq<FMT>(v));
    if (G > 1) {
      if (lane == 0) red[parity][group][warp_in_group] = ss;
      if (S::kGroupsPerCta == 1) __syncthreads();
      else group_barrier(1 + group, GT);
      ss = 0.f;
#pragma unroll
      for (int i = 0; i < G; ++i) ss += red[parity][group][i];
      parity ^= 1;
    }
    const RowTables* early = kEarly && shares_columns(m)        ? &tb
                             : kTableNext && shares_columns(m) ? &tbc
                                                               : nullptr;
    const unsigned char* cond_s = nullptr;
    if constexpr (kStageCond) {
      if (cond_base != nullptr && div_fast(row, a.rows_per_cond, a.cond_mul) == staged_cond)
        cond_s = cond_base;
    }
    if (a.w != nullptr)
      row_epilogue<MODE, VPL, GT, FMT, true, kWRegs>(a, row, v, m, inv_rms_of(ss, a), early,
                                                     cond_s, wreg);
    else
      row_epilogue<MODE, VPL, GT, FMT, false>(a, row, v, m, inv_rms_of(ss, a), early, cond_s);
    if constexpr (kPipe) {
#pragma unroll
      for (int k = 0; k < VPL; ++k) v[k] = nv[k];
      if constexpr (kTableNext) tbc = tbn;
    }
  }
}

// ---- TMA ring kernel: one warp per row, rows streamed through shared memory -
//
// Each warp owns a ring of `stages` row buffers in shared memory.  Lane 0
// keeps up to `stages` rows of x in flight with 1-D bulk copies
// (cp.async.bulk, completion counted in bytes on one mbarrier per buffer).
// For each row the warp waits for its buffer, copies the row into registers
// (the same slot map as above), immediately hands the buffer back to the
// copy engine for the row `stages` positions later, and only then reduces,
// scales and stores.  HBM reads therefore keep flowing while rows are being
// reduced and written, with no registers held for the rows in flight.
//
// Every wait is bounded (a %globaltimer limit).  A wait that runs out sets
// bit 0 of the device fault word, waits (again bounded) for the copies this
// warp still has in flight, and returns; the host reads the word with
// ltxk_fault_status().

constexpr int kTmaWarps = 8;
constexpr int kTmaMaxStages = 8;
constexpr uint32_t kTmaBarBytes = kTmaWarps * kTmaMaxStages * 8;   // 512

struct TmaArgs {
  RowArgs a;
  int stages;               // row buffers per warp (1..kTmaMaxStages)
  uint32_t stage_stride;    // bytes between buffers (row bytes rounded to 128)
  uint64_t wait_limit_ns;   // bound on every mbarrier wait
  int skip_first_copy;      // diagnostic: never issue the copy of a warp's
                            // first row (its wait then runs out)
  unsigned int* fault;      // device fault word
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done) : "r"(bar), "r"(parity) : "memory");
  return done != 0;
}

// Wait for phase `parity` of the barrier to complete, for at most limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// One elected lane: expect `bytes` on the barrier, then start the copy.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(bar), "r"(bytes) : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ uint4 ld_shared16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

template <int MODE, int VPL>
__global__ void __launch_bounds__(kTmaWarps * 32)
rows_tma_kernel(const TmaArgs ta) {
  extern __shared__ __align__(128) unsigned char smem[];
  const RowArgs& a = ta.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = ta.stages;
  const uint32_t row_bytes = static_cast<uint32_t>(a.hidden) * 2u;
  const uint32_t bars = smem_u32(smem) + warp * kTmaMaxStages * 8;
  const uint32_t ring = smem_u32(smem) + kTmaBarBytes + warp * S * ta.stage_stride;
  const SlotMap<MODE, VPL, 32> m(a, lane);

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(bars + 8 * s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kTmaWarps;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kTmaWarps + warp;
  // rows of this warp: first + i * nwarps, i = 0, 1, ...; row i uses buffer
  // i % S in phase (i / S) & 1.
  if (lane == 0) {
    for (int i = 0; i < S; ++i) {
      const int64_t r = first + i * nwarps;
      if (r >= a.rows) break;
      if (i == 0 && ta.skip_first_copy) continue;
      bulk_load(ring + i * ta.stage_stride, static_cast<const uint16_t*>(a.x) + r * a.hidden,
                row_bytes, bars + 8 * i);
    }
  }

  int64_t i = 0;
  for (int64_t row = first; row < a.rows; row += nwarps, ++i) {
    const int s = static_cast<int>(i % S);
    const uint32_t parity = static_cast<uint32_t>((i / S) & 1);
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bars + 8 * s, parity,
                                                              ta.wait_limit_ns));
    if (!ok) {
      // Record the fault, then wait (bounded) for this warp's other copies
      // in flight (rows i+1 .. i+S-1) so that none lands after the CTA exits.
      if (lane == 0) {
        atomicOr(ta.fault, 1u);
        for (int64_t j = i + 1; j < i + S && first + j * nwarps < a.rows; ++j)
          mbar_wait_bounded(bars + 8 * static_cast<int>(j % S),
                            static_cast<uint32_t>((j / S) & 1), ta.wait_limit_ns);
      }
      __syncwarp();
      return;
    }
    uint4 v[VPL];
    const uint32_t buf = ring + s * ta.stage_stride;
    m.load(v, [&](int off) { return ld_shared16(buf + off * 2); });
    __syncwarp();
    if (lane == 0) {
      const int64_t next = row + S * nwarps;
      if (next < a.rows) {
        // order this warp's generic-proxy reads of the buffer before the
        // async-proxy write that refills it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        bulk_load(buf, static_cast<const uint16_t*>(a.x) + next * a.hidden, row_bytes,
                  bars + 8 * s);
      }
    }
    const float ss = warp_sum(slots_sumsq<kBf16>(v));
    if (a.w != nullptr) row_epilogue<MODE, VPL, 32, kBf16, true>(a, row, v, m, inv_rms_of(ss, a));
    else row_epilogue<MODE, VPL, 32, kBf16, false>(a, row, v, m, inv_rms_of(ss, a));
  }
}

// ---- element-wise kernel (any alignment, any hidden) ---------------------
//
// One CTA per row (persistent stride over rows), two passes: the first sums
// the squares, the second re-reads the row and writes it.  In the fused
// modes each thread owns whole rotation pairs, so out may alias x in place.

constexpr int kElemBlock = 256;

__device__ __forceinline__ float block_sum(float v, float* scratch /* [32] */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float t = 0.f;
  const int nw = blockDim.x >> 5;
  for (int i = 0; i < nw; ++i) t += scratch[i];
  __syncthreads();
  return t;
}

template <int MODE, int FMT>
__global__ void __launch_bounds__(kElemBlock)
rows_elem_kernel(const RowArgs a) {
  using I = Io<FMT>;
  __shared__ float scratch[32];
  const int64_t H = a.hidden;
  const bool has_w = a.w != nullptr;
  for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
    const int64_t rb = row * H;
    float ss = 0.f;
    if (MODE == kAddNorm) {
      // h = round(x + res), stored as the new residual stream; each thread
      // reads back only the elements it wrote itself
      for (int64_t j = threadIdx.x; j < H; j += blockDim.x) {
        I::put(a.h_out, rb + j, __fadd_rn(I::get(a.x, rb + j), I::get(a.res, rb + j)));
        const float v = I::get(a.h_out, rb + j);
        ss = __fmaf_rn(v, v, ss);
      }
    } else {
      for (int64_t j = threadIdx.x; j < H; j += blockDim.x) {
        const float v = I::get(a.x, rb + j);
        ss = __fmaf_rn(v, v, ss);
      }
    }
    // block_sum ends with a barrier, so every read of this row is done
    // before any thread writes it (in-place safe), and scratch is free for
    // the next row.
    ss = block_sum(ss, scratch);
    const float inv_rms = rsqrtf(__fdiv_rn(ss, static_cast<float>(H)) + a.eps);
    if (MODE == kPlain || MODE == kAddNorm) {
      const void* src = MODE == kAddNorm ? static_cast<const void*>(a.h_out) : a.x;
      for (int64_t j = threadIdx.x; j < H; j += blockDim.x) {
        const float wj = has_w ? I::get(a.w, j) : 1.f;
        I::put(a.out, rb + j, __fmul_rn(__fmul_rn(I::get(src, rb + j), wj), inv_rms));
      }
    } else if (MODE == kAdaLN) {
      const int64_t cb = (row / a.rows_per_cond) * H;
      for (int64_t j = threadIdx.x; j < H; j += blockDim.x) {
        const float wj = has_w ? I::get(a.w, j) : 1.f;
        const float n = __fmul_rn(__fmul_rn(I::get(a.x, rb + j), wj), inv_rms);
        const float sc = __fadd_rn(1.f, I::get(a.scale, cb + j));
        I::put(a.out, rb + j, __fmaf_rn(n, sc, I::get(a.shift, cb + j)));
      }
    } else {
      const int64_t D = a.head_dim, P = D >> 1;
      const int64_t pos = row % a.table_rows;
      const float* ct = a.cos_t + pos * P;
      const float* st = a.sin_t + pos * P;
      for (int64_t q = threadIdx.x; q < (H >> 1); q += blockDim.x) {
        const int64_t head = q / P, p = q - head * P;
        const int64_t ia = MODE == kInterleaved ? head * D + 2 * p : head * D + p;
        const int64_t ib = MODE == kInterleaved ? ia + 1 : ia + P;
        const float wa = has_w ? I::get(a.w, ia) : 1.f;
        const float wb = has_w ? I::get(a.w, ib) : 1.f;
        const float u = __fmul_rn(I::get(a.x, rb + ia), wa);
        const float v = __fmul_rn(I::get(a.x, rb + ib), wb);
        const float c = ct[p], s = st[p];
        const float ra = __fmul_rn(diff_of_products(u, c, v, s), inv_rms);
        const float rb2 = __fmul_rn(sum_of_products(u, s, v, c), inv_rms);
        I::put(a.out, rb + ia, ra);
        I::put(a.out, rb + ib, rb2);
      }
    }
  }
}

}  // namespace ltxk
