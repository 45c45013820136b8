// ltxk_kernels.cuh -- device code for bf16 RMSNorm and fused RMSNorm + RoPE
// on sm_103a (GB300).
//
// The operation (no formula is printed on the pages; this is the definition
// the library implements):
//   per row r:  ms = (1/H) sum_j x_j^2,  n_j = x_j * w_j / sqrt(ms + eps)
//   fused:      per head and pair (a, b):  a' = a c - b s,  b' = a s + b c
//   one round-to-nearest-even to bfloat16 at the end.
// Sources: "cuda-kernels" skill page (Hugging Face), "Kernel-Specific
// Guidelines / RMSNorm" and "/ RoPE", "Core Kernel Patterns / Vectorized
// Memory Access" and "/ Warp Shuffle Reductions"; "ltx-kernels" README,
// opening list (`ops_cpp`: rms_norm_rope, rms_norm_split_rope).
//
// The path is bound by HBM bandwidth (4 bytes moved per element against a
// handful of fp32 operations), so it uses no tensor cores.  Design:
//   * Each row is read from HBM exactly once, as 16-byte vectors, into
//     registers; a group of G warps owns one row (G = 1 for hidden <= 4096).
//   * fp32 sum of squares: per-lane partials, an xor-butterfly over the
//     warp, then (G > 1) a fixed-order sum of the G warp totals through
//     shared memory.  Every thread ends with the same bit-identical total.
//   * inv_rms = rsqrtf(ss / H + eps); y = (x * w) * inv_rms, where x * w is
//     exact in fp32 (two 8-bit significands), so each output is one fp32
//     rounding away from (x w) * inv_rms before the final bf16 rounding.
//   * RoPE rotates (u, v) = (x_a w_a, x_b w_b) (both exact) and scales by
//     inv_rms afterwards; u c - v s and u s + v c are evaluated with Kahan's
//     2x2-determinant algorithm (W. Kahan; error bound in Jeannerod, Louvet &
//     Muller, "Further analysis of Kahan's algorithm for the accurate
//     computation of 2x2 determinants", Math. Comp. 82, 2013), which keeps
//     the relative error of a rotated value at a few fp32 ulps even when the
//     two products nearly cancel.
//   * Persistent grid: CTAs stride over rows, so any row count (ragged
//     tails included) is spread over all SMs.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ltxk {

enum Mode : int { kPlain = 0, kInterleaved = 1, kSplitHalf = 2, kAdaLN = 3, kAddNorm = 4 };

struct RowArgs {
  uint16_t* out;            // [rows, hidden] bf16
  const uint16_t* x;        // [rows, hidden] bf16
  const uint16_t* w;        // [hidden] bf16 or nullptr (ones)
  const float* cos_t;       // [table_rows, head_dim/2] fp32 (fused only)
  const float* sin_t;
  int64_t rows;
  int64_t table_rows;       // row r uses table row r % table_rows
  int hidden;
  int head_dim;
  float eps;
  const uint16_t* scale;    // AdaLN: [n_cond, hidden] bf16
  const uint16_t* shift;    // AdaLN: [n_cond, hidden] bf16
  int64_t rows_per_cond;    // AdaLN: row r uses conditioning row r / rows_per_cond
  const uint16_t* res;      // residual add: [rows, hidden] bf16 residual in
  uint16_t* h_out;          // residual add: [rows, hidden] bf16 h = x + res out
};

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

// bf16(a + b) for the 8 bf16 lanes of two vectors.  The fp32 sum of two
// bf16 values is exact unless their exponents differ by 16 or more, and then
// the smaller one is far below half a bf16 spacing of the larger, so the one
// RNE conversion gives the correctly rounded bf16 sum.
__device__ __forceinline__ uint4 add_bf16x8(uint4 a, uint4 b) {
  return make_uint4(pack_f2(__fadd2_rn(bf2_of(a.x), bf2_of(b.x))),
                    pack_f2(__fadd2_rn(bf2_of(a.y), bf2_of(b.y))),
                    pack_f2(__fadd2_rn(bf2_of(a.z), bf2_of(b.z))),
                    pack_f2(__fadd2_rn(bf2_of(a.w), bf2_of(b.w))));
}

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

// Rows ahead that the register kernel asks the bulk-copy engine to bring
// into L2 (0 = off).
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

// Sum of squares of 8 bf16 values, as two fp32 partial sums (even, odd).
__device__ __forceinline__ float2 sumsq8(uint4 v, float2 s) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = bf2_of(u[i]);
    s = __ffma2_rn(p, p, s);
  }
  return s;
}

constexpr uint32_t kOnes2 = 0x3F803F80u;   // two bf16 1.0 values

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

  // Load this thread's slots of one row (fetch(off) returns 16 bytes).
  template <class Fetch>
  __device__ __forceinline__ void load(uint4 (&v)[VPL], Fetch&& fetch) const {
    if constexpr (MODE == kSplitHalf) {
      each_pair([&](int j, int lo, int hi, int, bool ok) {
        v[2 * j] = ok ? fetch(lo) : make_uint4(0u, 0u, 0u, 0u);
        v[2 * j + 1] = ok ? fetch(hi) : make_uint4(0u, 0u, 0u, 0u);
      });
    } else {
      each_slot([&](int k, int off, int, bool ok) {
        v[k] = ok ? fetch(off) : make_uint4(0u, 0u, 0u, 0u);
      });
    }
  }
};

template <int VPL>
__device__ __forceinline__ float slots_sumsq(const uint4 (&v)[VPL]) {
  float2 ss = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < VPL; ++k) ss = sumsq8(v[k], ss);
  return ss.x + ss.y;
}

__device__ __forceinline__ float inv_rms_of(float ss, const RowArgs& a) {
  return rsqrtf(__fdiv_rn(ss, static_cast<float>(a.hidden)) + a.eps);
}

// Scale (and rotate) the thread's slots of one row and store them.
template <int MODE, int VPL, int GT>
__device__ __forceinline__ void row_epilogue(const RowArgs& a, int64_t row,
                                             uint4 (&v)[VPL], const SlotMap<MODE, VPL, GT>& m,
                                             float inv_rms) {
#pragma unroll
  for (int k = 0; k < VPL; ++k) launder(v[k]);
  const bool has_w = a.w != nullptr;
  uint16_t* yr = a.out + row * a.hidden;
  const uint4 ones = make_uint4(kOnes2, kOnes2, kOnes2, kOnes2);
  const float2 inv2 = make_float2(inv_rms, inv_rms);
  if constexpr (MODE == kPlain || MODE == kAddNorm) {
    m.each_slot([&](int k, int off, int, bool ok) {
      if (!ok) return;
      const uint4 wv = has_w ? ld_ro16(a.w + off) : ones;
      const uint32_t xu[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
      const uint32_t wu[4] = {wv.x, wv.y, wv.z, wv.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)   // (x * w) is exact; one rounding by inv_rms
        o[i] = pack_f2(__fmul2_rn(__fmul2_rn(bf2_of(xu[i]), bf2_of(wu[i])), inv2));
      st16(yr + off, make_uint4(o[0], o[1], o[2], o[3]));
    });
    return;
  } else if constexpr (MODE == kAdaLN) {
    // y = n * (1 + scale) + shift with n = (x * w) * inv_rms; one conditioning
    // row serves rows_per_cond rows, so its vectors come from L1/L2
    const int64_t c = row / a.rows_per_cond;
    const uint16_t* scr = a.scale + c * a.hidden;
    const uint16_t* shr = a.shift + c * a.hidden;
    const float2 one2 = make_float2(1.f, 1.f);
    m.each_slot([&](int k, int off, int, bool ok) {
      if (!ok) return;
      const uint4 wv = has_w ? ld_ro16(a.w + off) : ones;
      const uint4 sv = ld_ro16(scr + off);
      const uint4 tv = ld_ro16(shr + off);
      const uint32_t xu[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
      const uint32_t wu[4] = {wv.x, wv.y, wv.z, wv.w};
      const uint32_t su[4] = {sv.x, sv.y, sv.z, sv.w};
      const uint32_t tu[4] = {tv.x, tv.y, tv.z, tv.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 n = __fmul2_rn(__fmul2_rn(bf2_of(xu[i]), bf2_of(wu[i])), inv2);
        o[i] = pack_f2(__ffma2_rn(n, __fadd2_rn(one2, bf2_of(su[i])), bf2_of(tu[i])));
      }
      st16(yr + off, make_uint4(o[0], o[1], o[2], o[3]));
    });
    return;
  } else {
    const int64_t pos = row % a.table_rows;
    const float* ct = a.cos_t + pos * m.P;
    const float* st = a.sin_t + pos * m.P;
    if constexpr (MODE == kInterleaved) {
      // When the slot stride is a multiple of head_dim (a1 == 0), every slot
      // of this thread uses the same four rotation columns: load them once.
      const bool same_cols = m.a1 == 0;
      float4 c4h = make_float4(0.f, 0.f, 0.f, 0.f), s4h = c4h;
      if (same_cols) {
        c4h = ld_ro16f(ct + (m.a0 >> 1));
        s4h = ld_ro16f(st + (m.a0 >> 1));
      }
      m.each_slot([&](int k, int off, int pair0, bool ok) {
        if (!ok) return;
        const uint4 wv = has_w ? ld_ro16(a.w + off) : ones;
        const float4 c4 = same_cols ? c4h : ld_ro16f(ct + pair0);
        const float4 s4 = same_cols ? s4h : ld_ro16f(st + pair0);
        const float2 c[2] = {make_float2(c4.x, c4.y), make_float2(c4.z, c4.w)};
        const float2 s[2] = {make_float2(s4.x, s4.y), make_float2(s4.z, s4.w)};
        const uint32_t xu[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
        const uint32_t wu[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // words 2h and 2h+1 hold pairs 2h and 2h+1: lane x of each float2
          // is the first pair, lane y the second
          const uint32_t x0 = xu[2 * h], x1 = xu[2 * h + 1];
          const uint32_t w0 = wu[2 * h], w1 = wu[2 * h + 1];
          const float2 u = __fmul2_rn(make_float2(bf_lo(x0), bf_lo(x1)),
                                      make_float2(bf_lo(w0), bf_lo(w1)));   // a * w, exact
          const float2 q = __fmul2_rn(make_float2(bf_hi(x0), bf_hi(x1)),
                                      make_float2(bf_hi(w0), bf_hi(w1)));   // b * w, exact
          const float2 ra = __fmul2_rn(diff_of_products2(u, c[h], q, s[h]), inv2);
          const float2 rb = __fmul2_rn(diff_of_products2(u, s[h], neg2(q), c[h]), inv2);
          o[2 * h] = pack_bf2(ra.x, rb.x);
          o[2 * h + 1] = pack_bf2(ra.y, rb.y);
        }
        st16(yr + off, make_uint4(o[0], o[1], o[2], o[3]));
      });
    } else {
      // Same idea: when the pair-vector stride is a multiple of the vectors
      // per half-head (b1 == 0), the columns are the same for every pair.
      const bool same_cols = m.b1 == 0;
      float4 c0h = make_float4(0.f, 0.f, 0.f, 0.f), c1h = c0h, s0h = c0h, s1h = c0h;
      if (same_cols) {
        c0h = ld_ro16f(ct + m.b0 * 8);
        c1h = ld_ro16f(ct + m.b0 * 8 + 4);
        s0h = ld_ro16f(st + m.b0 * 8);
        s1h = ld_ro16f(st + m.b0 * 8 + 4);
      }
      m.each_pair([&](int j, int lo_off, int hi_off, int pair0, bool ok) {
        if (!ok) return;
        const int kl = 2 * j, kh = 2 * j + 1;
        const uint4 wl = has_w ? ld_ro16(a.w + lo_off) : ones;
        const uint4 wh = has_w ? ld_ro16(a.w + hi_off) : ones;
        const float4 c0 = same_cols ? c0h : ld_ro16f(ct + pair0);
        const float4 c1 = same_cols ? c1h : ld_ro16f(ct + pair0 + 4);
        const float4 s0 = same_cols ? s0h : ld_ro16f(st + pair0);
        const float4 s1 = same_cols ? s1h : ld_ro16f(st + pair0 + 4);
        const float2 c[4] = {make_float2(c0.x, c0.y), make_float2(c0.z, c0.w),
                             make_float2(c1.x, c1.y), make_float2(c1.z, c1.w)};
        const float2 s[4] = {make_float2(s0.x, s0.y), make_float2(s0.z, s0.w),
                             make_float2(s1.x, s1.y), make_float2(s1.z, s1.w)};
        const uint32_t xl[4] = {v[kl].x, v[kl].y, v[kl].z, v[kl].w};
        const uint32_t xh[4] = {v[kh].x, v[kh].y, v[kh].z, v[kh].w};
        const uint32_t wlu[4] = {wl.x, wl.y, wl.z, wl.w};
        const uint32_t whu[4] = {wh.x, wh.y, wh.z, wh.w};
        uint32_t ol[4], oh[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {   // pairs 2i, 2i+1: (lo word i, hi word i)
          const float2 u = __fmul2_rn(bf2_of(xl[i]), bf2_of(wlu[i]));   // exact
          const float2 q = __fmul2_rn(bf2_of(xh[i]), bf2_of(whu[i]));   // exact
          ol[i] = pack_f2(__fmul2_rn(diff_of_products2(u, c[i], q, s[i]), inv2));
          oh[i] = pack_f2(__fmul2_rn(diff_of_products2(u, s[i], neg2(q), c[i]), inv2));
        }
        st16(yr + lo_off, make_uint4(ol[0], ol[1], ol[2], ol[3]));
        st16(yr + hi_off, make_uint4(oh[0], oh[1], oh[2], oh[3]));
      });
    }
  }
}

// ---- register kernel: G warps per row, row loaded straight into registers -

// Threads per CTA of the register kernel when a row group is smaller.
#ifndef LTXK_VEC_BLOCK
#define LTXK_VEC_BLOCK 128
#endif

template <int G>
struct GroupShape {
  static constexpr int kThreadsPerGroup = 32 * G;
  static constexpr int kBlock = 32 * G >= LTXK_VEC_BLOCK ? 32 * G : LTXK_VEC_BLOCK;
  static constexpr int kGroupsPerCta = kBlock / kThreadsPerGroup;
};

// Register budget per thread of the register kernel: the row's 4*VPL words
// plus what the epilogue needs (weights, and for RoPE the cos/sin vectors).
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
template <int MODE, int VPL>
struct RegBudget {
  static constexpr int kRegs =
      4 * VPL + (MODE == kPlain          ? LTXK_REG_EXTRA_PLAIN
                 : MODE == kInterleaved  ? LTXK_REG_EXTRA_INTERLEAVED
                 : MODE == kSplitHalf    ? LTXK_REG_EXTRA_SPLIT
                 : MODE == kAddNorm      ? 4 * VPL + LTXK_REG_EXTRA_PLAIN  // x and res in flight
                                         : LTXK_REG_EXTRA_PLAIN + 16);
};
template <int MODE, int G, int VPL>
struct VecLaunch {
  static constexpr int kBlock = GroupShape<G>::kBlock;
  static constexpr int kMin = 65536 / (kBlock * RegBudget<MODE, VPL>::kRegs);
  static constexpr int kMinBlocks = kMin < 1 ? 1 : kMin;
};

template <int MODE, int G, int VPL>
__global__ void __launch_bounds__(VecLaunch<MODE, G, VPL>::kBlock,
                                  VecLaunch<MODE, G, VPL>::kMinBlocks)
rows_vec_kernel(const RowArgs a) {
  using S = GroupShape<G>;
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
  int parity = 0;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * S::kGroupsPerCta + group;
       row < a.rows; row += row_step) {
    const uint16_t* xr = a.x + row * a.hidden;
    if (LTXK_L2_PREFETCH_ROWS > 0 && t == 0 && (a.hidden & 7) == 0) {
      const int64_t ahead = row + LTXK_L2_PREFETCH_ROWS * row_step;
      if (ahead < a.rows) prefetch_l2(a.x + ahead * a.hidden, static_cast<uint32_t>(a.hidden) * 2u);
    }
    uint4 v[VPL];
    m.load(v, [&](int off) { return ld_stream16(xr + off); });
    if constexpr (MODE == kAddNorm) {
      // h = bf16(x + res): stored as the new residual stream, then normalised
      const uint16_t* rr = a.res + row * a.hidden;
      uint16_t* hr = a.h_out + row * a.hidden;
      uint4 rv[VPL];
      m.load(rv, [&](int off) { return ld_stream16(rr + off); });
#pragma unroll
      for (int k = 0; k < VPL; ++k) v[k] = add_bf16x8(v[k], rv[k]);
      m.each_slot([&](int k, int off, int, bool ok) {
        if (ok) st16(hr + off, v[k]);
      });
    }

    float ss = warp_sum(slots_sumsq(v));
    if (G > 1) {
      if (lane == 0) red[parity][group][warp_in_group] = ss;
      if (S::kGroupsPerCta == 1) __syncthreads();
      else group_barrier(1 + group, GT);
      ss = 0.f;
#pragma unroll
      for (int i = 0; i < G; ++i) ss += red[parity][group][i];
      parity ^= 1;
    }
    row_epilogue<MODE, VPL, GT>(a, row, v, m, inv_rms_of(ss, a));
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
      bulk_load(ring + i * ta.stage_stride, a.x + r * a.hidden, row_bytes, bars + 8 * i);
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
        bulk_load(buf, a.x + next * a.hidden, row_bytes, bars + 8 * s);
      }
    }
    const float ss = warp_sum(slots_sumsq(v));
    row_epilogue<MODE, VPL, 32>(a, row, v, m, inv_rms_of(ss, a));
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

template <int MODE>
__global__ void __launch_bounds__(kElemBlock)
rows_elem_kernel(const RowArgs a) {
  __shared__ float scratch[32];
  const int64_t H = a.hidden;
  const bool has_w = a.w != nullptr;
  for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
    const uint16_t* xr = a.x + row * H;
    uint16_t* yr = a.out + row * H;
    float ss = 0.f;
    if (MODE == kAddNorm) {
      // h = bf16(x + res), stored as the new residual stream; each thread
      // reads back only the elements it wrote itself
      const uint16_t* rr = a.res + row * H;
      uint16_t* hr = a.h_out + row * H;
      for (int64_t j = threadIdx.x; j < H; j += blockDim.x) {
        const uint16_t hb = f_to_bf(__fadd_rn(bf_to_f(xr[j]), bf_to_f(rr[j])));
        hr[j] = hb;
        const float v = bf_to_f(hb);
        ss = __fmaf_rn(v, v, ss);
      }
    } else {
      for (int64_t j = threadIdx.x; j < H; j += blockDim.x) {
        const float v = bf_to_f(xr[j]);
        ss = __fmaf_rn(v, v, ss);
      }
    }
    // block_sum ends with a barrier, so every read of this row is done
    // before any thread writes it (in-place safe), and scratch is free for
    // the next row.
    ss = block_sum(ss, scratch);
    const float inv_rms = rsqrtf(__fdiv_rn(ss, static_cast<float>(H)) + a.eps);
    if (MODE == kPlain || MODE == kAddNorm) {
      const uint16_t* src = MODE == kAddNorm ? a.h_out + row * H : xr;
      for (int64_t j = threadIdx.x; j < H; j += blockDim.x) {
        const float wj = has_w ? bf_to_f(a.w[j]) : 1.f;
        yr[j] = f_to_bf(__fmul_rn(__fmul_rn(bf_to_f(src[j]), wj), inv_rms));
      }
    } else if (MODE == kAdaLN) {
      const int64_t c = row / a.rows_per_cond;
      for (int64_t j = threadIdx.x; j < H; j += blockDim.x) {
        const float wj = has_w ? bf_to_f(a.w[j]) : 1.f;
        const float n = __fmul_rn(__fmul_rn(bf_to_f(xr[j]), wj), inv_rms);
        const float sc = __fadd_rn(1.f, bf_to_f(a.scale[c * H + j]));
        yr[j] = f_to_bf(__fmaf_rn(n, sc, bf_to_f(a.shift[c * H + j])));
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
        const float wa = has_w ? bf_to_f(a.w[ia]) : 1.f;
        const float wb = has_w ? bf_to_f(a.w[ib]) : 1.f;
        const float u = __fmul_rn(bf_to_f(xr[ia]), wa);
        const float v = __fmul_rn(bf_to_f(xr[ib]), wb);
        const float c = ct[p], s = st[p];
        const float ra = __fmul_rn(diff_of_products(u, c, v, s), inv_rms);
        const float rb = __fmul_rn(sum_of_products(u, s, v, c), inv_rms);
        yr[ia] = f_to_bf(ra);
        yr[ib] = f_to_bf(rb);
      }
    }
  }
}

}  // namespace ltxk
