/*
 * oracle.c -- plain, slow, fp64 CPU oracle for RMSNorm, the fused RMSNorm +
 * rotary-embedding (RoPE) forms, the AdaLN and residual-add norms, the
 * standalone RoPE with angles from token positions, and the tanh GELU and
 * GEGLU, each in bfloat16, IEEE binary16 and binary32.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent definition that the
 * CUDA path is checked against.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it.  It shares no code, header,
 * constant or helper with the CUDA library, and it includes no CUDA header.
 *
 * What it follows:
 *   - "cuda-kernels" skill page (Hugging Face), section "Kernel-Specific
 *     Guidelines / RMSNorm": the input layout is [..., hidden_size], the
 *     default epsilon is 1e-6, and the weight may be absent (treated as ones).
 *   - same page, "Kernel-Specific Guidelines / RoPE": the per-head layouts
 *     [batch, seq, heads, head_dim] (1D text) and [batch, t*h*w, heads,
 *     head_dim] (3D video).
 *   - "ltx-kernels" README, opening list (`ops_cpp`): the two fused ops
 *     rms_norm_rope (interleaved pairs) and rms_norm_split_rope (split-half
 *     pairs).
 *   - The pages print no formula for either operation.  The definition used:
 *       ms   = (1/H) * sum_j x_j^2                     (mean over exactly H)
 *       n_j  = x_j * w_j / sqrt(ms + eps)               (eps inside the root)
 *       RoPE, per head h and pair p with c = cos[pos,p], s = sin[pos,p]:
 *         a' = a*c - b*s,   b' = a*s + b*c
 *         interleaved: (a, b) = (n[h*D + 2p], n[h*D + 2p + 1])
 *         split-half : (a, b) = (n[h*D + p],  n[h*D + p + D/2])
 *       output = one round-to-nearest-even of the exact value to bfloat16.
 *     The RMSNorm is taken over the full hidden size before any rotation, and
 *     the rotation acts on the unrounded normalised values.
 *
 * All arithmetic is IEEE-754 binary64, summed in plain sequential order, with
 * no blocking, fusion or reordering.  The build compiles this file with
 * -ffp-contract=off so that no multiply-add is fused on any host.
 *
 *   - same page, "Supported Data Types" / "Kernel-Specific Guidelines /
 *     RMSNorm" in the block context of "Diffusers Critical Pitfalls": the
 *     residual add that precedes each block norm, fused here as
 *     h = bf16(x + residual), y = RMSNorm(h) -- the norm reads the rounded
 *     residual stream h, exactly as the unfused add-then-norm does.
 *   - same page, "Kernel-Specific Guidelines / GEGLU vs GELU": LTX-Video's
 *     tanh-approximated GELU ("gelu-approximate"),
 *       gelu(x) = x/2 * (1 + tanh(z)),  z = sqrt(2/pi) * (x + 0.044715 x^3),
 *     evaluated through the identity (1 + tanh(z))/2 = 1/(1 + exp(-2z)),
 *     which stays accurate where 1 + tanh(z) cancels (z < about -18); and
 *     GEGLU [.., 2h] -> [.., h]: the first half of the last axis is the
 *     value, the second half the gate, y = value * gelu(gate) (the diffusers
 *     GEGLU convention the page's LTX-Video discussion refers to).
 *   - same page, "Kernel-Specific Guidelines / AdaLN": the DiT conditioning
 *     norm(x) * weight * (1 + scale) + shift, with norm the RMSNorm above;
 *     scale and shift are one hidden-sized vector per conditioning row (one
 *     per batch item), shared by the rows_per_cond consecutive rows of x.
 *
 * Every exported function is re-entrant (no global state), so callers may run
 * disjoint row ranges on several threads at once.
 *
 * Parity pins (tests in tests/test_oracle.py; tests/test_oracle_mutants.py
 * checks that a plausible mistake in each part fails one of them):
 *   - rounding: brute force over all 65536 bfloat16 and binary16 patterns,
 *     ties to even, specials, numpy's and the hardware's own conversions;
 *   - RMSNorm: hand-computed cases at hidden = 4, the unit-RMS closed form,
 *     exact power-of-two scale invariance, the fp64 library RMSNorm of
 *     PyTorch;
 *   - RoPE on tables: identity / quarter-turn / half-turn rotations,
 *     pair-norm preservation, the permutation that maps split-half pairing
 *     to interleaved pairing, the table row of each row;
 *   - AdaLN and the residual add: hand cases, the reductions to plain
 *     RMSNorm, affinity in scale and shift, h as the rounded sum;
 *   - RoPE from positions: identity at token 0, the closed-form
 *     frequencies, the 3-axis coordinates, additivity of the angle in the
 *     position, norms and the pairing permutation;
 *   - GELU / GEGLU: the odd-part identity gelu(x) - gelu(-x) = x, PyTorch's
 *     fp64 tanh form, the log-sigmoid form of the far tail, value times
 *     gelu(gate), in every format;
 *   - formats: inputs every format holds exactly give the same exact
 *     results in every format.
 * No function here is left unpinned.
 */
#define _DEFAULT_SOURCE 1
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* A bfloat16 value is the upper 16 bits of an IEEE-754 binary32 value, so
 * widening is exact: place the bits on top of a binary32 and convert. */
static double widen_bf16(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---- element formats ---------------------------------------------------
 *
 * "cuda-kernels" skill page, "Supported Data Types": every kernel comes in
 * three precision modes, __half (IEEE binary16), __nv_bfloat16 and float
 * (IEEE binary32).  Format codes used below: */
enum { FMT_BF16 = 0, FMT_F16 = 1, FMT_F32 = 2 };

/* Round a binary64 value to the nearest value of a binary floating-point
 * format with `prec` significant bits, smallest normal exponent `emin` and
 * largest exponent `emax`, ties to even, straight from the IEEE-754
 * definition (no intermediate rounding).  For |v| in [2^(e-1), 2^e) the
 * spacing of representable values is 2^(e-prec); below 2^emin it stays
 * 2^(emin-prec+1) (subnormals).  Results beyond the largest finite value
 * (2 - 2^(1-prec)) * 2^emax become infinities; NaN, zeros and infinities
 * pass through. */
static double round_binary(double v, int prec, int emin, int emax) {
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    const double a = fabs(v);
    int e;
    (void)frexp(a, &e);                 /* a = m * 2^e, m in [0.5, 1) */
    if (e - 1 < emin) e = emin + 1;     /* subnormal range: fixed spacing */
    const double q = ldexp(1.0, e - prec);
    const double n = a / q;             /* exact: q is a power of two */
    double k = floor(n);
    const double frac = n - k;          /* exact */
    if (frac > 0.5 || (frac == 0.5 && fmod(k, 2.0) != 0.0)) k += 1.0;
    double r = k * q;                   /* exact */
    if (r > ldexp(2.0 - ldexp(1.0, 1 - prec), emax)) r = INFINITY;
    return signbit(v) ? -r : r;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits, so 8
 * significant bits; normal range from 2^-126, subnormal spacing 2^-133.
 * The rounded value is exactly representable in binary32 (or infinite), so
 * its encoding is the top half of the binary32 encoding. */
static uint16_t round_to_bf16(double v) {
    if (isnan(v)) return (uint16_t)(signbit(v) ? 0xFFC0u : 0x7FC0u);
    const float rf = (float)round_binary(v, 8, -126, 127);
    uint32_t u;
    memcpy(&u, &rf, sizeof u);
    return (uint16_t)(u >> 16);
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits:
 * 11 significant bits, normal range 2^-14 .. 65504, subnormal spacing 2^-24. */
static double widen_f16(uint16_t bits) {
    const int E = (bits >> 10) & 31;
    const int M = bits & 1023;
    double v;
    if (E == 0) v = ldexp((double)M, -24);
    else if (E == 31) v = M ? NAN : INFINITY;
    else v = ldexp((double)(1024 + M), E - 25);
    return (bits & 0x8000u) ? -v : v;
}

static uint16_t round_to_f16(double v) {
    if (isnan(v)) return (uint16_t)(signbit(v) ? 0xFE00u : 0x7E00u);
    const double r = round_binary(v, 11, -14, 15);
    const uint16_t sign = (uint16_t)(signbit(r) ? 0x8000u : 0u);
    const double a = fabs(r);
    if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
    if (a < ldexp(1.0, -14)) return (uint16_t)(sign | (uint16_t)(a * 16777216.0)); /* a / 2^-24 */
    int e;
    const double m = frexp(a, &e);      /* a = m * 2^e, m in [0.5, 1) */
    const int E = e - 1 + 15;
    const int M = (int)(m * 2048.0) - 1024;
    return (uint16_t)(sign | (uint16_t)(E << 10) | (uint16_t)M);
}

/* IEEE binary32: 24 significant bits, normal range from 2^-126, subnormal
 * spacing 2^-149.  The rounded value converts to float exactly. */
static float round_to_f32(double v) {
    if (isnan(v)) return signbit(v) ? -NAN : NAN;
    return (float)round_binary(v, 24, -126, 127);
}

/* Element i of an array in format fmt, exactly, as binary64. */
static double load_elem(int fmt, const void* p, int64_t i) {
    if (fmt == FMT_F32) return (double)((const float*)p)[i];
    const uint16_t b = ((const uint16_t*)p)[i];
    return fmt == FMT_F16 ? widen_f16(b) : widen_bf16(b);
}

/* Store v into element i of an array in format fmt, rounded once (RNE). */
static void store_elem(int fmt, void* p, int64_t i, double v) {
    if (fmt == FMT_F32) ((float*)p)[i] = round_to_f32(v);
    else if (fmt == FMT_F16) ((uint16_t*)p)[i] = round_to_f16(v);
    else ((uint16_t*)p)[i] = round_to_bf16(v);
}

/* ---- element conversions, exported for the pins ------------------------ */

void oracle_widen_bf16(const uint16_t* in, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = widen_bf16(in[i]);
}

void oracle_round_bf16(const double* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = round_to_bf16(in[i]);
}

/* Widen / round n elements of format fmt (for the pins). */
void oracle_widen_fmt(int fmt, const void* in, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = load_elem(fmt, in, i);
}

void oracle_round_fmt(int fmt, const double* in, void* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) store_elem(fmt, out, i, in[i]);
}

/* ---- RMSNorm ----------------------------------------------------------- */

/* Normalise row r of x [.., H] (format fmt) into n[0..H).  w == NULL means
 * all ones. */
static void normalise_row(int fmt, const void* x, int64_t r, const void* w, int64_t H,
                          float eps, double* n) {
    double ss = 0.0;
    for (int64_t j = 0; j < H; ++j) {
        const double v = load_elem(fmt, x, r * H + j);
        ss += v * v;
    }
    const double ms = ss / (double)H;
    const double denom = sqrt(ms + (double)eps);
    for (int64_t j = 0; j < H; ++j) {
        const double wj = w ? load_elem(fmt, w, j) : 1.0;
        n[j] = load_elem(fmt, x, r * H + j) * wj / denom;
    }
}

/* y[r, j] = round( x[r, j] * w[j] / sqrt(mean_j x[r, j]^2 + eps) ).
 *
 * x, y: row-major [rows, H] in format fmt.  w: [H] or NULL (ones).
 * y_exact: optional [rows, H] binary64 copy of the values before rounding.
 * Returns 0, -1 if scratch memory could not be allocated, -2 for an unknown
 * format. */
int oracle_rms_norm_fmt(int fmt, void* y, const void* x, const void* w,
                        int64_t rows, int64_t H, float eps, double* y_exact) {
    if (fmt < FMT_BF16 || fmt > FMT_F32) return -2;
    double* n = (double*)malloc((size_t)(H > 0 ? H : 1) * sizeof(double));
    if (!n) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        normalise_row(fmt, x, r, w, H, eps, n);
        for (int64_t j = 0; j < H; ++j) {
            if (y_exact) y_exact[r * H + j] = n[j];
            store_elem(fmt, y, r * H + j, n[j]);
        }
    }
    free(n);
    return 0;
}

int oracle_rms_norm(uint16_t* y, const uint16_t* x, const uint16_t* w,
                    int64_t rows, int64_t H, float eps, double* y_exact) {
    return oracle_rms_norm_fmt(FMT_BF16, y, x, w, rows, H, eps, y_exact);
}

/* Fused RMSNorm then RoPE.
 *
 * x, y: row-major [rows, heads*head_dim] in format fmt.  w: [heads*head_dim]
 * or NULL.  cos_t, sin_t: binary32 tables [table_rows, head_dim/2]; row r of
 * x (counted from first_row, the global index of the first row passed) uses
 * table row ((first_row + r) mod table_rows), i.e. x is [batch, table_rows,
 * hidden] with the sequence position as the inner row index.
 * mode 0 pairs (2p, 2p+1) inside each head; mode 1 pairs (p, p + head_dim/2).
 * Returns 0; -1 on allocation failure; -2 on an invalid argument. */
int oracle_rms_norm_rope_fmt(int fmt, void* y, const void* x, const void* w,
                             const float* cos_t, const float* sin_t,
                             int64_t rows, int64_t heads, int64_t head_dim,
                             int mode, float eps, int64_t table_rows,
                             int64_t first_row, double* y_exact) {
    if (fmt < FMT_BF16 || fmt > FMT_F32) return -2;
    if (head_dim <= 0 || head_dim % 2 != 0 || heads <= 0 || table_rows <= 0 ||
        first_row < 0)
        return -2;
    if (mode != 0 && mode != 1) return -2;
    const int64_t H = heads * head_dim;
    const int64_t P = head_dim / 2;
    double* n = (double*)malloc((size_t)H * sizeof(double));
    double* o = (double*)malloc((size_t)H * sizeof(double));
    if (!n || !o) { free(n); free(o); return -1; }

    for (int64_t r = 0; r < rows; ++r) {
        normalise_row(fmt, x, r, w, H, eps, n);
        const int64_t pos = (first_row + r) % table_rows;
        for (int64_t h = 0; h < heads; ++h) {
            for (int64_t p = 0; p < P; ++p) {
                int64_t ia, ib;
                if (mode == 0) { ia = h * head_dim + 2 * p; ib = ia + 1; }
                else           { ia = h * head_dim + p;     ib = ia + P; }
                const double c = (double)cos_t[pos * P + p];
                const double s = (double)sin_t[pos * P + p];
                const double a = n[ia];
                const double b = n[ib];
                o[ia] = a * c - b * s;
                o[ib] = a * s + b * c;
            }
        }
        for (int64_t j = 0; j < H; ++j) {
            if (y_exact) y_exact[r * H + j] = o[j];
            store_elem(fmt, y, r * H + j, o[j]);
        }
    }
    free(n);
    free(o);
    return 0;
}

int oracle_rms_norm_rope(uint16_t* y, const uint16_t* x, const uint16_t* w,
                         const float* cos_t, const float* sin_t,
                         int64_t rows, int64_t heads, int64_t head_dim,
                         int mode, float eps, int64_t table_rows,
                         int64_t first_row, double* y_exact) {
    return oracle_rms_norm_rope_fmt(FMT_BF16, y, x, w, cos_t, sin_t, rows, heads, head_dim,
                                    mode, eps, table_rows, first_row, y_exact);
}

/* AdaLN-modulated RMSNorm:
 *   y[r, j] = round( n[r, j] * (1 + scale[c, j]) + shift[c, j] ),
 *   n = the RMSNorm above (with w, or ones when w == NULL),
 *   c = r / rows_per_cond (x is [n_cond, rows_per_cond, H]).
 * scale, shift: [n_cond, H] in the format of x.  first_row is the global
 * index of the first row passed, so that row blocks keep their conditioning
 * row.  Returns 0; -1 on allocation failure; -2 on an invalid argument. */
int oracle_rms_norm_adaln_fmt(int fmt, void* y, const void* x, const void* w,
                              const void* scale, const void* shift,
                              int64_t rows, int64_t H, int64_t rows_per_cond,
                              int64_t first_row, float eps, double* y_exact) {
    if (fmt < FMT_BF16 || fmt > FMT_F32) return -2;
    if (H <= 0 || rows_per_cond <= 0 || first_row < 0) return -2;
    double* n = (double*)malloc((size_t)H * sizeof(double));
    if (!n) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        normalise_row(fmt, x, r, w, H, eps, n);
        const int64_t c = (first_row + r) / rows_per_cond;
        for (int64_t j = 0; j < H; ++j) {
            const double sc = load_elem(fmt, scale, c * H + j);
            const double sh = load_elem(fmt, shift, c * H + j);
            const double v = n[j] * (1.0 + sc) + sh;
            if (y_exact) y_exact[r * H + j] = v;
            store_elem(fmt, y, r * H + j, v);
        }
    }
    free(n);
    return 0;
}

int oracle_rms_norm_adaln(uint16_t* y, const uint16_t* x, const uint16_t* w,
                          const uint16_t* scale, const uint16_t* shift,
                          int64_t rows, int64_t H, int64_t rows_per_cond,
                          int64_t first_row, float eps, double* y_exact) {
    return oracle_rms_norm_adaln_fmt(FMT_BF16, y, x, w, scale, shift, rows, H, rows_per_cond,
                                     first_row, eps, y_exact);
}

/* Fused residual add + RMSNorm:
 *   h[r, j] = round( x[r, j] + res[r, j] )        (the new residual stream)
 *   y[r, j] = round( h[r, j] * w[j] / sqrt(mean_j h[r, j]^2 + eps) )
 * x, res, h, y: row-major [rows, H] in format fmt.  w: [H] or NULL.
 * Returns 0, -1 on allocation failure, -2 for an unknown format. */
int oracle_add_rms_norm_fmt(int fmt, void* y, void* h, const void* x, const void* res,
                            const void* w, int64_t rows, int64_t H, float eps,
                            double* y_exact) {
    if (fmt < FMT_BF16 || fmt > FMT_F32) return -2;
    double* n = (double*)malloc((size_t)(H > 0 ? H : 1) * sizeof(double));
    if (!n) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < H; ++j)
            store_elem(fmt, h, r * H + j,
                       load_elem(fmt, x, r * H + j) + load_elem(fmt, res, r * H + j));
        normalise_row(fmt, h, r, w, H, eps, n);
        for (int64_t j = 0; j < H; ++j) {
            if (y_exact) y_exact[r * H + j] = n[j];
            store_elem(fmt, y, r * H + j, n[j]);
        }
    }
    free(n);
    return 0;
}

int oracle_add_rms_norm(uint16_t* y, uint16_t* h, const uint16_t* x,
                        const uint16_t* res, const uint16_t* w, int64_t rows,
                        int64_t H, float eps, double* y_exact) {
    return oracle_add_rms_norm_fmt(FMT_BF16, y, h, x, res, w, rows, H, eps, y_exact);
}

/* ---- standalone RoPE with angles from token positions -------------------
 *
 * "cuda-kernels" page, "Kernel-Specific Guidelines / RoPE": x is
 * [batch, seq, heads, head_dim] (1D text) or [batch, t*h*w, heads, head_dim]
 * (3D video), and LTX-Video computes its own rotary angles.  The pages give
 * no frequency formula; the definition used (the one the table inputs of the
 * fused form are built with):
 *   token s = r mod (T*H*W) of row r has coordinates
 *     (ct, ch, cw) = (s / (H*W), (s / W) mod H, s mod W);
 *   the head_dim/2 pairs split into consecutive groups of nt, nh, nw pairs
 *   (axis t, then h, then w; 1D text is nt = head_dim/2 with H = W = 1);
 *   pair k of an axis with n pairs turns by angle = coordinate * theta^(-k/n);
 *   a' = a cos - b sin, b' = a sin + b cos on the pairs of every head, with
 *   the pairing of `mode` as for the fused form; one rounding to the format.
 * No normalisation: y is x rotated. */
static void rope_angles(int64_t s, int64_t T, int64_t H, int64_t W,
                        int64_t nt, int64_t nh, int64_t nw, double theta,
                        double* c, double* sn) {
    (void)T;
    const int64_t coord[3] = {s / (H * W), (s / W) % H, s % W};
    const int64_t n[3] = {nt, nh, nw};
    int64_t p = 0;
    for (int axis = 0; axis < 3; ++axis) {
        for (int64_t k = 0; k < n[axis]; ++k, ++p) {
            const double ang = (double)coord[axis] * pow(theta, -(double)k / (double)n[axis]);
            c[p] = cos(ang);
            sn[p] = sin(ang);
        }
    }
}

/* cos and sin tables [tokens, head_dim/2] of the same angles: row s holds
 * token s mod (T*H*W).  Returns 0, or -2 on an invalid argument. */
int oracle_rope_tables(double* cos_out, double* sin_out, int64_t tokens, int64_t head_dim,
                       int64_t T, int64_t H, int64_t W, int64_t nt, int64_t nh, int64_t nw,
                       double theta) {
    if (tokens < 0 || head_dim <= 0 || head_dim % 2 != 0) return -2;
    if (T <= 0 || H <= 0 || W <= 0 || nt < 0 || nh < 0 || nw < 0 ||
        nt + nh + nw != head_dim / 2 || !(theta > 0.0))
        return -2;
    const int64_t P = head_dim / 2;
    for (int64_t s = 0; s < tokens; ++s)
        rope_angles(s % (T * H * W), T, H, W, nt, nh, nw, theta, cos_out + s * P,
                    sin_out + s * P);
    return 0;
}

/* x, y: [rows, heads*head_dim] in format fmt; row r is token
 * (first_row + r) mod (T*H*W).  Returns 0, -1 on allocation failure, -2 on
 * an invalid argument. */
int oracle_rope_positions(int fmt, void* y, const void* x, int64_t rows,
                          int64_t heads, int64_t head_dim, int mode,
                          int64_t T, int64_t H, int64_t W,
                          int64_t nt, int64_t nh, int64_t nw, double theta,
                          int64_t first_row, double* y_exact) {
    if (fmt < FMT_BF16 || fmt > FMT_F32) return -2;
    if (heads <= 0 || head_dim <= 0 || head_dim % 2 != 0 || (mode != 0 && mode != 1))
        return -2;
    if (T <= 0 || H <= 0 || W <= 0 || nt < 0 || nh < 0 || nw < 0 ||
        nt + nh + nw != head_dim / 2 || !(theta > 0.0) || first_row < 0)
        return -2;
    const int64_t P = head_dim / 2, HD = heads * head_dim;
    double* c = (double*)malloc((size_t)P * sizeof(double));
    double* sn = (double*)malloc((size_t)P * sizeof(double));
    if (!c || !sn) { free(c); free(sn); return -1; }
    for (int64_t r = 0; r < rows; ++r) {
        rope_angles((first_row + r) % (T * H * W), T, H, W, nt, nh, nw, theta, c, sn);
        for (int64_t h = 0; h < heads; ++h) {
            for (int64_t p = 0; p < P; ++p) {
                int64_t ia, ib;
                if (mode == 0) { ia = h * head_dim + 2 * p; ib = ia + 1; }
                else           { ia = h * head_dim + p;     ib = ia + P; }
                const double a = load_elem(fmt, x, r * HD + ia);
                const double b = load_elem(fmt, x, r * HD + ib);
                const double ya = a * c[p] - b * sn[p];
                const double yb = a * sn[p] + b * c[p];
                if (y_exact) { y_exact[r * HD + ia] = ya; y_exact[r * HD + ib] = yb; }
                store_elem(fmt, y, r * HD + ia, ya);
                store_elem(fmt, y, r * HD + ib, yb);
            }
        }
    }
    free(c);
    free(sn);
    return 0;
}

/* tanh-approximated GELU of one value, binary64. */
static double gelu_tanh(double x) {
    const double z = sqrt(2.0 / M_PI) * (x + 0.044715 * x * x * x);
    /* x/2 (1 + tanh z) = x / (1 + exp(-2z)) */
    if (z >= 0.0) return x / (1.0 + exp(-2.0 * z));
    const double e = exp(2.0 * z);
    return x * e / (1.0 + e);
}

/* y = round(gelu(x)) elementwise over n values of format fmt (x and y of
 * that format); y_exact optional. */
void oracle_gelu_tanh_fmt(int fmt, void* y, const void* x, int64_t n, double* y_exact) {
    for (int64_t i = 0; i < n; ++i) {
        const double v = gelu_tanh(load_elem(fmt, x, i));
        if (y_exact) y_exact[i] = v;
        store_elem(fmt, y, i, v);
    }
}

void oracle_gelu_tanh(uint16_t* y, const uint16_t* x, int64_t n, double* y_exact) {
    oracle_gelu_tanh_fmt(FMT_BF16, y, x, n, y_exact);
}

/* GEGLU: x [rows, 2h] -> y [rows, h], y[r, j] = round(x[r, j] * gelu(x[r, h + j]))
 * in format fmt. */
void oracle_geglu_fmt(int fmt, void* y, const void* x, int64_t rows, int64_t h,
                      double* y_exact) {
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < h; ++j) {
            const double value = load_elem(fmt, x, r * 2 * h + j);
            const double gate = load_elem(fmt, x, r * 2 * h + h + j);
            const double v = value * gelu_tanh(gate);
            if (y_exact) y_exact[r * h + j] = v;
            store_elem(fmt, y, r * h + j, v);
        }
    }
}

void oracle_geglu(uint16_t* y, const uint16_t* x, int64_t rows, int64_t h, double* y_exact) {
    oracle_geglu_fmt(FMT_BF16, y, x, rows, h, y_exact);
}
