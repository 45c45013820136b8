// ltxk_abi.cu -- the C ABI declared in include/ltxk.h: argument validation
// (host only, before any CUDA call), the launch plan, and the launches.
//
// Operations: RMSNorm ("cuda-kernels" skill page, "Kernel-Specific
// Guidelines / RMSNorm"), the fused RMSNorm + RoPE forms ("ltx-kernels"
// README, opening list: rms_norm_rope, rms_norm_split_rope), the AdaLN and
// residual-add forms, in bf16, fp16 or fp32 ("Supported Data Types").  The
// launch configuration replaces the page's "Thread Configuration" rule (one
// block of min(hidden/2, max) threads per row) with warps-per-row and slot
// counts from a register budget, and grids sized by measurement: one CTA
// per row group for the row-only forms, persistent CTAs (from the SM count
// and each kernel's occupancy) for the fused ones.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include "ltxk.h"
#include "ltxk_kernels.cuh"
#include "ltxk_launch.h"

// Device fault word set by a TMA-ring wait that ran out (one per device).
static __device__ unsigned int g_ltxk_fault_word;

namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<int> g_path{LTXK_PATH_AUTO};

constexpr int kMaxVplSlots = 16;   // fp32 rows: 8 (twice the registers per slot)
constexpr int kGroupChoices[] = {1, 2, 4, 8, 16, 32};
constexpr int64_t kSmallRows = 2432;   // 152 SMs x 16 two-warp rows
// Dynamic shared memory a TMA-ring CTA aims for: two CTAs per SM share the
// 228 KB of an SM, so each keeps about 100 KB of rows in flight.
#ifndef LTXK_TMA_SMEM_TARGET
#define LTXK_TMA_SMEM_TARGET (100u * 1024u)
#endif
constexpr uint32_t kTmaSmemTarget = LTXK_TMA_SMEM_TARGET;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per mbarrier wait

bool aligned_to(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// Do [a, a + na) and [b, b + nb) share a byte?
bool overlaps(const void* a, uint64_t na, const void* b, uint64_t nb) {
  if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a);
  const uintptr_t b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

// Multiplier for the kernels' div_fast: floor((2^64 - 1) / d) + 1 for
// 2 <= d < 2^32, else 0 (the kernel divides).
uint64_t div_mul(int64_t d) {
  return (d < 2 || d >= (int64_t{1} << 32)) ? 0 : UINT64_MAX / static_cast<uint64_t>(d) + 1;
}

int max_vpl(int fmt) { return fmt == ltxk::kF32 ? 8 : kMaxVplSlots; }

int elem_bytes(int fmt) { return fmt == ltxk::kF32 ? 4 : 2; }

int bucket_vpl(int need) {
  if (need <= 4) return 4;
  if (need <= 8) return 8;
  if (need <= 12) return 12;
  return 16;
}

// Threads per CTA of the register kernel of kernel mode km with g warps per
// row (the kernels' own rule, ltxk::vec_block).
int block_for_group(int km, int g) { return ltxk::vec_block(km, g); }

// Grid shape.  1: at most the resident CTAs, striding over the rows
// (persistent); 0: one CTA per row group, scheduled by the hardware.
// Measured on GB300: plain RMSNorm is faster with one CTA per row group
// (no rounding of the last pass over the rows), the fused kernels with
// persistent CTAs (their per-CTA set-up is amortised).
#ifndef LTXK_PERSISTENT
#define LTXK_PERSISTENT 0
#endif
// Most vector slots per lane for the fused kernels before a row is split
// over more warps.  The rotation makes these kernels issue-heavy, so more
// warps with fewer registers each hide memory latency better; measured on
// GB300 for [2 x 4096 x 32 x 128] interleaved and [6144 x 32 x 64]
// split-half.
// Plain RMSNorm: 0 = fewest warps per row; 1 = four warps when a row is
// exactly 3 or 4 vectors per lane; 2 = any g >= 4 with such an exact fit
// (measured on GB300: copy speed or better for hidden 3072, 4096, 6144 and
// 8192, at 16384-65536 rows); 3 = as 2, from g >= 2.
#ifndef LTXK_PLAIN_SPLIT_RULE
#define LTXK_PLAIN_SPLIT_RULE 2
#endif
#ifndef LTXK_PLAIN_MAX_SLOTS
#define LTXK_PLAIN_MAX_SLOTS 16
#endif
#ifndef LTXK_ROPE_MAX_SLOTS_INTERLEAVED
#define LTXK_ROPE_MAX_SLOTS_INTERLEAVED 4
#endif
#ifndef LTXK_ROPE_MAX_SLOTS_SPLIT
#define LTXK_ROPE_MAX_SLOTS_SPLIT 8
#endif
#ifndef LTXK_ADALN_STAGE
#define LTXK_ADALN_STAGE 1
#endif
#ifndef LTXK_PERSISTENT_ROPE
#define LTXK_PERSISTENT_ROPE 1
#endif

int kernel_mode(int op, int mode) {
  if (op == LTXK_OP_RMS_NORM) return ltxk::kPlain;
  if (op == LTXK_OP_RMS_NORM_ADALN) return ltxk::kAdaLN;
  if (op == LTXK_OP_ADD_RMS_NORM) return ltxk::kAddNorm;
  return mode == LTXK_ROPE_INTERLEAVED ? ltxk::kInterleaved : ltxk::kSplitHalf;
}

int fail_cuda(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return LTXK_ERR_CUDA;
}

uint32_t tma_stride(int64_t hidden) {
  return static_cast<uint32_t>((hidden * 2 + 127) / 128 * 128);
}

// ---- per-device facts, queried once ---------------------------------------

struct DeviceCache {
  std::mutex mu;
  std::map<int, int> sms;
  std::map<int, unsigned int*> fault_word;
  std::map<std::tuple<int, const void*, int>, int> occupancy;   // (dev, fn, smem)
  std::map<std::pair<int, const void*>, int> smem_opt_in;        // bytes set
};
DeviceCache& cache() {
  static DeviceCache c;
  return c;
}

cudaError_t device_facts(int* dev, int* sms, unsigned int** fault) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return e;
  DeviceCache& c = cache();
  std::lock_guard<std::mutex> lock(c.mu);
  auto it = c.sms.find(*dev);
  if (it == c.sms.end()) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, *dev);
    if (e != cudaSuccess) return e;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_ltxk_fault_word);
    if (e != cudaSuccess) return e;
    c.fault_word[*dev] = static_cast<unsigned int*>(p);
    it = c.sms.emplace(*dev, n).first;
  }
  *sms = it->second;
  if (fault) *fault = c.fault_word[*dev];
  return cudaSuccess;
}

}  // namespace

namespace ltxk {
// Resident CTAs per SM of `fn` with `block` threads and `smem` dynamic bytes;
// opts the function in to that much dynamic shared memory first.
cudaError_t resident_ctas(int dev, const void* fn, int block, int smem, int* per_sm) {
  DeviceCache& c = cache();
  std::lock_guard<std::mutex> lock(c.mu);
  cudaError_t e;
  if (smem > 48 * 1024) {
    int& set = c.smem_opt_in[{dev, fn}];
    if (set < smem) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      set = smem;
    }
  }
  auto key = std::make_tuple(dev, fn, smem);
  auto it = c.occupancy.find(key);
  if (it == c.occupancy.end()) {
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, block, smem);
    if (e != cudaSuccess) return e;
    it = c.occupancy.emplace(key, n < 1 ? 1 : n).first;
  }
  *per_sm = it->second;
  return cudaSuccess;
}
}  // namespace ltxk

namespace {
using ltxk::resident_ctas;

// ---- planning -------------------------------------------------------------

int check_shape(int op, int64_t rows, int64_t hidden, int head_dim, int mode) {
  if (rows < 0 || hidden <= 0 || hidden > LTXK_MAX_HIDDEN) return LTXK_ERR_SHAPE;
  if (rows > 0 && rows > INT64_MAX / 4 / hidden) return LTXK_ERR_SHAPE;
  if (op == LTXK_OP_RMS_NORM_ROPE) {
    if (head_dim < 2 || head_dim % 2 != 0 || hidden % head_dim != 0) return LTXK_ERR_SHAPE;
    if (mode != LTXK_ROPE_INTERLEAVED && mode != LTXK_ROPE_SPLIT_HALF) return LTXK_ERR_MODE;
  } else if (op != LTXK_OP_RMS_NORM && op != LTXK_OP_RMS_NORM_ADALN &&
             op != LTXK_OP_ADD_RMS_NORM) {
    return LTXK_ERR_MODE;
  }
  return LTXK_OK;
}

int make_plan_core(int op, int fmt, int64_t rows, int64_t hidden, int head_dim, int mode,
                   bool vector_ok, int path, ltxk_plan* p) {
  if (fmt != ltxk::kBf16 && fmt != ltxk::kF16 && fmt != ltxk::kF32) return LTXK_ERR_DTYPE;
  const int st = check_shape(op, rows, hidden, head_dim, mode);
  if (st != LTXK_OK) return st;
  *p = ltxk_plan{LTXK_KERNEL_NONE, 0, 0, 0, 0, 0, 0};
  if (rows == 0) return LTXK_OK;
  const int km = kernel_mode(op, mode);
  bool vec = vector_ok && hidden % 8 == 0;
  if (km == ltxk::kInterleaved) vec = vec && head_dim % 8 == 0;
  if (km == ltxk::kSplitHalf) vec = vec && head_dim % 16 == 0;
  const bool row_only = km == ltxk::kPlain || km == ltxk::kAdaLN || km == ltxk::kAddNorm;
  if (vec && row_only && LTXK_PLAIN_SPLIT_RULE > 0) {
    // Split the row over g >= 4 warps when it divides into exactly 3 or 4
    // vectors per lane: a light per-warp share (about 45 registers) lets far
    // more warps be resident.
    const int64_t nv = hidden / 8;
    for (int g : kGroupChoices) {
      if (g < (LTXK_PLAIN_SPLIT_RULE >= 3 ? 2 : 4) || (LTXK_PLAIN_SPLIT_RULE == 1 && g != 4))
        continue;
      if (nv % (32 * g) != 0) continue;
      const int64_t s = nv / (32 * g);
      if (s == 3 || s == 4) {
        p->kernel = LTXK_KERNEL_ROWS_VEC;
        p->group_warps = g;
        p->vec_per_lane = 4;
        p->block_threads = block_for_group(km, g);
        p->rows_per_cta = p->block_threads / (32 * g);
        return LTXK_OK;
      }
    }
    // Few rows: when two-warp rows still fit in one wave (about 32 resident
    // warps per SM on 152 SMs), an exact two-warp split doubles the loads in
    // flight of a problem too small to fill the GPU.  Measured on GB300 at
    // hidden 2048: 1024 rows 9.3 -> 8.5 us, 2048 rows 10.7 -> 10.3 us; at
    // 4096 rows (more than one wave) one warp per row stays faster.
    if (path != LTXK_PATH_TMA && rows <= kSmallRows && nv % 64 == 0 &&
        (nv / 64 == 3 || nv / 64 == 4)) {
      p->kernel = LTXK_KERNEL_ROWS_VEC;
      p->group_warps = 2;
      p->vec_per_lane = 4;
      p->block_threads = block_for_group(km, 2);
      p->rows_per_cta = p->block_threads / 64;
      return LTXK_OK;
    }
  }
  if (vec) {
    const int64_t nv = hidden / 8;
    // split-half slots are (lo, hi) pairs: nv/2 units of two slots each
    const int64_t units = km == ltxk::kSplitHalf ? nv / 2 : nv;
    const int slots_per_unit = km == ltxk::kSplitHalf ? 2 : 1;
    const int cap = max_vpl(fmt);
    int max_slots = row_only                   ? LTXK_PLAIN_MAX_SLOTS
                    : km == ltxk::kInterleaved ? LTXK_ROPE_MAX_SLOTS_INTERLEAVED
                                               : LTXK_ROPE_MAX_SLOTS_SPLIT;
    if (max_slots > cap) max_slots = cap;
    for (int g : kGroupChoices) {
      const int64_t need = (units + 32 * g - 1) / (32 * g) * slots_per_unit;
      if (need > max_slots && g < 32) continue;
      if (need > cap) continue;
      p->group_warps = g;
      p->vec_per_lane = bucket_vpl(static_cast<int>(need));
      // The TMA ring is used only on request: measured on GB300 it trails
      // the register kernel on every workload here.
      if (g == 1 && path == LTXK_PATH_TMA && km != ltxk::kAdaLN && km != ltxk::kAddNorm &&
          fmt == ltxk::kBf16) {
        const uint32_t stride = tma_stride(hidden);
        int stages = static_cast<int>((kTmaSmemTarget - ltxk::kTmaBarBytes) /
                                      (ltxk::kTmaWarps * stride));
        stages = stages < 1 ? 1 : (stages > ltxk::kTmaMaxStages ? ltxk::kTmaMaxStages : stages);
        p->kernel = LTXK_KERNEL_ROWS_TMA;
        p->block_threads = ltxk::kTmaWarps * 32;
        p->rows_per_cta = ltxk::kTmaWarps;
        p->stages = stages;
        p->smem_bytes = static_cast<int>(ltxk::kTmaBarBytes + ltxk::kTmaWarps * stages * stride);
      } else {
        p->kernel = LTXK_KERNEL_ROWS_VEC;
        p->block_threads = block_for_group(km, g);
        p->rows_per_cta = p->block_threads / (32 * g);
      }
      return LTXK_OK;
    }
  }
  p->kernel = LTXK_KERNEL_ROWS_ELEM;
  p->group_warps = ltxk::kElemBlock / 32;
  p->block_threads = ltxk::kElemBlock;
  p->rows_per_cta = 1;
  return LTXK_OK;
}

// Dynamic shared memory of a register-kernel launch: AdaLN's conditioning
// row on 16-bit rows (scale and shift, 2 * e * hidden bytes), which each CTA
// stages when it fits without an opt-in (48 KB); 0 otherwise.
int stage_cond_bytes(int km, int fmt, int64_t hidden) {
  if (LTXK_ADALN_STAGE == 0 || km != ltxk::kAdaLN || fmt == ltxk::kF32) return 0;
  const int64_t b = 2 * hidden * elem_bytes(fmt);
  return b <= 48 * 1024 ? static_cast<int>(b) : 0;
}

int make_plan(int op, int fmt, int64_t rows, int64_t hidden, int head_dim, int mode,
              bool vector_ok, int path, ltxk_plan* p) {
  const int st = make_plan_core(op, fmt, rows, hidden, head_dim, mode, vector_ok, path, p);
  if (st == LTXK_OK && p->kernel == LTXK_KERNEL_ROWS_VEC) {
    const int km = kernel_mode(op, mode);
    p->smem_bytes = stage_cond_bytes(km, fmt, hidden);
  }
  return st;
}

template <int FMT>
const void* vec_fn(int km, int g, int vpl) {
  switch (km) {
    case ltxk::kPlain: return ltxk::rows_vec_ptr<ltxk::kPlain, FMT>(g, vpl);
    case ltxk::kInterleaved: return ltxk::rows_vec_ptr<ltxk::kInterleaved, FMT>(g, vpl);
    case ltxk::kSplitHalf: return ltxk::rows_vec_ptr<ltxk::kSplitHalf, FMT>(g, vpl);
    case ltxk::kAdaLN: return ltxk::rows_vec_ptr<ltxk::kAdaLN, FMT>(g, vpl);
    case ltxk::kAddNorm: return ltxk::rows_vec_ptr<ltxk::kAddNorm, FMT>(g, vpl);
    default: return nullptr;
  }
}

template <int FMT>
const void* elem_fn(int km) {
  switch (km) {
    case ltxk::kPlain: return ltxk::rows_elem_ptr<ltxk::kPlain, FMT>();
    case ltxk::kInterleaved: return ltxk::rows_elem_ptr<ltxk::kInterleaved, FMT>();
    case ltxk::kSplitHalf: return ltxk::rows_elem_ptr<ltxk::kSplitHalf, FMT>();
    case ltxk::kAdaLN: return ltxk::rows_elem_ptr<ltxk::kAdaLN, FMT>();
    case ltxk::kAddNorm: return ltxk::rows_elem_ptr<ltxk::kAddNorm, FMT>();
    default: return nullptr;
  }
}

const void* kernel_fn(const ltxk_plan& p, int km, int fmt) {
  switch (p.kernel) {
    case LTXK_KERNEL_ROWS_VEC:
      if (fmt == ltxk::kF16) return vec_fn<ltxk::kF16>(km, p.group_warps, p.vec_per_lane);
      if (fmt == ltxk::kF32) return vec_fn<ltxk::kF32>(km, p.group_warps, p.vec_per_lane);
      return vec_fn<ltxk::kBf16>(km, p.group_warps, p.vec_per_lane);
    case LTXK_KERNEL_ROWS_TMA:
      if (km == ltxk::kPlain) return ltxk::rows_tma_plain_ptr(p.vec_per_lane);
      if (km == ltxk::kInterleaved) return ltxk::rows_tma_interleaved_ptr(p.vec_per_lane);
      return ltxk::rows_tma_split_ptr(p.vec_per_lane);
    case LTXK_KERNEL_ROWS_ELEM:
      if (fmt == ltxk::kF16) return elem_fn<ltxk::kF16>(km);
      if (fmt == ltxk::kF32) return elem_fn<ltxk::kF32>(km);
      return elem_fn<ltxk::kBf16>(km);
    default:
      return nullptr;
  }
}

int launch(int op, int mode, int fmt, const ltxk::RowArgs& args, bool vector_ok,
           cudaStream_t stream, int path, int skip_first_copy = 0,
           uint64_t wait_limit_ns = kWaitLimitNs) {
  ltxk_plan p;
  int st = make_plan(op, fmt, args.rows, args.hidden, args.head_dim, mode, vector_ok, path, &p);
  if (st != LTXK_OK || p.kernel == LTXK_KERNEL_NONE) return st;
  const int km = kernel_mode(op, mode);
  const void* fn = kernel_fn(p, km, fmt);
  if (fn == nullptr) return fail_cuda(cudaErrorInvalidDeviceFunction);
  int dev = 0, sms = 0, per_sm = 0;
  unsigned int* fault = nullptr;
  cudaError_t e = device_facts(&dev, &sms, &fault);
  if (e != cudaSuccess) return fail_cuda(e);
  // the register kernel's dynamic shared memory holds AdaLN's staged
  // conditioning row (the plan sizes it; 0 otherwise)
  const int dyn_smem = p.smem_bytes;
  ltxk::RowArgs a = args;
  a.stage_cond = p.kernel == LTXK_KERNEL_ROWS_VEC && p.smem_bytes > 0 ? 1 : 0;
  e = resident_ctas(dev, fn, p.block_threads, dyn_smem, &per_sm);
  if (e != cudaSuccess) return fail_cuda(e);
  const int64_t needed = (args.rows + p.rows_per_cta - 1) / p.rows_per_cta;
  const bool persistent =
      (km == ltxk::kPlain || km == ltxk::kAdaLN || km == ltxk::kAddNorm) ? LTXK_PERSISTENT
                                                                         : LTXK_PERSISTENT_ROPE;
  const int64_t cap = (persistent || p.kernel == LTXK_KERNEL_ROWS_TMA)
                          ? static_cast<int64_t>(sms) * per_sm
                          : int64_t{2147483647};
  const unsigned grid = static_cast<unsigned>(needed < cap ? needed : cap);
  if (p.kernel == LTXK_KERNEL_ROWS_TMA) {
    ltxk::TmaArgs ta{args, p.stages, tma_stride(args.hidden), wait_limit_ns, skip_first_copy,
                     fault};
    void* params[] = {&ta};
    e = cudaLaunchKernel(fn, dim3(grid), dim3(p.block_threads), params,
                         static_cast<size_t>(p.smem_bytes), stream);
  } else {
    void* params[] = {&a};
    e = cudaLaunchKernel(fn, dim3(grid), dim3(p.block_threads), params,
                         static_cast<size_t>(dyn_smem), stream);
  }
  if (e != cudaSuccess) return fail_cuda(e);
  return LTXK_OK;
}

// Element format of an LTXK_DTYPE_* code, or -1.
int fmt_of(int dtype) {
  switch (dtype) {
    case LTXK_DTYPE_BF16: return ltxk::kBf16;
    case LTXK_DTYPE_F16: return ltxk::kF16;
    case LTXK_DTYPE_F32: return ltxk::kF32;
    default: return -1;
  }
}

int rope_common(void* out, const void* x, const void* w, const float* cos, const float* sin,
                int64_t rows, int heads, int head_dim, int mode, float eps, int64_t table_rows,
                int fmt, cudaStream_t stream) {
  if (fmt < 0) return LTXK_ERR_DTYPE;
  if (out == nullptr || x == nullptr || cos == nullptr || sin == nullptr) return LTXK_ERR_NULL;
  if (heads < 1 || head_dim < 2 || head_dim % 2 != 0 || table_rows < 1) return LTXK_ERR_SHAPE;
  const int64_t hidden = static_cast<int64_t>(heads) * head_dim;
  int st = check_shape(LTXK_OP_RMS_NORM_ROPE, rows, hidden, head_dim, mode);
  if (st != LTXK_OK) return st;
  if (table_rows > INT64_MAX / 8 / head_dim) return LTXK_ERR_SHAPE;
  const int esz = elem_bytes(fmt);
  if (!aligned_to(out, esz) || !aligned_to(x, esz) || (w && !aligned_to(w, esz)) ||
      !aligned_to(cos, 4) || !aligned_to(sin, 4))
    return LTXK_ERR_ALIGN;
  const uint64_t xbytes = static_cast<uint64_t>(rows) * hidden * esz;
  const uint64_t tbytes = static_cast<uint64_t>(table_rows) * (head_dim / 2) * 4;
  if (out != x && overlaps(out, xbytes, x, xbytes)) return LTXK_ERR_OVERLAP;
  if (overlaps(out, xbytes, w, static_cast<uint64_t>(hidden) * esz) ||
      overlaps(out, xbytes, cos, tbytes) || overlaps(out, xbytes, sin, tbytes))
    return LTXK_ERR_OVERLAP;
  if (rows == 0) return LTXK_OK;
  const bool vector_ok = aligned_to(out, 16) && aligned_to(x, 16) && (!w || aligned_to(w, 16)) &&
                         aligned_to(cos, 16) && aligned_to(sin, 16);
  ltxk::RowArgs a{out, x, w, cos, sin, rows, table_rows, static_cast<int>(hidden), head_dim, eps};
  a.table_mul = div_mul(table_rows);
  return launch(LTXK_OP_RMS_NORM_ROPE, mode, fmt, a, vector_ok, stream, g_path.load());
}

int norm_checks(void* out, const void* x, const void* w, int64_t rows, int64_t hidden, int fmt) {
  if (fmt < 0) return LTXK_ERR_DTYPE;
  if (out == nullptr || x == nullptr) return LTXK_ERR_NULL;
  int st = check_shape(LTXK_OP_RMS_NORM, rows, hidden, 0, 0);
  if (st != LTXK_OK) return st;
  const int esz = elem_bytes(fmt);
  if (!aligned_to(out, esz) || !aligned_to(x, esz) || (w && !aligned_to(w, esz)))
    return LTXK_ERR_ALIGN;
  const uint64_t xbytes = static_cast<uint64_t>(rows) * hidden * esz;
  if (out != x && overlaps(out, xbytes, x, xbytes)) return LTXK_ERR_OVERLAP;
  if (overlaps(out, xbytes, w, static_cast<uint64_t>(hidden) * esz)) return LTXK_ERR_OVERLAP;
  return LTXK_OK;
}

int rms_norm_fmt(void* out, const void* x, const void* w, int64_t rows, int64_t hidden,
                 float eps, int fmt, cudaStream_t stream) {
  int st = norm_checks(out, x, w, rows, hidden, fmt);
  if (st != LTXK_OK || rows == 0) return st;
  const bool vector_ok = aligned_to(out, 16) && aligned_to(x, 16) && (!w || aligned_to(w, 16));
  ltxk::RowArgs a{out, x, w, nullptr, nullptr, rows, 1, static_cast<int>(hidden), 0, eps};
  return launch(LTXK_OP_RMS_NORM, 0, fmt, a, vector_ok, stream, g_path.load());
}

int adaln_fmt(void* out, const void* x, const void* w, const void* scale, const void* shift,
              int64_t rows, int64_t hidden, int64_t rows_per_cond, float eps, int fmt,
              cudaStream_t stream) {
  if (fmt < 0) return LTXK_ERR_DTYPE;
  if (scale == nullptr || shift == nullptr) return LTXK_ERR_NULL;
  int st = norm_checks(out, x, w, rows, hidden, fmt);
  if (st != LTXK_OK) return st;
  if (rows_per_cond < 1) return LTXK_ERR_SHAPE;
  const int esz = elem_bytes(fmt);
  if (!aligned_to(scale, esz) || !aligned_to(shift, esz)) return LTXK_ERR_ALIGN;
  const int64_t n_cond = rows == 0 ? 0 : (rows - 1) / rows_per_cond + 1;
  const uint64_t xbytes = static_cast<uint64_t>(rows) * hidden * esz;
  const uint64_t cbytes = static_cast<uint64_t>(n_cond) * hidden * esz;
  if (overlaps(out, xbytes, scale, cbytes) || overlaps(out, xbytes, shift, cbytes))
    return LTXK_ERR_OVERLAP;
  if (rows == 0) return LTXK_OK;
  const bool vector_ok = aligned_to(out, 16) && aligned_to(x, 16) && (!w || aligned_to(w, 16)) &&
                         aligned_to(scale, 16) && aligned_to(shift, 16);
  ltxk::RowArgs a{out, x, w, nullptr, nullptr, rows, 1, static_cast<int>(hidden), 0, eps, 0,
                  scale, shift, rows_per_cond};
  a.cond_mul = div_mul(rows_per_cond);
  return launch(LTXK_OP_RMS_NORM_ADALN, 0, fmt, a, vector_ok, stream, g_path.load());
}

int add_norm_fmt(void* out, void* residual_out, const void* x, const void* residual,
                 const void* w, int64_t rows, int64_t hidden, float eps, int fmt,
                 cudaStream_t stream) {
  if (fmt < 0) return LTXK_ERR_DTYPE;
  if (residual_out == nullptr || residual == nullptr) return LTXK_ERR_NULL;
  int st = norm_checks(out, x, w, rows, hidden, fmt);
  if (st != LTXK_OK) return st;
  const int esz = elem_bytes(fmt);
  if (!aligned_to(residual_out, esz) || !aligned_to(residual, esz)) return LTXK_ERR_ALIGN;
  const uint64_t bytes = static_cast<uint64_t>(rows) * hidden * esz;
  const uint64_t wbytes = static_cast<uint64_t>(hidden) * esz;
  // the two outputs must be disjoint; an output may coincide exactly with an
  // input (every row is read before it is written) but not partly overlap one
  if (overlaps(out, bytes, residual_out, bytes)) return LTXK_ERR_OVERLAP;
  if (residual_out != x && overlaps(residual_out, bytes, x, bytes)) return LTXK_ERR_OVERLAP;
  if (residual_out != residual && overlaps(residual_out, bytes, residual, bytes))
    return LTXK_ERR_OVERLAP;
  if (out != residual && overlaps(out, bytes, residual, bytes)) return LTXK_ERR_OVERLAP;
  if (overlaps(residual_out, bytes, w, wbytes)) return LTXK_ERR_OVERLAP;
  if (rows == 0) return LTXK_OK;
  const bool vector_ok = aligned_to(out, 16) && aligned_to(x, 16) && (!w || aligned_to(w, 16)) &&
                         aligned_to(residual, 16) && aligned_to(residual_out, 16);
  ltxk::RowArgs a{out, x, w, nullptr, nullptr, rows, 1, static_cast<int>(hidden), 0, eps, 0,
                  nullptr, nullptr, 0, residual, residual_out};
  return launch(LTXK_OP_ADD_RMS_NORM, 0, fmt, a, vector_ok, stream, g_path.load());
}

}  // namespace

namespace ltxk {
void record_cuda_error(int e) { g_last_cuda_error = e; }
int current_path() { return g_path.load(); }
}  // namespace ltxk

extern "C" {

int ltxk_rms_norm(void* out, const void* x, const void* w, int64_t rows, int64_t hidden,
                  float eps, ltxk_stream_t stream) {
  return rms_norm_fmt(out, x, w, rows, hidden, eps, ltxk::kBf16, stream);
}

int ltxk_rms_norm_dt(void* out, const void* x, const void* w, int64_t rows, int64_t hidden,
                     float eps, int dtype, ltxk_stream_t stream) {
  return rms_norm_fmt(out, x, w, rows, hidden, eps, fmt_of(dtype), stream);
}

int ltxk_rms_norm_rope(void* out, const void* x, const void* w, const float* cos,
                       const float* sin, int64_t rows, int heads, int head_dim, int mode,
                       float eps, ltxk_stream_t stream) {
  // Per-row tables: row r uses table row r.  With rows == 0 there is no
  // table at all; any positive table_rows gives the same (empty) launch.
  return rope_common(out, x, w, cos, sin, rows, heads, head_dim, mode, eps,
                     rows > 0 ? rows : 1, ltxk::kBf16, stream);
}

int ltxk_rms_norm_rope_seq(void* out, const void* x, const void* w, const float* cos,
                           const float* sin, int64_t rows, int heads, int head_dim, int mode,
                           float eps, int64_t seq_len, ltxk_stream_t stream) {
  return rope_common(out, x, w, cos, sin, rows, heads, head_dim, mode, eps, seq_len,
                     ltxk::kBf16, stream);
}

int ltxk_rms_norm_rope_dt(void* out, const void* x, const void* w, const float* cos,
                          const float* sin, int64_t rows, int heads, int head_dim, int mode,
                          float eps, int64_t seq_len, int dtype, ltxk_stream_t stream) {
  return rope_common(out, x, w, cos, sin, rows, heads, head_dim, mode, eps, seq_len,
                     fmt_of(dtype), stream);
}

int ltxk_rms_norm_adaln(void* out, const void* x, const void* w, const void* scale,
                        const void* shift, int64_t rows, int64_t hidden, int64_t rows_per_cond,
                        float eps, ltxk_stream_t stream) {
  return adaln_fmt(out, x, w, scale, shift, rows, hidden, rows_per_cond, eps, ltxk::kBf16,
                   stream);
}

int ltxk_rms_norm_adaln_dt(void* out, const void* x, const void* w, const void* scale,
                           const void* shift, int64_t rows, int64_t hidden,
                           int64_t rows_per_cond, float eps, int dtype, ltxk_stream_t stream) {
  return adaln_fmt(out, x, w, scale, shift, rows, hidden, rows_per_cond, eps, fmt_of(dtype),
                   stream);
}

int ltxk_add_rms_norm(void* out, void* residual_out, const void* x, const void* residual,
                      const void* w, int64_t rows, int64_t hidden, float eps,
                      ltxk_stream_t stream) {
  return add_norm_fmt(out, residual_out, x, residual, w, rows, hidden, eps, ltxk::kBf16, stream);
}

int ltxk_add_rms_norm_dt(void* out, void* residual_out, const void* x, const void* residual,
                         const void* w, int64_t rows, int64_t hidden, float eps, int dtype,
                         ltxk_stream_t stream) {
  return add_norm_fmt(out, residual_out, x, residual, w, rows, hidden, eps, fmt_of(dtype),
                      stream);
}

int ltxk_fault_status(void) {
  int dev = 0, sms = 0;
  unsigned int* fault = nullptr;
  cudaError_t e = device_facts(&dev, &sms, &fault);
  if (e != cudaSuccess) return fail_cuda(e);
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail_cuda(e);
  unsigned int word = 0;
  e = cudaMemcpy(&word, fault, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e);
  if (word != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpy(fault, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail_cuda(e);
    return LTXK_ERR_TIMEOUT;
  }
  return LTXK_OK;
}

int ltxk_set_path(int path) {
  if (path != LTXK_PATH_AUTO && path != LTXK_PATH_REGISTERS && path != LTXK_PATH_TMA) return -1;
  return g_path.exchange(path);
}

int ltxk_diag_missing_copy(void* out, const void* x, int64_t rows, int64_t hidden,
                           uint64_t wait_limit_ns, ltxk_stream_t stream) {
  int st = norm_checks(out, x, nullptr, rows, hidden, ltxk::kBf16);
  if (st != LTXK_OK) return st;
  if (hidden % 8 != 0 || hidden > 4096 || wait_limit_ns < 1000ull ||
      wait_limit_ns > 10000000000ull)
    return LTXK_ERR_SHAPE;
  if (!aligned_to(out, 16) || !aligned_to(x, 16)) return LTXK_ERR_ALIGN;
  if (rows == 0) return LTXK_OK;
  ltxk::RowArgs a{out, x, nullptr, nullptr, nullptr, rows, 1, static_cast<int>(hidden), 0, 1e-6f};
  return launch(LTXK_OP_RMS_NORM, 0, ltxk::kBf16, a, true, stream, LTXK_PATH_TMA, 1,
                wait_limit_ns);
}

const char* ltxk_status_string(int status) {
  switch (status) {
    case LTXK_OK: return "ok";
    case LTXK_ERR_NULL: return "a required pointer is NULL";
    case LTXK_ERR_SHAPE: return "invalid shape";
    case LTXK_ERR_ALIGN: return "pointer not aligned to its element size";
    case LTXK_ERR_MODE: return "unknown RoPE pairing mode";
    case LTXK_ERR_OVERLAP: return "output overlaps an input (other than exactly in place)";
    case LTXK_ERR_CUDA: return "CUDA runtime error (see ltxk_last_cuda_error)";
    case LTXK_ERR_TIMEOUT: return "a kernel gave up waiting for a bulk copy";
    case LTXK_ERR_DTYPE: return "unknown element type";
    default: return "unknown status";
  }
}

int ltxk_last_cuda_error(void) { return g_last_cuda_error; }

int ltxk_plan_launch(int op, int64_t rows, int64_t hidden, int head_dim, int mode, int vector_ok,
                     ltxk_plan* plan) {
  if (plan == nullptr) return LTXK_ERR_NULL;
  return make_plan(op, ltxk::kBf16, rows, hidden, head_dim, mode, vector_ok != 0, g_path.load(),
                   plan);
}

int ltxk_plan_launch_dt(int op, int dtype, int64_t rows, int64_t hidden, int head_dim, int mode,
                        int vector_ok, ltxk_plan* plan) {
  if (plan == nullptr) return LTXK_ERR_NULL;
  const int fmt = fmt_of(dtype);
  if (fmt < 0) return LTXK_ERR_DTYPE;
  return make_plan(op, fmt, rows, hidden, head_dim, mode, vector_ok != 0, g_path.load(), plan);
}

}  // extern "C"
