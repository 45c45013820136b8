// ltxk_noalloc.cu -- ltxk_rms_norm_noalloc: RMSNorm through the TMA-ring
// kernel for callers that must not allocate device memory, and the reader
// of its fault word.
//
// Who needs this: code that runs where cudaMalloc is unavailable or
// unwelcome. Examples are an engine whose device memory all comes from its
// own pre-sized pool, and a latency-critical loop where an allocation's
// implicit device synchronisation is not acceptable.  The ring kernel needs
// one word of device memory beyond its inputs and outputs: the fault word
// its bounded waits set.  Here that word lives in this file's static device
// array, so this entry point, like the rest of the library, never allocates.
//
// The pages have no counterpart to these entry points.
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>

#include "ltxk.h"
#include "ltxk_kernels.cuh"
#include "ltxk_launch.h"

// Static scratch: 64 words (256 bytes) per device, held from the first use
// of the library on that device until the process exits.  Word 0 is the
// ring kernel's fault word; the rest is reserved.  In host code this name
// is only a stand-in for the symbol: its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned int g_ltxk_noalloc_scratch[LTXK_NOALLOC_SCRATCH_WORDS];

namespace {

constexpr uint32_t kSmemTarget = 100u * 1024u;     // same ring budget as the library
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per mbarrier wait
constexpr int kScratchWordsNeeded = 1;             // the fault word
static_assert(kScratchWordsNeeded <= LTXK_NOALLOC_SCRATCH_WORDS, "scratch too small");

struct NoAllocDevice {
  unsigned int* scratch = nullptr;   // device address of g_ltxk_noalloc_scratch
  int sms = 0;
};

std::mutex g_mu;
std::map<int, NoAllocDevice> g_dev;

int fail(cudaError_t e) {
  ltxk::record_cuda_error(static_cast<int>(e));   // seen by ltxk_last_cuda_error()
  return LTXK_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, uint64_t na, const void* b, uint64_t nb) {
  if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

// Set-up, once per device, with that device current: resolve the scratch
// symbol's device address and the SM count.
cudaError_t device_setup(int dev, NoAllocDevice* out) {
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_dev.find(dev);
  if (it == g_dev.end()) {
    NoAllocDevice d;
    unsigned int* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_ltxk_noalloc_scratch);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    d.scratch = ptr;
    it = g_dev.emplace(dev, d).first;
  }
  *out = it->second;
  return cudaSuccess;
}

// The call, with the diagnostic's two knobs: skip_first_copy leaves every
// warp's first bulk copy unissued, so its wait runs out after wait_limit_ns.
int noalloc_call(void* out, const void* x, const void* w, int64_t rows, int64_t hidden,
                 float eps, ltxk_stream_t stream, int skip_first_copy, uint64_t wait_limit_ns) {
  if (out == nullptr || x == nullptr) return LTXK_ERR_NULL;
  if (rows < 0 || hidden <= 0) return LTXK_ERR_SHAPE;
  // Beyond the maximum this entry point handles: rows longer than one warp's
  // ring buffer slots (4096 elements) or not a whole number of 16-byte vectors.
  if (hidden > LTXK_NOALLOC_MAX_HIDDEN || hidden % 8 != 0) return LTXK_ERR_SHAPE;
  if (rows > INT64_MAX / 4 / hidden) return LTXK_ERR_SHAPE;
  if (!aligned16(out) || !aligned16(x) || (w != nullptr && !aligned16(w))) return LTXK_ERR_ALIGN;
  const uint64_t xbytes = static_cast<uint64_t>(rows) * hidden * 2;
  if (out != x && overlaps(out, xbytes, x, xbytes)) return LTXK_ERR_OVERLAP;
  if (overlaps(out, xbytes, w, static_cast<uint64_t>(hidden) * 2)) return LTXK_ERR_OVERLAP;
  if (rows == 0) return LTXK_OK;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(e);
  NoAllocDevice d;
  e = device_setup(dev, &d);
  if (e != cudaSuccess) return fail(e);

  const int nv = static_cast<int>(hidden / 8);
  const int need = (nv + 31) / 32;
  const int vpl = need <= 4 ? 4 : need <= 8 ? 8 : need <= 12 ? 12 : 16;
  const uint32_t stride = static_cast<uint32_t>((hidden * 2 + 127) / 128 * 128);
  int stages = static_cast<int>((kSmemTarget - ltxk::kTmaBarBytes) / (ltxk::kTmaWarps * stride));
  stages = stages < 1 ? 1 : (stages > ltxk::kTmaMaxStages ? ltxk::kTmaMaxStages : stages);
  const int smem = static_cast<int>(ltxk::kTmaBarBytes + ltxk::kTmaWarps * stages * stride);
  const void* fn = ltxk::rows_tma_plain_ptr(vpl);
  if (fn == nullptr) return fail(cudaErrorInvalidDeviceFunction);
  // The library's one record per (device, kernel) opts the kernel in to this
  // much shared memory (only ever raising the limit) and caches the
  // occupancy per shared-memory size.
  int per_sm = 0;
  e = ltxk::resident_ctas(dev, fn, ltxk::kTmaWarps * 32, smem, &per_sm);
  if (e != cudaSuccess) return fail(e);
  const int64_t needed = (rows + ltxk::kTmaWarps - 1) / ltxk::kTmaWarps;
  const int64_t cap = static_cast<int64_t>(d.sms) * per_sm;
  const unsigned grid = static_cast<unsigned>(needed < cap ? needed : cap);

  // The fault word must start at zero: clear it on the caller's stream.
  e = cudaMemsetAsync(d.scratch, 0, kScratchWordsNeeded * sizeof(unsigned int), stream);
  if (e != cudaSuccess) return fail(e);
  ltxk::RowArgs a{static_cast<uint16_t*>(out), static_cast<const uint16_t*>(x),
                  static_cast<const uint16_t*>(w), nullptr, nullptr, rows, 1,
                  static_cast<int>(hidden), 0, eps};
  ltxk::TmaArgs ta{a, stages, stride, wait_limit_ns, skip_first_copy, d.scratch};
  void* params[] = {&ta};
  e = cudaLaunchKernel(fn, dim3(grid), dim3(ltxk::kTmaWarps * 32), params,
                       static_cast<size_t>(smem), stream);
  if (e != cudaSuccess) return fail(e);
  return LTXK_OK;
}

}  // namespace

extern "C" int ltxk_rms_norm_noalloc(void* out, const void* x, const void* w, int64_t rows,
                                     int64_t hidden, float eps, ltxk_stream_t stream) {
  return noalloc_call(out, x, w, rows, hidden, eps, stream, 0, kWaitLimitNs);
}

extern "C" int ltxk_noalloc_fault_status(void) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(e);
  NoAllocDevice d;
  e = device_setup(dev, &d);
  if (e != cudaSuccess) return fail(e);
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(e);
  unsigned int word = 0;
  e = cudaMemcpy(&word, d.scratch, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(e);
  if (word == 0) return LTXK_OK;
  const unsigned int zero = 0;
  e = cudaMemcpy(d.scratch, &zero, sizeof zero, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail(e);
  return LTXK_ERR_TIMEOUT;
}

extern "C" int ltxk_diag_noalloc_missing_copy(void* out, const void* x, int64_t rows,
                                              int64_t hidden, uint64_t wait_limit_ns,
                                              ltxk_stream_t stream) {
  if (wait_limit_ns < 1000ull || wait_limit_ns > 10000000000ull) return LTXK_ERR_SHAPE;
  return noalloc_call(out, x, nullptr, rows, hidden, 1e-6f, stream, 1, wait_limit_ns);
}
