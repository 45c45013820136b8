// ltxk_pipeline.cu -- ltxk_rms_norm_host: RMSNorm of rows held in host
// memory.
//
// Page-locked host memory that the GPU can address (cudaHostAlloc, torch's
// pin_memory, cudaHostRegister): one kernel on streams[0] reads x and writes
// y across the host link itself (zero-copy).  On GB300 the link to the Grace
// CPU (NVLink-C2C) then carries both directions at once, at the rate of two
// concurrent copies, with no staging and no copy engine.
//
// Any other host memory is pipelined over caller-provided streams and device
// staging memory:
// The rows are cut into chunks.  Chunk i goes to stream i % n and staging
// slot i % n: copy x in (host -> device), normalise in place in the slot,
// copy y out (device -> host).  Consecutive chunks run on different streams,
// so the copy-in of one chunk, the kernel of another and the copy-out of a
// third proceed together on the GPU's copy engines and SMs.  A slot is only
// reused by the next chunk on the same stream, after that stream finished
// the previous chunk's copy-out, so stream order alone makes the reuse safe:
// no events, no allocation.
#include <cuda_runtime.h>

#include <cstdint>

#include "ltxk.h"
#include "ltxk_launch.h"

namespace {

int fail(cudaError_t e) {
  ltxk::record_cuda_error(static_cast<int>(e));
  return LTXK_ERR_CUDA;
}

// The current device's address of [p, p + bytes) if the whole range is host
// memory it can access directly (page-locked and mapped, or managed), with
// the device addresses of both ends the same distance apart; else nullptr.
void* device_view(const void* p, int64_t bytes) {
  const char* c = static_cast<const char*>(p);
  cudaPointerAttributes a0, a1;
  if (cudaPointerGetAttributes(&a0, c) != cudaSuccess ||
      cudaPointerGetAttributes(&a1, c + bytes - 1) != cudaSuccess) {
    cudaGetLastError();   // an unknown pointer is not an error here
    return nullptr;
  }
  const bool host0 = a0.type == cudaMemoryTypeHost || a0.type == cudaMemoryTypeManaged;
  const bool host1 = a1.type == cudaMemoryTypeHost || a1.type == cudaMemoryTypeManaged;
  if (!host0 || !host1 || a0.devicePointer == nullptr || a1.devicePointer == nullptr)
    return nullptr;
  if (static_cast<char*>(a1.devicePointer) - static_cast<char*>(a0.devicePointer) != bytes - 1)
    return nullptr;
  return a0.devicePointer;
}

}  // namespace

extern "C" int ltxk_rms_norm_host(void* out_host, const void* x_host, const void* w,
                                  int64_t rows, int64_t hidden, float eps, void* staging,
                                  int64_t staging_bytes, const ltxk_stream_t* streams,
                                  int n_streams) {
  if (out_host == nullptr || x_host == nullptr || staging == nullptr || streams == nullptr)
    return LTXK_ERR_NULL;
  if (rows < 0 || hidden <= 0 || hidden > LTXK_MAX_HIDDEN) return LTXK_ERR_SHAPE;
  if (rows > 0 && rows > INT64_MAX / 4 / hidden) return LTXK_ERR_SHAPE;
  if (n_streams < 1 || n_streams > LTXK_HOST_MAX_STREAMS) return LTXK_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(staging) & 255u) != 0) return LTXK_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(x_host) & 1u) != 0 ||
      (reinterpret_cast<uintptr_t>(out_host) & 1u) != 0 ||
      (reinterpret_cast<uintptr_t>(w) & 1u) != 0)
    return LTXK_ERR_ALIGN;
  const int64_t row_bytes = hidden * 2;
  // each slot starts on a 256-byte boundary so the kernel's vector path applies
  const int64_t slot_bytes = (staging_bytes / n_streams) / 256 * 256;
  const int64_t chunk_rows = slot_bytes / row_bytes;
  if (chunk_rows < 1) return LTXK_ERR_SHAPE;   // staging too small for one row per slot
  // the kernels write the staging slots in place: w must lie outside them
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(staging);
  const uintptr_t w0 = reinterpret_cast<uintptr_t>(w);
  if (w != nullptr && w0 < s0 + static_cast<uint64_t>(staging_bytes) &&
      s0 < w0 + static_cast<uint64_t>(hidden) * 2)
    return LTXK_ERR_OVERLAP;
  // out may be x exactly (in place), never partly
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x_host), ya = reinterpret_cast<uintptr_t>(out_host);
  const uint64_t total = static_cast<uint64_t>(rows) * hidden * 2;
  if (xa != ya && total != 0 && xa < ya + total && ya < xa + total) return LTXK_ERR_OVERLAP;
  if (rows == 0) return LTXK_OK;

  // zero-copy when both buffers are device-accessible host memory (the TMA
  // ring, selectable for tests, always stages)
  if (ltxk::current_path() != LTXK_PATH_TMA) {
    void* yd = device_view(out_host, static_cast<int64_t>(total));
    const void* xd = yd == nullptr ? nullptr : device_view(x_host, static_cast<int64_t>(total));
    if (xd != nullptr) return ltxk_rms_norm(yd, xd, w, rows, hidden, eps, streams[0]);
  }

  const char* xh = static_cast<const char*>(x_host);
  char* yh = static_cast<char*>(out_host);
  char* base = static_cast<char*>(staging);
  int64_t chunk = 0;
  for (int64_t r0 = 0; r0 < rows; r0 += chunk_rows, ++chunk) {
    const int64_t n = rows - r0 < chunk_rows ? rows - r0 : chunk_rows;
    const int k = static_cast<int>(chunk % n_streams);
    ltxk_stream_t s = streams[k];
    char* slot = base + k * slot_bytes;
    const size_t bytes = static_cast<size_t>(n * row_bytes);
    cudaError_t e = cudaMemcpyAsync(slot, xh + r0 * row_bytes, bytes, cudaMemcpyHostToDevice,
                                    reinterpret_cast<cudaStream_t>(s));
    if (e != cudaSuccess) return fail(e);
    const int st = ltxk_rms_norm(slot, slot, w, n, hidden, eps, s);
    if (st != LTXK_OK) return st;
    e = cudaMemcpyAsync(yh + r0 * row_bytes, slot, bytes, cudaMemcpyDeviceToHost,
                        reinterpret_cast<cudaStream_t>(s));
    if (e != cudaSuccess) return fail(e);
  }
  return LTXK_OK;
}
