// ltxk_launch.h -- internal interface between the C-ABI front end
// (ltxk_abi.cu) and the translation units that instantiate the kernels.
#pragma once

#include "ltxk_kernels.cuh"

namespace ltxk {

// Register kernel of a pairing mode and element format for (group warps,
// vector slots per lane), or nullptr if that combination is not
// instantiated; element-wise kernel of a mode and format.  The instance
// file of each mode defines them for the format it is compiled for.
template <int MODE, int FMT>
const void* rows_vec_ptr(int group_warps, int vec_per_lane);
template <int MODE, int FMT>
const void* rows_elem_ptr();

#define LTXK_DECLARE_ROW_GETTERS(MODE, FMT)                      \
  template <>                                                    \
  const void* rows_vec_ptr<MODE, FMT>(int group_warps, int vec_per_lane); \
  template <>                                                    \
  const void* rows_elem_ptr<MODE, FMT>();
#define LTXK_DECLARE_FMT_GETTERS(FMT)          \
  LTXK_DECLARE_ROW_GETTERS(kPlain, FMT)        \
  LTXK_DECLARE_ROW_GETTERS(kInterleaved, FMT)  \
  LTXK_DECLARE_ROW_GETTERS(kSplitHalf, FMT)    \
  LTXK_DECLARE_ROW_GETTERS(kAdaLN, FMT)        \
  LTXK_DECLARE_ROW_GETTERS(kAddNorm, FMT)
LTXK_DECLARE_FMT_GETTERS(kBf16)
LTXK_DECLARE_FMT_GETTERS(kF16)
LTXK_DECLARE_FMT_GETTERS(kF32)
#undef LTXK_DECLARE_FMT_GETTERS
#undef LTXK_DECLARE_ROW_GETTERS

// TMA ring kernel (bf16 rows) for vector slots per lane, or nullptr.
const void* rows_tma_plain_ptr(int vec_per_lane);
const void* rows_tma_interleaved_ptr(int vec_per_lane);
const void* rows_tma_split_ptr(int vec_per_lane);

// Record a cudaError_t for ltxk_last_cuda_error() (calling thread).
void record_cuda_error(int e);

// Resident CTAs per SM of kernel `fn` with `block` threads and `smem` bytes
// of dynamic shared memory on device `dev`, after opting the kernel in to
// that much dynamic shared memory.  One record per (device, kernel) keeps
// the opt-in monotonic (it is only ever raised), under one lock, for every
// entry point that launches the kernel.
cudaError_t resident_ctas(int dev, const void* fn, int block, int smem, int* per_sm);

// The kernel-family setting of ltxk_set_path (LTXK_PATH_*).
int current_path();

}  // namespace ltxk
