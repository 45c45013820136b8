// ltxk_launch.h -- internal interface between the C-ABI front end
// (ltxk_abi.cu) and the translation units that instantiate the kernels.
#pragma once

namespace ltxk {

// Kernel function for (group warps, vector slots per lane), or nullptr if
// that combination is not instantiated.  One function per pairing mode.
const void* rows_vec_plain_ptr(int group_warps, int vec_per_lane);
const void* rows_vec_interleaved_ptr(int group_warps, int vec_per_lane);
const void* rows_vec_split_ptr(int group_warps, int vec_per_lane);
const void* rows_vec_adaln_ptr(int group_warps, int vec_per_lane);
const void* rows_vec_addnorm_ptr(int group_warps, int vec_per_lane);

// TMA ring kernel for vector slots per lane, or nullptr.
const void* rows_tma_plain_ptr(int vec_per_lane);
const void* rows_tma_interleaved_ptr(int vec_per_lane);
const void* rows_tma_split_ptr(int vec_per_lane);

// Record a cudaError_t for ltxk_last_cuda_error() (calling thread).
void record_cuda_error(int e);

// Element-wise kernel for a mode (0 plain, 1 interleaved, 2 split-half,
// 3 AdaLN, 4 residual add + RMSNorm).
const void* rows_elem_kernel_ptr(int mode);

}  // namespace ltxk
