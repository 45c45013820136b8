// Instances of the vectorised row kernel for RMSNorm + split-half RoPE, and
// of the element-wise kernel for all three modes.
#include "ltxk_instances.cuh"
#include "ltxk_launch.h"

namespace ltxk {
const void* rows_tma_split_ptr(int vpl) { return select_rows_tma<kSplitHalf>(vpl); }
const void* rows_vec_split_ptr(int g, int vpl) { return select_rows_vec<kSplitHalf>(g, vpl); }

const void* rows_elem_kernel_ptr(int mode) {
  switch (mode) {
    case kPlain: return reinterpret_cast<const void*>(&rows_elem_kernel<kPlain>);
    case kInterleaved: return reinterpret_cast<const void*>(&rows_elem_kernel<kInterleaved>);
    case kSplitHalf: return reinterpret_cast<const void*>(&rows_elem_kernel<kSplitHalf>);
    case kAdaLN: return reinterpret_cast<const void*>(&rows_elem_kernel<kAdaLN>);
    case kAddNorm: return reinterpret_cast<const void*>(&rows_elem_kernel<kAddNorm>);
    default: return nullptr;
  }
}
}  // namespace ltxk
