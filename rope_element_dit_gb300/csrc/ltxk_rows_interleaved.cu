// Instances of the vectorised row kernel for RMSNorm + interleaved RoPE.
#include "ltxk_instances.cuh"
#include "ltxk_launch.h"

namespace ltxk {
const void* rows_tma_interleaved_ptr(int vpl) { return select_rows_tma<kInterleaved>(vpl); }
const void* rows_vec_interleaved_ptr(int g, int vpl) {
  return select_rows_vec<kInterleaved>(g, vpl);
}
}  // namespace ltxk
