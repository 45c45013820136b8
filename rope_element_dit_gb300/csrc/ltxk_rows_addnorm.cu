// Instances of the vectorised row kernel for the fused residual add + RMSNorm.
#include "ltxk_instances.cuh"
#include "ltxk_launch.h"

namespace ltxk {
const void* rows_vec_addnorm_ptr(int g, int vpl) { return select_rows_vec<kAddNorm>(g, vpl); }
}  // namespace ltxk
