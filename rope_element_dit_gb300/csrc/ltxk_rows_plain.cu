// Instances of the vectorised row kernel for plain RMSNorm.
#include "ltxk_instances.cuh"
#include "ltxk_launch.h"

namespace ltxk {
const void* rows_tma_plain_ptr(int vpl) { return select_rows_tma<kPlain>(vpl); }
const void* rows_vec_plain_ptr(int g, int vpl) { return select_rows_vec<kPlain>(g, vpl); }
}  // namespace ltxk
