// Instances of the vectorised row kernel for the AdaLN-modulated RMSNorm.
#include "ltxk_instances.cuh"
#include "ltxk_launch.h"

namespace ltxk {
const void* rows_vec_adaln_ptr(int g, int vpl) { return select_rows_vec<kAdaLN>(g, vpl); }
}  // namespace ltxk
