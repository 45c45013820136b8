// Instances of the row kernels for RMSNorm + interleaved RoPE, in the
// element format given by LTXK_FMT (this file is compiled once per format).
#include "ltxk_instances.cuh"
#include "ltxk_launch.h"

LTXK_DEFINE_ROW_GETTERS(kInterleaved)

#if LTXK_FMT == 0
namespace ltxk {
const void* rows_tma_interleaved_ptr(int vpl) { return select_rows_tma<kInterleaved>(vpl); }
}  // namespace ltxk
#endif
