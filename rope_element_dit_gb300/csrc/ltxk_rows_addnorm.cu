// Instances of the row kernels for the fused residual add + RMSNorm, in the
// element format given by LTXK_FMT (this file is compiled once per format).
#include "ltxk_instances.cuh"
#include "ltxk_launch.h"

LTXK_DEFINE_ROW_GETTERS(kAddNorm)
