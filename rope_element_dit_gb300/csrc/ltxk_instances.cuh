// ltxk_instances.cuh -- the instances of the vectorised kernels.  Register
// kernel: (group warps, vector slots per lane); group sizes 1..32 warps cover
// hidden up to 32 warps * 32 lanes * 16 slots * 8 = 131072 elements per row.
// TMA ring kernel: one warp per row, up to 16 slots (hidden <= 4096).
#pragma once

#include "ltxk_kernels.cuh"

namespace ltxk {

template <int MODE, int G>
const void* select_vpl(int vpl) {
  switch (vpl) {
    case 4: return reinterpret_cast<const void*>(&rows_vec_kernel<MODE, G, 4>);
    case 8: return reinterpret_cast<const void*>(&rows_vec_kernel<MODE, G, 8>);
    case 12: return reinterpret_cast<const void*>(&rows_vec_kernel<MODE, G, 12>);
    case 16: return reinterpret_cast<const void*>(&rows_vec_kernel<MODE, G, 16>);
    default: return nullptr;
  }
}

template <int MODE>
const void* select_rows_vec(int g, int vpl) {
  switch (g) {
    case 1: return select_vpl<MODE, 1>(vpl);
    case 2: return select_vpl<MODE, 2>(vpl);
    case 4: return select_vpl<MODE, 4>(vpl);
    case 8: return select_vpl<MODE, 8>(vpl);
    case 16: return select_vpl<MODE, 16>(vpl);
    case 32: return select_vpl<MODE, 32>(vpl);
    default: return nullptr;
  }
}

template <int MODE>
const void* select_rows_tma(int vpl) {
  switch (vpl) {
    case 4: return reinterpret_cast<const void*>(&rows_tma_kernel<MODE, 4>);
    case 8: return reinterpret_cast<const void*>(&rows_tma_kernel<MODE, 8>);
    case 12: return reinterpret_cast<const void*>(&rows_tma_kernel<MODE, 12>);
    case 16: return reinterpret_cast<const void*>(&rows_tma_kernel<MODE, 16>);
    default: return nullptr;
  }
}

}  // namespace ltxk
