// ltxk_instances.cuh -- the instances of the vectorised kernels.  Register
// kernel: (group warps, vector slots per lane, element format); group sizes
// 1..32 warps cover hidden up to 32 warps * 32 lanes * 16 slots * 8 =
// 131072 elements per row (fp32 rows: 8 slots, 65536 elements).
// TMA ring kernel: bf16 rows, one warp per row, up to 16 slots (hidden <=
// 4096).
#pragma once

#include "ltxk_kernels.cuh"

namespace ltxk {

template <int MODE, int G, int FMT>
const void* select_vpl(int vpl) {
  switch (vpl) {
    case 4: return reinterpret_cast<const void*>(&rows_vec_kernel<MODE, G, 4, FMT>);
    case 8: return reinterpret_cast<const void*>(&rows_vec_kernel<MODE, G, 8, FMT>);
    default: break;
  }
  if constexpr (FMT != kF32) {   // fp32 slots are twice the registers: at most 8
    switch (vpl) {
      case 12: return reinterpret_cast<const void*>(&rows_vec_kernel<MODE, G, 12, FMT>);
      case 16: return reinterpret_cast<const void*>(&rows_vec_kernel<MODE, G, 16, FMT>);
      default: break;
    }
  }
  return nullptr;
}

template <int MODE, int FMT>
const void* select_rows_vec(int g, int vpl) {
  switch (g) {
    case 1: return select_vpl<MODE, 1, FMT>(vpl);
    case 2: return select_vpl<MODE, 2, FMT>(vpl);
    case 4: return select_vpl<MODE, 4, FMT>(vpl);
    case 8: return select_vpl<MODE, 8, FMT>(vpl);
    case 16: return select_vpl<MODE, 16, FMT>(vpl);
    case 32: return select_vpl<MODE, 32, FMT>(vpl);
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

// Each instance file is compiled once per element format, with
// -DLTXK_FMT=<Fmt>, and defines the getters of its mode for that format.
#ifndef LTXK_FMT
#define LTXK_FMT 0
#endif

#define LTXK_DEFINE_ROW_GETTERS(MODE)                                          \
  namespace ltxk {                                                             \
  template <>                                                                  \
  const void* rows_vec_ptr<MODE, LTXK_FMT>(int group_warps, int vec_per_lane) { \
    return select_rows_vec<MODE, LTXK_FMT>(group_warps, vec_per_lane);         \
  }                                                                            \
  template <>                                                                  \
  const void* rows_elem_ptr<MODE, LTXK_FMT>() {                                \
    return reinterpret_cast<const void*>(&rows_elem_kernel<MODE, LTXK_FMT>);   \
  }                                                                            \
  }
