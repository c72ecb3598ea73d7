// kvq_split_inst.cuh -- the table from (V bits, G, step, packed-block
// halves, general) to one instantiation of split_mma_kernel, for a K width
// KB and a mode (kCl: cluster mode, where a unit's CTAs combine through
// distributed shared memory; else global mode).  Each kvq_split_*.cu
// translation unit instantiates one (KB, mode) so that they compile in
// parallel; the two modes are separate kernels so that neither carries the
// other's code (instruction-cache footprint).
#pragma once

#include "kvq_split.cuh"

namespace kvq {
namespace split_inst {

template <int KB, bool kCl, int VB, int G, bool kStep>
const void* by_halves(int halves, bool general) {
  if (general) return reinterpret_cast<const void*>(&split_mma_kernel<KB, VB, G, kStep, 2, true, kCl>);
  if constexpr (packed_block_halves(KB, VB, G) == 4) {
    if (halves == 4) return reinterpret_cast<const void*>(&split_mma_kernel<KB, VB, G, kStep, 4, false, kCl>);
  }
  return reinterpret_cast<const void*>(&split_mma_kernel<KB, VB, G, kStep, 2, false, kCl>);
}

template <int KB, bool kCl, int VB, bool kStep>
const void* by_group(int G, int halves, bool general) {
  switch (G) {
    case 32: return by_halves<KB, kCl, VB, 32, kStep>(halves, general);
    case 64: return by_halves<KB, kCl, VB, 64, kStep>(halves, general);
    case 128: return by_halves<KB, kCl, VB, 128, kStep>(halves, general);
  }
  return nullptr;
}

template <int KB, bool kCl, bool kStep>
const void* by_vbits(int vb, int G, int halves, bool general) {
  switch (vb) {
    case 2: return by_group<KB, kCl, 2, kStep>(G, halves, general);
    case 4: return by_group<KB, kCl, 4, kStep>(G, halves, general);
    case 8: return by_group<KB, kCl, 8, kStep>(G, halves, general);
    case 16: return by_group<KB, kCl, 16, kStep>(G, halves, general);
  }
  return nullptr;
}

template <int KB, bool kCl>
const void* dispatch(int vb, int G, bool step, int halves, bool general) {
  return step ? by_vbits<KB, kCl, true>(vb, G, halves, general) : by_vbits<KB, kCl, false>(vb, G, halves, general);
}

}  // namespace split_inst
}  // namespace kvq
