// Instantiations of the split-KV kernel for K bit-width 16 (all V widths,
// group sizes, both the plain split pass and the fused decode step, the
// 64-position packed blocks where a tile holds them, and the general
// variants for layouts with K-only protected heads and for multi-query
// calls); one translation unit per K width so that they compile in parallel.
#include "kvq_split.cuh"

namespace kvq {
namespace {
template <int VB, int G, bool kStep>
const void* by_halves(int halves, bool general) {
  if (general) return reinterpret_cast<const void*>(&split_mma_kernel<16, VB, G, kStep, 2, true>);
  if constexpr (packed_block_halves(16, VB, G) == 4) {
    if (halves == 4) return reinterpret_cast<const void*>(&split_mma_kernel<16, VB, G, kStep, 4, false>);
  }
  return reinterpret_cast<const void*>(&split_mma_kernel<16, VB, G, kStep, 2, false>);
}
template <int VB, bool kStep>
const void* by_group(int G, int halves, bool general) {
  switch (G) {
    case 32: return by_halves<VB, 32, kStep>(halves, general);
    case 64: return by_halves<VB, 64, kStep>(halves, general);
    case 128: return by_halves<VB, 128, kStep>(halves, general);
  }
  return nullptr;
}
template <bool kStep>
const void* by_vbits(int vb, int G, int halves, bool general) {
  switch (vb) {
    case 2: return by_group<2, kStep>(G, halves, general);
    case 4: return by_group<4, kStep>(G, halves, general);
    case 8: return by_group<8, kStep>(G, halves, general);
    case 16: return by_group<16, kStep>(G, halves, general);
  }
  return nullptr;
}
}  // namespace

const void* split_kernel_k16(int vb, int G, bool step, int halves, bool general) {
  return step ? by_vbits<true>(vb, G, halves, general) : by_vbits<false>(vb, G, halves, general);
}
}  // namespace kvq
