// Instantiations of the split-KV kernel for K bit-width 4 (all V widths,
// group sizes, both the plain split pass and the fused decode step, and the
// 64-position packed blocks where a tile holds them); one translation unit per
// K width so that they compile in parallel.
#include "kvq_split.cuh"

namespace kvq {
namespace {
template <int VB, int G, bool kStep>
const void* by_halves(int halves) {
  if constexpr (packed_block_halves(4, VB, G) == 4) {
    if (halves == 4) return reinterpret_cast<const void*>(&split_mma_kernel<4, VB, G, kStep, 4>);
  }
  return reinterpret_cast<const void*>(&split_mma_kernel<4, VB, G, kStep, 2>);
}
template <int VB, bool kStep>
const void* by_group(int G, int halves) {
  switch (G) {
    case 32: return by_halves<VB, 32, kStep>(halves);
    case 64: return by_halves<VB, 64, kStep>(halves);
    case 128: return by_halves<VB, 128, kStep>(halves);
  }
  return nullptr;
}
template <bool kStep>
const void* by_vbits(int vb, int G, int halves) {
  switch (vb) {
    case 2: return by_group<2, kStep>(G, halves);
    case 4: return by_group<4, kStep>(G, halves);
    case 8: return by_group<8, kStep>(G, halves);
    case 16: return by_group<16, kStep>(G, halves);
  }
  return nullptr;
}
}  // namespace

const void* split_kernel_k4(int vb, int G, bool step, int halves) {
  return step ? by_vbits<true>(vb, G, halves) : by_vbits<false>(vb, G, halves);
}
}  // namespace kvq
