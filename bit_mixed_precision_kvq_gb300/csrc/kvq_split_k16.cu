// Instantiations of the split-KV kernel for K bit-width 16 (all V widths,
// group sizes, and both the plain split pass and the fused decode step); one
// translation unit per K width so that they compile in parallel.
#include "kvq_split.cuh"

namespace kvq {
namespace {
template <int VB, bool kStep>
const void* by_group(int G) {
  switch (G) {
    case 32: return reinterpret_cast<const void*>(&split_mma_kernel<16, VB, 32, kStep>);
    case 64: return reinterpret_cast<const void*>(&split_mma_kernel<16, VB, 64, kStep>);
    case 128: return reinterpret_cast<const void*>(&split_mma_kernel<16, VB, 128, kStep>);
  }
  return nullptr;
}
template <bool kStep>
const void* by_vbits(int vb, int G) {
  switch (vb) {
    case 2: return by_group<2, kStep>(G);
    case 4: return by_group<4, kStep>(G);
    case 8: return by_group<8, kStep>(G);
    case 16: return by_group<16, kStep>(G);
  }
  return nullptr;
}
}  // namespace

const void* split_kernel_k16(int vb, int G, bool step) {
  return step ? by_vbits<true>(vb, G) : by_vbits<false>(vb, G);
}
}  // namespace kvq
