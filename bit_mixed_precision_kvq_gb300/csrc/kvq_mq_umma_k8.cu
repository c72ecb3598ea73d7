// Instantiations of the multi-query tensor-core kernel for K bit-width 8
// (all V widths and group sizes); one translation unit per K width so that
// they compile in parallel.
#include "kvq_mq_umma.cuh"

namespace kvq {
namespace {
template <int VB>
const void* by_group(int G) {
  switch (G) {
    case 32: return reinterpret_cast<const void*>(&mq::mq_umma_kernel<8, VB, 32>);
    case 64: return reinterpret_cast<const void*>(&mq::mq_umma_kernel<8, VB, 64>);
    case 128: return reinterpret_cast<const void*>(&mq::mq_umma_kernel<8, VB, 128>);
  }
  return nullptr;
}
}  // namespace

const void* mq_umma_kernel_k8(int vb, int G) {
  switch (vb) {
    case 2: return by_group<2>(G);
    case 4: return by_group<4>(G);
    case 8: return by_group<8>(G);
    case 16: return by_group<16>(G);
  }
  return nullptr;
}
}  // namespace kvq
