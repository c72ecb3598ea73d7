// Instantiations of the split-KV kernel for K bit-width 16 (all V widths);
// one translation unit per K width so that they compile in parallel.
#include "kvq_split.cuh"

namespace kvq {
const void* split_kernel_k16(int vb) {
  switch (vb) {
    case 2: return reinterpret_cast<const void*>(&split_mma_kernel<16, 2>);
    case 4: return reinterpret_cast<const void*>(&split_mma_kernel<16, 4>);
    case 8: return reinterpret_cast<const void*>(&split_mma_kernel<16, 8>);
    case 16: return reinterpret_cast<const void*>(&split_mma_kernel<16, 16>);
  }
  return nullptr;
}
}  // namespace kvq
