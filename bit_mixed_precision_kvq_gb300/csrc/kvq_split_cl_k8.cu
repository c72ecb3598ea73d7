// Cluster-mode instantiations of the split-KV kernel for K bit-width 8
// (the same variants as the global-mode ones).
#include "kvq_split_inst.cuh"

namespace kvq {
const void* split_kernel_cl_k8(int vb, int G, bool step, int halves, bool general) {
  return split_inst::dispatch<8, true>(vb, G, step, halves, general);
}
}  // namespace kvq
