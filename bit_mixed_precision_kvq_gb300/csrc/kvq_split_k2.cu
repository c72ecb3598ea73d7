// Global-mode instantiations of the split-KV kernel for K bit-width 2 (all
// V widths, group sizes, the plain split pass and the fused decode step,
// the 64-position packed blocks where a tile holds them, and the general
// variants for layouts with K-only protected heads and for multi-query
// calls).
#include "kvq_split_inst.cuh"

namespace kvq {
const void* split_kernel_k2(int vb, int G, bool step, int halves, bool general) {
  return split_inst::dispatch<2, false>(vb, G, step, halves, general);
}
}  // namespace kvq
