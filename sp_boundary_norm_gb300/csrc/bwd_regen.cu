// The mask-free backward: instantiations of the backward kernel template that
// draw the dropout keep decisions again from Philox4x32-10 (the forward's
// seed and offset) instead of reading the stored 1-byte mask.
#include "bwd_dispatch.cuh"

namespace spb {

const void* bwd_regen_kernel(int threads, int maxc, int ring) {
  return bwd_kernel_any<true>(threads, maxc, ring);
}

}  // namespace spb
