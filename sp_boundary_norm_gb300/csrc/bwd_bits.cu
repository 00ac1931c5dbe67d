// The backward of the bit-packed mask: instantiations of the backward kernel
// template that read the dropout keep decisions one bit per element (byte j
// of a row holds channels [8j, 8j + 8), bit e channel 8j + e) instead of one
// byte per element.
#include "bwd_dispatch.cuh"

namespace spb {

const void* bwd_bits_kernel(int threads, int maxc, int ring) {
  return bwd_kernel_any<false, false, true>(threads, maxc, ring);
}

}  // namespace spb
