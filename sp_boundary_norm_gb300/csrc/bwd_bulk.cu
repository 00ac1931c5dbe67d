// The backward with the gathered dYpre copies sent by bulk copies from a
// shared-memory copy of each row (stored mask), for calls with several
// gathered copies.
#include "bwd_dispatch.cuh"

namespace spb {

const void* bwd_bulk_kernel(int threads, int maxc, int ring) {
  return bwd_kernel_any<false, true>(threads, maxc, ring);
}

}  // namespace spb
