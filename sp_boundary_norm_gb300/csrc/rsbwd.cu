// Instantiations of the backward entered through g (rsbwd_kernel.cuh) with the
// dropout mask stored one byte per element.
#include "rsbwd_kernel.cuh"

namespace spb {

const void* rs_bwd_kernel(int threads, int maxc, int t, int stages) {
  return rs_bwd_any<false>(threads, maxc, t, stages);
}

}  // namespace spb
