// The middle step of the unfused boundary (bias, dropout, residual, norm on
// shards reduced by a separate reduce-scatter): instantiations of the forward
// kernel template with one input stream and per-shard output.
#include "fwd_kernel.cuh"

namespace spb {

template <int NTHR>
static const void* fwd_shard_s(int stages) {
  switch (stages) {
    case 2: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, 2, 1, true>);
    case 3: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, 3, 1, true>);
    default: return nullptr;
  }
}

const void* fwd_shard_kernel(int threads, int stages) {
  switch (threads) {
    case 64: return fwd_shard_s<64>(stages);
    case 128: return fwd_shard_s<128>(stages);
    case 160: return fwd_shard_s<160>(stages);
    case 256: return fwd_shard_s<256>(stages);
    default: return nullptr;
  }
}

}  // namespace spb
