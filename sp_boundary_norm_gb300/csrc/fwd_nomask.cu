// The forwards of the mask-free pipeline: the fused boundary and the shard
// step of the unfused one, storing no dropout mask (the backward draws the
// keep decisions again from the same counter-based generator).  Same shapes
// as the stored-mask instantiations, without the 2-CTA row split.
#include "fwd_kernel.cuh"

namespace spb {

template <int NTHR, int TT, bool SHARD>
static const void* fwd_nomask_s(int stages) {
  switch (stages) {
    case 2: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, 2, TT, SHARD, 1, false>);
    case 3: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, 3, TT, SHARD, 1, false>);
    default: return nullptr;
  }
}

const void* fwd_nomask_kernel(int threads, int t, int stages) {
  const bool t8 = (t == 8);
  switch (threads) {
    case 64: return t8 ? fwd_nomask_s<64, 8, false>(stages) : fwd_nomask_s<64, 0, false>(stages);
    case 128: return t8 ? fwd_nomask_s<128, 8, false>(stages) : fwd_nomask_s<128, 0, false>(stages);
    case 160: return t8 ? fwd_nomask_s<160, 8, false>(stages) : fwd_nomask_s<160, 0, false>(stages);
    case 256: return t8 ? fwd_nomask_s<256, 8, false>(stages) : fwd_nomask_s<256, 0, false>(stages);
    default: return nullptr;
  }
}

const void* fwd_shard_nomask_kernel(int threads, int stages) {
  switch (threads) {
    case 64: return fwd_nomask_s<64, 1, true>(stages);
    case 128: return fwd_nomask_s<128, 1, true>(stages);
    case 160: return fwd_nomask_s<160, 1, true>(stages);
    case 256: return fwd_nomask_s<256, 1, true>(stages);
    default: return nullptr;
  }
}

}  // namespace spb
