// The forwards that store the dropout mask other than one byte per element:
// not at all (the mask-free pipeline: the fused boundary and the shard step
// of the unfused one; the backward draws the keep decisions again from the
// same counter-based generator), or one bit per element (the fused
// boundary).  Same shapes as the byte-mask instantiations, without the 2-CTA
// row split.
#include "fwd_kernel.cuh"

namespace spb {

template <int NTHR, int TT, bool SHARD, int MASKF>
static const void* fwd_fmt_s(int stages) {
  switch (stages) {
    case 2: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, 2, TT, SHARD, 1, MASKF>);
    case 3: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, 3, TT, SHARD, 1, MASKF>);
    default: return nullptr;
  }
}

template <int MASKF>
static const void* fwd_fmt(int threads, int t, int stages) {
  const bool t8 = (t == 8);
  switch (threads) {
    case 64: return t8 ? fwd_fmt_s<64, 8, false, MASKF>(stages) : fwd_fmt_s<64, 0, false, MASKF>(stages);
    case 128: return t8 ? fwd_fmt_s<128, 8, false, MASKF>(stages) : fwd_fmt_s<128, 0, false, MASKF>(stages);
    case 160: return t8 ? fwd_fmt_s<160, 8, false, MASKF>(stages) : fwd_fmt_s<160, 0, false, MASKF>(stages);
    case 256: return t8 ? fwd_fmt_s<256, 8, false, MASKF>(stages) : fwd_fmt_s<256, 0, false, MASKF>(stages);
    default: return nullptr;
  }
}

const void* fwd_nomask_kernel(int threads, int t, int stages) {
  return fwd_fmt<kMaskNone>(threads, t, stages);
}

const void* fwd_bits_kernel(int threads, int t, int stages) {
  return fwd_fmt<kMaskBits>(threads, t, stages);
}

const void* fwd_shard_nomask_kernel(int threads, int stages) {
  switch (threads) {
    case 64: return fwd_fmt_s<64, 1, true, kMaskNone>(stages);
    case 128: return fwd_fmt_s<128, 1, true, kMaskNone>(stages);
    case 160: return fwd_fmt_s<160, 1, true, kMaskNone>(stages);
    case 256: return fwd_fmt_s<256, 1, true, kMaskNone>(stages);
    default: return nullptr;
  }
}

}  // namespace spb
