// Launch-shape dispatch of the backward kernel template.
#pragma once

#include "bwd_kernel.cuh"

namespace spb {

template <int NTHR, int MAXC, bool REGEN, bool BULK, bool BITS>
static const void* bwd_kernel_s(int ring) {
  switch (ring) {
    case 1: return reinterpret_cast<const void*>(norm_bwd_kernel<NTHR, MAXC, 1, REGEN, BULK, BITS>);
    case 2: return reinterpret_cast<const void*>(norm_bwd_kernel<NTHR, MAXC, 2, REGEN, BULK, BITS>);
    case 3: return reinterpret_cast<const void*>(norm_bwd_kernel<NTHR, MAXC, 3, REGEN, BULK, BITS>);
    default: return nullptr;
  }
}

// Instantiated shapes (threads, chunks per row): (64, 1), (128, 2), (256, 1),
// (256, 2), (512, 1), (512, 2), (512, 4), (640, 1) with the parameter-gradient
// terms in registers, (128, 4), (256, 4), (320, 2) with them in tensor memory;
// ring of 1, 2 or 3 rows; dYpre stored per thread or (BULK) sent by bulk copies;
// the mask read as bytes, as bits (BITS) or drawn again (REGEN).
template <bool REGEN, bool BULK = false, bool BITS = false>
static const void* bwd_kernel_any(int threads, int maxc, int ring) {
  switch (threads * 8 + maxc) {
    case 64 * 8 + 1: return bwd_kernel_s<64, 1, REGEN, BULK, BITS>(ring);
    case 128 * 8 + 2: return bwd_kernel_s<128, 2, REGEN, BULK, BITS>(ring);
    case 256 * 8 + 1: return bwd_kernel_s<256, 1, REGEN, BULK, BITS>(ring);
    case 256 * 8 + 2: return bwd_kernel_s<256, 2, REGEN, BULK, BITS>(ring);
    case 128 * 8 + 4: return bwd_kernel_s<128, 4, REGEN, BULK, BITS>(ring);
    case 256 * 8 + 4: return bwd_kernel_s<256, 4, REGEN, BULK, BITS>(ring);
    case 320 * 8 + 2: return bwd_kernel_s<320, 2, REGEN, BULK, BITS>(ring);
    case 512 * 8 + 1: return bwd_kernel_s<512, 1, REGEN, BULK, BITS>(ring);
    case 512 * 8 + 2: return bwd_kernel_s<512, 2, REGEN, BULK, BITS>(ring);
    case 512 * 8 + 4: return bwd_kernel_s<512, 4, REGEN, BULK, BITS>(ring);
    case 640 * 8 + 1: return bwd_kernel_s<640, 1, REGEN, BULK, BITS>(ring);
    default: return nullptr;
  }
}

}  // namespace spb
