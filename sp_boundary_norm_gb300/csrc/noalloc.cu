// sp_norm_bwd_noalloc: the boundary backward for callers that cannot hand the
// library a workspace.
//
// Some callers have no way to obtain device memory on their own: code that
// runs inside a host framework which reserves every byte of device memory up
// front and offers no scratch to its plugins, or a path where the implicit
// device synchronisation of cudaMalloc is not acceptable.  For them the
// per-block parameter-gradient partials live in a fixed array in the
// library's own device memory, declared below, instead of in a caller buffer.
// The array is allocated when the library's device code is loaded on a GPU
// and stays until the process exits (SP_NOALLOC_WORKSPACE_BYTES per GPU).
#include <mutex>

#include "sp_internal.h"

namespace {

// Scratch of the allocate-nothing backward, one per GPU that loads the
// library.  Only its device address, looked up with cudaGetSymbolAddress on
// the device in question, is handed to the kernels; the host-side symbol
// itself is not a device address.
static __device__ __align__(256) float g_noalloc_ws[SP_NOALLOC_WORKSPACE_BYTES / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ws_addr[kMaxDevices] = {};

// Device address of g_noalloc_ws on the current device.  Outside stream
// capture it is looked up on every call (a host-side query, no device work),
// so a module reloaded at another address after cudaDeviceReset is seen; the
// address is remembered per device for calls made while `stream` is being
// captured, where the lookup is not made.  A device's first call must
// therefore come before any capture on it.
sp_status_t scratch_address(cudaStream_t stream, void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return spb::record_error(SP_ERR_CUDA, "sp_norm_bwd_noalloc: no usable current device");
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    cudaGetLastError();
    cap = cudaStreamCaptureStatusActive;   // e.g. the legacy stream during a global capture
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_ws);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return spb::record_error(SP_ERR_CUDA,
                               "sp_norm_bwd_noalloc: cudaGetSymbolAddress of the scratch failed");
    }
    g_ws_addr[dev] = p;
  } else if (g_ws_addr[dev] == nullptr) {
    return spb::record_error(SP_ERR_INVALID_ARG,
                             "sp_norm_bwd_noalloc: the first call on a device must come before "
                             "any stream capture on it");
  }
  *out = g_ws_addr[dev];
  return SP_OK;
}

}  // namespace

extern "C" sp_status_t sp_norm_bwd_noalloc(
    const void* const* dy, const void* const* z, const uint8_t* const* mask,
    const float* const* mean, const float* const* rstd, const void* gamma,
    const void* const* dz_skip, int64_t b, int64_t s, int64_t h, int32_t t, double p,
    const int32_t* cu_seqlens, int32_t n_seqs, sp_norm_t norm, void* const* dresidual,
    void* const* dgathered, int32_t n_gather, float* dgamma, float* dbeta, float* dbias,
    int32_t* dev_status, void* stream) {
  const bool valid_shape = b > 0 && s > 0 && h >= 8 && h % 8 == 0 && h <= SP_MAX_HIDDEN;
  const size_t need = valid_shape ? spb::stored_mask_bwd_workspace_bytes(b * s, h, dz_skip != nullptr)
                                  : 0;
  if (need > SP_NOALLOC_WORKSPACE_BYTES) {
    return spb::record_error(
        SP_ERR_UNSUPPORTED,
        "sp_norm_bwd_noalloc: this shape needs more parameter-gradient scratch than the "
        "library's fixed SP_NOALLOC_WORKSPACE_BYTES; use sp_norm_bwd with a workspace");
  }
  void* ws = nullptr;
  const sp_status_t st = scratch_address(static_cast<cudaStream_t>(stream), &ws);
  if (st != SP_OK) return st;
  // The partials are overwritten in full by every call (nothing is
  // accumulated into the scratch), so it needs no clearing between calls.
  return sp_norm_bwd(dy, z, mask, mean, rstd, gamma, dz_skip, b, s, h, t, p, cu_seqlens,
                     n_seqs, norm, dresidual, dgathered, n_gather, dgamma, dbeta, dbias, ws,
                     SP_NOALLOC_WORKSPACE_BYTES, dev_status, stream);
}
