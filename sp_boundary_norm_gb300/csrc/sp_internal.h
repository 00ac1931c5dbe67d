// Internal declarations shared by the host entry points and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sp_boundary.h"

namespace spb {

// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As
// Easy as 1, 2, 3", SC'11): the two round multipliers and the Weyl key
// increments (golden ratio, sqrt(3) - 1).
constexpr uint32_t kPhiloxMul0 = 0xD2511F53u;
constexpr uint32_t kPhiloxMul1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxWeyl0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxWeyl1 = 0xBB67AE85u;

// The key of each of the ten rounds, (k0 + r * W0, k1 + r * W1) mod 2^32 for
// round r: fixed per seed, so it is computed once on the host and read by the
// kernels from their parameters.
// Backward launch shapes (threads, chunks per row) whose per-thread
// parameter-gradient terms live in tensor memory instead of registers, and
// the tensor-memory columns one block of them allocates: 24 columns per chunk
// (dgamma, dbeta, dbias terms of 8 channels) for each warp sharing a lane
// quarter, rounded up to a power of two.  512 / columns blocks fit an SM.
__host__ __device__ constexpr bool bwd_tmem_shape(int nthr, int maxc) {
  return (nthr == 256 && maxc == 4) || (nthr == 128 && maxc == 4) || (nthr == 320 && maxc == 2);
}
__host__ __device__ constexpr int bwd_tmem_cols(int nthr, int maxc) {
  int need = ((nthr / 32 + 3) / 4) * 24 * maxc, c = 32;
  while (c < need) c <<= 1;
  return c;
}

// The backward's staged chunk of one row ("item"), shared by the kernel's
// shared-memory layout and the host's launch-shape choice: dY and Z (16 bytes
// per thread each), then the mask (8 bytes per thread as bytes, one byte per
// thread as bits, none when drawn again), then the optional skip gradient
// (16 bytes per thread).  Offsets of the mask and the skip gradient inside it:
__host__ __device__ constexpr int bwd_item_mask_offset(int nthr) { return 2 * nthr * 16; }
__host__ __device__ constexpr int bwd_item_skip_offset(int nthr, bool regen, bool bits) {
  return bwd_item_mask_offset(nthr) + (regen ? 0 : bits ? nthr : nthr * 8);
}
__host__ __device__ constexpr int bwd_item_bytes(int nthr, bool has_skip, bool regen, bool bits) {
  return bwd_item_skip_offset(nthr, regen, bits) + (has_skip ? nthr * 16 : 0);
}

// The backward entered through g keeps each row's Z, mask and optional skip
// gradient in a row buffer of MAXC such items, shared by its kernel and the
// host: Z (16 bytes per thread), the mask (8 bytes per thread as bytes, one
// byte per thread as bits), the skip gradient (16 bytes per thread).
__host__ __device__ constexpr int rsbwd_rb_skip_offset(int nthr, bool bits) {
  return nthr * 16 + (bits ? nthr : nthr * 8);
}
__host__ __device__ constexpr int rsbwd_rb_item_bytes(int nthr, bool has_skip, bool bits) {
  return rsbwd_rb_skip_offset(nthr, bits) + (has_skip ? nthr * 16 : 0);
}

struct PhiloxKeys {
  uint32_t k0[10], k1[10];
};

inline void philox_round_keys(uint64_t seed, PhiloxKeys* rk) {
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    rk->k0[r] = k0;
    rk->k1[r] = k1;
    k0 += kPhiloxWeyl0;
    k1 += kPhiloxWeyl1;
  }
}

// Where each token of the (b, s) token grid lives: sequence shard k holds
// positions [off[k], off[k+1]) of every batch row (o_k = floor(k*s/t)).
struct ShardMap {
  int64_t off[SP_MAX_RANKS + 1];
  int64_t b, s, h;
  int32_t t;
};

// How a forward stores the dropout mask.
constexpr int kMaskNone = 0;    // not at all
constexpr int kMaskBytes = 1;   // one byte per element, 1 = kept
constexpr int kMaskBits = 2;    // one bit per element, 8 channels per byte

// The forward's blocks add one copy-producer warp to their compute threads.
constexpr int kFwdProducerThreads = 32;

struct FwdParams {
  ShardMap map;
  const uint16_t* partials[SP_MAX_RANKS];
  const uint16_t* residual[SP_MAX_RANKS];
  uint16_t* z[SP_MAX_RANKS];
  uint8_t* mask[SP_MAX_RANKS];
  float* mean[SP_MAX_RANKS];
  float* rstd[SP_MAX_RANKS];
  uint16_t* gathered[SP_MAX_RANKS];
  const uint16_t* bias;
  const uint16_t* gamma;
  const uint16_t* beta;
  const int32_t* cu_seqlens;
  int32_t n_seqs;
  int32_t n_gather;
  int32_t norm;          // sp_norm_t
  uint32_t thr;          // keep iff draw >= thr; 0 disables dropout
  float scale;           // float(1/(1-p))
  float eps;
  PhiloxKeys rk;         // Philox round keys of the seed
  int32_t withhold;      // test hook: block 0 never stages its first chunk
  uint32_t off0, off1;   // Philox counter words 2, 3 = offset
  int64_t rows;          // b * s
  int32_t* status;
};

struct BwdParams {
  ShardMap map;
  const uint16_t* dy[SP_MAX_RANKS];
  const uint16_t* z[SP_MAX_RANKS];
  const uint8_t* mask[SP_MAX_RANKS];
  const float* mean[SP_MAX_RANKS];
  const float* rstd[SP_MAX_RANKS];
  const uint16_t* dz_skip[SP_MAX_RANKS];
  uint16_t* dresidual[SP_MAX_RANKS];
  uint16_t* dgathered[SP_MAX_RANKS];
  const uint16_t* gamma;
  const int32_t* cu_seqlens;
  int32_t n_seqs;
  int32_t n_gather;
  int32_t norm;
  int32_t has_skip;
  float scale;
  uint32_t thr;          // mask regeneration (mask-free backward): keep iff draw >= thr
  PhiloxKeys rk;         // Philox round keys of the forward's seed
  uint32_t off0, off1;   // Philox counter offset = the forward's offset
  int64_t rows;
  float* ws;             // [gridDim.x][3][h] per-block parameter-gradient partials
  int32_t* status;
};

struct ParamReduceParams {
  const float* ws;       // [nblk][3][h]
  int32_t nblk;
  int64_t h;
  float* out[3];         // dgamma, dbeta, dbias (NULL = skip)
};

struct CopyParams {
  ShardMap map;
  const uint16_t* src[SP_MAX_RANKS];
  uint16_t* dst[SP_MAX_RANKS];
  int32_t n_dst;
  const int32_t* cu_seqlens;
  int32_t n_seqs;
  int64_t rows;
  int32_t* status;
};

// Launch shapes chosen on the host.
struct LaunchShape {
  int threads;     // threads per block (consumers of one token row)
  int maxc;        // chunks per row (backward: its compile-time bound)
  int stages;      // cp.async pipeline depth (forward: chunks; backward: rows)
  int grid;        // blocks
  size_t smem;     // dynamic shared memory bytes
  bool fits;       // false: no instantiated shape fits this SM's shared memory
  int cluster;     // CTAs per thread-block cluster (forward: CTAs sharing a row); 1 = none
};

int device_sm_count();

// Launches kernel `fn` (one parameter-struct argument per entry of `args`)
// with programmatic stream serialisation, and a cluster dimension of
// `cluster` CTAs when above 1: its blocks are placed as soon as every block
// of the previous kernel on the stream has exited, and every kernel of the
// library waits for that kernel's memory operations (pdl_wait) before its
// first global memory access.
cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, void** args,
                       cudaStream_t st, int cluster = 1);

// Sets the thread's sp_last_error() text; returns `code`.
sp_status_t record_error(sp_status_t code, const char* message);

// Kernel entry of a launch shape, or nullptr if that shape is not instantiated.
// Forward: (threads, ranks t, pipeline stages); backward: (threads, chunks per
// row, ring rows).
const void* fwd_kernel(int threads, int t, int stages);
// The forward with each row split over a cluster of two CTAs (threads 128 or 256).
const void* fwd_kernel_pair(int threads, int t, int stages);
const void* fwd_shard_kernel(int threads, int stages);
// The same two forwards storing no dropout mask (no cluster variant).
const void* fwd_nomask_kernel(int threads, int t, int stages);
const void* fwd_shard_nomask_kernel(int threads, int stages);
// The fused forward storing the mask one bit per element (no cluster variant).
const void* fwd_bits_kernel(int threads, int t, int stages);
const void* bwd_kernel(int threads, int maxc, int ring);
const void* bwd_regen_kernel(int threads, int maxc, int ring);
// The stored-mask backward sending dYpre to its gathered copies with bulk copies.
const void* bwd_bulk_kernel(int threads, int maxc, int ring);
// The backward reading the mask stored one bit per element.
const void* bwd_bits_kernel(int threads, int maxc, int ring);
// Backward entered through g (reduce-scatter of t partial gradients fused):
// (threads, chunks per row, ranks t, chunk stages).
const void* rs_bwd_kernel(int threads, int maxc, int t, int stages);
// The same reading the mask stored one bit per element.
const void* rs_bwd_bits_kernel(int threads, int maxc, int t, int stages);

// Workspace bytes of one sp_norm_bwd call (stored mask) of `rows` tokens of
// width h (0 for shapes outside the limits): its own launch grid, not the
// maximum over the backward variants that sp_norm_bwd_workspace_bytes reports.
size_t stored_mask_bwd_workspace_bytes(int64_t rows, int64_t h, bool has_skip);
cudaError_t launch_param_reduce(const ParamReduceParams& p, cudaStream_t st);
cudaError_t launch_allgather(const CopyParams& p, cudaStream_t st);
cudaError_t launch_reduce_scatter(const CopyParams& p, int t, cudaStream_t st);
cudaError_t launch_debug_philox(const uint32_t* in, uint32_t* out, int64_t n, cudaStream_t st);

}  // namespace spb
