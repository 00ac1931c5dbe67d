// Fused forward of the SP boundary: g* reduce-scatter + bias + dropout +
// residual + LayerNorm/RMSNorm + g all-gather, one pass over HBM.
//
// "第 7 课：序列并行 SP" §3.A: the reduce-scatter that ends the TP region sums
// the t row-linear partials and leaves each rank its s/t tokens; the
// token-wise ops of the SP region then need nothing from other tokens, so a
// block can own a whole token row: it reads the t partials and the residual
// of that token once, and writes Z, the mask, the statistics and the
// normalised row straight into the all-gather destination(s).
//
// Work layout: a persistent grid (16 compute warps per SM); block b of G
// processes tokens b, b + G, b + 2G, ... when every block gets at least 32
// rows (the blocks then stream neighbouring rows together), else a
// contiguous range of about rows/G tokens; either way the walk moves the
// shard and the row inside it by increments (no per-row division or shard
// search).  A row of h channels is cut into chunks of 8*T channels (T =
// compute threads); in each chunk thread i owns channels [8i, 8i+8).
//
// Staging: one extra warp per block is the copy producer.  For every (row,
// chunk) item in order it waits until the compute warps have released the
// item's stage (an mbarrier each warp arrives on once it has read the stage),
// then arms the stage's "full" mbarrier with the item's byte count and issues
// one bulk global -> shared copy per input stream (the t partial rows and the
// residual row of the chunk, cp.async.bulk completing on that mbarrier).  The
// compute warps wait on "full", read their own 16 bytes of every stream, sum
// the partials, release the stage at once and only then run the dropout and
// the rest, so the next chunks are in flight while a chunk is computed.  The
// only block-wide barriers are the row reductions of the norm, on a named
// barrier of the compute warps.  Every wait is bounded (about a second of
// %globaltimer, then SP_ERR_TIMEOUT in the status word and no further waits).
// The chunk loop is not unrolled (the Philox rounds make its body long): Z of
// the row waits for the statistics in the thread's own shared-memory slots
// rather than in registers.
//
// A tuning option (not the default: measured slower on GB300) splits every
// row over a thread-block cluster of two CTAs, each staging and computing
// h / 2 channels; the halves of the row sums meet through distributed shared
// memory (fwd_kernel_pair).
#include "fwd_kernel.cuh"

namespace spb {

template <int NTHR, int TT, int CL = 1>
static const void* fwd_kernel_s(int stages) {
  switch (stages) {
    case 2: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, 2, TT, false, CL>);
    case 3: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, 3, TT, false, CL>);
    default: return nullptr;
  }
}

// Instantiated shapes: 64, 128, 160 or 256 threads per block; pipeline depth
// 2 or 3 chunks; t either a run-time value or the compile-time 8.
const void* fwd_kernel(int threads, int t, int stages) {
  const bool t8 = (t == 8);
  switch (threads) {
    case 64: return t8 ? fwd_kernel_s<64, 8>(stages) : fwd_kernel_s<64, 0>(stages);
    case 128: return t8 ? fwd_kernel_s<128, 8>(stages) : fwd_kernel_s<128, 0>(stages);
    case 160: return t8 ? fwd_kernel_s<160, 8>(stages) : fwd_kernel_s<160, 0>(stages);
    case 256: return t8 ? fwd_kernel_s<256, 8>(stages) : fwd_kernel_s<256, 0>(stages);
    default: return nullptr;
  }
}

// Rows split over clusters of two CTAs (the distributed-shared-memory
// exchange of the row sums): 128 or 256 threads per CTA.
const void* fwd_kernel_pair(int threads, int t, int stages) {
  const bool t8 = (t == 8);
  switch (threads) {
    case 128: return t8 ? fwd_kernel_s<128, 8, 2>(stages) : fwd_kernel_s<128, 0, 2>(stages);
    case 256: return t8 ? fwd_kernel_s<256, 8, 2>(stages) : fwd_kernel_s<256, 0, 2>(stages);
    default: return nullptr;
  }
}

}  // namespace spb
