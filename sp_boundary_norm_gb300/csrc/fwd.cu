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
// Work layout: a persistent grid (16 warps per SM); block b of G processes
// tokens b, b + G, b + 2G, ... when every block gets at least 32 rows (the
// blocks then stream neighbouring rows together: 0.7 % faster on the 70B
// shape), else a contiguous range of about rows/G tokens; either way the walk
// moves the shard and the row inside it by increments (no per-row division or
// shard search).  A row of h channels is cut into chunks of 8*T
// channels (T = threads); in each chunk thread i owns channels [8i, 8i+8).
// Every thread streams its own 16-byte pieces of the t + 1 input rows into
// its own shared-memory slots with cp.async, STAGES - 1 chunks ahead, so the
// loads of the next chunks are in flight while the current one is summed,
// dropped out, normalised and stored.  A thread only reads back what it
// copied itself, so the pipeline needs no block barrier; the only barriers
// are the row reductions of the norm.  The chunk loop is not unrolled (the
// Philox rounds make its body long): Z of the row waits for the statistics
// in the thread's own shared-memory slots rather than in registers.
#include "fwd_kernel.cuh"

namespace spb {

template <int NTHR, int TT>
static const void* fwd_kernel_s(int stages) {
  switch (stages) {
    case 2: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, 2, TT, false>);
    case 3: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, 3, TT, false>);
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

}  // namespace spb
