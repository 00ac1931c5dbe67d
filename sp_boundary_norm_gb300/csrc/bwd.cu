// Backward of the SP boundary: LayerNorm/RMSNorm + residual + dropout backward
// on each shard, the all-gather of the partials' gradient (the transpose of
// g*), and the parameter gradients.
//
// "第 7 课：序列并行 SP" §3.B: the backward pass is the adjoint of the forward;
// the gradient of a reduce-scatter along s is an all-gather along s.  Every
// rank's row-linear partial entered the sum with weight one, so each receives
// the full-sequence gradient of the pre-dropout sum, dYpre.
//
// Work layout mirrors the forward: a persistent grid, a contiguous range of
// token rows per block, chunks of 8*T channels with thread i owning channels
// [8i, 8i+8) of each chunk.  Each thread stages its own pieces of dY, Z, the
// mask (and the optional skip-path gradient) of whole rows with cp.async into
// a ring of RING rows in shared memory, RING - 1 rows ahead (a bit-packed
// mask is staged by 8 lanes per warp for the whole warp); the row's
// statistics are loaded when it is staged and wait in registers.  The two
// passes a row needs (the row sums mean(dxh) and mean(dxh * x_hat), then the
// gradients) both read the row from there.  The two sums are reduced
// together: one block barrier per row.  Because a thread owns the same
// channels in every row, it accumulates its channels' parameter-gradient
// terms in registers across all rows of its block and writes one float32
// partial per block and channel at the end; a second kernel sums the
// partials over blocks in a fixed order (eight float32 warp sums, combined in
// float64), so results are bit-reproducible without atomics.
#include "bwd_dispatch.cuh"

namespace spb {

// out[q][c] = sum over blocks b of ws[b][q][c], in a fixed order.  A block
// owns 32 consecutive columns of one quantity q; warp w sums the partials
// b = w, w + 8, w + 16, ... of its lane's column (float32, in that order;
// each warp row is one coalesced 128-byte read) and the 8 warp sums are then
// added in warp order in float64.  Same inputs, same bits.
constexpr int kReduceWarps = 8;

__global__ void __launch_bounds__(32 * kReduceWarps) param_reduce_kernel(const ParamReduceParams P) {
  __shared__ float part[kReduceWarps][32];
  pdl_wait();
  const int q = blockIdx.y;
  float* out = P.out[q];
  if (out == nullptr) return;   // uniform per block
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  const int64_t stride = 3 * P.h;
  float acc = 0.f;
  if (c < P.h) {
    const float* src = P.ws + q * P.h + c;
    int b = warp;
    // eight, then four independent loads in flight per step; the adds keep
    // the order b = w, w + 8, w + 16, ...
    for (; b + 7 * kReduceWarps < P.nblk; b += 8 * kReduceWarps) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = src[(b + j * kReduceWarps) * stride];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc += v[j];
    }
    if (b + 3 * kReduceWarps < P.nblk) {
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = src[(b + j * kReduceWarps) * stride];
#pragma unroll
      for (int j = 0; j < 4; ++j) acc += v[j];
      b += 4 * kReduceWarps;
    }
    for (; b < P.nblk; b += kReduceWarps) acc += src[b * stride];
  }
  part[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && c < P.h) {
    double sum = 0.0;
#pragma unroll
    for (int w = 0; w < kReduceWarps; ++w) sum += static_cast<double>(part[w][lane]);
    out[c] = static_cast<float>(sum);
  }
}

const void* bwd_kernel(int threads, int maxc, int ring) {
  return bwd_kernel_any<false>(threads, maxc, ring);
}

cudaError_t launch_param_reduce(const ParamReduceParams& p, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>((p.h + 31) / 32), 3);
  void* args[] = {const_cast<ParamReduceParams*>(&p)};
  return launch_pdl(reinterpret_cast<const void*>(&param_reduce_kernel), grid,
                    dim3(32 * kReduceWarps), 0, args, st);
}

}  // namespace spb
