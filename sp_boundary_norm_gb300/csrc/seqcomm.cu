// Unfused sequence-dimension collectives over emulated rank buffers:
// g (all-gather along s) and g* (reduce-scatter along s) on their own, as in
// "第 7 课：序列并行 SP" §3.A, plus a device Philox probe for tests.
//
// On one GPU a "rank" is a buffer, so an all-gather is a strided copy of
// each shard into the full buffer(s) and a reduce-scatter reads shard k's
// rows from all t partials.  Both are pure HBM streams: a persistent grid,
// a contiguous range of token rows per block, 16-byte loads that bypass L1 and
// streaming 16-byte stores, several loads in flight per thread.
#include "sp_device.cuh"

namespace spb {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads) allgather_kernel(const CopyParams P) {
  pdl_wait();
  if (blockIdx.x == 0 && threadIdx.x < 32)
    check_cu_seqlens(P.cu_seqlens, P.n_seqs, P.rows, P.status);
  const int64_t h = P.map.h;
  const int64_t nvec = h / 8;
  int64_t r0, nrows;
  block_rows(P.rows, blockIdx.x, gridDim.x, &r0, &nrows);
  RowWalk cur;
  cur.init(P.map, r0);
  for (int64_t ri = 0; ri < nrows; ++ri) {
    if (ri > 0) cur.next(P.map);
    const int64_t row = cur.row;
    const uint16_t* src = P.src[cur.k] + cur.local * h;
    for (int64_t v0 = threadIdx.x; v0 < nvec; v0 += kCopyThreads * kCopyUnroll) {
      uint4 buf[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t v = v0 + u * kCopyThreads;
        if (v < nvec) buf[u] = ldg16_stream(src + v * 8);
      }
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t v = v0 + u * kCopyThreads;
        if (v < nvec)
          for (int j = 0; j < P.n_dst; ++j) st16_stream(P.dst[j] + row * h + v * 8, buf[u]);
      }
    }
  }
}

// shards[k][local] = bf16(sum over r ascending of partials[r][row]), float32
// (each add widens its bf16 operand exactly: ((P_0 + P_1) + P_2) + ...).  A
// thread issues the loads of all the partials of its 8 channels before it
// adds them (TT = t known at compile time), or groups of four (TT = 0), so
// several loads are in flight per thread.
template <int TT>
__global__ void __launch_bounds__(kCopyThreads) reduce_scatter_kernel(const CopyParams P,
                                                                      int t) {
  pdl_wait();
  if (blockIdx.x == 0 && threadIdx.x < 32)
    check_cu_seqlens(P.cu_seqlens, P.n_seqs, P.rows, P.status);
  const int64_t h = P.map.h;
  const int64_t nvec = h / 8;
  int64_t r0, nrows;
  block_rows(P.rows, blockIdx.x, gridDim.x, &r0, &nrows);
  RowWalk cur;
  cur.init(P.map, r0);
  for (int64_t ri = 0; ri < nrows; ++ri) {
    if (ri > 0) cur.next(P.map);
    const int64_t row = cur.row;
    uint16_t* dst = P.dst[cur.k] + cur.local * h;
    for (int64_t v = threadIdx.x; v < nvec; v += kCopyThreads) {
      const int64_t off = row * h + v * 8;
      float y[8];
      if constexpr (TT > 0) {
        uint4 raw[TT];
#pragma unroll
        for (int r = 0; r < TT; ++r) raw[r] = ldg16_stream(P.src[r] + off);
        unpack8(raw[0], y);
#pragma unroll
        for (int r = 1; r < TT; ++r) add8_bf16(raw[r], y);
      } else {
        unpack8(ldg16_stream(P.src[0] + off), y);
        for (int rb = 1; rb < t; rb += 4) {
          uint4 raw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (rb + i < t) raw[i] = ldg16_stream(P.src[rb + i] + off);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (rb + i < t) add8_bf16(raw[i], y);
        }
      }
      st16_stream(dst + v * 8, pack8(y));
    }
  }
}

__global__ void debug_philox_kernel(const uint32_t* in, uint32_t* out, int64_t n) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t* a = in + 6 * i;
  const uint4 r = philox4x32_10(make_uint4(a[0], a[1], a[2], a[3]), a[4], a[5]);
  out[4 * i + 0] = r.x;
  out[4 * i + 1] = r.y;
  out[4 * i + 2] = r.z;
  out[4 * i + 3] = r.w;
}

static int copy_grid(int64_t rows) {
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  return static_cast<int>(rows < cap ? rows : cap);
}

cudaError_t launch_allgather(const CopyParams& p, cudaStream_t st) {
  void* args[] = {const_cast<CopyParams*>(&p)};
  return launch_pdl(reinterpret_cast<const void*>(&allgather_kernel), dim3(copy_grid(p.rows)),
                    dim3(kCopyThreads), 0, args, st);
}

cudaError_t launch_reduce_scatter(const CopyParams& p, int t, cudaStream_t st) {
  void* args[] = {const_cast<CopyParams*>(&p), &t};
  const void* fn = t == 8 ? reinterpret_cast<const void*>(&reduce_scatter_kernel<8>)
                          : reinterpret_cast<const void*>(&reduce_scatter_kernel<0>);
  return launch_pdl(fn, dim3(copy_grid(p.rows)), dim3(kCopyThreads), 0, args, st);
}

cudaError_t launch_debug_philox(const uint32_t* in, uint32_t* out, int64_t n, cudaStream_t st) {
  const int64_t blocks = (n + 255) / 256;
  debug_philox_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(in, out, n);
  return cudaGetLastError();
}

}  // namespace spb
