// Backward of the SP boundary: LayerNorm/RMSNorm + residual + dropout backward
// on each shard, the all-gather of the partials' gradient (the transpose of
// g*), and the parameter gradients.
//
// "第 7 课：序列并行 SP" §3.B: the backward pass is the adjoint of the forward;
// the gradient of a reduce-scatter along s is an all-gather along s.  Every
// rank's row-linear partial entered the sum with weight one, so each receives
// the full-sequence gradient of the pre-dropout sum, dYpre.
//
// Work layout mirrors the forward: a persistent grid, one token row per block
// iteration, chunks of 8*T channels with thread i owning channels
// [8i, 8i+8) of each chunk.  Each thread stages its own pieces of dY, Z, the
// mask (and the optional skip-path gradient) of whole rows with cp.async into
// a ring of RING rows in shared memory, RING - 1 rows ahead; the two passes a
// row needs (the row sums mean(dxh) and mean(dxh * x_hat), then the
// gradients) both read the row from there.  The two sums are reduced
// together: one block barrier per row.  Because a thread owns the same
// channels in every row, it accumulates its channels' parameter-gradient
// terms in registers across all rows of its block and writes one float32
// partial per block and channel at the end; a second kernel sums the
// partials over blocks in a fixed order (eight float32 warp sums, combined in
// float64), so results are bit-reproducible without atomics.
#include "sp_device.cuh"

namespace spb {

// REGEN = true: the mask-free variant; the dropout keep decisions are drawn
// again from Philox4x32-10 at the element's global index (the forward's seed
// and offset) instead of being read from the stored 1-byte mask.
template <int NTHR, int MAXC, int RING, bool REGEN>
__global__ void __launch_bounds__(NTHR, 1) norm_bwd_kernel(const BwdParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int h = static_cast<int>(P.map.h);   // <= SP_MAX_HIDDEN
  constexpr int kChunk = 8 * NTHR;
  const int nchunk = (h + kChunk - 1) / kChunk;
  const bool is_ln = (P.norm == SP_NORM_LAYERNORM);
  const bool has_skip = P.has_skip != 0;
  // one staged chunk ("item") of all threads: [dY | Z | mask | skip (optional)]
  // (no mask slots in the mask-free variant)
  constexpr int v16 = NTHR * 16;
  constexpr int off_mask = 2 * v16;
  constexpr int off_skip = off_mask + (REGEN ? 0 : NTHR * 8);
  const int item_bytes = off_skip + (has_skip ? v16 : 0);
  const int row_bytes = MAXC * item_bytes;
  float2* red = reinterpret_cast<float2*>(smem + RING * row_bytes);   // [2][32]
  const int c0 = tid * 8;
  uint32_t valid = 0;   // bit ch: this thread has channels in chunk ch
#pragma unroll
  for (int ch = 0; ch < MAXC; ++ch)
    if (ch < nchunk && ch * kChunk + c0 < h) valid |= 1u << ch;

  if (blockIdx.x == 0 && tid < 32) check_cu_seqlens(P.cu_seqlens, P.n_seqs, P.rows, P.status);

  const int64_t G = gridDim.x;
  const int64_t nrows = (P.rows > blockIdx.x) ? (P.rows - 1 - blockIdx.x) / G + 1 : 0;

  // gamma of this thread's channels, kept for every row
  uint4 gam[MAXC];
#pragma unroll
  for (int ch = 0; ch < MAXC; ++ch)
    gam[ch] = ((valid >> ch) & 1u) ? ldg16(P.gamma + ch * kChunk + c0) : make_uint4(0, 0, 0, 0);

  // Stage the next row (all of its chunks, one cp.async group) into the next
  // ring slot; rows are issued in order, so one cursor walks them.
  RowCursor pf;
  pf.init(P.map, blockIdx.x);
  int64_t pf_ri = 0;
  int pf_slot = 0;
  auto issue_row = [&]() {
    if (pf_ri < nrows) {
      const int k = pf.k;
      const int64_t lo0 = pf.local(P.map) * h + c0;
      const uint16_t* dyp = P.dy[k] + lo0;
      const uint16_t* zp = P.z[k] + lo0;
      const uint8_t* mp = REGEN ? nullptr : P.mask[k] + lo0;
      uint8_t* it0 = smem + pf_slot * row_bytes + tid * 16;
#pragma unroll
      for (int ch = 0; ch < MAXC; ++ch) {
        if ((valid >> ch) & 1u) {
          uint8_t* it = it0 + ch * item_bytes;
          cp_async16(it, dyp + ch * kChunk);
          cp_async16(it + v16, zp + ch * kChunk);
          if (!REGEN) cp_async8(it + off_mask - tid * 8, mp + ch * kChunk);   // 8 B apart
          if (has_skip) cp_async16(it + off_skip, P.dz_skip[k] + lo0 + ch * kChunk);
        }
      }
      if (++pf_ri < nrows) pf.advance(P.map, G);
    }
    cp_async_commit();
    pf_slot = (pf_slot + 1 == RING) ? 0 : pf_slot + 1;
  };

#pragma unroll
  for (int i = 0; i < RING - 1; ++i) issue_row();

  float acc_g[MAXC][8], acc_b[MAXC][8], acc_bias[MAXC][8];
#pragma unroll
  for (int ch = 0; ch < MAXC; ++ch)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc_g[ch][e] = acc_b[ch][e] = acc_bias[ch][e] = 0.f;

  // statistics of the current row, loaded one row ahead
  RowCursor cur, nxt;
  cur.init(P.map, blockIdx.x);
  nxt = cur;
  float cur_mean = 0.f, cur_rstd = 0.f;
  if (nrows > 0) {
    const int64_t l0 = cur.local(P.map);
    cur_rstd = P.rstd[cur.k][l0];
    if (is_ln) cur_mean = P.mean[cur.k][l0];
  }

  int slot_sel = 0;
  int slot = 0;   // ring slot of the current row
  const float fh = static_cast<float>(h);
  for (int64_t ri = 0; ri < nrows; ++ri) {
    if (ri > 0) cur = nxt;
    const int64_t row = cur.row;
    const int k = cur.k;
    const int64_t local = cur.local(P.map);
    float nx_mean = 0.f, nx_rstd = 0.f;
    if (ri + 1 < nrows) {
      nxt.advance(P.map, G);
      const int64_t l1 = nxt.local(P.map);
      nx_rstd = P.rstd[nxt.k][l1];
      if (is_ln) nx_mean = P.mean[nxt.k][l1];
    }
    const float mean = cur_mean, rstd = cur_rstd;

    issue_row();                    // row ri + RING - 1 refills the slot row ri - 1 used
    cp_async_wait<RING - 1>();      // row ri has landed
    const uint8_t* it0 = smem + slot * row_bytes + tid * 16;
    slot = (slot + 1 == RING) ? 0 : slot + 1;

    // ---- pass 1: the two row sums, and dgamma / dbeta terms --------------
    // x_hat = (z - mean) * rstd (LN) or z * rstd (RMS); dxh = dY * gamma is an
    // exact product of two bf16 values
    const float nmean = is_ln ? -mean : 0.f;
    float s1a = 0.f, s1b = 0.f, s2a = 0.f, s2b = 0.f;
#pragma unroll
    for (int ch = 0; ch < MAXC; ++ch) {
      if ((valid >> ch) & 1u) {
        const uint8_t* it = it0 + ch * item_bytes;
        const uint4 dyv = lds16(it);
        const uint4 zv = lds16(it + v16);
        float xh[8], dxh[8], dy[8];
        add8_bf16_bcast(zv, nmean, xh);             // z - mean
        fma8_bf16_bcast(dyv, gam[ch], 0.f, dxh);    // dY * gamma
        if (is_ln) add8_bf16(dyv, acc_b[ch]);       // dbeta terms
        unpack8(dyv, dy);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          mul2(xh[e], xh[e + 1], rstd, rstd);
          add2(s1a, s1b, dxh[e], dxh[e + 1]);
          fma2(s2a, s2b, dxh[e], dxh[e + 1], xh[e], xh[e + 1]);
          fma2(acc_g[ch][e], acc_g[ch][e + 1], dy[e], dy[e + 1], xh[e], xh[e + 1]);
        }
      }
    }

    const float2 s = block_sum2(s1a + s1b, s2a + s2b, red + 32 * slot_sel);
    slot_sel ^= 1;
    const float nm1 = is_ln ? -(s.x / fh) : 0.f;
    const float nm2r = -(s.y / fh) * rstd;

    // ---- pass 2: dZ, dResidual, dYpre (gathered), dbias terms ------------
    // dZ = rstd * (dxh - m1 - (z - mean) * rstd * m2)
    uint16_t* dres_row = P.dresidual[k] + local * h + c0;
    const int64_t grow = row * h + c0;
    uint16_t* dg0_row = P.n_gather > 0 ? P.dgathered[0] + grow : nullptr;
#pragma unroll
    for (int ch = 0; ch < MAXC; ++ch) {
      if ((valid >> ch) & 1u) {
        const uint8_t* it = it0 + ch * item_bytes;
        const uint4 dyv = lds16(it);
        const uint4 zv = lds16(it + v16);
        uint2 mk;
        if (REGEN) {
          const uint64_t q = static_cast<uint64_t>(grow + ch * kChunk) >> 2;
          const uint4 a = philox4x32_10(make_uint4(static_cast<uint32_t>(q),
                                                   static_cast<uint32_t>(q >> 32), P.off0, P.off1),
                                        P.key0, P.key1);
          const uint4 b = philox4x32_10(make_uint4(static_cast<uint32_t>(q + 1),
                                                   static_cast<uint32_t>((q + 1) >> 32), P.off0,
                                                   P.off1),
                                        P.key0, P.key1);
          mk = make_uint2(keep_bytes4(a, P.thr), keep_bytes4(b, P.thr));
        } else {
          mk = lds8(it + off_mask - tid * 8);
        }
        float zc[8], dz[8], dp[8];
        add8_bf16_bcast(zv, nmean, zc);           // z - mean
        fma8_bf16_bcast(dyv, gam[ch], nm1, dz);  // dxh - m1
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          fma2(dz[e], dz[e + 1], zc[e], zc[e + 1], nm2r, nm2r);
          mul2(dz[e], dz[e + 1], rstd, rstd);
        }
        if (has_skip) add8_bf16(lds16(it + off_skip), dz);
#pragma unroll
        for (int e = 0; e < 8; e += 2) mul2_to(dz[e], dz[e + 1], P.scale, dp[e], dp[e + 1]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          // mask bytes are 0 or 1: bit 0 of byte e decides
          const bool kept = ((e < 4 ? mk.x : mk.y) & (1u << (8 * (e & 3)))) != 0u;
          dp[e] = kept ? dp[e] : 0.f;
        }
#pragma unroll
        for (int e = 0; e < 8; e += 2) add2(acc_bias[ch][e], acc_bias[ch][e + 1], dp[e], dp[e + 1]);
        st16_stream(dres_row + ch * kChunk, pack8(dz));
        const uint4 pb = pack8(dp);
        if (dg0_row != nullptr) st16_stream(dg0_row + ch * kChunk, pb);
        for (int j = 1; j < P.n_gather; ++j) st16_stream(P.dgathered[j] + grow + ch * kChunk, pb);
      }
    }
    cur_mean = nx_mean;
    cur_rstd = nx_rstd;
  }
  cp_async_wait<0>();

  // per-block partials: ws[block][0|1|2][c] = dgamma | dbeta | dbias terms
  float* wsb = P.ws + static_cast<int64_t>(blockIdx.x) * 3 * h;
#pragma unroll
  for (int ch = 0; ch < MAXC; ++ch) {
    const int c = ch * kChunk + c0;
    if ((valid >> ch) & 1u) {
      float4* dg = reinterpret_cast<float4*>(wsb + c);
      float4* db = reinterpret_cast<float4*>(wsb + h + c);
      float4* dc = reinterpret_cast<float4*>(wsb + 2 * h + c);
      dg[0] = make_float4(acc_g[ch][0], acc_g[ch][1], acc_g[ch][2], acc_g[ch][3]);
      dg[1] = make_float4(acc_g[ch][4], acc_g[ch][5], acc_g[ch][6], acc_g[ch][7]);
      db[0] = make_float4(acc_b[ch][0], acc_b[ch][1], acc_b[ch][2], acc_b[ch][3]);
      db[1] = make_float4(acc_b[ch][4], acc_b[ch][5], acc_b[ch][6], acc_b[ch][7]);
      dc[0] = make_float4(acc_bias[ch][0], acc_bias[ch][1], acc_bias[ch][2], acc_bias[ch][3]);
      dc[1] = make_float4(acc_bias[ch][4], acc_bias[ch][5], acc_bias[ch][6], acc_bias[ch][7]);
    }
  }
}

// out[q][c] = sum over blocks b of ws[b][q][c], in a fixed order.  A block
// owns 32 consecutive columns of one quantity q; warp w sums the partials
// b = w, w + 8, w + 16, ... of its lane's column (float32, in that order;
// each warp row is one coalesced 128-byte read) and the 8 warp sums are then
// added in warp order in float64.  Same inputs, same bits.
constexpr int kReduceWarps = 8;

__global__ void __launch_bounds__(32 * kReduceWarps) param_reduce_kernel(const ParamReduceParams P) {
  __shared__ float part[kReduceWarps][32];
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
    // four independent loads in flight per step
    for (; b + 3 * kReduceWarps < P.nblk; b += 4 * kReduceWarps) {
      const float v0 = src[b * stride];
      const float v1 = src[(b + kReduceWarps) * stride];
      const float v2 = src[(b + 2 * kReduceWarps) * stride];
      const float v3 = src[(b + 3 * kReduceWarps) * stride];
      acc += v0;
      acc += v1;
      acc += v2;
      acc += v3;
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

template <int NTHR, int MAXC, bool REGEN>
static const void* bwd_kernel_s(int ring) {
  switch (ring) {
    case 2: return reinterpret_cast<const void*>(norm_bwd_kernel<NTHR, MAXC, 2, REGEN>);
    case 3: return reinterpret_cast<const void*>(norm_bwd_kernel<NTHR, MAXC, 3, REGEN>);
    case 4: return reinterpret_cast<const void*>(norm_bwd_kernel<NTHR, MAXC, 4, REGEN>);
    default: return nullptr;
  }
}

template <bool REGEN>
static const void* bwd_kernel_any(int threads, int maxc, int ring) {
  if (threads == 64) return maxc == 1 ? bwd_kernel_s<64, 1, REGEN>(ring) : nullptr;
  if (threads == 256) return maxc == 1 ? bwd_kernel_s<256, 1, REGEN>(ring) : nullptr;
  if (threads != 512) return nullptr;
  switch (maxc) {
    case 1: return bwd_kernel_s<512, 1, REGEN>(ring);
    case 2: return bwd_kernel_s<512, 2, REGEN>(ring);
    case 4: return bwd_kernel_s<512, 4, REGEN>(ring);
    default: return nullptr;
  }
}

// Instantiated shapes (threads, chunks per row): (64, 1) for h <= 512,
// (256, 1) for h <= 2048, (512, 1 | 2 | 4) above; ring of 2, 3 or 4 rows.
const void* bwd_kernel(int threads, int maxc, int ring) {
  return bwd_kernel_any<false>(threads, maxc, ring);
}

const void* bwd_regen_kernel(int threads, int maxc, int ring) {
  return bwd_kernel_any<true>(threads, maxc, ring);
}

cudaError_t launch_param_reduce(const ParamReduceParams& p, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>((p.h + 31) / 32), 3);
  param_reduce_kernel<<<grid, 32 * kReduceWarps, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace spb
