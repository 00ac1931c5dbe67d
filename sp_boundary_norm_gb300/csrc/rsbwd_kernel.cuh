// Backward of the SP boundary entered through g (the kernel template;
// instantiated in rsbwd.cu with the byte mask and in rsbwd_bits.cu with the
// bit mask): the reduce-scatter of the t
// ranks' partial gradients of the gathered input (the transpose of the
// all-gather, "第 7 课：序列并行 SP" §3.B) fused into the prologue of the norm /
// dropout backward -- the mirror of the fused forward.
//
// Each rank's column-parallel linear leaves a partial gradient of the full
// (b, s, h) gathered input; rank k's dY on its tokens is their float32 sum in
// rank order, used unrounded.  Per token row a block needs the t partial rows
// (t times the bytes of one row) in the first pass only, while the second pass
// needs Z, the mask and dY again.  So there are two staging areas in shared
// memory, both filled per thread with cp.async (each thread reads back only
// what it copied, except the bit-packed mask's bytes, see BITS below):
//   - a ring of STAGES chunk stages for the t partial pieces (streamed through
//     the first pass);
//   - two row buffers (the current row, the next) for Z, the mask and the
//     optional skip gradient, copied together with the row's first chunk.
// The reduced dY waits in the thread's own float32 slots for the second pass.
// Parameter gradients: per-thread registers over the block's rows, one fp32
// partial per block, summed by param_reduce_kernel (as in norm_bwd_kernel).
// BITS = true: the mask is stored one bit per element (h % 32 == 0); lanes 0-7
// of each warp copy the warp's 32 mask bytes of each chunk into the row
// buffer in 4-byte pieces, every lane reads its own byte after the row's
// block barrier, and a warp passes a __syncwarp before a row buffer is
// refilled (as in norm_bwd_kernel).
#pragma once

#include "sp_device.cuh"

namespace spb {

template <int NTHR, int MAXC, int STAGES, int TT, bool BITS = false>
__global__ void __launch_bounds__(NTHR, 1) rs_norm_bwd_kernel(const BwdParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int t = TT > 0 ? TT : P.map.t;
  const int h = static_cast<int>(P.map.h);
  constexpr int kChunk = 8 * NTHR;
  const int nchunk = (h + kChunk - 1) / kChunk;
  const bool is_ln = (P.norm == SP_NORM_LAYERNORM);
  const bool has_skip = P.has_skip != 0;
  constexpr int v16 = NTHR * 16;
  // shared-memory map
  const int stage_bytes = t * v16;                       // [t][NTHR][16 B]
  const int rb_item = rsbwd_rb_item_bytes(NTHR, has_skip, BITS);   // [Z | mask | skip]
  constexpr int rb_skip = rsbwd_rb_skip_offset(NTHR, BITS);
  uint8_t* stages = smem;
  uint8_t* rowbuf = smem + STAGES * stage_bytes;         // [2][MAXC] items
  uint8_t* dybuf = rowbuf + 2 * MAXC * rb_item;          // [MAXC][2][NTHR][16 B]
  float2* red = reinterpret_cast<float2*>(dybuf + MAXC * 2 * v16);   // [2][32]
  const int c0 = tid * 8;
  uint32_t valid = 0;
#pragma unroll
  for (int ch = 0; ch < MAXC; ++ch)
    if (ch < nchunk && ch * kChunk + c0 < h) valid |= 1u << ch;

  pdl_wait();
  if (blockIdx.x == 0 && tid < 32) check_cu_seqlens(P.cu_seqlens, P.n_seqs, P.rows, P.status);

  // this block's rows: a contiguous range
  int64_t r0, nrows;
  block_rows(P.rows, blockIdx.x, gridDim.x, &r0, &nrows);

  uint4 gam[MAXC];
#pragma unroll
  for (int ch = 0; ch < MAXC; ++ch)
    gam[ch] = ((valid >> ch) & 1u) ? ldg16(P.gamma + ch * kChunk + c0) : make_uint4(0, 0, 0, 0);

  // ---- prefetch cursor over (row, chunk) items ---------------------------
  // P.dy[r] holds rank r's full (b, s, h) partial gradient here.
  RowWalk pf;
  pf.init(P.map, r0);
  int64_t pf_ri = 0;
  int pf_chunk = 0, pf_stage = 0, pf_buf = 0;
  auto issue_next = [&]() {
    if (pf_ri < nrows) {
      const int64_t goff = pf.row * h + c0 + pf_chunk * kChunk;
      if (pf_chunk * kChunk + c0 < h) {
        uint8_t* slot = stages + pf_stage * stage_bytes + tid * 16;
#pragma unroll
        for (int r = 0; r < (TT > 0 ? TT : SP_MAX_RANKS); ++r)
          if (TT > 0 || r < t) cp_async16(slot + r * v16, P.dy[r] + goff);
      }
      if (pf_chunk == 0) {
        // the row's Z, mask (and skip gradient), all chunks, ride with chunk 0
        const int k = pf.k;
        const int64_t lo0 = pf.local * h + c0;
        uint8_t* rb = rowbuf + pf_buf * MAXC * rb_item + tid * 16;
#pragma unroll
        for (int ch = 0; ch < MAXC; ++ch) {
          if ((valid >> ch) & 1u) {
            uint8_t* it = rb + ch * rb_item;
            cp_async16(it, P.z[k] + lo0 + ch * kChunk);
            if (!BITS) cp_async8(it + v16 - tid * 8, P.mask[k] + lo0 + ch * kChunk);   // 8 B apart
            if (has_skip) cp_async16(it + rb_skip, P.dz_skip[k] + lo0 + ch * kChunk);
          }
          if (BITS && (tid & 31) < 8) {
            // bytes [4 l, 4 l + 4) of this warp's 32 (lane l), wholly inside
            // the row or wholly past its end (h % 32 == 0)
            const int byte0 = ch * NTHR + (tid & ~31) + 4 * (tid & 31);
            if (byte0 < h / 8)
              cp_async4(rb - tid * 16 + ch * rb_item + v16 + (byte0 - ch * NTHR),
                        P.mask[k] + (pf.local * h) / 8 + byte0);
          }
        }
        pf_buf ^= 1;
      }
      if (++pf_chunk == nchunk) {
        pf_chunk = 0;
        if (++pf_ri < nrows) pf.next(P.map);
      }
    }
    cp_async_commit();
    pf_stage = (pf_stage + 1 == STAGES) ? 0 : pf_stage + 1;
  };

#pragma unroll
  for (int i = 0; i < STAGES - 1; ++i) issue_next();

  float acc_g[MAXC][8], acc_b[MAXC][8], acc_bias[MAXC][8];
#pragma unroll
  for (int ch = 0; ch < MAXC; ++ch)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc_g[ch][e] = acc_b[ch][e] = acc_bias[ch][e] = 0.f;

  RowWalk cur, nxt;
  cur.init(P.map, r0);
  nxt = cur;
  float cur_mean = 0.f, cur_rstd = 0.f;
  if (nrows > 0) {
    const int64_t l0 = cur.local;
    cur_rstd = P.rstd[cur.k][l0];
    if (is_ln) cur_mean = P.mean[cur.k][l0];
  }

  int stage = 0, buf = 0, slot_sel = 0;
  const float inv_h = 1.f / static_cast<float>(h);
  for (int64_t ri = 0; ri < nrows; ++ri) {
    if constexpr (BITS) __syncwarp();   // the lanes have read the bytes a refill replaces
    if (ri > 0) cur = nxt;
    const int64_t row = cur.row;
    const int k = cur.k;
    const int64_t local = cur.local;
    float nx_mean = 0.f, nx_rstd = 0.f;
    if (ri + 1 < nrows) {
      nxt.next(P.map);
      const int64_t l1 = nxt.local;
      nx_rstd = P.rstd[nxt.k][l1];
      if (is_ln) nx_mean = P.mean[nxt.k][l1];
    }
    const float mean = cur_mean, rstd = cur_rstd;
    const float nmean = is_ln ? -mean : 0.f;
    const uint8_t* rb = rowbuf + buf * MAXC * rb_item + tid * 16;
    buf ^= 1;

    // ---- pass 1: reduce the t partials into dY, the row sums, dgamma/dbeta
    float s1a = 0.f, s1b = 0.f, s2a = 0.f, s2b = 0.f;
#pragma unroll
    for (int ch = 0; ch < MAXC; ++ch) {
      if (ch < nchunk) {
        issue_next();
        cp_async_wait<STAGES - 1>();
        if ((valid >> ch) & 1u) {
          const uint8_t* slot = stages + stage * stage_bytes + tid * 16;
          float dy[8];
          unpack8(lds16(slot), dy);
#pragma unroll
          for (int r = 1; r < (TT > 0 ? TT : SP_MAX_RANKS); ++r)
            if (TT > 0 || r < t) add8_bf16(lds16(slot + r * v16), dy);
          float4* dys = reinterpret_cast<float4*>(dybuf + (ch * 2) * v16 + tid * 16);
          dys[0] = make_float4(dy[0], dy[1], dy[2], dy[3]);
          *reinterpret_cast<float4*>(dybuf + (ch * 2 + 1) * v16 + tid * 16) =
              make_float4(dy[4], dy[5], dy[6], dy[7]);
          const uint4 zv = lds16(rb + ch * rb_item);
          float xh[8], g[8];
          add8_bf16_bcast(zv, nmean, xh);   // z - mean
          unpack8(gam[ch], g);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            float dxh0, dxh1;
            mul2_pair(dy[e], dy[e + 1], g[e], g[e + 1], dxh0, dxh1);   // dY * gamma
            mul2(xh[e], xh[e + 1], rstd, rstd);              // x_hat
            add2(s1a, s1b, dxh0, dxh1);
            fma2(s2a, s2b, dxh0, dxh1, xh[e], xh[e + 1]);
            fma2(acc_g[ch][e], acc_g[ch][e + 1], dy[e], dy[e + 1], xh[e], xh[e + 1]);
            if (is_ln) add2(acc_b[ch][e], acc_b[ch][e + 1], dy[e], dy[e + 1]);
          }
        }
        stage = (stage + 1 == STAGES) ? 0 : stage + 1;
      }
    }

    const float2 s = block_sum2(s1a + s1b, s2a + s2b, red + 32 * slot_sel);
    slot_sel ^= 1;
    const float nm1 = is_ln ? -(s.x * inv_h) : 0.f;
    const float nm2r = -(s.y * inv_h) * rstd;

    // ---- pass 2: dZ, dResidual, dYpre (gathered), dbias terms ------------
    uint16_t* dres_row = P.dresidual[k] + local * h + c0;
    const int64_t grow = row * h + c0;
    uint16_t* dg0_row = P.n_gather > 0 ? P.dgathered[0] + grow : nullptr;
#pragma unroll
    for (int ch = 0; ch < MAXC; ++ch) {
      if ((valid >> ch) & 1u) {
        const uint8_t* it = rb + ch * rb_item;
        const uint4 zv = lds16(it);
        uint2 mk;   // the 8 keep flags: bytes (bit 0 of byte e) or, for BITS, nibbles
        if (BITS) {
          const uint32_t mbyte = it[v16 - tid * 15];   // own byte of the staged bits
          mk = make_uint2(mbyte, mbyte >> 4);   // element e's flag: bit (e & 3) of word e >> 2
        } else {
          mk = lds8(it + v16 - tid * 8);
        }
        const float4 d0 = *reinterpret_cast<const float4*>(dybuf + (ch * 2) * v16 + tid * 16);
        const float4 d1 =
            *reinterpret_cast<const float4*>(dybuf + (ch * 2 + 1) * v16 + tid * 16);
        const float dy[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
        float zc[8], g[8], dz[8], dp[8];
        add8_bf16_bcast(zv, nmean, zc);   // z - mean
        unpack8(gam[ch], g);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          dz[e] = nm1;
          dz[e + 1] = nm1;
          fma2(dz[e], dz[e + 1], dy[e], dy[e + 1], g[e], g[e + 1]);      // dxh - m1
          fma2(dz[e], dz[e + 1], zc[e], zc[e + 1], nm2r, nm2r);
          mul2(dz[e], dz[e + 1], rstd, rstd);
        }
        if (has_skip) add8_bf16(lds16(it + rb_skip), dz);   // skip slot
#pragma unroll
        for (int e = 0; e < 8; e += 2) mul2_to(dz[e], dz[e + 1], P.scale, dp[e], dp[e + 1]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t bit = BITS ? (1u << (e & 3)) : (1u << (8 * (e & 3)));
          const bool kept = ((e < 4 ? mk.x : mk.y) & bit) != 0u;
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

// Instantiated shapes (threads, chunks per row): (64, 1) for h <= 512,
// (256, 1) for h <= 2048, (512, 1 | 2) for h <= 8192; t run-time or 8;
// 1 to 3 chunk stages.
template <int NTHR, int MAXC, int TT, bool BITS>
static const void* rsbwd_s(int stages) {
  switch (stages) {
    case 1: return reinterpret_cast<const void*>(rs_norm_bwd_kernel<NTHR, MAXC, 1, TT, BITS>);
    case 2: return reinterpret_cast<const void*>(rs_norm_bwd_kernel<NTHR, MAXC, 2, TT, BITS>);
    case 3: return reinterpret_cast<const void*>(rs_norm_bwd_kernel<NTHR, MAXC, 3, TT, BITS>);
    default: return nullptr;
  }
}

template <bool BITS>
static const void* rs_bwd_any(int threads, int maxc, int t, int stages) {
  const bool t8 = (t == 8);
  if (threads == 64 && maxc == 1)
    return t8 ? rsbwd_s<64, 1, 8, BITS>(stages) : rsbwd_s<64, 1, 0, BITS>(stages);
  if (threads == 256 && maxc == 1)
    return t8 ? rsbwd_s<256, 1, 8, BITS>(stages) : rsbwd_s<256, 1, 0, BITS>(stages);
  if (threads == 512 && maxc == 1)
    return t8 ? rsbwd_s<512, 1, 8, BITS>(stages) : rsbwd_s<512, 1, 0, BITS>(stages);
  if (threads == 512 && maxc == 2)
    return t8 ? rsbwd_s<512, 2, 8, BITS>(stages) : rsbwd_s<512, 2, 0, BITS>(stages);
  return nullptr;
}

}  // namespace spb
