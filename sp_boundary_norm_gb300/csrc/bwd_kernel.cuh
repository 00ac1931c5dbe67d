// Norm / dropout backward kernel template (see bwd.cu for the design);
// instantiated in bwd.cu (stored mask) and bwd_regen.cu (mask drawn again).
#pragma once

#include "sp_device.cuh"

namespace spb {

// REGEN = true: the mask-free variant; the dropout keep decisions are drawn
// again from Philox4x32-10 at the element's global index (the forward's seed
// and offset) instead of being read from the stored 1-byte mask.
// Shapes with bwd_tmem_shape(NTHR, MAXC) keep each thread's dgamma / dbeta /
// dbias terms in tensor memory (its lane, 24 columns per chunk), which frees
// the registers for wider rows per thread at 16 warps per SM; the others keep
// them in registers.
// BULK = true (used when dYpre goes to several gathered copies): each thread
// writes its dYpre values once, into a shared-memory copy of the row (two
// such rows, alternating), and thread 0 sends the whole row to every
// gathered copy with bulk copies (one per copy, h * 2 bytes each) right
// after the next row's block barrier, so the threads issue one shared store
// instead of n_gather global stores per 8 elements and no barrier is added.
// A row buffer is rewritten two rows later, after thread 0 has seen its
// copies finish reading it (before that row's barrier).
// BITS = true: the mask is stored one bit per element (byte j of a row holds
// channels [8j, 8j + 8), bit e channel 8j + e; h % 32 == 0); a thread needs
// one byte per chunk.  The bytes are staged with the row: lanes 0-7 of each
// warp copy the warp's 32 bytes of each chunk in 4-byte pieces, and every
// lane reads its byte after the row's block barrier (which follows the
// copying lanes' waits); a warp passes a __syncwarp before it refills a ring
// slot, so no lane still reads the bytes being replaced.
template <int NTHR, int MAXC, int RING, bool REGEN, bool BULK = false, bool BITS = false>
__global__ void __launch_bounds__(NTHR, bwd_tmem_shape(NTHR, MAXC)
                                            ? 512 / bwd_tmem_cols(NTHR, MAXC)
                                            : (NTHR <= 256 ? 512 / NTHR : 1))
    norm_bwd_kernel(const BwdParams P) {
  constexpr bool TACC = bwd_tmem_shape(NTHR, MAXC);
  constexpr uint32_t kCols = bwd_tmem_cols(NTHR, MAXC);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x;
  pdl_wait();   // before tensor memory is taken, too
  // tensor memory: allocated by warp 0 before anything can diverge
  uint32_t tacc = 0;   // this thread's lane, first of its columns
  if constexpr (TACC) {
    if (tid < 32) tmem_alloc(&tmem_base, kCols);
    tmem_sync_block();
    const int w = tid >> 5;
    tacc = tmem_base + (static_cast<uint32_t>(32 * (w & 3)) << 16) +
           static_cast<uint32_t>((w >> 2) * 24 * MAXC);
    const float zero[16] = {};
#pragma unroll
    for (int ch = 0; ch < MAXC; ++ch) {
      tmem_st16(tacc + 24 * ch, zero);
      tmem_st8(tacc + 24 * ch + 16, zero);
    }
  }
  const int h = static_cast<int>(P.map.h);   // <= SP_MAX_HIDDEN
  constexpr int kChunk = 8 * NTHR;
  const int nchunk = (h + kChunk - 1) / kChunk;
  const bool is_ln = (P.norm == SP_NORM_LAYERNORM);
  const bool has_skip = P.has_skip != 0;
  // one staged chunk ("item") of all threads: [dY | Z | mask | skip (optional)]
  // (no mask slots in the mask-free variant)
  constexpr int v16 = NTHR * 16;
  constexpr int off_mask = bwd_item_mask_offset(NTHR);
  constexpr int off_skip = bwd_item_skip_offset(NTHR, REGEN, BITS);
  const int item_bytes = bwd_item_bytes(NTHR, has_skip, REGEN, BITS);
  const int row_bytes = MAXC * item_bytes;
  float2* red = reinterpret_cast<float2*>(smem + RING * row_bytes);   // [2][32]
  // BULK: two shared copies of a row's dYpre, h bf16 each (16-byte aligned)
  uint8_t* const stage0 = smem + RING * row_bytes + 2 * 32 * sizeof(float2);
  const int stage_bytes = ((h * 2 + 15) / 16) * 16;
  const int c0 = tid * 8;
  uint32_t valid = 0;   // bit ch: this thread has channels in chunk ch
#pragma unroll
  for (int ch = 0; ch < MAXC; ++ch)
    if (ch < nchunk && ch * kChunk + c0 < h) valid |= 1u << ch;
  // BITS: lane l < 8 of warp w copies bytes [32 w + 4 l, 32 w + 4 l + 4) of
  // each chunk's NTHR mask bytes; bit ch: that piece lies inside the row
  const int bits_lane = (tid & ~31) + 4 * (tid & 31);
  uint32_t bits_copy = 0;
#pragma unroll
  for (int ch = 0; ch < MAXC; ++ch)
    if (BITS && (tid & 31) < 8 && ch * NTHR + bits_lane < h / 8) bits_copy |= 1u << ch;

  if (blockIdx.x == 0 && tid < 32) check_cu_seqlens(P.cu_seqlens, P.n_seqs, P.rows, P.status);

  // this block's rows: a contiguous range
  int64_t r0, nrows;
  block_rows(P.rows, blockIdx.x, gridDim.x, &r0, &nrows);

  // gamma of this thread's channels, kept for every row
  uint4 gam[MAXC];
#pragma unroll
  for (int ch = 0; ch < MAXC; ++ch)
    gam[ch] = ((valid >> ch) & 1u) ? ldg16(P.gamma + ch * kChunk + c0) : make_uint4(0, 0, 0, 0);

  // Stage the next row (all of its chunks, one cp.async group) into the next
  // ring slot and load its statistics; the row's shard, position and
  // statistics travel with it in a register queue of RING - 1 entries.
  struct RowRec {
    int64_t row, local;
    int k;
    float mean, rstd;
  };
  RowWalk pw;
  pw.init(P.map, r0);
  int64_t pf_ri = 0;
  int pf_slot = 0;
  auto issue_row = [&](RowRec& rec) {
    if (pf_ri < nrows) {
      const int k = pw.k;
      const int64_t lo0 = pw.local * h + c0;
      const uint16_t* dyp = P.dy[k] + lo0;
      const uint16_t* zp = P.z[k] + lo0;
      const uint8_t* mp = REGEN || BITS ? nullptr : P.mask[k] + lo0;
      uint8_t* it0 = smem + pf_slot * row_bytes + tid * 16;
#pragma unroll
      for (int ch = 0; ch < MAXC; ++ch) {
        if ((valid >> ch) & 1u) {
          uint8_t* it = it0 + ch * item_bytes;
          cp_async16(it, dyp + ch * kChunk);
          cp_async16(it + v16, zp + ch * kChunk);
          if (!REGEN && !BITS) cp_async8(it + off_mask - tid * 8, mp + ch * kChunk);   // 8 B apart
          if (has_skip) cp_async16(it + off_skip, P.dz_skip[k] + lo0 + ch * kChunk);
        }
        if (BITS && ((bits_copy >> ch) & 1u)) {
          // (h % 32 == 0: a 4-byte piece is wholly inside the row or past it)
          cp_async4(it0 - tid * 16 + ch * item_bytes + off_mask + bits_lane,
                    P.mask[k] + (static_cast<uint64_t>(pw.local) * h >> 3) + ch * NTHR + bits_lane);
        }
      }
      rec.row = pw.row;
      rec.local = pw.local;
      rec.k = k;
      rec.rstd = __ldg(P.rstd[k] + pw.local);
      rec.mean = is_ln ? __ldg(P.mean[k] + pw.local) : 0.f;
      if (++pf_ri < nrows) pw.next(P.map);
    }
    cp_async_commit();
    pf_slot = (pf_slot + 1 == RING) ? 0 : pf_slot + 1;
  };

  constexpr int kQ = RING > 1 ? RING - 1 : 1;
  RowRec q[kQ];
#pragma unroll
  for (int i = 0; i < RING - 1; ++i) issue_row(q[i]);

  float acc_g[MAXC][8], acc_b[MAXC][8], acc_bias[MAXC][8];
#pragma unroll
  for (int ch = 0; ch < MAXC; ++ch)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc_g[ch][e] = acc_b[ch][e] = acc_bias[ch][e] = 0.f;

  int slot_sel = 0;
  int slot = 0;   // ring slot of the current row
  int64_t prev_grow = 0;   // BULK: first element of the previous row in the gathered buffers
  const float inv_h = 1.f / static_cast<float>(h);
  for (int64_t ri = 0; ri < nrows; ++ri) {
    // row ri + RING - 1 refills the slot row ri - 1 used
    if constexpr (BITS) __syncwarp();   // the lanes have read the bytes it replaces
    RowRec cur;
    if (RING > 1) {
      cur = q[0];
#pragma unroll
      for (int i = 0; i + 1 < kQ; ++i) q[i] = q[i + 1];
      issue_row(q[kQ - 1]);
    } else {
      issue_row(cur);
    }
    cp_async_wait<RING - 1>();      // row ri has landed
    const int64_t row = cur.row;
    const int k = cur.k;
    const int64_t local = cur.local;
    const float mean = cur.mean, rstd = cur.rstd;
    const uint8_t* it0 = smem + slot * row_bytes + tid * 16;
    slot = (slot + 1 == RING) ? 0 : slot + 1;

    // ---- pass 1: the two row sums, and dgamma / dbeta terms --------------
    // x_hat = (z - mean) * rstd (LN) or z * rstd (RMS); dxh = dY * gamma is an
    // exact product of two bf16 values
    const float nmean = is_ln ? -mean : 0.f;
    float s1a = 0.f, s1b = 0.f, s2a = 0.f, s2b = 0.f;
    if constexpr (TACC) tmem_wait_st();   // the previous row's stores have landed
#pragma unroll
    for (int ch = 0; ch < MAXC; ++ch) {
      float gb[16];   // this chunk's dgamma terms, then its dbeta terms
      if constexpr (TACC) {
        tmem_ld16(tacc + 24 * ch, gb);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) gb[e] = acc_g[ch][e], gb[8 + e] = acc_b[ch][e];
      }
      if ((valid >> ch) & 1u) {
        const uint8_t* it = it0 + ch * item_bytes;
        const uint4 dyv = lds16(it);
        const uint4 zv = lds16(it + v16);
        float xh[8], dxh[8], dy[8];
        add8_bf16_bcast(zv, nmean, xh);             // z - mean
        fma8_bf16_bcast(dyv, gam[ch], 0.f, dxh);    // dY * gamma
        unpack8(dyv, dy);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          mul2(xh[e], xh[e + 1], rstd, rstd);
          add2(s1a, s1b, dxh[e], dxh[e + 1]);
          fma2(s2a, s2b, dxh[e], dxh[e + 1], xh[e], xh[e + 1]);
          fma2(gb[e], gb[e + 1], dy[e], dy[e + 1], xh[e], xh[e + 1]);
          if (is_ln) add2(gb[8 + e], gb[9 + e], dy[e], dy[e + 1]);   // dbeta terms
        }
      }
      if constexpr (TACC) {
        tmem_st16(tacc + 24 * ch, gb);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc_g[ch][e] = gb[e], acc_b[ch][e] = gb[8 + e];
      }
    }

    // BULK: the copies of row ri - 2 must have read their row buffer before
    // this barrier (row ri writes it again after it); row ri - 1, complete
    // in its buffer once every thread has passed the barrier, is sent after it
    if (BULK && tid == 0) bulk_wait_read_all();
    const float2 s = block_sum2(s1a + s1b, s2a + s2b, red + 32 * slot_sel);
    slot_sel ^= 1;
    if (BULK && tid == 0 && ri > 0) {
      const uint8_t* src = stage0 + ((ri - 1) & 1) * stage_bytes;
      for (int j = 0; j < P.n_gather; ++j)
        bulk_s2g(P.dgathered[j] + prev_grow, src, static_cast<uint32_t>(h) * 2u);
      bulk_commit();
    }
    const float nm1 = is_ln ? -(s.x * inv_h) : 0.f;
    const float nm2r = -(s.y * inv_h) * rstd;

    // ---- pass 2: dZ, dResidual, dYpre (gathered), dbias terms ------------
    // dZ = rstd * (dxh - m1 - (z - mean) * rstd * m2)
    uint16_t* dres_row = P.dresidual[k] + local * h + c0;
    const int64_t grow = row * h + c0;
    uint16_t* dg0_row = P.n_gather > 0 ? P.dgathered[0] + grow : nullptr;
    uint8_t* const stage_row = stage0 + (ri & 1) * stage_bytes + tid * 16;
    // REGEN: Philox words [chunk of the group][call].  In the shapes whose
    // parameter-gradient terms live in tensor memory the draws of two chunks
    // are made together (four independent Philox chains in flight instead of
    // two); the register shapes have no registers to spare for it, and each
    // chunk draws its own.
    constexpr int kDrawGroup = (TACC && MAXC >= 2) ? 2 : 1;
    uint4 draws[kDrawGroup][2];
#pragma unroll
    for (int ch = 0; ch < MAXC; ++ch) {
      if (REGEN && kDrawGroup > 1 && ch % kDrawGroup == 0) {
#pragma unroll
        for (int k = 0; k < kDrawGroup; ++k) {
          if (ch + k < MAXC) {
            const uint64_t q = static_cast<uint64_t>(grow + (ch + k) * kChunk) >> 2;
            draws[k][0] = philox4x32_10(make_uint4(static_cast<uint32_t>(q),
                                                   static_cast<uint32_t>(q >> 32), P.off0,
                                                   P.off1),
                                        P.rk);
            draws[k][1] = philox4x32_10(make_uint4(static_cast<uint32_t>(q + 1),
                                                   static_cast<uint32_t>((q + 1) >> 32), P.off0,
                                                   P.off1),
                                        P.rk);
          }
        }
      }
      float bt[8];   // this chunk's dbias terms
      if constexpr (TACC) {
        tmem_ld8(tacc + 24 * ch + 16, bt);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) bt[e] = acc_bias[ch][e];
      }
      if ((valid >> ch) & 1u) {
        const uint8_t* it = it0 + ch * item_bytes;
        const uint4 dyv = lds16(it);
        const uint4 zv = lds16(it + v16);
        bool kept[8];   // the forward's keep decisions of these 8 elements
        if (REGEN) {
          // drawn again: element e is kept iff its Philox word >= thr
          if (kDrawGroup == 1) {
            const uint64_t q = static_cast<uint64_t>(grow + ch * kChunk) >> 2;
            draws[0][0] = philox4x32_10(make_uint4(static_cast<uint32_t>(q),
                                                   static_cast<uint32_t>(q >> 32), P.off0,
                                                   P.off1),
                                        P.rk);
            draws[0][1] = philox4x32_10(make_uint4(static_cast<uint32_t>(q + 1),
                                                   static_cast<uint32_t>((q + 1) >> 32), P.off0,
                                                   P.off1),
                                        P.rk);
          }
          const uint4 a = draws[ch % kDrawGroup][0], b = draws[ch % kDrawGroup][1];
          const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) kept[e] = u[e] >= P.thr;
        } else if (BITS) {
          const uint32_t mbyte = it0[ch * item_bytes + off_mask - tid * 15];   // own byte
#pragma unroll
          for (int e = 0; e < 8; ++e) kept[e] = ((mbyte >> e) & 1u) != 0u;
        } else {
          // stored mask bytes are 0 or 1: bit 0 of byte e decides
          const uint2 mk = lds8(it + off_mask - tid * 8);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            kept[e] = ((e < 4 ? mk.x : mk.y) & (1u << (8 * (e & 3)))) != 0u;
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
        for (int e = 0; e < 8; ++e) dp[e] = kept[e] ? dp[e] : 0.f;
#pragma unroll
        for (int e = 0; e < 8; e += 2) add2(bt[e], bt[e + 1], dp[e], dp[e + 1]);
        st16_stream(dres_row + ch * kChunk, pack8(dz));
        const uint4 pb = pack8(dp);
        if (BULK) {
          *reinterpret_cast<uint4*>(stage_row + ch * (NTHR * 16)) = pb;
        } else {
          if (dg0_row != nullptr) st16_stream(dg0_row + ch * kChunk, pb);
          for (int j = 1; j < P.n_gather; ++j)
            st16_stream(P.dgathered[j] + grow + ch * kChunk, pb);
        }
      }
      if constexpr (TACC) {
        tmem_st8(tacc + 24 * ch + 16, bt);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc_bias[ch][e] = bt[e];
      }
    }
    if (BULK) {
      fence_proxy_async_smem();   // this row's shared dYpre, visible to the copy engine
      prev_grow = row * h;
    }
  }
  if (BULK) {
    // the last row: every thread has written and fenced its part
    __syncthreads();
    if (tid == 0) {
      if (nrows > 0) {
        bulk_wait_read_all();
        const uint8_t* src = stage0 + ((nrows - 1) & 1) * stage_bytes;
        for (int j = 0; j < P.n_gather; ++j)
          bulk_s2g(P.dgathered[j] + prev_grow, src, static_cast<uint32_t>(h) * 2u);
        bulk_commit();
      }
      bulk_wait_all();   // no copy may still read this block's shared memory at exit
    }
  }
  cp_async_wait<0>();
  if constexpr (TACC) {
    tmem_wait_st();
#pragma unroll
    for (int ch = 0; ch < MAXC; ++ch) {
      float gb[16], bt[8];
      tmem_ld16(tacc + 24 * ch, gb);
      tmem_ld8(tacc + 24 * ch + 16, bt);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        acc_g[ch][e] = gb[e];
        acc_b[ch][e] = gb[8 + e];
        acc_bias[ch][e] = bt[e];
      }
    }
    tmem_sync_block();   // every warp is done with tensor memory
    if (tid < 32) tmem_dealloc(tmem_base, kCols);
  }

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

}  // namespace spb
