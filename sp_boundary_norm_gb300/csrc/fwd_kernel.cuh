// Fused forward kernel template (see fwd.cu for the design); instantiated in
// fwd.cu (the fused boundary) and fwd_shard.cu (the unfused middle step).
#pragma once

#include "sp_device.cuh"

namespace spb {

// Blocks are sized for 16 resident compute warps per SM: 512 / NTHR blocks of
// NTHR compute threads plus one copy-producer warp.
// SHARD = false: the fused boundary (inputs: the t full partials; output:
// the gathered full buffers).  SHARD = true: the middle step of the unfused
// boundary (input: each rank's already reduced shard, one stream; output: O
// of each shard in its own buffer; P.partials / P.gathered hold per-shard
// pointers).  Dropout draws use the token's index in the full sequence in
// both cases.
// CL = 2: the kernel runs in clusters of two CTAs that split every token row
// in halves of h / 2 channels (h a multiple of 16); each CTA reduces its half
// of the row sums, the two exchange them through distributed shared memory
// (one mbarrier hand-off per reduction, bounded waits) and both add them in
// the same order (CTA 0's part first), so both normalise with the same
// statistics.  Launched with a cluster dimension of 2; CTA 0 stores mean and
// rstd.
// MASKF: how the dropout mask is stored -- kMaskBytes (one byte per element,
// 1 = kept), kMaskNone (not at all: the mask-free pipeline, whose backward
// draws the keep decisions again) or kMaskBits (one bit per element: byte j
// of a row holds channels [8j, 8j + 8), bit e channel 8j + e).
template <int NTHR, int STAGES, int TT, bool SHARD, int CL = 1, int MASKF = kMaskBytes>
__global__ void __launch_bounds__(NTHR + kFwdProducerThreads, 512 / NTHR)
    rs_norm_fwd_kernel(const FwdParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar_full[STAGES], bar_empty[STAGES];
  __shared__ __align__(8) uint64_t xbar[2];   // CL > 1: the partner's row sums arrived
  __shared__ __align__(8) float2 xpub[2];     // CL > 1: this CTA's row sums, published
  constexpr int kWarps = NTHR / 32;   // compute warps; warp kWarps issues the copies
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  // input streams summed per element (compile-time when specialised)
  const int t = SHARD ? 1 : (TT > 0 ? TT : P.map.t);
  const int64_t h = P.map.h;
  const uint32_t crank = CL > 1 ? cluster_ctarank() : 0u;
  const int64_t hl = h / CL;          // channels of a row this CTA handles
  const int64_t coff = crank * hl;    // their first channel
  constexpr int kChunk = 8 * NTHR;
  const int nchunk = static_cast<int>((hl + kChunk - 1) / kChunk);
  constexpr int kStream = NTHR * 16;
  const int stage_bytes = (t + 1) * kStream;
  uint8_t* zbuf = smem + STAGES * stage_bytes + tid * 16;   // own slots, stride kStream
  float2* red = reinterpret_cast<float2*>(smem + STAGES * stage_bytes + nchunk * kStream);   // [2][32]
  const bool is_ln = (P.norm == SP_NORM_LAYERNORM);

  if (tid == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], kWarps);
    }
    if (CL > 1) {
      mbar_init(&xbar[0], 1);
      mbar_init(&xbar[1], 1);
    }
    mbar_fence_init();
  }
  if (CL > 1)
    cluster_sync_all();   // the partner's mbarriers are initialised too
  else
    __syncthreads();
  pdl_wait();
  if (blockIdx.x == 0 && tid < 32) check_cu_seqlens(P.cu_seqlens, P.n_seqs, P.rows, P.status);

  // this block's rows (a cluster's: both CTAs walk the same rows): every G-th
  // token when blocks get many rows (neighbouring tokens are then in flight
  // together), else a contiguous range
  const int64_t G = gridDim.x / CL;
  const int64_t bid = blockIdx.x / CL;
  const bool strided = P.rows >= 32 * G;
  const int64_t step = strided ? G : 1;
  int64_t r0, nrows;
  if (strided) {
    r0 = bid;
    nrows = (P.rows - 1 - r0) / G + 1;
  } else {
    block_rows(P.rows, bid, G, &r0, &nrows);
  }
  const int64_t c0 = tid * 8;   // this thread's first channel in every chunk

  // ---- producer warp: stage every (row, chunk) item in order ------------
  // Lane 0 of the producer warp stages item j into stage j % STAGES as soon as
  // the compute warps have released the stage's previous item (they do so
  // right after reading it, so a stage refills while the previous chunk is
  // still being computed): it arms the stage's full barrier with the item's
  // byte count and issues one bulk copy per stream.
  // Giving up is well defined: a compute thread whose wait runs out stops
  // waiting, and its warp stops releasing stages, from then on.  The
  // producer issues an item only after every compute warp has released the
  // stage's previous item, which a warp does only once that item's copies
  // have landed, so no stage is refilled while its phase has bytes pending;
  // when the producer's own wait runs out it issues nothing more, and before
  // the block ends it waits (bounded) for exactly the copies it did issue,
  // so no copy lands in shared memory after the block has gone.  A failure
  // costs at most two wait limits; the call then reports SP_ERR_TIMEOUT and
  // its outputs are undefined.
  bool timed_out = false;   // this thread's own wait ran out
  if (tid >= NTHR) {
    if (lane == 0) {
      RowWalk pf;
      pf.init(P.map, r0);
      int64_t item = 0;   // items attempted so far, in order; all but a withheld one issued
      for (int64_t ri = 0; ri < nrows; ++ri) {
        if (ri > 0) pf.next(P.map, step);
        const int64_t goff = pf.row * h + coff, roff = pf.local * h + coff;
        const int kk = pf.k;
        int ch = 0;
        for (; ch < nchunk; ++ch, ++item) {
          const int s = static_cast<int>(item % STAGES);
          const int64_t use = item / STAGES;
          if (use > 0 && !mbar_wait(&bar_empty[s], static_cast<uint32_t>((use - 1) & 1))) {
            timed_out = true;
            break;
          }
          if (P.withhold != 0 && blockIdx.x == 0 && item == 0) continue;   // test hook
          const int cc = ch * kChunk;
          const int n = (hl - cc < kChunk) ? static_cast<int>(hl - cc) : kChunk;
          const uint32_t bytes = static_cast<uint32_t>(n) * 2u;
          uint8_t* dst = smem + s * stage_bytes;
          mbar_arrive_expect_tx(&bar_full[s], bytes * static_cast<uint32_t>(t + 1));
          if (SHARD) {
            bulk_g2s(dst, P.partials[kk] + roff + cc, bytes, &bar_full[s]);
          } else {
#pragma unroll
            for (int r = 0; r < (TT > 0 ? TT : SP_MAX_RANKS); ++r)
              if (TT > 0 || r < t) bulk_g2s(dst + r * kStream, P.partials[r] + goff + cc, bytes,
                                            &bar_full[s]);
          }
          bulk_g2s(dst + t * kStream, P.residual[kk] + roff + cc, bytes, &bar_full[s]);
        }
        if (ch < nchunk) break;   // gave up
      }
      // Drain: the copies of the last STAGES items issued must land before the
      // block may end.  Item j was issued only after the stage's previous
      // item had completed its phase, so its copies complete phase
      // (j / STAGES) & 1 of its stage; a withheld item issued nothing.
      for (int64_t j = (item > STAGES ? item - STAGES : 0); j < item; ++j) {
        if (P.withhold != 0 && blockIdx.x == 0 && j == 0) continue;
        if (!mbar_wait(&bar_full[j % STAGES], static_cast<uint32_t>((j / STAGES) & 1)))
          timed_out = true;
      }
      if (timed_out && P.status != nullptr) *P.status = SP_ERR_TIMEOUT;
    }
    __syncwarp();
    if (CL > 1) cluster_sync_all();
    return;
  }

  RowWalk cur;
  cur.init(P.map, r0);
  bool gave_up = false;   // this thread's wait ran out: it waits and releases no more
  int slot_sel = 0;
  const float inv_h = 1.f / static_cast<float>(h);

  // CL > 1: adds the partner CTA's part of a row sum to this CTA's part, in
  // CTA order.  Exchange xi uses slot xi & 1 and that slot's phase parity
  // (xi >> 1) & 1; a slot is reused two exchanges later, which the partner
  // can reach only after this CTA's next exchange, i.e. after every warp here
  // has read the slot.
  uint32_t xi = 0;
  auto pair_sum = [&](float2 part) -> float2 {
    if constexpr (CL == 1) {
      return part;
    } else {
      const uint32_t peer = crank ^ 1u;
      const int slot = static_cast<int>(xi & 1u);
      const uint32_t par = (xi >> 1) & 1u;
      ++xi;
      if (tid == 0) {
        xpub[slot] = part;
        mbar_arrive_remote(cluster_map(&xbar[slot], peer));
      }
      float2 other = make_float2(0.f, 0.f);
      if (lane == 0 && !gave_up) {
        if (mbar_wait_cluster(&xbar[slot], par)) {
          other = ld_cluster_f2(cluster_map(&xpub[slot], peer));
        } else {
          gave_up = true;
          timed_out = true;
        }
      }
      other.x = __shfl_sync(0xFFFFFFFFu, other.x, 0);
      other.y = __shfl_sync(0xFFFFFFFFu, other.y, 0);
      return crank == 0 ? make_float2(part.x + other.x, part.y + other.y)
                        : make_float2(other.x + part.x, other.y + part.y);
    }
  };
  for (int64_t ri = 0; ri < nrows; ++ri) {
    if (ri > 0) cur.next(P.map, step);
    const int64_t row = cur.row;
    const int k = cur.k;
    const int64_t local = cur.local;
    uint16_t* zrow = P.z[k] + local * h + coff + c0;
    uint8_t* mrow = MASKF == kMaskBytes ? P.mask[k] + local * h + coff + c0
                    : MASKF == kMaskBits ? P.mask[k] + (local * h + coff + c0) / 8
                                         : nullptr;
    const uint64_t e_row = static_cast<uint64_t>(row * h + coff + c0);   // global element index

    // ---- pass 1: g* sum, bias, dropout, residual -> Z (stored) ----------
    float lsum = 0.f, lsq = 0.f;
#pragma unroll 1
    for (int ch = 0; ch < nchunk; ++ch) {
      const int64_t item = ri * nchunk + ch;
      const int stage = static_cast<int>(item % STAGES);
      // the item has landed (after a give-up the thread reads whatever the
      // stage holds: the outputs are undefined then, and it releases nothing)
      bool have = !gave_up;
      if (have && !mbar_wait(&bar_full[stage], static_cast<uint32_t>((item / STAGES) & 1))) {
        have = false;
        gave_up = true;
        timed_out = true;
      }
      const int cc = ch * kChunk;
      // g*: float32 sum of the t partials, ranks in ascending order
      // ((P_0 + P_1) + P_2) + ...; each add widens its bf16 operand exactly
      float y[8];
      uint4 rv = make_uint4(0, 0, 0, 0);
      if (cc + c0 < hl) {
        const uint8_t* slot = smem + stage * stage_bytes + tid * 16;
        unpack8(lds16(slot), y);
        if (!SHARD) {
#pragma unroll
          for (int r = 1; r < (TT > 0 ? TT : SP_MAX_RANKS); ++r)
            if (TT > 0 || r < t) add8_bf16(lds16(slot + r * kStream), y);
        }
        rv = lds16(slot + t * kStream);   // the residual, used after the dropout
      }
      __syncwarp();
      if (lane == 0 && have) mbar_arrive(&bar_empty[stage]);   // the stage is free again
      if (cc + c0 < hl) {
        const uint4 bv = ldg16(P.bias + coff + cc + c0);
        add8_bf16(bv, y);   // + bias
        // dropout: element e keeps iff its Philox word >= thr
        [[maybe_unused]] uint2 keep = make_uint2(0x01010101u, 0x01010101u);   // mask bytes
        if (P.thr) {
          const uint64_t q = (e_row + cc) >> 2;
          const uint4 a = philox4x32_10(make_uint4(static_cast<uint32_t>(q),
                                                   static_cast<uint32_t>(q >> 32), P.off0, P.off1),
                                        P.rk);
          const uint4 b = philox4x32_10(make_uint4(static_cast<uint32_t>(q + 1),
                                                   static_cast<uint32_t>((q + 1) >> 32), P.off0,
                                                   P.off1),
                                        P.rk);
          const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
          float ys[8];
#pragma unroll
          for (int e = 0; e < 8; e += 2) mul2_to(y[e], y[e + 1], P.scale, ys[e], ys[e + 1]);
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = (u[e] >= P.thr) ? ys[e] : 0.f;
          if constexpr (MASKF != kMaskNone)
            keep = make_uint2(keep_bytes4(a, P.thr), keep_bytes4(b, P.thr));
        }
        // (with p == 0 the scale is exactly 1 and y * 1 == y)
        add8_bf16(rv, y);   // + residual -> Z in fp32
        const uint4 zb = pack8(y);                 // Z = bf16_rne(...)
        st16_stream(zrow + cc, zb);
        if constexpr (MASKF == kMaskBytes) st8_stream(mrow + cc, keep);
        if constexpr (MASKF == kMaskBits) st1_stream(mrow + cc / 8, keep_bits8(keep));
        *reinterpret_cast<uint4*>(zbuf + ch * kStream) = zb;
        // the norm sees the stored bf16 values: sum of Z (LayerNorm) and sum
        // of Z^2 (both norms)
        float q2[2] = {0.f, 0.f};
        fma2_bf16(zb.x, zb.x, q2[0], q2[1]);
        fma2_bf16(zb.y, zb.y, q2[0], q2[1]);
        fma2_bf16(zb.z, zb.z, q2[0], q2[1]);
        fma2_bf16(zb.w, zb.w, q2[0], q2[1]);
        lsq += q2[0] + q2[1];
        if (is_ln) {
          float l2[2] = {0.f, 0.f};
          add2_bf16(zb.x, l2[0], l2[1]);
          add2_bf16(zb.y, l2[0], l2[1]);
          add2_bf16(zb.z, l2[0], l2[1]);
          add2_bf16(zb.w, l2[0], l2[1]);
          lsum += l2[0] + l2[1];
        }
      }
    }

    // ---- token-wise statistics over h ------------------------------------
    // LayerNorm: the two sums are reduced together (one block barrier) and
    // the biased variance is taken as E[Z^2] - mean^2 when mean^2 <= var / 4:
    // there the float32 cancellation error stays within a few 1e-6 of var
    // (the terms are at most 1.25 var).  Otherwise (a row whose mean is large
    // against its spread, or a non-finite value) the variance is recomputed
    // in a second pass as the mean of (Z - mean)^2.
    float mean = 0.f, rstd;
    if (is_ln) {
      const float2 sums = pair_sum(warps_sum2<kWarps>(lsum, lsq, red + 32 * slot_sel));
      slot_sel ^= 1;
      mean = sums.x * inv_h;
      const float var1 = sums.y * inv_h - mean * mean;
      if (mean * mean <= 0.25f * var1) {
        rstd = rsqrtf(var1 + P.eps);
      } else {
        float lsqa = 0.f, lsqb = 0.f;
        const float nmean = -mean;
#pragma unroll 1
        for (int ch = 0; ch < nchunk; ++ch) {
          if (ch * kChunk + c0 < hl) {
            float d[8];
            add8_bf16_bcast(lds16(zbuf + ch * kStream), nmean, d);   // z - mean
#pragma unroll
            for (int e = 0; e < 8; e += 2) fma2(lsqa, lsqb, d[e], d[e + 1], d[e], d[e + 1]);
          }
        }
        const float var =
            pair_sum(make_float2(warps_sum<kWarps>(lsqa + lsqb,
                                                   reinterpret_cast<float*>(red + 32 * slot_sel)),
                                 0.f)).x * inv_h;
        slot_sel ^= 1;
        rstd = rsqrtf(var + P.eps);
      }
    } else {
      const float ms =
          pair_sum(make_float2(warps_sum<kWarps>(lsq, reinterpret_cast<float*>(red + 32 * slot_sel)),
                               0.f)).x * inv_h;
      slot_sel ^= 1;
      rstd = rsqrtf(ms + P.eps);
    }

    // ---- normalise and write into the all-gather destination(s) ----------
    const int64_t orow = row * h + coff + c0;
    uint16_t* g0_row = SHARD ? P.gathered[k] + local * h + coff + c0
                             : (P.n_gather > 0 ? P.gathered[0] + orow : nullptr);
#pragma unroll 1
    for (int ch = 0; ch < nchunk; ++ch) {
      const int cc = ch * kChunk;
      if (cc + c0 < hl) {
        const uint4 zv = lds16(zbuf + ch * kStream);
        const uint4 gv = ldg16(P.gamma + coff + cc + c0);
        float o[8];
        if (is_ln) {
          float g[8], bt[8];
          unpack8(gv, g);
          unpack8(ldg16(P.beta + coff + cc + c0), bt);
          add8_bf16_bcast(zv, -mean, o);   // z - mean
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            mul2(o[e], o[e + 1], rstd, rstd);
            fma2(bt[e], bt[e + 1], o[e], o[e + 1], g[e], g[e + 1]);   // * gamma + beta
            o[e] = bt[e];
            o[e + 1] = bt[e + 1];
          }
        } else {
          fma8_bf16_bcast(zv, gv, 0.f, o);   // z * gamma, exact
#pragma unroll
          for (int e = 0; e < 8; e += 2) mul2(o[e], o[e + 1], rstd, rstd);
        }
        const uint4 ob = pack8(o);
        if (g0_row != nullptr) st16_stream(g0_row + cc, ob);
        if (!SHARD)
          for (int j = 1; j < P.n_gather; ++j) st16_stream(P.gathered[j] + orow + cc, ob);
      }
    }
    if (tid == 0 && crank == 0) {
      if (is_ln) P.mean[k][local] = mean;
      P.rstd[k][local] = rstd;
    }
  }
  if (timed_out && P.status != nullptr) *P.status = SP_ERR_TIMEOUT;
  if (CL > 1) cluster_sync_all();   // no partner reads this CTA's shared memory any more
}

}  // namespace spb
