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
// Work layout: a persistent grid (two blocks per SM); block b processes
// tokens b, b + G, b + 2G, ...  A row of h channels is cut into chunks of 8*T
// channels (T = threads); in each chunk thread i owns channels [8i, 8i+8).
// Every thread streams its own 16-byte pieces of the t + 1 input rows into
// its own shared-memory slots with cp.async, STAGES - 1 chunks ahead, so the
// loads of the next chunks are in flight while the current one is summed,
// dropped out, normalised and stored.  A thread only reads back what it
// copied itself, so the pipeline needs no block barrier; the only barriers
// are the row reductions of the norm.  The chunk loop is not unrolled (the
// Philox rounds make its body long): Z of the row waits for the statistics
// in the thread's own shared-memory slots rather than in registers.
#include "sp_device.cuh"

namespace spb {

template <int NTHR, int STAGES, int TT>
__global__ void __launch_bounds__(NTHR, (NTHR >= 256 ? 2 : 4))
    rs_norm_fwd_kernel(const FwdParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int t = TT > 0 ? TT : P.map.t;     // compile-time rank count when specialised
  const int64_t h = P.map.h;
  constexpr int64_t kChunk = 8LL * NTHR;
  const int nchunk = static_cast<int>((h + kChunk - 1) / kChunk);
  constexpr size_t kStream = static_cast<size_t>(NTHR) * 16;
  const size_t stage_bytes = static_cast<size_t>(t + 1) * kStream;
  uint8_t* zbuf = smem + STAGES * stage_bytes;                       // [nchunk][NTHR][16 B]
  float* red = reinterpret_cast<float*>(zbuf + nchunk * kStream);   // [2][32]
  const bool is_ln = (P.norm == SP_NORM_LAYERNORM);

  if (blockIdx.x == 0 && tid < 32) check_cu_seqlens(P.cu_seqlens, P.n_seqs, P.rows, P.status);

  const int64_t G = gridDim.x;
  const int64_t nrows = (P.rows > blockIdx.x) ? (P.rows - 1 - blockIdx.x) / G + 1 : 0;

  // ---- prefetch cursor: the next (row, chunk) item to stage -------------
  int64_t pf_ri = 0;
  int pf_chunk = 0, pf_stage = 0, pf_k = 0;
  int64_t pf_local = 0;
  if (nrows > 0) locate(P.map, blockIdx.x, pf_k, pf_local);

  auto issue_next = [&]() {
    if (pf_ri < nrows) {
      const int64_t row = blockIdx.x + pf_ri * G;
      const int64_t c = pf_chunk * kChunk + tid * 8;
      if (c < h) {
        uint8_t* slot = smem + pf_stage * stage_bytes + tid * 16;
        const int64_t goff = row * h + c;
#pragma unroll
        for (int r = 0; r < (TT > 0 ? TT : SP_MAX_RANKS); ++r)
          if (TT > 0 || r < t) cp_async16(slot + r * kStream, P.partials[r] + goff);
        cp_async16(slot + t * kStream, P.residual[pf_k] + pf_local * h + c);
      }
      if (++pf_chunk == nchunk) {
        pf_chunk = 0;
        if (++pf_ri < nrows) locate(P.map, blockIdx.x + pf_ri * G, pf_k, pf_local);
      }
    }
    cp_async_commit();
    pf_stage = (pf_stage + 1 == STAGES) ? 0 : pf_stage + 1;
  };

#pragma unroll
  for (int i = 0; i < STAGES - 1; ++i) issue_next();

  int stage = 0;
  int slot_sel = 0;
  const float fh = static_cast<float>(h);
  for (int64_t ri = 0; ri < nrows; ++ri) {
    const int64_t row = blockIdx.x + ri * G;
    int k;
    int64_t local;
    locate(P.map, row, k, local);
    uint16_t* zrow = P.z[k] + local * h;
    uint8_t* mrow = P.mask[k] + local * h;

    // ---- pass 1: g* sum, bias, dropout, residual -> Z (stored) ----------
    float lsum = 0.f;
#pragma unroll 1
    for (int ch = 0; ch < nchunk; ++ch) {
      issue_next();
      cp_async_wait<STAGES - 1>();
      const int64_t c = ch * kChunk + tid * 8;
      if (c < h) {
        const uint8_t* slot = smem + stage * stage_bytes + tid * 16;
        const uint4 bv = ldg16(P.bias + c);
        uint2 keep = make_uint2(0x01010101u, 0x01010101u);
        if (P.thr) keep = keep_mask8(static_cast<uint64_t>(row * h + c), P.thr, P.key0, P.key1,
                                     P.off0, P.off1);
        // g*: float32 sum of the t partials, ranks in ascending order
        float y[8], q[8];
        unpack8(lds16(slot), y);
#pragma unroll
        for (int r = 1; r < (TT > 0 ? TT : SP_MAX_RANKS); ++r) {
          if (TT > 0 || r < t) {
            unpack8(lds16(slot + r * kStream), q);
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = __fadd_rn(y[e], q[e]);
          }
        }
        unpack8(bv, q);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = __fadd_rn(y[e], q[e]);
        unpack8(lds16(slot + t * kStream), q);   // residual
        float zr[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t kb = ((e < 4 ? keep.x : keep.y) >> (8 * (e & 3))) & 0xFFu;
          const float d = kb ? __fmul_rn(y[e], P.scale) : 0.f;
          zr[e] = __fadd_rn(d, q[e]);
        }
        const uint4 zb = pack8(zr);
        st16_stream(zrow + c, zb);
        st8_stream(mrow + c, keep);
        *reinterpret_cast<uint4*>(zbuf + ch * kStream + tid * 16) = zb;
        float zf[8];
        unpack8(zb, zf);   // the norm sees the stored bf16 values
#pragma unroll
        for (int e = 0; e < 8; ++e) lsum += is_ln ? zf[e] : zf[e] * zf[e];
      }
      stage = (stage + 1 == STAGES) ? 0 : stage + 1;
    }

    // ---- token-wise statistics over h ------------------------------------
    float mean = 0.f, rstd;
    if (is_ln) {
      mean = block_sum(lsum, red + 32 * slot_sel) / fh;
      slot_sel ^= 1;
      float lsq = 0.f;
#pragma unroll 1
      for (int ch = 0; ch < nchunk; ++ch) {
        if (ch * kChunk + tid * 8 < h) {
          float zf[8];
          unpack8(lds16(zbuf + ch * kStream + tid * 16), zf);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float d = zf[e] - mean;
            lsq += d * d;
          }
        }
      }
      const float var = block_sum(lsq, red + 32 * slot_sel) / fh;
      slot_sel ^= 1;
      rstd = rsqrtf(var + P.eps);
    } else {
      const float ms = block_sum(lsum, red + 32 * slot_sel) / fh;
      slot_sel ^= 1;
      rstd = rsqrtf(ms + P.eps);
    }

    // ---- normalise and write into the all-gather destination(s) ----------
#pragma unroll 1
    for (int ch = 0; ch < nchunk; ++ch) {
      const int64_t c = ch * kChunk + tid * 8;
      if (c < h) {
        float zf[8], g[8], o[8];
        unpack8(lds16(zbuf + ch * kStream + tid * 16), zf);
        unpack8(ldg16(P.gamma + c), g);
        if (is_ln) {
          float bt[8];
          unpack8(ldg16(P.beta + c), bt);
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = fmaf((zf[e] - mean) * rstd, g[e], bt[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = (zf[e] * rstd) * g[e];
        }
        const uint4 ob = pack8(o);
        for (int j = 0; j < P.n_gather; ++j) st16_stream(P.gathered[j] + row * h + c, ob);
      }
    }
    if (tid == 0) {
      if (is_ln) P.mean[k][local] = mean;
      P.rstd[k][local] = rstd;
    }
  }
  cp_async_wait<0>();
}

template <int NTHR, int TT>
static const void* fwd_kernel_s(int stages) {
  switch (stages) {
    case 2: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, 2, TT>);
    case 3: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, 3, TT>);
    case 4: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, 4, TT>);
    default: return nullptr;
  }
}

// Instantiated shapes: 64 threads for h <= 512, else 256; pipeline depth 2, 3
// or 4 chunks; t either a run-time value or the compile-time 8.
const void* fwd_kernel(int threads, int t, int stages) {
  const bool t8 = (t == 8);
  if (threads == 64) return t8 ? fwd_kernel_s<64, 8>(stages) : fwd_kernel_s<64, 0>(stages);
  if (threads == 256) return t8 ? fwd_kernel_s<256, 8>(stages) : fwd_kernel_s<256, 0>(stages);
  return nullptr;
}

}  // namespace spb
