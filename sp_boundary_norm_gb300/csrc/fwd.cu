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
// Layout of the work: a persistent grid; block b processes tokens
// b, b + G, b + 2G, ...  A row of h channels is cut into chunks of 8*T
// channels (T = threads); in each chunk thread i owns channels
// [8i, 8i+8).  Every thread streams its own 16-byte pieces of the t + 1 input
// rows into its own shared-memory slots with cp.async, STAGES chunks ahead,
// so the loads of the next chunks are in flight while the current one is
// reduced, normalised and stored.  Since a thread only reads back what it
// copied itself, the pipeline needs no block barrier; the only barriers are
// the two row reductions (mean, variance) of the norm.
#include "sp_device.cuh"

namespace spb {

template <int NTHR, int MAXC, int STAGES>
__global__ void __launch_bounds__(NTHR, 1) rs_norm_fwd_kernel(const FwdParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  constexpr int nthr = NTHR;
  const int t = P.map.t;
  const int64_t h = P.map.h;
  const int64_t chunk_ch = 8LL * nthr;
  const int nchunk = static_cast<int>((h + chunk_ch - 1) / chunk_ch);
  const size_t stream_bytes = static_cast<size_t>(nthr) * 16;
  const size_t stage_bytes = static_cast<size_t>(t + 1) * stream_bytes;
  float* red = reinterpret_cast<float*>(smem + STAGES * stage_bytes);   // [2][32]
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
      const int64_t c = pf_chunk * chunk_ch + tid * 8;
      if (c < h) {
        uint8_t* slot = smem + pf_stage * stage_bytes + tid * 16;
        const int64_t goff = row * h + c;
        for (int r = 0; r < t; ++r) cp_async16(slot + r * stream_bytes, P.partials[r] + goff);
        cp_async16(slot + t * stream_bytes, P.residual[pf_k] + pf_local * h + c);
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
  for (int64_t ri = 0; ri < nrows; ++ri) {
    const int64_t row = blockIdx.x + ri * G;
    int k;
    int64_t local;
    locate(P.map, row, k, local);
    uint16_t* zrow = P.z[k] + local * h;
    uint8_t* mrow = P.mask[k] + local * h;

    float z[MAXC][8];
    float lsum = 0.f;
#pragma unroll
    for (int ch = 0; ch < MAXC; ++ch) {
#pragma unroll
      for (int e = 0; e < 8; ++e) z[ch][e] = 0.f;
      if (ch < nchunk) {
        issue_next();
        cp_async_wait<STAGES - 1>();
        const int64_t c = ch * chunk_ch + tid * 8;
        if (c < h) {
          const uint8_t* slot = smem + stage * stage_bytes + tid * 16;
          // g*: float32 sum of the t partials, ranks in ascending order
          float y[8], q[8];
          unpack8(lds16(slot), y);
          for (int r = 1; r < t; ++r) {
            unpack8(lds16(slot + r * stream_bytes), q);
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = __fadd_rn(y[e], q[e]);
          }
          unpack8(ldg16(P.bias + c), q);
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = __fadd_rn(y[e], q[e]);
          const uint32_t keep =
              P.thr ? keep_bits8(static_cast<uint64_t>(row * h + c), P.thr, P.key0, P.key1,
                                 P.off0, P.off1)
                    : 0xFFu;
          unpack8(lds16(slot + t * stream_bytes), q);   // residual
          float zr[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float d = ((keep >> e) & 1u) ? __fmul_rn(y[e], P.scale) : 0.f;
            zr[e] = __fadd_rn(d, q[e]);
          }
          const uint4 zb = pack8(zr);
          st16_stream(zrow + c, zb);
          st8_stream(mrow + c, bits_to_bytes8(keep));
          unpack8(zb, z[ch]);   // the norm sees the stored bf16 values
#pragma unroll
          for (int e = 0; e < 8; ++e) lsum += is_ln ? z[ch][e] : z[ch][e] * z[ch][e];
        }
        stage = (stage + 1 == STAGES) ? 0 : stage + 1;
      }
    }

    // ---- token-wise statistics over h ------------------------------------
    float mean = 0.f, rstd;
    const float fh = static_cast<float>(h);
    if (is_ln) {
      mean = block_sum(lsum, red + 32 * slot_sel) / fh;
      slot_sel ^= 1;
      float lsq = 0.f;
#pragma unroll
      for (int ch = 0; ch < MAXC; ++ch) {
        if (ch < nchunk && ch * chunk_ch + tid * 8 < h) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float d = z[ch][e] - mean;
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
#pragma unroll
    for (int ch = 0; ch < MAXC; ++ch) {
      const int64_t c = ch * chunk_ch + tid * 8;
      if (ch < nchunk && c < h) {
        float g[8], o[8];
        unpack8(ldg16(P.gamma + c), g);
        if (is_ln) {
          float bt[8];
          unpack8(ldg16(P.beta + c), bt);
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = fmaf((z[ch][e] - mean) * rstd, g[e], bt[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = (z[ch][e] * rstd) * g[e];
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

template <int NTHR, int MAXC>
static const void* fwd_kernel_s(int stages) {
  switch (stages) {
    case 2: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, MAXC, 2>);
    case 3: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, MAXC, 3>);
    case 4: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, MAXC, 4>);
    case 6: return reinterpret_cast<const void*>(rs_norm_fwd_kernel<NTHR, MAXC, 6>);
    default: return nullptr;
  }
}

// Instantiated shapes: (threads, chunks) = (64, 1) for h <= 512, else
// (256, 1 | 2 | 4 | 8) for h <= 2048 * chunks; pipeline depth 2, 3, 4 or 6.
const void* fwd_kernel(int threads, int maxc, int stages) {
  if (threads == 64) return maxc == 1 ? fwd_kernel_s<64, 1>(stages) : nullptr;
  if (threads != 256) return nullptr;
  switch (maxc) {
    case 1: return fwd_kernel_s<256, 1>(stages);
    case 2: return fwd_kernel_s<256, 2>(stages);
    case 4: return fwd_kernel_s<256, 4>(stages);
    case 8: return fwd_kernel_s<256, 8>(stages);
    default: return nullptr;
  }
}

}  // namespace spb
