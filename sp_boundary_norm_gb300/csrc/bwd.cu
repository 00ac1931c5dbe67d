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
// [8i, 8i+8) of each chunk, and a per-thread cp.async pipeline that stages
// dY, Z, the mask (and the optional skip-path gradient) of the next chunks.
// A row needs two reductions over h (mean(dxh), mean(dxh * x_hat)); they are
// done together, so one block barrier per row.  Because a thread owns the same
// channels in every row, it accumulates its channels' parameter-gradient
// terms in registers across all rows of its block and writes one float32
// partial per block and channel at the end; a second kernel sums the
// partials over blocks in a fixed order (float64), so results are
// bit-reproducible without atomics.
#include "sp_device.cuh"

namespace spb {

template <int NTHR, int MAXC, int STAGES>
__global__ void __launch_bounds__(NTHR, 1) norm_bwd_kernel(const BwdParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  constexpr int nthr = NTHR;
  const int64_t h = P.map.h;
  const int64_t chunk_ch = 8LL * nthr;
  const int nchunk = static_cast<int>((h + chunk_ch - 1) / chunk_ch);
  const bool is_ln = (P.norm == SP_NORM_LAYERNORM);
  const bool has_skip = P.has_skip != 0;
  const size_t v16 = static_cast<size_t>(nthr) * 16;
  const size_t off_z = v16;
  const size_t off_skip = 2 * v16;
  const size_t off_mask = (has_skip ? 3 : 2) * v16;
  const size_t stage_bytes = off_mask + static_cast<size_t>(nthr) * 8;
  float2* red = reinterpret_cast<float2*>(smem + STAGES * stage_bytes);   // [2][32]

  if (blockIdx.x == 0 && tid < 32) check_cu_seqlens(P.cu_seqlens, P.n_seqs, P.rows, P.status);

  const int64_t G = gridDim.x;
  const int64_t nrows = (P.rows > blockIdx.x) ? (P.rows - 1 - blockIdx.x) / G + 1 : 0;

  // gamma of this thread's channels, kept for every row
  uint4 gam[MAXC];
#pragma unroll
  for (int ch = 0; ch < MAXC; ++ch) {
    const int64_t c = ch * chunk_ch + tid * 8;
    gam[ch] = (ch < nchunk && c < h) ? ldg16(P.gamma + c) : make_uint4(0, 0, 0, 0);
  }

  int64_t pf_ri = 0;
  int pf_chunk = 0, pf_stage = 0, pf_k = 0;
  int64_t pf_local = 0;
  if (nrows > 0) locate(P.map, blockIdx.x, pf_k, pf_local);

  auto issue_next = [&]() {
    if (pf_ri < nrows) {
      const int64_t c = pf_chunk * chunk_ch + tid * 8;
      if (c < h) {
        uint8_t* slot = smem + pf_stage * stage_bytes;
        const int64_t lo = pf_local * h + c;
        cp_async16(slot + tid * 16, P.dy[pf_k] + lo);
        cp_async16(slot + off_z + tid * 16, P.z[pf_k] + lo);
        if (has_skip) cp_async16(slot + off_skip + tid * 16, P.dz_skip[pf_k] + lo);
        cp_async8(slot + off_mask + tid * 8, P.mask[pf_k] + lo);
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

  float acc_g[MAXC][8], acc_b[MAXC][8], acc_bias[MAXC][8];
#pragma unroll
  for (int ch = 0; ch < MAXC; ++ch)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc_g[ch][e] = acc_b[ch][e] = acc_bias[ch][e] = 0.f;

  // statistics of the current row, loaded one row ahead
  float cur_mean = 0.f, cur_rstd = 0.f;
  if (nrows > 0) {
    int k0;
    int64_t l0;
    locate(P.map, blockIdx.x, k0, l0);
    cur_rstd = P.rstd[k0][l0];
    if (is_ln) cur_mean = P.mean[k0][l0];
  }

  int stage = 0;
  int slot_sel = 0;
  for (int64_t ri = 0; ri < nrows; ++ri) {
    const int64_t row = blockIdx.x + ri * G;
    int k;
    int64_t local;
    locate(P.map, row, k, local);
    float nx_mean = 0.f, nx_rstd = 0.f;
    if (ri + 1 < nrows) {
      int k1;
      int64_t l1;
      locate(P.map, row + G, k1, l1);
      nx_rstd = P.rstd[k1][l1];
      if (is_ln) nx_mean = P.mean[k1][l1];
    }
    const float mean = cur_mean, rstd = cur_rstd;

    uint4 dyv[MAXC], zv[MAXC], skv[MAXC];
    uint2 mkv[MAXC];
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int ch = 0; ch < MAXC; ++ch) {
      dyv[ch] = zv[ch] = skv[ch] = make_uint4(0, 0, 0, 0);
      mkv[ch] = make_uint2(0, 0);
      if (ch < nchunk) {
        issue_next();
        cp_async_wait<STAGES - 1>();
        const int64_t c = ch * chunk_ch + tid * 8;
        if (c < h) {
          const uint8_t* slot = smem + stage * stage_bytes;
          dyv[ch] = lds16(slot + tid * 16);
          zv[ch] = lds16(slot + off_z + tid * 16);
          if (has_skip) skv[ch] = lds16(slot + off_skip + tid * 16);
          mkv[ch] = lds8(slot + off_mask + tid * 8);
          float dy[8], zf[8], g[8];
          unpack8(dyv[ch], dy);
          unpack8(zv[ch], zf);
          unpack8(gam[ch], g);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float xh = is_ln ? (zf[e] - mean) * rstd : zf[e] * rstd;
            const float dxh = dy[e] * g[e];
            s1 += dxh;
            s2 += dxh * xh;
            acc_g[ch][e] += dy[e] * xh;
            acc_b[ch][e] += dy[e];
          }
        }
        stage = (stage + 1 == STAGES) ? 0 : stage + 1;
      }
    }

    const float2 s = block_sum2(s1, s2, red + 32 * slot_sel);
    slot_sel ^= 1;
    const float fh = static_cast<float>(h);
    const float m1 = is_ln ? s.x / fh : 0.f;
    const float m2 = s.y / fh;

#pragma unroll
    for (int ch = 0; ch < MAXC; ++ch) {
      const int64_t c = ch * chunk_ch + tid * 8;
      if (ch < nchunk && c < h) {
        float dy[8], zf[8], g[8], sk[8], dz[8], dp[8];
        unpack8(dyv[ch], dy);
        unpack8(zv[ch], zf);
        unpack8(gam[ch], g);
        unpack8(skv[ch], sk);   // zeros when there is no skip gradient
        const uint32_t keep = bytes8_to_bits(mkv[ch]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float xh = is_ln ? (zf[e] - mean) * rstd : zf[e] * rstd;
          const float dxh = dy[e] * g[e];
          dz[e] = rstd * (dxh - m1 - xh * m2) + sk[e];
          dp[e] = ((keep >> e) & 1u) ? dz[e] * P.scale : 0.f;
          acc_bias[ch][e] += dp[e];
        }
        st16_stream(P.dresidual[k] + local * h + c, pack8(dz));
        const uint4 pb = pack8(dp);
        for (int j = 0; j < P.n_gather; ++j) st16_stream(P.dgathered[j] + row * h + c, pb);
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
    const int64_t c = ch * chunk_ch + tid * 8;
    if (ch < nchunk && c < h) {
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

// out[q][c] = sum over blocks (in block order, float64) of ws[block][q][c].
__global__ void __launch_bounds__(256) param_reduce_kernel(const ParamReduceParams P) {
  const int q = blockIdx.y;
  float* out = P.out[q];
  const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (out == nullptr || c >= P.h) return;
  double acc = 0.0;
  const float* src = P.ws + q * P.h + c;
  const int64_t stride = 3 * P.h;
  for (int b = 0; b < P.nblk; ++b) acc += static_cast<double>(src[b * stride]);
  out[c] = static_cast<float>(acc);
}

template <int NTHR, int MAXC>
static const void* bwd_kernel_s(int stages) {
  switch (stages) {
    case 2: return reinterpret_cast<const void*>(norm_bwd_kernel<NTHR, MAXC, 2>);
    case 4: return reinterpret_cast<const void*>(norm_bwd_kernel<NTHR, MAXC, 4>);
    case 8: return reinterpret_cast<const void*>(norm_bwd_kernel<NTHR, MAXC, 8>);
    default: return nullptr;
  }
}

// Instantiated shapes: (threads, chunks) = (64, 1) for h <= 512, else
// (256, 1 | 2 | 4 | 8); pipeline depth 2, 4 or 8.
const void* bwd_kernel(int threads, int maxc, int stages) {
  if (threads == 64) return maxc == 1 ? bwd_kernel_s<64, 1>(stages) : nullptr;
  if (threads != 256) return nullptr;
  switch (maxc) {
    case 1: return bwd_kernel_s<256, 1>(stages);
    case 2: return bwd_kernel_s<256, 2>(stages);
    case 4: return bwd_kernel_s<256, 4>(stages);
    case 8: return bwd_kernel_s<256, 8>(stages);
    default: return nullptr;
  }
}

cudaError_t launch_param_reduce(const ParamReduceParams& p, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>((p.h + 255) / 256), 3);
  param_reduce_kernel<<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace spb
