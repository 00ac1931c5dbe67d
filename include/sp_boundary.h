/*
 * sp_boundary.h -- C ABI of the GB300 (sm_103a) sequence-parallel boundary.
 *
 * The boundary between the sequence-parallel (SP) region and the
 * tensor-parallel (TP) region of a transformer block under Megatron-style
 * TP+SP, as taught in "第 7 课：序列并行 SP" (hpc.payai.win/train/lesson07.html,
 * cited as L7).  The t tensor-parallel ranks are emulated on one GPU as t
 * separate device buffers: "rank k" is nothing more than the k-th pointer of
 * each pointer array below.
 *
 * Common conventions (every entry point):
 *  - All tensors are dense, row-major, caller-allocated device memory.  The
 *    library never allocates, frees or keeps a pointer after the call returns
 *    (except where an entry point says otherwise).
 *  - Pointer arrays ("[t]", "[n_gather]") are HOST arrays of DEVICE pointers;
 *    they are copied by value into kernel parameters, hence t <= SP_MAX_RANKS.
 *  - bf16 tensors are IEEE bfloat16 bit patterns (2 bytes per element); every
 *    bf16 / uint8 tensor pointer must be 16-byte aligned; h % 8 == 0.
 *  - Shapes: a "full" tensor is (b, s, h); the sequence axis s is split into
 *    t shards at o_k = floor(k*s/t), shard k is tokens [o_k, o_{k+1}) of every
 *    batch row and is stored as its own (b, s_k, h) tensor, s_k = o_{k+1}-o_k
 *    (L7 §3: LayerNorm / dropout / residual are token-wise, so each rank keeps
 *    only its (b, s/t, h) slice).  Without cu_seqlens the split must be even
 *    (s % t == 0, L7 §3 "均分").  With cu_seqlens (packed, padding-free
 *    sequences) b must be 1, s is the total token count cu_seqlens[n_seqs] and
 *    shards may differ by one token.
 *  - Calls are asynchronous: they validate on the host, enqueue on `stream`
 *    (a cudaStream_t; NULL = the legacy default stream) and return.  A host
 *    validation failure returns an error code before anything is enqueued.
 *    Kernels are launched with programmatic stream serialisation: a call's
 *    kernel may start on the SMs while the kernel before it on `stream` is
 *    completing, but touches no global memory before that kernel's writes
 *    are visible, so stream order holds as for plain launches (also when the
 *    calls are captured into a CUDA graph).
 *    Device-side checks (cu_seqlens contents) write a nonzero sp_status_t into
 *    `dev_status` (a caller-owned device int32, may be NULL) and never clear it.
 *  - Outputs must not overlap inputs or each other (checked on the host).
 *  - On error, sp_last_error() returns a thread-local description.
 */
#ifndef SP_BOUNDARY_H
#define SP_BOUNDARY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SP_ABI_VERSION 1
#define SP_MAX_RANKS 16
#define SP_MAX_HIDDEN 16384

typedef enum sp_status {
  SP_OK = 0,
  SP_ERR_INVALID_ARG = 1,   /* a size, count, probability or pointer is invalid */
  SP_ERR_MISALIGNED = 2,    /* a tensor pointer is not 16-byte aligned */
  SP_ERR_UNSUPPORTED = 3,   /* valid request outside this build (h > SP_MAX_HIDDEN, or no
                               launch shape of the kernel fits one SM's shared memory) */
  SP_ERR_CUDA = 4,          /* a CUDA runtime error (text in sp_last_error) */
  SP_ERR_TIMEOUT = 5,       /* a bounded device-side wait expired (via dev_status): the
                               forward's staging waits give up after about a second of
                               wall time (also if the context was preempted that long
                               mid-kernel); the call's outputs are then undefined and
                               the call may simply be repeated */
  SP_ERR_DEVICE_CHECK = 6,  /* device-side validation failed (via dev_status) */
  SP_ERR_OVERLAP = 7        /* an output buffer overlaps another buffer */
} sp_status_t;

typedef enum sp_norm {
  SP_NORM_LAYERNORM = 0,    /* (z - mean) * rstd * gamma + beta, L7 §2 */
  SP_NORM_RMSNORM = 1       /* z * rstd * gamma, rstd = 1/sqrt(mean(z^2) + eps) */
} sp_norm_t;

/*
 * sp_rs_norm_fwd -- the forward boundary, fused: g* (reduce-scatter along s),
 * bias-add, dropout, residual-add, LayerNorm/RMSNorm, g (all-gather along s).
 *
 * L7 §3.A: after the row-parallel linear each rank holds a partial sum
 * (b, s, h); g* both sums the partials and leaves each rank its (b, s/t, h)
 * shard ("一石二鸟"); the token-wise ops then run on the shard; g all-gathers
 * the normalised shards into the (b, s, h) input of the next column-parallel
 * linear.  L7 §2 gives the LayerNorm formula (biased variance, eps inside the
 * square root).  Dropout follows L7's answer to Q1: one seed on every rank, so
 * the mask of an element does not depend on which rank computes it.
 *
 * Per token g (global index bi*s + si) of shard k, channel c:
 *   Y  = (((P_0 + P_1) + ...) + P_{t-1})[g,c] + bias[c]      float32, this order
 *   u  = word (i mod 4) of Philox4x32-10(key = (seed lo, seed hi),
 *        counter = (q lo, q hi, offset lo, offset hi)),  i = g*h + c,  q = i >> 2
 *   keep = u >= floor(p * 2^32);  D = keep ? Y * float(1/(1-p)) : 0
 *   Z  = bf16_rne(D + R[g,c])                                 (stored)
 *   LN : mean, var (biased) of Z over h; rstd = 1/sqrt(var + eps)
 *        O = (Z - mean) * rstd * gamma + beta
 *   RMS: rstd = 1/sqrt(mean(Z^2) + eps);  O = Z * rstd * gamma
 *   gathered[j][g,:] = bf16_rne(O)  for every j < n_gather
 *
 * partials  [t]  (b, s, h)   bf16  rank r's row-linear partial sum (input)
 * residual  [t]  (b, s_k, h) bf16  shard k of the residual stream (input)
 * bias, gamma    (h)         bf16  replicated parameters (input)
 * beta           (h)         bf16  LayerNorm only; ignored (may be NULL) for RMS
 * eps            > 0
 * p              dropout probability in [0, 1); p == 0 disables dropout
 * seed, offset   Philox key and counter offset (advance offset per call to
 *                draw fresh masks; the pair makes a run reproducible)
 * cu_seqlens     NULL (dense) or device int32 [n_seqs + 1] prefix sums of the
 *                packed sequence lengths; requires b == 1 and
 *                cu_seqlens[n_seqs] == s (checked on the device)
 * z_out     [t]  (b, s_k, h) bf16  Z, saved for the backward (output)
 * mask_out  [t]  (b, s_k, h) u8    1 = kept, 0 = dropped (output); NULL (the
 *                array): no mask is stored, h bytes less per token written and
 *                kept -- the backward is then sp_norm_bwd_philox, which draws
 *                the keep decisions again from (seed, offset, p)
 * mean_out  [t]  (b, s_k)    f32   LayerNorm mean; NULL (the array) for RMS
 * rstd_out  [t]  (b, s_k)    f32   rstd (output)
 * gathered  [n_gather] (b, s, h) bf16  full-sequence copies of O (output);
 *                n_gather in [0, SP_MAX_RANKS]; 0 skips the all-gather
 */
sp_status_t sp_rs_norm_fwd(const void* const* partials, const void* const* residual,
                           const void* bias, const void* gamma, const void* beta,
                           int64_t b, int64_t s, int64_t h, int32_t t, float eps,
                           double p, uint64_t seed, uint64_t offset,
                           const int32_t* cu_seqlens, int32_t n_seqs, sp_norm_t norm,
                           void* const* z_out, uint8_t* const* mask_out,
                           float* const* mean_out, float* const* rstd_out,
                           void* const* gathered, int32_t n_gather,
                           int32_t* dev_status, void* stream);

/*
 * sp_allgather_seq -- g alone: all-gather along s (L7 §3.A, "前向转入 TP 区域"),
 * and, in the backward, the transpose of g* (L7 §3.B: the gradient of a
 * reduce-scatter along s is an all-gather along s).
 *
 * shards    [t]  (b, s_k, h) bf16  (input)
 * gathered  [n_gather] (b, s, h) bf16: gathered[j][bi, o_k + i, :] =
 *                shards[k][bi, i, :] (output), n_gather in [1, SP_MAX_RANKS]
 */
sp_status_t sp_allgather_seq(const void* const* shards, int64_t b, int64_t s, int64_t h,
                             int32_t t, const int32_t* cu_seqlens, int32_t n_seqs,
                             void* const* gathered, int32_t n_gather,
                             int32_t* dev_status, void* stream);

/*
 * sp_shard_norm_fwd -- the middle step of the unfused boundary: bias,
 * dropout, residual-add and LayerNorm/RMSNorm on shards that were already
 * reduced by a separate reduce-scatter (sp_reduce_scatter_seq, whose bf16
 * output is the input here), writing O per shard for a separate all-gather
 * (sp_allgather_seq).  The three calls together are the boundary without
 * fusion (L7 §3.A applied step by step); they exist to measure what fusing
 * them into sp_rs_norm_fwd saves.  Per token the arithmetic is that of
 * sp_rs_norm_fwd with Y = the bf16 shard value (no rank sum); dropout draws
 * use the token's index in the full sequence, so the mask equals the fused
 * one.
 *
 * y_shards  [t]  (b, s_k, h) bf16  reduced partial sums of shard k (input)
 * residual, bias, gamma, beta, eps, p, seed, offset, cu_seqlens, norm,
 * z_out, mask_out, mean_out, rstd_out: as for sp_rs_norm_fwd
 * o_shards  [t]  (b, s_k, h) bf16  normalised shard (output)
 */
sp_status_t sp_shard_norm_fwd(const void* const* y_shards, const void* const* residual,
                              const void* bias, const void* gamma, const void* beta,
                              int64_t b, int64_t s, int64_t h, int32_t t, float eps, double p,
                              uint64_t seed, uint64_t offset, const int32_t* cu_seqlens,
                              int32_t n_seqs, sp_norm_t norm, void* const* z_out,
                              uint8_t* const* mask_out, float* const* mean_out,
                              float* const* rstd_out, void* const* o_shards,
                              int32_t* dev_status, void* stream);

/*
 * sp_reduce_scatter_seq -- g* alone, unfused: shards[k] = bf16_rne(sum over r
 * of partials[r] restricted to shard k), float32 sum in ascending r
 * (L7 §3.A, "前向转出 TP 区域").  In the backward it is the transpose of g
 * (L7 §3.B).
 *
 * partials  [t]  (b, s, h)   bf16  (input)
 * shards    [t]  (b, s_k, h) bf16  (output)
 */
sp_status_t sp_reduce_scatter_seq(const void* const* partials, int64_t b, int64_t s,
                                  int64_t h, int32_t t, const int32_t* cu_seqlens,
                                  int32_t n_seqs, void* const* shards,
                                  int32_t* dev_status, void* stream);

/*
 * sp_norm_bwd_workspace_bytes -- bytes of device workspace sp_norm_bwd needs
 * on the current device for this shape (0 when b*s == 0).  The workspace
 * holds per-block float32 partial sums of the parameter gradients.
 */
size_t sp_norm_bwd_workspace_bytes(int64_t b, int64_t s, int64_t h, int32_t t,
                                   sp_norm_t norm);

/*
 * sp_norm_bwd -- the backward boundary: the transpose of sp_rs_norm_fwd from
 * dY (the gradient of the normalised shard O) back to the residual and to the
 * row-linear partials (L7 §3.B: backward is the adjoint of the forward; the
 * gradient of g* is an all-gather along s).
 *
 * Per token of shard k (x_hat from the saved Z, mean, rstd):
 *   x_hat = (Z - mean) * rstd  (LN)   |   Z * rstd  (RMS)
 *   dxh   = dY * gamma
 *   LN : dZ = rstd * (dxh - mean_h(dxh) - x_hat * mean_h(dxh * x_hat))
 *   RMS: dZ = rstd * (dxh - x_hat * mean_h(dxh * x_hat))
 *   dZ += dz_skip (if given)
 *   dresidual = bf16_rne(dZ);   dYpre = dZ * mask * float(1/(1-p))
 *   dgathered[j][g,:] = bf16_rne(dYpre)  (each rank's partial gets the same)
 *   dgamma[c] = sum_g dY*x_hat,  dbeta[c] = sum_g dY (LN),  dbias[c] = sum_g dYpre
 *   (sums over every token of every shard: the parameters are replicated)
 *
 * dy        [t]  (b, s_k, h) bf16  (input)
 * z         [t]  (b, s_k, h) bf16  saved Z (input)
 * mask      [t]  (b, s_k, h) u8    saved mask (input)
 * mean      [t]  (b, s_k)    f32   saved mean (LN); NULL (the array) for RMS
 * rstd      [t]  (b, s_k)    f32   saved rstd (input)
 * gamma          (h)         bf16
 * dz_skip   [t]  (b, s_k, h) bf16  or NULL: gradient reaching Z by the skip path
 * p              the forward's dropout probability
 * dresidual [t]  (b, s_k, h) bf16  (output)
 * dgathered [n_gather] (b, s, h) bf16 (output); n_gather in [0, SP_MAX_RANKS]
 * dgamma, dbeta, dbias  (h) f32 (output); each may be NULL to skip it; dbeta
 *                is ignored for RMS.  Deterministic: same inputs, same device
 *                -> same bits.
 * workspace      device memory of at least sp_norm_bwd_workspace_bytes(...),
 *                16-byte aligned, owned by the caller, clobbered by the call
 */
sp_status_t sp_norm_bwd(const void* const* dy, const void* const* z,
                        const uint8_t* const* mask, const float* const* mean,
                        const float* const* rstd, const void* gamma,
                        const void* const* dz_skip, int64_t b, int64_t s, int64_t h,
                        int32_t t, double p, const int32_t* cu_seqlens, int32_t n_seqs,
                        sp_norm_t norm, void* const* dresidual, void* const* dgathered,
                        int32_t n_gather, float* dgamma, float* dbeta, float* dbias,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        void* stream);

/*
 * sp_norm_bwd_noalloc -- sp_norm_bwd for callers that cannot allocate device
 * memory.  The lesson has no counterpart to this entry point: it exists for
 * callers that cannot obtain a workspace themselves, such as a plugin inside
 * a host framework that reserves all device memory up front and hands its
 * plugins no scratch, or a path where cudaMalloc's implicit device
 * synchronisation is not acceptable.
 *
 * Arguments and results are those of sp_norm_bwd, minus the workspace.  The
 * per-block parameter-gradient partials go to a fixed array in the library's
 * own device memory (SP_NOALLOC_WORKSPACE_BYTES on every GPU that loads the
 * library, held until the process exits).  Nothing is allocated or freed by
 * the call.
 *  - Shapes whose partials (one float32 row of 3*h per block of this call's
 *    own launch: the stored-mask backward, with or without dz_skip) exceed
 *    SP_NOALLOC_WORKSPACE_BYTES are rejected with SP_ERR_UNSUPPORTED before
 *    anything is enqueued.  h = 8192 (152 blocks on a 152-SM GPU) fits;
 *    h = 5120 (304 blocks) and h = 16384 do not.
 *  - Outside stream capture every call looks up the array's device address
 *    on the current device (cudaGetSymbolAddress, a host-side query), so an
 *    address that changed after cudaDeviceReset is picked up; a call made
 *    while `stream` is being captured reuses the address of the device's
 *    last uncaptured call instead.  Make the first call on each device (and
 *    the first after a cudaDeviceReset) before any stream capture on it; a
 *    captured first call returns SP_ERR_INVALID_ARG.
 *  - All calls on a device share the one array: calls that may overlap on the
 *    GPU (different streams, no ordering between them) race on it.  Serialise
 *    them (one stream, or events).  Every call overwrites the partials it
 *    reads, so no clearing is needed between calls.
 */
#define SP_NOALLOC_WORKSPACE_BYTES (16u << 20)
sp_status_t sp_norm_bwd_noalloc(const void* const* dy, const void* const* z,
                                const uint8_t* const* mask, const float* const* mean,
                                const float* const* rstd, const void* gamma,
                                const void* const* dz_skip, int64_t b, int64_t s, int64_t h,
                                int32_t t, double p, const int32_t* cu_seqlens,
                                int32_t n_seqs, sp_norm_t norm, void* const* dresidual,
                                void* const* dgathered, int32_t n_gather, float* dgamma,
                                float* dbeta, float* dbias, int32_t* dev_status, void* stream);

/*
 * sp_rs_norm_bwd -- the backward entered through g, fused: the reduce-scatter
 * of the t ranks' partial gradients of the gathered input (the gradient of an
 * all-gather along s is a reduce-scatter along s, L7 §3.B) runs in the
 * prologue of the norm / dropout backward, so no reduced dY is written or
 * read.  Rank k's dY on its tokens is the float32 sum over r (ascending) of
 * dy_partials[r], used unrounded; the rest is sp_norm_bwd.
 *
 * dy_partials [t] (b, s, h) bf16  rank r's partial gradient of the gathered
 *                column-linear input (input)
 * other arguments as for sp_norm_bwd (same workspace size); h <= 8192
 * (SP_ERR_UNSUPPORTED above).
 */
sp_status_t sp_rs_norm_bwd(const void* const* dy_partials, const void* const* z,
                           const uint8_t* const* mask, const float* const* mean,
                           const float* const* rstd, const void* gamma,
                           const void* const* dz_skip, int64_t b, int64_t s, int64_t h,
                           int32_t t, double p, const int32_t* cu_seqlens, int32_t n_seqs,
                           sp_norm_t norm, void* const* dresidual, void* const* dgathered,
                           int32_t n_gather, float* dgamma, float* dbeta, float* dbias,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           void* stream);

/*
 * sp_norm_bwd_philox -- the mask-free backward: sp_norm_bwd with the dropout
 * keep decisions drawn again from Philox4x32-10 instead of read from the
 * stored 1-byte mask.  Because the forward's generator is counter-based and
 * keyed on the element's global index (L7 answer to Q1: one seed on every
 * rank), the same (seed, offset, p) reproduce the forward's mask exactly; the
 * backward then reads h bytes less per token, and a forward called with
 * mask_out == NULL need not write or keep the mask at all (h bytes less per
 * token in the forward and in the saved activations).  Arguments as for sp_norm_bwd,
 * minus `mask`, plus the forward's `seed` and `offset`; the workspace size is
 * sp_norm_bwd_workspace_bytes.
 */
sp_status_t sp_norm_bwd_philox(const void* const* dy, const void* const* z,
                               const float* const* mean, const float* const* rstd,
                               const void* gamma, const void* const* dz_skip, int64_t b,
                               int64_t s, int64_t h, int32_t t, double p, uint64_t seed,
                               uint64_t offset, const int32_t* cu_seqlens, int32_t n_seqs,
                               sp_norm_t norm, void* const* dresidual, void* const* dgathered,
                               int32_t n_gather, float* dgamma, float* dbeta, float* dbias,
                               void* workspace, size_t workspace_bytes, int32_t* dev_status,
                               void* stream);

/*
 * sp_rs_norm_fwd_bitmask / sp_norm_bwd_bitmask / sp_rs_norm_bwd_bitmask --
 * the boundary with the dropout mask stored one bit per element instead of
 * one byte: the same keep decisions, h / 8 bytes per token written, kept and
 * read instead of h.  Arguments as for sp_rs_norm_fwd, sp_norm_bwd and
 * sp_rs_norm_bwd, except:
 *
 * mask_bits_out / mask_bits  [t]  (b, s_k, h / 8) u8, 16-byte aligned: byte
 *                j of a token row holds channels [8j, 8j + 8), bit e (value
 *                2^e) is channel 8j + e, 1 = kept.  Never NULL.
 * h              a multiple of 32 (rows of whole 4-byte words of bits, staged
 *                with the row's other inputs); other widths: SP_ERR_UNSUPPORTED
 *                before anything is enqueued
 *
 * The forward's other outputs are bit for bit those of sp_rs_norm_fwd; the
 * backwards' are bit for bit those of sp_norm_bwd and sp_rs_norm_bwd given the
 * byte mask of the same decisions (same launch shapes, same summation order).
 */
sp_status_t sp_rs_norm_fwd_bitmask(const void* const* partials, const void* const* residual,
                                   const void* bias, const void* gamma, const void* beta,
                                   int64_t b, int64_t s, int64_t h, int32_t t, float eps,
                                   double p, uint64_t seed, uint64_t offset,
                                   const int32_t* cu_seqlens, int32_t n_seqs, sp_norm_t norm,
                                   void* const* z_out, uint8_t* const* mask_bits_out,
                                   float* const* mean_out, float* const* rstd_out,
                                   void* const* gathered, int32_t n_gather,
                                   int32_t* dev_status, void* stream);
sp_status_t sp_rs_norm_bwd_bitmask(const void* const* dy_partials, const void* const* z,
                                   const uint8_t* const* mask_bits, const float* const* mean,
                                   const float* const* rstd, const void* gamma,
                                   const void* const* dz_skip, int64_t b, int64_t s, int64_t h,
                                   int32_t t, double p, const int32_t* cu_seqlens,
                                   int32_t n_seqs, sp_norm_t norm, void* const* dresidual,
                                   void* const* dgathered, int32_t n_gather, float* dgamma,
                                   float* dbeta, float* dbias, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_status, void* stream);
sp_status_t sp_norm_bwd_bitmask(const void* const* dy, const void* const* z,
                                const uint8_t* const* mask_bits, const float* const* mean,
                                const float* const* rstd, const void* gamma,
                                const void* const* dz_skip, int64_t b, int64_t s, int64_t h,
                                int32_t t, double p, const int32_t* cu_seqlens, int32_t n_seqs,
                                sp_norm_t norm, void* const* dresidual, void* const* dgathered,
                                int32_t n_gather, float* dgamma, float* dbeta, float* dbias,
                                void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                void* stream);

/* Thread-local text of the last non-OK status returned on this thread. */
const char* sp_last_error(void);

/* SP_ABI_VERSION of the built library. */
int32_t sp_abi_version(void);

/*
 * sp_debug_inject -- test hook: the next entry-point call on any thread
 * returns `code` (without validating or enqueuing anything) and the hook
 * disarms itself.  SP_OK disarms it.  SP_ERR_TIMEOUT is the exception when
 * the next call is sp_rs_norm_fwd or sp_shard_norm_fwd: that call launches
 * normally except that block 0's copy producer never stages the block's
 * first chunk, so the block's bounded waits run out (one to two seconds) and
 * the call's dev_status reads SP_ERR_TIMEOUT; that block's rows hold undefined
 * values.  It shows the waits are bounded, without faulting or hanging.
 */
sp_status_t sp_debug_inject(sp_status_t code);

/*
 * sp_debug_tune -- tuning hook: override the launch shape chosen for the
 * forward (kernel 0) or backward (kernel 1) row kernels: `stages` = cp.async
 * pipeline depth, `blocks_per_sm` = resident blocks per SM the grid is sized
 * for, `threads` = threads per block (forward: 64, 128, 160 or 256), `chunks`
 * = chunks per row (backward, with `threads`: one of the instantiated pairs;
 * forward: 2 splits every token row over a thread-block cluster of two CTAs
 * of h / 2 channels each, which exchange their parts of the row sums through
 * distributed shared memory -- taken when h % 16 == 0 and the CTA has 128 or
 * 256 threads, else ignored); 0 keeps the default rule for that field.  Values that do not fit shared
 * memory are reduced; shapes that are not instantiated are ignored.  Affects
 * sp_norm_bwd_workspace_bytes, so set it before sizing the workspace.  Results
 * do not depend on it except the float rounding of sums whose partition
 * changes (row statistics with the thread count, parameter gradients with the
 * grid).
 */
sp_status_t sp_debug_tune(int32_t kernel, int32_t stages, int32_t blocks_per_sm,
                          int32_t threads, int32_t chunks);

/*
 * sp_debug_last_shape -- test hook: the launch shape of the calling thread's
 * last sp_rs_norm_fwd (kernel 0) or backward (kernel 1: sp_norm_bwd,
 * sp_norm_bwd_philox, sp_norm_bwd_noalloc, sp_rs_norm_bwd) call, whether or
 * not it launched.  out: host int32 [6] = compute threads per block, chunks
 * per row (backward) or row chunks of one CTA (forward), pipeline stages,
 * grid (blocks), CTAs per cluster, dynamic shared memory bytes; all zero
 * before the first call.
 */
sp_status_t sp_debug_last_shape(int32_t kernel, int32_t* out);

/*
 * sp_debug_philox -- evaluate the library's device Philox4x32-10 on n
 * counter/key sets, for checking it against an independent implementation.
 * in  : device uint32 [n][6] = (c0, c1, c2, c3, k0, k1)
 * out : device uint32 [n][4]
 */
sp_status_t sp_debug_philox(const uint32_t* in, uint32_t* out, int64_t n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SP_BOUNDARY_H */
