// Host side of the C ABI: argument validation, launch-shape choice, launch.
//
// Nothing here allocates device memory; every buffer is the caller's.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "sp_internal.h"

namespace spb {

namespace {

thread_local char g_err[512] = "";
std::atomic<int> g_inject{SP_OK};
// Launch-shape overrides for tuning sweeps: [kernel][stages, blocks per SM,
// threads, chunks per row (backward only)]; 0 = the default rule.
std::atomic<int> g_tune[2][4] = {{{0}, {0}, {0}, {0}}, {{0}, {0}, {0}, {0}}};
// The launch shape of this thread's last forward (0) and backward (1) call.
thread_local LaunchShape g_last_shape[2] = {};

sp_status_t fail(sp_status_t code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

sp_status_t fail_cuda(cudaError_t e, const char* where) {
  if (e == cudaErrorInvalidConfiguration)
    return fail(SP_ERR_UNSUPPORTED, "%s: no launch shape of this kernel fits the shared memory "
                "of one SM for these sizes", where);
  return fail(SP_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorString(e), cudaGetErrorName(e));
}

bool take_injected(sp_status_t* out) {
  const int code = g_inject.exchange(SP_OK);
  if (code == SP_OK) return false;
  *out = fail(static_cast<sp_status_t>(code), "injected failure (sp_debug_inject)");
  return true;
}

// An injected SP_ERR_TIMEOUT is not returned by the host: the next forward
// launches with its device-side withhold hook set instead (block 0's copy
// producer never stages its first chunk, so that block's waits run out and
// the call's status word reads SP_ERR_TIMEOUT).
bool take_injected_timeout() {
  int expect = SP_ERR_TIMEOUT;
  return g_inject.compare_exchange_strong(expect, SP_OK);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A list of device byte ranges; outputs must not overlap anything else.
struct Ranges {
  struct R {
    uintptr_t lo, hi;
    bool out;
    const char* what;
    int idx;
  };
  std::vector<R> v;
  void add(const void* p, size_t bytes, bool out, const char* what, int idx) {
    if (p == nullptr || bytes == 0) return;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    v.push_back({lo, lo + bytes, out, what, idx});
  }
  sp_status_t check() const {
    for (size_t i = 0; i < v.size(); ++i) {
      if (!v[i].out) continue;
      for (size_t j = 0; j < v.size(); ++j) {
        if (i == j) continue;
        if (v[i].lo < v[j].hi && v[j].lo < v[i].hi)
          return fail(SP_ERR_OVERLAP, "output %s[%d] overlaps %s[%d]", v[i].what, v[i].idx,
                      v[j].what, v[j].idx);
      }
    }
    return SP_OK;
  }
};

// Shapes common to every entry point.
sp_status_t check_shape(int64_t b, int64_t s, int64_t h, int32_t t, const int32_t* cu_seqlens,
                        int32_t n_seqs) {
  if (t < 1 || t > SP_MAX_RANKS)
    return fail(SP_ERR_INVALID_ARG, "t = %d outside [1, %d]", t, SP_MAX_RANKS);
  if (b < 0 || s < 0) return fail(SP_ERR_INVALID_ARG, "negative b or s");
  if (h < 8 || h % 8 != 0) return fail(SP_ERR_INVALID_ARG, "h = %lld must be a positive multiple of 8", (long long)h);
  if (h > SP_MAX_HIDDEN)
    return fail(SP_ERR_UNSUPPORTED, "h = %lld above SP_MAX_HIDDEN = %d", (long long)h, SP_MAX_HIDDEN);
  if (cu_seqlens != nullptr) {
    if (b != 1) return fail(SP_ERR_INVALID_ARG, "cu_seqlens requires b == 1 (got %lld)", (long long)b);
    if (n_seqs < 1) return fail(SP_ERR_INVALID_ARG, "n_seqs = %d must be >= 1", n_seqs);
    if (!aligned16(cu_seqlens) && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
      return fail(SP_ERR_MISALIGNED, "cu_seqlens not 4-byte aligned");
  } else if (t > 0 && s % t != 0) {
    return fail(SP_ERR_INVALID_ARG, "s = %lld not divisible by t = %d (dense shards are even)",
                (long long)s, t);
  }
  const int64_t elems_limit = int64_t(1) << 60;
  if (b > 0 && s > 0 && (b > elems_limit / s || b * s > elems_limit / h))
    return fail(SP_ERR_INVALID_ARG, "b*s*h overflows");
  return SP_OK;
}

ShardMap make_map(int64_t b, int64_t s, int64_t h, int32_t t) {
  ShardMap m{};
  for (int k = 0; k <= t; ++k) m.off[k] = (k * s) / t;
  for (int k = t + 1; k <= SP_MAX_RANKS; ++k) m.off[k] = s;
  m.b = b;
  m.s = s;
  m.h = h;
  m.t = t;
  return m;
}

int64_t shard_rows(const ShardMap& m, int k) { return m.b * (m.off[k + 1] - m.off[k]); }

// Per-rank pointer arrays: non-NULL and aligned, except that the pointer of a
// shard with no token (possible when t > s) is never used and may be anything.
template <typename T>
sp_status_t check_ptrs(const T* const* arr, int n, const char* what, bool need16,
                       const ShardMap* shards = nullptr) {
  if (n > 0 && arr == nullptr) return fail(SP_ERR_INVALID_ARG, "%s array is NULL", what);
  for (int i = 0; i < n; ++i) {
    if (shards != nullptr && shard_rows(*shards, i) == 0) continue;
    if (arr[i] == nullptr) return fail(SP_ERR_INVALID_ARG, "%s[%d] is NULL", what, i);
    if (need16 ? !aligned16(arr[i]) : (reinterpret_cast<uintptr_t>(arr[i]) & 3u))
      return fail(SP_ERR_MISALIGNED, "%s[%d] misaligned", what, i);
  }
  return SP_OK;
}

sp_status_t check_vec(const void* p, const char* what) {
  if (p == nullptr) return fail(SP_ERR_INVALID_ARG, "%s is NULL", what);
  if (!aligned16(p)) return fail(SP_ERR_MISALIGNED, "%s misaligned", what);
  return SP_OK;
}

int pow2_at_least(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

constexpr size_t kSmemPerSm = 228 * 1024;     // sm_100-class shared memory per SM
constexpr size_t kSmemPerBlock = 227 * 1024;  // opt-in maximum per block
constexpr size_t kReserve = 1024;             // per-block reservation

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = -1;
  }
  return dev;
}

// The dynamic shared-memory opt-in of each kernel, per (kernel, device): it is
// only ever raised, to the largest size requested so far, and every setter
// goes through here so the cache always matches the driver's value.
struct AttrCache {
  std::mutex mu;
  static constexpr int kSlots = 256;
  const void* fn[kSlots];
  int device[kSlots];
  size_t smem[kSlots];
  int used = 0;
};
AttrCache g_attr;

cudaError_t ensure_smem_attr(const void* fn, size_t smem) {
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(g_attr.mu);
  int i = 0;
  for (; i < g_attr.used; ++i)
    if (g_attr.fn[i] == fn && g_attr.device[i] == dev) break;
  if (i < g_attr.used && g_attr.smem[i] >= smem) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (i == g_attr.used) {
    if (g_attr.used == AttrCache::kSlots) return cudaSuccess;   // full: just do not cache
    ++g_attr.used;
    g_attr.fn[i] = fn;
    g_attr.device[i] = dev;
  }
  g_attr.smem[i] = smem;
  return cudaSuccess;
}

// Launch shapes are pure functions of (kernel kind, rows, h, t, flags, device,
// tuning overrides); caching them keeps the per-call host cost to the
// argument checks, which matters for short kernels.
struct ShapeKey {
  int kind, t, flags, device, tune;
  int64_t rows, h;
  bool operator==(const ShapeKey& o) const {
    return kind == o.kind && t == o.t && flags == o.flags && device == o.device &&
           tune == o.tune && rows == o.rows && h == o.h;
  }
};

struct ShapeCache {
  std::mutex mu;
  static constexpr int kSlots = 64;
  ShapeKey key[kSlots];
  LaunchShape val[kSlots];
  int used = 0, next = 0;
};

ShapeCache g_shapes;
std::atomic<int> g_tune_epoch{0};

template <typename Make>
LaunchShape cached_shape(int kind, int64_t rows, int64_t h, int t, int flags, Make make) {
  const ShapeKey k{kind, t, flags, current_device(), g_tune_epoch.load(), rows, h};
  {
    std::lock_guard<std::mutex> lock(g_shapes.mu);
    for (int i = 0; i < g_shapes.used; ++i)
      if (g_shapes.key[i] == k) return g_shapes.val[i];
  }
  const LaunchShape ls = make();
  std::lock_guard<std::mutex> lock(g_shapes.mu);
  const int slot = g_shapes.used < ShapeCache::kSlots ? g_shapes.used++ : g_shapes.next;
  g_shapes.next = (slot + 1) % ShapeCache::kSlots;
  g_shapes.key[slot] = k;
  g_shapes.val[slot] = ls;
  return ls;
}

// Choose the pipeline depth (`stages`: chunks for the forward, rows for the
// backward) and blocks per SM: start from the requested pair and shrink, blocks
// first, until the shared memory fits; then cap the grid at what the
// occupancy calculator says is resident (persistent kernels: no block waits
// for another, so a larger grid would only queue).
template <typename KernelOf>
LaunchShape pick_shape(int which, int threads, int maxc, int64_t rows, size_t unit_bytes,
                       size_t fixed_bytes, const int* opts, int n_opts, int want_stages,
                       int want_blocks, KernelOf kernel_of) {
  LaunchShape ls{};
  ls.threads = threads;
  ls.maxc = maxc;
  ls.cluster = 1;
  int stages = g_tune[which][0].load();
  int bps = g_tune[which][1].load();
  if (stages == 0) stages = want_stages;
  if (bps == 0) bps = want_blocks;
  auto fits = [&](int st, int bp) {
    const size_t per_block = st * unit_bytes + fixed_bytes;
    return per_block <= kSmemPerBlock && bp * (per_block + kReserve) <= kSmemPerSm;
  };
  bool ok = false;
  for (int bp = bps; bp >= 1 && !ok; --bp) {
    for (int i = 0; i < n_opts && !ok; ++i) {
      if (opts[i] > stages || !fits(opts[i], bp)) continue;
      stages = opts[i];
      bps = bp;
      ok = true;
    }
  }
  if (!ok) {
    stages = opts[n_opts - 1];
    bps = 1;
  }
  ls.fits = ok;
  ls.stages = stages;
  ls.smem = stages * unit_bytes + fixed_bytes;
  const void* fn = kernel_of(stages);
  int occ = bps;
  if (fn != nullptr && ensure_smem_attr(fn, ls.smem) == cudaSuccess) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, ls.threads, ls.smem) ==
            cudaSuccess &&
        n > 0 && n < occ)
      occ = n;
  }
  cudaGetLastError();
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * occ;
  ls.grid = static_cast<int>(rows < cap ? rows : cap);
  if (ls.grid < 1) ls.grid = 1;
  return ls;
}

const int kFwdStages[] = {3, 2};
const int kBwdRing[] = {3, 2, 1};   // rows staged; 1 = no prefetch (very wide rows)

// Forward threads per block: the first of 256, 128, 64 that splits the row's
// h/8 vectors into at least 2 full chunks (no thread idles in a last partial
// chunk, and the blocks fill an SM's 16 warps exactly), else 160 (three blocks
// per SM); measured on GB300, fewer chunks of more threads beat more chunks of
// fewer threads (h = 4096: 256 x 2 over 128 x 4 over 64 x 8).
int fwd_threads(int64_t h) {
  const int64_t nvec = h / 8;
  const int forced = g_tune[0][2].load();
  if (forced != 0 && fwd_kernel(forced, 0, 2) != nullptr) return forced;
  static const int opts[] = {256, 128, 64, 160};
  for (int n : opts)
    if (nvec % n == 0 && nvec / n >= 2) return n;
  return nvec <= 64 ? 64 : 256;
}

// Backward (threads, chunks per row): a shape that covers the row exactly,
// in this order of preference (measured on GB300): two chunks per thread with
// the parameter-gradient terms in registers (512, 256, 128 threads); for the
// mask-free variant at h = 8192, four chunks of 256 threads with the terms in
// tensor memory (its Philox draws need the registers); two chunks of 320
// threads with the terms in tensor memory (h = 5120: 20 warps per SM instead
// of one 640-thread block); one chunk (640, 512, 256, 64 threads).  Other h:
// the smallest register shape that covers the row.
void bwd_threads(int64_t h, bool regen, int* threads, int* maxc) {
  const int64_t nvec = h / 8;
  const int ft = g_tune[1][2].load(), fc = g_tune[1][3].load();
  if (ft != 0 && fc != 0 && static_cast<int64_t>(ft) * fc * 8 >= h &&
      bwd_kernel(ft, fc, 2) != nullptr) {
    *threads = ft;
    *maxc = fc;
    return;
  }
  if (regen && nvec == 1024) {
    *threads = 256;
    *maxc = 4;
    return;
  }
  static const int opts[][2] = {{512, 2}, {256, 2}, {128, 2}, {320, 2}, {640, 1},
                                {512, 1}, {256, 1}, {64, 1}};
  for (const auto& o : opts) {
    if (nvec == static_cast<int64_t>(o[0]) * o[1]) {
      *threads = o[0];
      *maxc = o[1];
      return;
    }
  }
  *threads = nvec <= 64 ? 64 : nvec <= 256 ? 256 : 512;
  *maxc = nvec <= 512 ? 1 : nvec <= 1024 ? 2 : 4;
}

// Forward: every compute thread owns 8 channels of each chunk of 8 * threads
// channels, and the block adds one copy-producer warp; one pipeline stage
// holds the chunk of the t partials and the residual, and the row's Z waits
// in shared memory for the statistics.
//
// Tuning option (sp_debug_tune, forward `chunks` = 2): each row split over a
// cluster of two CTAs, each handling h / 2 channels; the grid is then as many
// clusters as the occupancy calculator says can be resident at once.
LaunchShape fwd_shape_uncached(int64_t rows, int64_t h, int t) {
  int pair = (g_tune[0][3].load() == 2 && h % 16 == 0) ? 2 : 1;
  int threads = fwd_threads(h / pair);
  if (pair > 1 && fwd_kernel_pair(threads, t, 2) == nullptr) {
    pair = 1;
    threads = fwd_threads(h);
  }
  const int64_t hl = h / pair;
  const int64_t nchunk = (hl + 8 * threads - 1) / (8 * threads);
  const size_t stage = static_cast<size_t>(t + 1) * threads * 16;
  const size_t fixed = static_cast<size_t>(nchunk) * threads * 16 + 2 * 32 * sizeof(float2);
  auto kernel_of = [&](int st) {
    return pair > 1 ? fwd_kernel_pair(threads, t, st) : fwd_kernel(threads, t, st);
  };
  LaunchShape ls = pick_shape(0, threads + kFwdProducerThreads, static_cast<int>(nchunk), rows,
                              stage, fixed, kFwdStages, 2, /*stages=*/3,
                              /*blocks per SM=*/512 / threads, kernel_of);
  if (pair > 1) {
    ls.cluster = pair;
    int64_t clusters = ls.grid / pair;
    const void* fn = kernel_of(ls.stages);
    if (fn != nullptr) {
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = pair;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(pair);
      cfg.blockDim = dim3(ls.threads);
      cfg.dynamicSmemBytes = ls.smem;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) == cudaSuccess && n > 0) clusters = n;
      cudaGetLastError();
    }
    if (clusters > rows) clusters = rows;
    if (clusters < 1) clusters = 1;
    ls.grid = static_cast<int>(clusters * pair);
  }
  return ls;
}

// The shard-input variant of the forward: two streams per stage.
LaunchShape fwd_shard_shape_uncached(int64_t rows, int64_t h) {
  const int threads = fwd_threads(h);
  const int64_t nchunk = (h + 8 * threads - 1) / (8 * threads);
  const size_t stage = static_cast<size_t>(2) * threads * 16;
  const size_t fixed = static_cast<size_t>(nchunk) * threads * 16 + 2 * 32 * sizeof(float2);
  return pick_shape(0, threads + kFwdProducerThreads, static_cast<int>(nchunk), rows, stage,
                    fixed, kFwdStages, 2,
                    /*stages=*/3, /*blocks per SM=*/512 / threads,
                    [&](int st) { return fwd_shard_kernel(threads, st); });
}

// Backward: a ring of whole rows (dY, Z, mask unless regenerated, optional
// skip gradient).
// Backward entered through g: t partial-gradient pieces per chunk stage, two
// row buffers (Z, mask, skip), the reduced dY in float32.  The row buffers are
// double-buffered, which is safe while the prefetch reaches at most one row
// ahead: stages - 1 <= chunks per row.
LaunchShape rs_bwd_shape_uncached(int64_t rows, int64_t h, int t, bool has_skip, bool bits) {
  const int64_t nvec = h / 8;
  int threads, maxc;
  if (nvec <= 64) {
    threads = 64;
    maxc = 1;
  } else if (nvec <= 256) {
    threads = 256;
    maxc = 1;
  } else {
    threads = 512;
    maxc = static_cast<int>((nvec + 511) / 512);
  }
  const size_t v16 = static_cast<size_t>(threads) * 16;
  const size_t stage = static_cast<size_t>(t) * v16;
  const size_t rb_item = static_cast<size_t>(rsbwd_rb_item_bytes(threads, has_skip, bits));
  const size_t fixed = 2 * maxc * rb_item + static_cast<size_t>(maxc) * 2 * v16 +
                       2 * 32 * sizeof(float2);
  static const int kOpts[] = {3, 2, 1};
  const int want = maxc + 1 < 3 ? maxc + 1 : 3;
  return pick_shape(1, threads, maxc, rows, stage, fixed, kOpts, 3, want, 1, [&](int st) {
    return bits ? rs_bwd_bits_kernel(threads, maxc, t, st) : rs_bwd_kernel(threads, maxc, t, st);
  });
}

// bulk: dYpre sent to the gathered copies by bulk copies from two shared
// copies of the row (stored mask only), for calls with several copies.
LaunchShape bwd_shape_uncached(int64_t rows, int64_t h, bool has_skip, bool regen, bool bulk,
                               bool bits) {
  int threads, maxc;
  bwd_threads(h, regen, &threads, &maxc);
  const size_t item = static_cast<size_t>(bwd_item_bytes(threads, has_skip, regen, bits));
  const size_t ring_row = item * maxc;
  const size_t stage_row = static_cast<size_t>((h * 2 + 15) / 16) * 16;
  const size_t fixed = 2 * 32 * sizeof(float2) + (bulk ? 2 * stage_row : 0);
  const bool tacc = bwd_tmem_shape(threads, maxc);
  const int cap = tacc ? 512 / bwd_tmem_cols(threads, maxc) : (threads <= 256 ? 512 / threads : 1);
  // rows staged: three when one block holds the SM (measured on GB300, h = 8192:
  // 0.191 against 0.194 ms), else two
  LaunchShape ls = pick_shape(1, threads, maxc, rows, ring_row, fixed, kBwdRing,
                              3, /*ring=*/cap == 1 ? 3 : 2, /*blocks per SM=*/cap, [&](int st) {
                                return regen  ? bwd_regen_kernel(threads, maxc, st)
                                       : bits ? bwd_bits_kernel(threads, maxc, st)
                                       : bulk ? bwd_bulk_kernel(threads, maxc, st)
                                              : bwd_kernel(threads, maxc, st);
                              });
  if (tacc && ls.fits) {
    // The blocks of an SM share its 512 tensor-memory columns: pad the shared
    // memory so that no more than `cap` blocks can be resident on one SM (an
    // allocation beyond the columns would wait for a block to finish).
    const size_t floor = kSmemPerSm / (cap + 1) - kReserve + 16;
    if (ls.smem < floor) ls.smem = floor;
    ls.fits = ls.smem <= kSmemPerBlock;
    const int64_t most = static_cast<int64_t>(device_sm_count()) * cap;
    ls.grid = static_cast<int>(rows < most ? (rows > 0 ? rows : 1) : most);
  }
  return ls;
}

LaunchShape fwd_shape(int64_t rows, int64_t h, int t) {
  return cached_shape(0, rows, h, t, 0, [&] { return fwd_shape_uncached(rows, h, t); });
}

LaunchShape fwd_shard_shape(int64_t rows, int64_t h) {
  return cached_shape(1, rows, h, 1, 0, [&] { return fwd_shard_shape_uncached(rows, h); });
}

LaunchShape rs_bwd_shape(int64_t rows, int64_t h, int t, bool has_skip, bool bits = false) {
  return cached_shape(2, rows, h, t, (has_skip ? 1 : 0) | (bits ? 2 : 0),
                      [&] { return rs_bwd_shape_uncached(rows, h, t, has_skip, bits); });
}

LaunchShape bwd_shape(int64_t rows, int64_t h, bool has_skip, bool regen = false,
                      bool bulk = false, bool bits = false) {
  return cached_shape(3, rows, h, 0,
                      (has_skip ? 1 : 0) | (regen ? 2 : 0) | (bulk ? 4 : 0) | (bits ? 8 : 0),
                      [&] { return bwd_shape_uncached(rows, h, has_skip, regen, bulk, bits); });
}

cudaError_t launch(const void* fn, const LaunchShape& ls, void* params, cudaStream_t st) {
  if (fn == nullptr) return cudaErrorInvalidDeviceFunction;
  if (!ls.fits) return cudaErrorInvalidConfiguration;   // reported as SP_ERR_UNSUPPORTED
  cudaError_t e = ensure_smem_attr(fn, ls.smem);
  if (e != cudaSuccess) return e;
  void* args[] = {params};
  return launch_pdl(fn, dim3(ls.grid), dim3(ls.threads), ls.smem, args, st, ls.cluster);
}

}  // namespace

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, void** args,
                       cudaStream_t st, int cluster) {
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

sp_status_t record_error(sp_status_t code, const char* message) {
  return fail(code, "%s", message);
}

size_t stored_mask_bwd_workspace_bytes(int64_t rows, int64_t h, bool has_skip) {
  const LaunchShape ls = bwd_shape(rows, h, has_skip, false);
  return static_cast<size_t>(ls.grid) * 3 * static_cast<size_t>(h) * sizeof(float);
}

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 1;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = 1;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace spb

using namespace spb;

extern "C" {

// The fused forward with the mask stored as `maskf` (kMaskBytes, kMaskBits, or
// kMaskNone when mask_out is NULL).
static sp_status_t rs_norm_fwd_impl(const void* const* partials, const void* const* residual,
                                    const void* bias, const void* gamma, const void* beta,
                                    int64_t b, int64_t s, int64_t h, int32_t t, float eps,
                                    double p, uint64_t seed, uint64_t offset,
                                    const int32_t* cu_seqlens, int32_t n_seqs, sp_norm_t norm,
                                    void* const* z_out, uint8_t* const* mask_out, int maskf,
                                    float* const* mean_out, float* const* rstd_out,
                                    void* const* gathered, int32_t n_gather,
                                    int32_t* dev_status, void* stream) {
  sp_status_t st;
  const bool withhold = take_injected_timeout();
  if (take_injected(&st)) return st;
  if ((st = check_shape(b, s, h, t, cu_seqlens, n_seqs)) != SP_OK) return st;
  if (norm != SP_NORM_LAYERNORM && norm != SP_NORM_RMSNORM)
    return fail(SP_ERR_INVALID_ARG, "unknown norm %d", (int)norm);
  if (!(eps > 0.f) || !std::isfinite(eps)) return fail(SP_ERR_INVALID_ARG, "eps must be > 0");
  if (!(p >= 0.0 && p < 1.0)) return fail(SP_ERR_INVALID_ARG, "p = %g outside [0, 1)", p);
  if (n_gather < 0 || n_gather > SP_MAX_RANKS)
    return fail(SP_ERR_INVALID_ARG, "n_gather = %d outside [0, %d]", n_gather, SP_MAX_RANKS);
  const bool ln = norm == SP_NORM_LAYERNORM;
  if (b * s == 0) return SP_OK;   // nothing to read or write: any pointers are fine
  const ShardMap map = make_map(b, s, h, t);
  if ((st = check_ptrs(partials, t, "partials", true)) != SP_OK) return st;
  if ((st = check_ptrs(residual, t, "residual", true, &map)) != SP_OK) return st;
  if ((st = check_ptrs(z_out, t, "z_out", true, &map)) != SP_OK) return st;
  const bool store_mask = maskf != kMaskNone;
  if (store_mask && (st = check_ptrs(mask_out, t, "mask_out", true, &map)) != SP_OK) return st;
  if ((st = check_ptrs(rstd_out, t, "rstd_out", false, &map)) != SP_OK) return st;
  if (ln && (st = check_ptrs(mean_out, t, "mean_out", false, &map)) != SP_OK) return st;
  if ((st = check_ptrs(gathered, n_gather, "gathered", true)) != SP_OK) return st;
  if ((st = check_vec(bias, "bias")) != SP_OK) return st;
  if ((st = check_vec(gamma, "gamma")) != SP_OK) return st;
  if (ln && (st = check_vec(beta, "beta")) != SP_OK) return st;
  if (dev_status != nullptr && (reinterpret_cast<uintptr_t>(dev_status) & 3u))
    return fail(SP_ERR_MISALIGNED, "dev_status misaligned");

  const size_t full = static_cast<size_t>(b * s * h) * 2;
  Ranges rg;
  for (int r = 0; r < t; ++r) rg.add(partials[r], full, false, "partials", r);
  for (int k = 0; k < t; ++k) {
    const size_t n = static_cast<size_t>(shard_rows(map, k));
    rg.add(residual[k], n * h * 2, false, "residual", k);
    rg.add(z_out[k], n * h * 2, true, "z_out", k);
    if (store_mask)
      rg.add(mask_out[k], maskf == kMaskBits ? n * h / 8 : n * h, true, "mask_out", k);
    rg.add(rstd_out[k], n * 4, true, "rstd_out", k);
    if (ln) rg.add(mean_out[k], n * 4, true, "mean_out", k);
  }
  for (int j = 0; j < n_gather; ++j) rg.add(gathered[j], full, true, "gathered", j);
  rg.add(bias, h * 2, false, "bias", 0);
  rg.add(gamma, h * 2, false, "gamma", 0);
  if (ln) rg.add(beta, h * 2, false, "beta", 0);
  if ((st = rg.check()) != SP_OK) return st;

  const int64_t rows = b * s;
  if (rows == 0) return SP_OK;

  FwdParams P{};
  P.map = map;
  for (int r = 0; r < t; ++r) P.partials[r] = static_cast<const uint16_t*>(partials[r]);
  for (int k = 0; k < t; ++k) {
    P.residual[k] = static_cast<const uint16_t*>(residual[k]);
    P.z[k] = static_cast<uint16_t*>(z_out[k]);
    P.mask[k] = store_mask ? mask_out[k] : nullptr;
    P.rstd[k] = rstd_out[k];
    P.mean[k] = ln ? mean_out[k] : nullptr;
  }
  for (int j = 0; j < n_gather; ++j) P.gathered[j] = static_cast<uint16_t*>(gathered[j]);
  P.bias = static_cast<const uint16_t*>(bias);
  P.gamma = static_cast<const uint16_t*>(gamma);
  P.beta = ln ? static_cast<const uint16_t*>(beta) : nullptr;
  P.cu_seqlens = cu_seqlens;
  P.n_seqs = n_seqs;
  P.n_gather = n_gather;
  P.norm = norm;
  // keep iff draw >= floor(p * 2^32): the drop probability is thr / 2^32
  P.thr = static_cast<uint32_t>(std::floor(p * 4294967296.0));
  P.scale = static_cast<float>(1.0 / (1.0 - p));
  P.eps = eps;
  philox_round_keys(seed, &P.rk);
  P.off0 = static_cast<uint32_t>(offset);
  P.off1 = static_cast<uint32_t>(offset >> 32);
  P.rows = rows;
  P.status = dev_status;
  P.withhold = withhold ? 1 : 0;

  const LaunchShape ls = fwd_shape(rows, h, t);
  g_last_shape[0] = ls;
  const int threads = ls.threads - kFwdProducerThreads;
  if (maskf != kMaskBytes && ls.cluster > 1)
    return fail(SP_ERR_UNSUPPORTED, "the row split over a CTA pair (a tuning option) stores "
                "the mask one byte per element only");
  const void* fn = maskf == kMaskNone   ? fwd_nomask_kernel(threads, t, ls.stages)
                   : maskf == kMaskBits ? fwd_bits_kernel(threads, t, ls.stages)
                   : ls.cluster > 1     ? fwd_kernel_pair(threads, t, ls.stages)
                                        : fwd_kernel(threads, t, ls.stages);
  const cudaError_t e = launch(fn, ls, &P, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "sp_rs_norm_fwd launch");
  return SP_OK;
}

sp_status_t sp_rs_norm_fwd(const void* const* partials, const void* const* residual,
                           const void* bias, const void* gamma, const void* beta, int64_t b,
                           int64_t s, int64_t h, int32_t t, float eps, double p, uint64_t seed,
                           uint64_t offset, const int32_t* cu_seqlens, int32_t n_seqs,
                           sp_norm_t norm, void* const* z_out, uint8_t* const* mask_out,
                           float* const* mean_out, float* const* rstd_out,
                           void* const* gathered, int32_t n_gather, int32_t* dev_status,
                           void* stream) {
  return rs_norm_fwd_impl(partials, residual, bias, gamma, beta, b, s, h, t, eps, p, seed,
                          offset, cu_seqlens, n_seqs, norm, z_out, mask_out,
                          mask_out != nullptr ? kMaskBytes : kMaskNone, mean_out, rstd_out,
                          gathered, n_gather, dev_status, stream);
}

sp_status_t sp_rs_norm_fwd_bitmask(const void* const* partials, const void* const* residual,
                                   const void* bias, const void* gamma, const void* beta,
                                   int64_t b, int64_t s, int64_t h, int32_t t, float eps,
                                   double p, uint64_t seed, uint64_t offset,
                                   const int32_t* cu_seqlens, int32_t n_seqs, sp_norm_t norm,
                                   void* const* z_out, uint8_t* const* mask_bits_out,
                                   float* const* mean_out, float* const* rstd_out,
                                   void* const* gathered, int32_t n_gather,
                                   int32_t* dev_status, void* stream) {
  if (mask_bits_out == nullptr)
    return fail(SP_ERR_INVALID_ARG, "mask_bits_out array is NULL");
  if (h % 32 != 0)
    return fail(SP_ERR_UNSUPPORTED, "bit-packed mask: h = %lld must be a multiple of 32",
                (long long)h);
  return rs_norm_fwd_impl(partials, residual, bias, gamma, beta, b, s, h, t, eps, p, seed,
                          offset, cu_seqlens, n_seqs, norm, z_out, mask_bits_out, kMaskBits,
                          mean_out, rstd_out, gathered, n_gather, dev_status, stream);
}

sp_status_t sp_shard_norm_fwd(const void* const* y_shards, const void* const* residual,
                              const void* bias, const void* gamma, const void* beta, int64_t b,
                              int64_t s, int64_t h, int32_t t, float eps, double p,
                              uint64_t seed, uint64_t offset, const int32_t* cu_seqlens,
                              int32_t n_seqs, sp_norm_t norm, void* const* z_out,
                              uint8_t* const* mask_out, float* const* mean_out,
                              float* const* rstd_out, void* const* o_shards,
                              int32_t* dev_status, void* stream) {
  sp_status_t st;
  const bool withhold = take_injected_timeout();
  if (take_injected(&st)) return st;
  if ((st = check_shape(b, s, h, t, cu_seqlens, n_seqs)) != SP_OK) return st;
  if (norm != SP_NORM_LAYERNORM && norm != SP_NORM_RMSNORM)
    return fail(SP_ERR_INVALID_ARG, "unknown norm %d", (int)norm);
  if (!(eps > 0.f) || !std::isfinite(eps)) return fail(SP_ERR_INVALID_ARG, "eps must be > 0");
  if (!(p >= 0.0 && p < 1.0)) return fail(SP_ERR_INVALID_ARG, "p = %g outside [0, 1)", p);
  const bool ln = norm == SP_NORM_LAYERNORM;
  if (b * s == 0) return SP_OK;
  const ShardMap map = make_map(b, s, h, t);
  if ((st = check_ptrs(y_shards, t, "y_shards", true, &map)) != SP_OK) return st;
  if ((st = check_ptrs(residual, t, "residual", true, &map)) != SP_OK) return st;
  if ((st = check_ptrs(z_out, t, "z_out", true, &map)) != SP_OK) return st;
  const bool store_mask = mask_out != nullptr;
  if (store_mask && (st = check_ptrs(mask_out, t, "mask_out", true, &map)) != SP_OK) return st;
  if ((st = check_ptrs(rstd_out, t, "rstd_out", false, &map)) != SP_OK) return st;
  if (ln && (st = check_ptrs(mean_out, t, "mean_out", false, &map)) != SP_OK) return st;
  if ((st = check_ptrs(o_shards, t, "o_shards", true, &map)) != SP_OK) return st;
  if ((st = check_vec(bias, "bias")) != SP_OK) return st;
  if ((st = check_vec(gamma, "gamma")) != SP_OK) return st;
  if (ln && (st = check_vec(beta, "beta")) != SP_OK) return st;
  if (dev_status != nullptr && (reinterpret_cast<uintptr_t>(dev_status) & 3u))
    return fail(SP_ERR_MISALIGNED, "dev_status misaligned");
  Ranges rg;
  for (int k = 0; k < t; ++k) {
    const size_t n = static_cast<size_t>(shard_rows(map, k));
    rg.add(y_shards[k], n * h * 2, false, "y_shards", k);
    rg.add(residual[k], n * h * 2, false, "residual", k);
    rg.add(z_out[k], n * h * 2, true, "z_out", k);
    if (store_mask) rg.add(mask_out[k], n * h, true, "mask_out", k);
    rg.add(rstd_out[k], n * 4, true, "rstd_out", k);
    if (ln) rg.add(mean_out[k], n * 4, true, "mean_out", k);
    rg.add(o_shards[k], n * h * 2, true, "o_shards", k);
  }
  rg.add(bias, h * 2, false, "bias", 0);
  rg.add(gamma, h * 2, false, "gamma", 0);
  if (ln) rg.add(beta, h * 2, false, "beta", 0);
  if ((st = rg.check()) != SP_OK) return st;

  FwdParams P{};
  P.map = map;
  for (int k = 0; k < t; ++k) {
    P.partials[k] = static_cast<const uint16_t*>(y_shards[k]);
    P.residual[k] = static_cast<const uint16_t*>(residual[k]);
    P.z[k] = static_cast<uint16_t*>(z_out[k]);
    P.mask[k] = store_mask ? mask_out[k] : nullptr;
    P.rstd[k] = rstd_out[k];
    P.mean[k] = ln ? mean_out[k] : nullptr;
    P.gathered[k] = static_cast<uint16_t*>(o_shards[k]);
  }
  P.bias = static_cast<const uint16_t*>(bias);
  P.gamma = static_cast<const uint16_t*>(gamma);
  P.beta = ln ? static_cast<const uint16_t*>(beta) : nullptr;
  P.cu_seqlens = cu_seqlens;
  P.n_seqs = n_seqs;
  P.n_gather = t;
  P.norm = norm;
  P.thr = static_cast<uint32_t>(std::floor(p * 4294967296.0));
  P.scale = static_cast<float>(1.0 / (1.0 - p));
  P.eps = eps;
  philox_round_keys(seed, &P.rk);
  P.off0 = static_cast<uint32_t>(offset);
  P.off1 = static_cast<uint32_t>(offset >> 32);
  P.rows = b * s;
  P.status = dev_status;
  P.withhold = withhold ? 1 : 0;
  const LaunchShape ls = fwd_shard_shape(P.rows, h);
  const int threads = ls.threads - kFwdProducerThreads;
  const void* fn = store_mask ? fwd_shard_kernel(threads, ls.stages)
                              : fwd_shard_nomask_kernel(threads, ls.stages);
  const cudaError_t e = launch(fn, ls, &P, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "sp_shard_norm_fwd launch");
  return SP_OK;
}

static sp_status_t seq_copy_common(const void* const* src, int n_src, const char* src_name,
                                   bool src_full, void* const* dst, int n_dst,
                                   const char* dst_name, bool dst_full, int64_t b, int64_t s,
                                   int64_t h, int32_t t, const int32_t* cu_seqlens,
                                   int32_t n_seqs, int32_t* dev_status, CopyParams* P) {
  sp_status_t st;
  if ((st = check_shape(b, s, h, t, cu_seqlens, n_seqs)) != SP_OK) return st;
  *P = CopyParams{};
  P->rows = b * s;
  if (P->rows == 0) return SP_OK;   // nothing to copy: any pointers are fine
  const ShardMap map = make_map(b, s, h, t);
  if ((st = check_ptrs(src, n_src, src_name, true, src_full ? nullptr : &map)) != SP_OK) return st;
  if ((st = check_ptrs(dst, n_dst, dst_name, true, dst_full ? nullptr : &map)) != SP_OK) return st;
  if (dev_status != nullptr && (reinterpret_cast<uintptr_t>(dev_status) & 3u))
    return fail(SP_ERR_MISALIGNED, "dev_status misaligned");
  const size_t full = static_cast<size_t>(b * s * h) * 2;
  Ranges rg;
  for (int i = 0; i < n_src; ++i)
    rg.add(src[i], src_full ? full : shard_rows(map, i) * h * 2, false, src_name, i);
  for (int i = 0; i < n_dst; ++i)
    rg.add(dst[i], dst_full ? full : shard_rows(map, i) * h * 2, true, dst_name, i);
  if ((st = rg.check()) != SP_OK) return st;
  P->map = map;
  for (int i = 0; i < n_src; ++i) P->src[i] = static_cast<const uint16_t*>(src[i]);
  for (int i = 0; i < n_dst; ++i) P->dst[i] = static_cast<uint16_t*>(dst[i]);
  P->n_dst = n_dst;
  P->cu_seqlens = cu_seqlens;
  P->n_seqs = n_seqs;
  P->status = dev_status;
  return SP_OK;
}

sp_status_t sp_allgather_seq(const void* const* shards, int64_t b, int64_t s, int64_t h,
                             int32_t t, const int32_t* cu_seqlens, int32_t n_seqs,
                             void* const* gathered, int32_t n_gather, int32_t* dev_status,
                             void* stream) {
  sp_status_t st;
  if (take_injected(&st)) return st;
  if (n_gather < 1 || n_gather > SP_MAX_RANKS)
    return fail(SP_ERR_INVALID_ARG, "n_gather = %d outside [1, %d]", n_gather, SP_MAX_RANKS);
  CopyParams P;
  if ((st = seq_copy_common(shards, t, "shards", false, gathered, n_gather, "gathered", true, b,
                            s, h, t, cu_seqlens, n_seqs, dev_status, &P)) != SP_OK)
    return st;
  if (P.rows == 0) return SP_OK;
  const cudaError_t e = launch_allgather(P, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "sp_allgather_seq launch");
  return SP_OK;
}

sp_status_t sp_reduce_scatter_seq(const void* const* partials, int64_t b, int64_t s, int64_t h,
                                  int32_t t, const int32_t* cu_seqlens, int32_t n_seqs,
                                  void* const* shards, int32_t* dev_status, void* stream) {
  sp_status_t st;
  if (take_injected(&st)) return st;
  CopyParams P;
  if ((st = seq_copy_common(partials, t, "partials", true, shards, t, "shards", false, b, s, h,
                            t, cu_seqlens, n_seqs, dev_status, &P)) != SP_OK)
    return st;
  if (P.rows == 0) return SP_OK;
  const cudaError_t e = launch_reduce_scatter(P, t, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "sp_reduce_scatter_seq launch");
  return SP_OK;
}

size_t sp_norm_bwd_workspace_bytes(int64_t b, int64_t s, int64_t h, int32_t t, sp_norm_t norm) {
  (void)norm;
  if (b <= 0 || s <= 0 || h < 8 || h % 8 != 0 || h > SP_MAX_HIDDEN || t < 1 || t > SP_MAX_RANKS)
    return 0;
  // the largest grid over the variants (skip gradient or not; stored mask,
  // regenerated mask, or dYpre sent by bulk copies): one workspace size serves
  // every backward entry point
  int grid = 0;
  for (int v = 0; v < 8; ++v) {   // skip gradient or not; byte mask, drawn again, bulk, bits
    const LaunchShape ls = bwd_shape(b * s, h, (v & 1) != 0, (v >> 1) == 1, (v >> 1) == 2,
                                     (v >> 1) == 3);
    if (ls.grid > grid) grid = ls.grid;
  }
  if (h <= 8192) {
    for (int v = 0; v < 4; ++v) {   // skip gradient or not; byte or bit mask
      const LaunchShape ls = rs_bwd_shape(b * s, h, t, (v & 1) != 0, (v & 2) != 0 && h % 32 == 0);
      if (ls.grid > grid) grid = ls.grid;
    }
  }
  return static_cast<size_t>(grid) * 3 * static_cast<size_t>(h) * sizeof(float);
}

static sp_status_t norm_bwd_common(
    const void* const* dy, const void* const* z, const uint8_t* const* mask,
    const float* const* mean, const float* const* rstd, const void* gamma,
    const void* const* dz_skip, int64_t b, int64_t s, int64_t h, int32_t t, double p,
    bool regen, bool bits, uint64_t seed, uint64_t offset, const int32_t* cu_seqlens,
    int32_t n_seqs,
    sp_norm_t norm, void* const* dresidual, void* const* dgathered, int32_t n_gather,
    float* dgamma, float* dbeta, float* dbias, void* workspace, size_t workspace_bytes,
    int32_t* dev_status, void* stream) {
  sp_status_t st;
  if ((st = check_shape(b, s, h, t, cu_seqlens, n_seqs)) != SP_OK) return st;
  if (norm != SP_NORM_LAYERNORM && norm != SP_NORM_RMSNORM)
    return fail(SP_ERR_INVALID_ARG, "unknown norm %d", (int)norm);
  if (!(p >= 0.0 && p < 1.0)) return fail(SP_ERR_INVALID_ARG, "p = %g outside [0, 1)", p);
  if (n_gather < 0 || n_gather > SP_MAX_RANKS)
    return fail(SP_ERR_INVALID_ARG, "n_gather = %d outside [0, %d]", n_gather, SP_MAX_RANKS);
  const bool ln = norm == SP_NORM_LAYERNORM;
  const int64_t rows = b * s;
  if (dgamma != nullptr && !aligned16(dgamma)) return fail(SP_ERR_MISALIGNED, "dgamma misaligned");
  if (dbeta != nullptr && !aligned16(dbeta)) return fail(SP_ERR_MISALIGNED, "dbeta misaligned");
  if (dbias != nullptr && !aligned16(dbias)) return fail(SP_ERR_MISALIGNED, "dbias misaligned");
  if (rows == 0) {
    // no token: the parameter gradients are exact zeros, nothing else is touched
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (dgamma) e = cudaMemsetAsync(dgamma, 0, h * 4, cs);
    if (e == cudaSuccess && dbeta && ln) e = cudaMemsetAsync(dbeta, 0, h * 4, cs);
    if (e == cudaSuccess && dbias) e = cudaMemsetAsync(dbias, 0, h * 4, cs);
    if (e != cudaSuccess) return fail_cuda(e, "sp_norm_bwd zero fill");
    return SP_OK;
  }
  const ShardMap map = make_map(b, s, h, t);
  if ((st = check_ptrs(dy, t, "dy", true, &map)) != SP_OK) return st;
  if ((st = check_ptrs(z, t, "z", true, &map)) != SP_OK) return st;
  if (!regen && (st = check_ptrs(mask, t, "mask", true, &map)) != SP_OK) return st;
  if ((st = check_ptrs(rstd, t, "rstd", false, &map)) != SP_OK) return st;
  if (ln && (st = check_ptrs(mean, t, "mean", false, &map)) != SP_OK) return st;
  if (dz_skip != nullptr && (st = check_ptrs(dz_skip, t, "dz_skip", true, &map)) != SP_OK)
    return st;
  if ((st = check_ptrs(dresidual, t, "dresidual", true, &map)) != SP_OK) return st;
  if ((st = check_ptrs(dgathered, n_gather, "dgathered", true)) != SP_OK) return st;
  if ((st = check_vec(gamma, "gamma")) != SP_OK) return st;
  if (dev_status != nullptr && (reinterpret_cast<uintptr_t>(dev_status) & 3u))
    return fail(SP_ERR_MISALIGNED, "dev_status misaligned");

  const bool has_skip = dz_skip != nullptr;
  // several gathered copies: the bulk-copy variant, if its shape fits (byte
  // mask only)
  bool bulk = !regen && !bits && n_gather > 1;
  LaunchShape ls = bwd_shape(rows, h, has_skip, regen, bulk, bits);
  if (bulk && !ls.fits) {
    bulk = false;
    ls = bwd_shape(rows, h, has_skip, regen, false, bits);
  }
  g_last_shape[1] = ls;
  const size_t need = static_cast<size_t>(ls.grid) * 3 * h * sizeof(float);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(SP_ERR_INVALID_ARG, "workspace of %zu bytes needed (got %zu)", need,
                workspace == nullptr ? (size_t)0 : workspace_bytes);
  if (!aligned16(workspace)) return fail(SP_ERR_MISALIGNED, "workspace misaligned");

  const size_t full = static_cast<size_t>(rows * h) * 2;
  Ranges rg;
  for (int k = 0; k < t; ++k) {
    const size_t n = static_cast<size_t>(shard_rows(map, k));
    rg.add(dy[k], n * h * 2, false, "dy", k);
    rg.add(z[k], n * h * 2, false, "z", k);
    if (!regen) rg.add(mask[k], bits ? n * h / 8 : n * h, false, "mask", k);
    rg.add(rstd[k], n * 4, false, "rstd", k);
    if (ln) rg.add(mean[k], n * 4, false, "mean", k);
    if (has_skip) rg.add(dz_skip[k], n * h * 2, false, "dz_skip", k);
    rg.add(dresidual[k], n * h * 2, true, "dresidual", k);
  }
  for (int j = 0; j < n_gather; ++j) rg.add(dgathered[j], full, true, "dgathered", j);
  rg.add(gamma, h * 2, false, "gamma", 0);
  rg.add(dgamma, h * 4, true, "dgamma", 0);
  if (ln) rg.add(dbeta, h * 4, true, "dbeta", 0);
  rg.add(dbias, h * 4, true, "dbias", 0);
  rg.add(workspace, need, true, "workspace", 0);
  if ((st = rg.check()) != SP_OK) return st;

  BwdParams P{};
  P.map = map;
  for (int k = 0; k < t; ++k) {
    P.dy[k] = static_cast<const uint16_t*>(dy[k]);
    P.z[k] = static_cast<const uint16_t*>(z[k]);
    P.mask[k] = regen ? nullptr : mask[k];
    P.rstd[k] = rstd[k];
    P.mean[k] = ln ? mean[k] : nullptr;
    P.dz_skip[k] = has_skip ? static_cast<const uint16_t*>(dz_skip[k]) : nullptr;
    P.dresidual[k] = static_cast<uint16_t*>(dresidual[k]);
  }
  for (int j = 0; j < n_gather; ++j) P.dgathered[j] = static_cast<uint16_t*>(dgathered[j]);
  P.gamma = static_cast<const uint16_t*>(gamma);
  P.cu_seqlens = cu_seqlens;
  P.n_seqs = n_seqs;
  P.n_gather = n_gather;
  P.norm = norm;
  P.has_skip = has_skip ? 1 : 0;
  P.scale = static_cast<float>(1.0 / (1.0 - p));
  // same keep rule as the forward: keep iff draw >= floor(p * 2^32)
  P.thr = static_cast<uint32_t>(std::floor(p * 4294967296.0));
  philox_round_keys(seed, &P.rk);
  P.off0 = static_cast<uint32_t>(offset);
  P.off1 = static_cast<uint32_t>(offset >> 32);
  P.rows = rows;
  P.ws = static_cast<float*>(workspace);
  P.status = dev_status;

  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const void* fn = regen ? bwd_regen_kernel(ls.threads, ls.maxc, ls.stages)
                   : bits  ? bwd_bits_kernel(ls.threads, ls.maxc, ls.stages)
                   : bulk  ? bwd_bulk_kernel(ls.threads, ls.maxc, ls.stages)
                           : bwd_kernel(ls.threads, ls.maxc, ls.stages);
  cudaError_t e = launch(fn, ls, &P, cs);
  if (e != cudaSuccess) return fail_cuda(e, "sp_norm_bwd launch");
  if (dgamma || (dbeta && ln) || dbias) {
    ParamReduceParams R{};
    R.ws = P.ws;
    R.nblk = ls.grid;
    R.h = h;
    R.out[0] = dgamma;
    R.out[1] = ln ? dbeta : nullptr;
    R.out[2] = dbias;
    e = launch_param_reduce(R, cs);
    if (e != cudaSuccess) return fail_cuda(e, "sp_norm_bwd parameter reduce launch");
  }
  return SP_OK;
}

// The backward entered through g, reading the mask as bytes or (bits) one
// bit per element.
static sp_status_t rs_norm_bwd_impl(const void* const* dy_partials, const void* const* z,
                                    const uint8_t* const* mask, bool bits, const float* const* mean,
                                    const float* const* rstd, const void* gamma,
                                    const void* const* dz_skip, int64_t b, int64_t s, int64_t h,
                                    int32_t t, double p, const int32_t* cu_seqlens,
                                    int32_t n_seqs, sp_norm_t norm, void* const* dresidual,
                                    void* const* dgathered, int32_t n_gather, float* dgamma,
                                    float* dbeta, float* dbias, void* workspace,
                                    size_t workspace_bytes, int32_t* dev_status, void* stream) {
  sp_status_t st;
  if (take_injected(&st)) return st;
  if ((st = check_shape(b, s, h, t, cu_seqlens, n_seqs)) != SP_OK) return st;
  if (h > 8192)
    return fail(SP_ERR_UNSUPPORTED, "sp_rs_norm_bwd: h = %lld above 8192", (long long)h);
  if (norm != SP_NORM_LAYERNORM && norm != SP_NORM_RMSNORM)
    return fail(SP_ERR_INVALID_ARG, "unknown norm %d", (int)norm);
  if (!(p >= 0.0 && p < 1.0)) return fail(SP_ERR_INVALID_ARG, "p = %g outside [0, 1)", p);
  if (n_gather < 0 || n_gather > SP_MAX_RANKS)
    return fail(SP_ERR_INVALID_ARG, "n_gather = %d outside [0, %d]", n_gather, SP_MAX_RANKS);
  const bool ln = norm == SP_NORM_LAYERNORM;
  const int64_t rows = b * s;
  if (dgamma != nullptr && !aligned16(dgamma)) return fail(SP_ERR_MISALIGNED, "dgamma misaligned");
  if (dbeta != nullptr && !aligned16(dbeta)) return fail(SP_ERR_MISALIGNED, "dbeta misaligned");
  if (dbias != nullptr && !aligned16(dbias)) return fail(SP_ERR_MISALIGNED, "dbias misaligned");
  if (rows == 0) {
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (dgamma) e = cudaMemsetAsync(dgamma, 0, h * 4, cs);
    if (e == cudaSuccess && dbeta && ln) e = cudaMemsetAsync(dbeta, 0, h * 4, cs);
    if (e == cudaSuccess && dbias) e = cudaMemsetAsync(dbias, 0, h * 4, cs);
    if (e != cudaSuccess) return fail_cuda(e, "sp_rs_norm_bwd zero fill");
    return SP_OK;
  }
  const ShardMap map = make_map(b, s, h, t);
  if ((st = check_ptrs(dy_partials, t, "dy_partials", true)) != SP_OK) return st;
  if ((st = check_ptrs(z, t, "z", true, &map)) != SP_OK) return st;
  if ((st = check_ptrs(mask, t, "mask", true, &map)) != SP_OK) return st;
  if ((st = check_ptrs(rstd, t, "rstd", false, &map)) != SP_OK) return st;
  if (ln && (st = check_ptrs(mean, t, "mean", false, &map)) != SP_OK) return st;
  if (dz_skip != nullptr && (st = check_ptrs(dz_skip, t, "dz_skip", true, &map)) != SP_OK)
    return st;
  if ((st = check_ptrs(dresidual, t, "dresidual", true, &map)) != SP_OK) return st;
  if ((st = check_ptrs(dgathered, n_gather, "dgathered", true)) != SP_OK) return st;
  if ((st = check_vec(gamma, "gamma")) != SP_OK) return st;
  if (dev_status != nullptr && (reinterpret_cast<uintptr_t>(dev_status) & 3u))
    return fail(SP_ERR_MISALIGNED, "dev_status misaligned");
  const bool has_skip = dz_skip != nullptr;
  const LaunchShape ls = rs_bwd_shape(rows, h, t, has_skip, bits);
  g_last_shape[1] = ls;
  const size_t need = static_cast<size_t>(ls.grid) * 3 * h * sizeof(float);
  if (workspace == nullptr || workspace_bytes < need)
    return fail(SP_ERR_INVALID_ARG, "workspace of %zu bytes needed (got %zu)", need,
                workspace == nullptr ? (size_t)0 : workspace_bytes);
  if (!aligned16(workspace)) return fail(SP_ERR_MISALIGNED, "workspace misaligned");
  const size_t full = static_cast<size_t>(rows * h) * 2;
  Ranges rg;
  for (int r = 0; r < t; ++r) rg.add(dy_partials[r], full, false, "dy_partials", r);
  for (int k = 0; k < t; ++k) {
    const size_t n = static_cast<size_t>(shard_rows(map, k));
    rg.add(z[k], n * h * 2, false, "z", k);
    rg.add(mask[k], bits ? n * h / 8 : n * h, false, "mask", k);
    rg.add(rstd[k], n * 4, false, "rstd", k);
    if (ln) rg.add(mean[k], n * 4, false, "mean", k);
    if (has_skip) rg.add(dz_skip[k], n * h * 2, false, "dz_skip", k);
    rg.add(dresidual[k], n * h * 2, true, "dresidual", k);
  }
  for (int j = 0; j < n_gather; ++j) rg.add(dgathered[j], full, true, "dgathered", j);
  rg.add(gamma, h * 2, false, "gamma", 0);
  rg.add(dgamma, h * 4, true, "dgamma", 0);
  if (ln) rg.add(dbeta, h * 4, true, "dbeta", 0);
  rg.add(dbias, h * 4, true, "dbias", 0);
  rg.add(workspace, need, true, "workspace", 0);
  if ((st = rg.check()) != SP_OK) return st;

  BwdParams P{};
  P.map = map;
  for (int r = 0; r < t; ++r) P.dy[r] = static_cast<const uint16_t*>(dy_partials[r]);
  for (int k = 0; k < t; ++k) {
    P.z[k] = static_cast<const uint16_t*>(z[k]);
    P.mask[k] = mask[k];
    P.rstd[k] = rstd[k];
    P.mean[k] = ln ? mean[k] : nullptr;
    P.dz_skip[k] = has_skip ? static_cast<const uint16_t*>(dz_skip[k]) : nullptr;
    P.dresidual[k] = static_cast<uint16_t*>(dresidual[k]);
  }
  for (int j = 0; j < n_gather; ++j) P.dgathered[j] = static_cast<uint16_t*>(dgathered[j]);
  P.gamma = static_cast<const uint16_t*>(gamma);
  P.cu_seqlens = cu_seqlens;
  P.n_seqs = n_seqs;
  P.n_gather = n_gather;
  P.norm = norm;
  P.has_skip = has_skip ? 1 : 0;
  P.scale = static_cast<float>(1.0 / (1.0 - p));
  P.rows = rows;
  P.ws = static_cast<float*>(workspace);
  P.status = dev_status;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch(bits ? rs_bwd_bits_kernel(ls.threads, ls.maxc, t, ls.stages)
                             : rs_bwd_kernel(ls.threads, ls.maxc, t, ls.stages),
                        ls, &P, cs);
  if (e != cudaSuccess) return fail_cuda(e, "sp_rs_norm_bwd launch");
  if (dgamma || (dbeta && ln) || dbias) {
    ParamReduceParams R{};
    R.ws = P.ws;
    R.nblk = ls.grid;
    R.h = h;
    R.out[0] = dgamma;
    R.out[1] = ln ? dbeta : nullptr;
    R.out[2] = dbias;
    e = launch_param_reduce(R, cs);
    if (e != cudaSuccess) return fail_cuda(e, "sp_rs_norm_bwd parameter reduce launch");
  }
  return SP_OK;
}

sp_status_t sp_rs_norm_bwd(const void* const* dy_partials, const void* const* z,
                           const uint8_t* const* mask, const float* const* mean,
                           const float* const* rstd, const void* gamma,
                           const void* const* dz_skip, int64_t b, int64_t s, int64_t h,
                           int32_t t, double p, const int32_t* cu_seqlens, int32_t n_seqs,
                           sp_norm_t norm, void* const* dresidual, void* const* dgathered,
                           int32_t n_gather, float* dgamma, float* dbeta, float* dbias,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           void* stream) {
  return rs_norm_bwd_impl(dy_partials, z, mask, false, mean, rstd, gamma, dz_skip, b, s, h, t,
                          p, cu_seqlens, n_seqs, norm, dresidual, dgathered, n_gather, dgamma,
                          dbeta, dbias, workspace, workspace_bytes, dev_status, stream);
}

sp_status_t sp_rs_norm_bwd_bitmask(const void* const* dy_partials, const void* const* z,
                                   const uint8_t* const* mask_bits, const float* const* mean,
                                   const float* const* rstd, const void* gamma,
                                   const void* const* dz_skip, int64_t b, int64_t s, int64_t h,
                                   int32_t t, double p, const int32_t* cu_seqlens,
                                   int32_t n_seqs, sp_norm_t norm, void* const* dresidual,
                                   void* const* dgathered, int32_t n_gather, float* dgamma,
                                   float* dbeta, float* dbias, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (h % 32 != 0)
    return fail(SP_ERR_UNSUPPORTED, "bit-packed mask: h = %lld must be a multiple of 32",
                (long long)h);
  return rs_norm_bwd_impl(dy_partials, z, mask_bits, true, mean, rstd, gamma, dz_skip, b, s, h,
                          t, p, cu_seqlens, n_seqs, norm, dresidual, dgathered, n_gather, dgamma,
                          dbeta, dbias, workspace, workspace_bytes, dev_status, stream);
}

sp_status_t sp_norm_bwd(const void* const* dy, const void* const* z, const uint8_t* const* mask,
                        const float* const* mean, const float* const* rstd, const void* gamma,
                        const void* const* dz_skip, int64_t b, int64_t s, int64_t h, int32_t t,
                        double p, const int32_t* cu_seqlens, int32_t n_seqs, sp_norm_t norm,
                        void* const* dresidual, void* const* dgathered, int32_t n_gather,
                        float* dgamma, float* dbeta, float* dbias, void* workspace,
                        size_t workspace_bytes, int32_t* dev_status, void* stream) {
  sp_status_t st;
  if (take_injected(&st)) return st;
  return norm_bwd_common(dy, z, mask, mean, rstd, gamma, dz_skip, b, s, h, t, p, false, false,
                         0, 0, cu_seqlens, n_seqs, norm, dresidual, dgathered, n_gather, dgamma,
                         dbeta, dbias, workspace, workspace_bytes, dev_status, stream);
}

sp_status_t sp_norm_bwd_bitmask(const void* const* dy, const void* const* z,
                                const uint8_t* const* mask_bits, const float* const* mean,
                                const float* const* rstd, const void* gamma,
                                const void* const* dz_skip, int64_t b, int64_t s, int64_t h,
                                int32_t t, double p, const int32_t* cu_seqlens, int32_t n_seqs,
                                sp_norm_t norm, void* const* dresidual, void* const* dgathered,
                                int32_t n_gather, float* dgamma, float* dbeta, float* dbias,
                                void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                void* stream) {
  sp_status_t st;
  if (take_injected(&st)) return st;
  if (h % 32 != 0)
    return fail(SP_ERR_UNSUPPORTED, "bit-packed mask: h = %lld must be a multiple of 32",
                (long long)h);
  return norm_bwd_common(dy, z, mask_bits, mean, rstd, gamma, dz_skip, b, s, h, t, p, false,
                         true, 0, 0, cu_seqlens, n_seqs, norm, dresidual, dgathered, n_gather,
                         dgamma, dbeta, dbias, workspace, workspace_bytes, dev_status, stream);
}

sp_status_t sp_norm_bwd_philox(const void* const* dy, const void* const* z,
                               const float* const* mean, const float* const* rstd,
                               const void* gamma, const void* const* dz_skip, int64_t b,
                               int64_t s, int64_t h, int32_t t, double p, uint64_t seed,
                               uint64_t offset, const int32_t* cu_seqlens, int32_t n_seqs,
                               sp_norm_t norm, void* const* dresidual, void* const* dgathered,
                               int32_t n_gather, float* dgamma, float* dbeta, float* dbias,
                               void* workspace, size_t workspace_bytes, int32_t* dev_status,
                               void* stream) {
  sp_status_t st;
  if (take_injected(&st)) return st;
  return norm_bwd_common(dy, z, nullptr, mean, rstd, gamma, dz_skip, b, s, h, t, p, true, false,
                         seed, offset, cu_seqlens, n_seqs, norm, dresidual, dgathered, n_gather,
                         dgamma, dbeta, dbias, workspace, workspace_bytes, dev_status, stream);
}

const char* sp_last_error(void) { return g_err; }

int32_t sp_abi_version(void) { return SP_ABI_VERSION; }

sp_status_t sp_debug_inject(sp_status_t code) {
  g_inject.store(static_cast<int>(code));
  return SP_OK;
}

sp_status_t sp_debug_tune(int32_t kernel, int32_t stages, int32_t blocks_per_sm,
                          int32_t threads, int32_t chunks) {
  if (kernel < 0 || kernel > 1 || stages < 0 || stages > 8 || blocks_per_sm < 0 ||
      blocks_per_sm > 16 || threads < 0 || threads > 1024 || chunks < 0 || chunks > 8)
    return fail(SP_ERR_INVALID_ARG, "sp_debug_tune: bad arguments");
  g_tune[kernel][0].store(stages);
  g_tune[kernel][1].store(blocks_per_sm);
  g_tune[kernel][2].store(threads);
  g_tune[kernel][3].store(chunks);
  g_tune_epoch.fetch_add(1);   // cached launch shapes are stale now
  return SP_OK;
}

sp_status_t sp_debug_last_shape(int32_t kernel, int32_t* out) {
  if ((kernel != 0 && kernel != 1) || out == nullptr)
    return fail(SP_ERR_INVALID_ARG, "sp_debug_last_shape: bad arguments");
  const LaunchShape& ls = g_last_shape[kernel];
  out[0] = kernel == 0 && ls.threads > 0 ? ls.threads - kFwdProducerThreads : ls.threads;
  out[1] = ls.maxc;
  out[2] = ls.stages;
  out[3] = ls.grid;
  out[4] = ls.cluster;
  out[5] = static_cast<int32_t>(ls.smem);
  return SP_OK;
}

sp_status_t sp_debug_philox(const uint32_t* in, uint32_t* out, int64_t n, void* stream) {
  sp_status_t st;
  if (take_injected(&st)) return st;
  if (n < 0) return fail(SP_ERR_INVALID_ARG, "n < 0");
  if (n == 0) return SP_OK;
  if (in == nullptr || out == nullptr) return fail(SP_ERR_INVALID_ARG, "NULL buffer");
  const cudaError_t e = launch_debug_philox(in, out, n, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "sp_debug_philox launch");
  return SP_OK;
}

}  // extern "C"
