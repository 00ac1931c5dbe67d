// Device helpers for the SP boundary kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "sp_internal.h"

namespace spb {

// ----------------------------------------------------------------- Philox --
// Philox4x32-10: per round, two 32x32->64-bit multiplies of counter words 0
// and 2 by the fixed odd multipliers; the high halves are xored with the
// other two counter words and the round key.  The round keys come from the
// kernel parameters (one constant operand of each xor, no key arithmetic).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKeys& rk) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint64_t p0 = static_cast<uint64_t>(kPhiloxMul0) * c.x;
    const uint64_t p1 = static_cast<uint64_t>(kPhiloxMul1) * c.z;
    const uint32_t hi0 = static_cast<uint32_t>(p0 >> 32), lo0 = static_cast<uint32_t>(p0);
    const uint32_t hi1 = static_cast<uint32_t>(p1 >> 32), lo1 = static_cast<uint32_t>(p1);
    c = make_uint4(hi1 ^ c.y ^ rk.k0[round], lo1, hi0 ^ c.w ^ rk.k1[round], lo0);
  }
  return c;
}

// The same from a bare key (k0, k1): the round keys are derived first.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
  PhiloxKeys rk;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    rk.k0[round] = k0;
    rk.k1[round] = k1;
    k0 += kPhiloxWeyl0;
    k1 += kPhiloxWeyl1;
  }
  return philox4x32_10(c, rk);
}

// ------------------------------------------------------------------- bf16 --
__device__ __forceinline__ void unpack8(const uint4 v, float f[8]) {
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xFFFF0000u);
  f[4] = __uint_as_float(v.z << 16);
  f[5] = __uint_as_float(v.z & 0xFFFF0000u);
  f[6] = __uint_as_float(v.w << 16);
  f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);   // round to nearest even
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint4 pack8(const float f[8]) {
  return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}

// ------------------------------------------- mixed bf16 / fp32 arithmetic --
// sm_100-class mixed-precision add / fma: bf16 operands are widened exactly
// inside the instruction and the fp32 result is rounded once (round to
// nearest even), so add_bf16(a, c) == __fadd_rn(float(a), c) bit for bit.
// A 32-bit register holds two bf16: element 2i in the low half.

// c[0] += lo(v), c[1] += hi(v)
__device__ __forceinline__ void add2_bf16(uint32_t v, float& c0, float& c1) {
  asm("{.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.bf16 %0, lo, %0;\n\t"
      "add.rn.f32.bf16 %1, hi, %1;}"
      : "+f"(c0), "+f"(c1)
      : "r"(v));
}

// c[e] += bf16 element e of v (8 elements)
__device__ __forceinline__ void add8_bf16(const uint4 v, float c[8]) {
  add2_bf16(v.x, c[0], c[1]);
  add2_bf16(v.y, c[2], c[3]);
  add2_bf16(v.z, c[4], c[5]);
  add2_bf16(v.w, c[6], c[7]);
}

// d0 = lo(v) + c0, d1 = hi(v) + c1 (non-destructive: no copy of c needed)
__device__ __forceinline__ void add2_bf16_to(uint32_t v, float c0, float c1, float& d0,
                                             float& d1) {
  asm("{.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.bf16 %0, lo, %3;\n\t"
      "add.rn.f32.bf16 %1, hi, %4;}"
      : "=f"(d0), "=f"(d1)
      : "r"(v), "f"(c0), "f"(c1));
}

// d[e] = bf16 element e of v + c (the same c for all 8)
__device__ __forceinline__ void add8_bf16_bcast(const uint4 v, float c, float d[8]) {
  add2_bf16_to(v.x, c, c, d[0], d[1]);
  add2_bf16_to(v.y, c, c, d[2], d[3]);
  add2_bf16_to(v.z, c, c, d[4], d[5]);
  add2_bf16_to(v.w, c, c, d[6], d[7]);
}

// d[e] = a[e] * b[e] + c (bf16 a, b; the same c for all 8)
__device__ __forceinline__ void fma8_bf16_bcast(const uint4 a, const uint4 b, float c,
                                                float d[8]) {
  const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    asm("{.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %2;\n\t"
        "mov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %4;\n\t"
        "fma.rn.f32.bf16 %1, ah, bh, %4;}"
        : "=f"(d[2 * i]), "=f"(d[2 * i + 1])
        : "r"(av[i]), "r"(bv[i]), "f"(c));
}

// c[e] = a[e] * b[e] + c[e] with a, b bf16 (the product of two bf16 is exact
// in fp32, so with c == 0 this is the exact product)
__device__ __forceinline__ void fma2_bf16(uint32_t a, uint32_t b, float& c0, float& c1) {
  asm("{.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %2;\n\t"
      "mov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %0;\n\t"
      "fma.rn.f32.bf16 %1, ah, bh, %1;}"
      : "+f"(c0), "+f"(c1)
      : "r"(a), "r"(b));
}

// ------------------------------------------------- packed fp32 (f32x2) --
// sm_100-class packed fp32 arithmetic: two independent IEEE fp32 operations
// (round to nearest even, no fusion beyond what is written) in one
// instruction.
__device__ __forceinline__ void mul2(float& a0, float& a1, float b0, float b1) {
  asm("{.reg .b64 a, b;\n\t"
      "mov.b64 a, {%0, %1};\n\t"
      "mov.b64 b, {%2, %3};\n\t"
      "mul.rn.f32x2 a, a, b;\n\t"
      "mov.b64 {%0, %1}, a;}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

// d = a * b + d, per lane, one rounding
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0,
                                     float b1) {
  asm("{.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %5};\n\t"
      "mov.b64 d, {%0, %1};\n\t"
      "fma.rn.f32x2 d, a, b, d;\n\t"
      "mov.b64 {%0, %1}, d;}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// (d0, d1) = (a0 * b, a1 * b)
__device__ __forceinline__ void mul2_to(float a0, float a1, float b, float& d0, float& d1) {
  asm("{.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %4};\n\t"
      "mul.rn.f32x2 d, a, b;\n\t"
      "mov.b64 {%0, %1}, d;}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b));
}

// (d0, d1) = (a0 * b0, a1 * b1)
__device__ __forceinline__ void mul2_pair(float a0, float a1, float b0, float b1, float& d0,
                                          float& d1) {
  asm("{.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 d, a, b;\n\t"
      "mov.b64 {%0, %1}, d;}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1) {
  asm("{.reg .b64 a, d;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 d, {%0, %1};\n\t"
      "add.rn.f32x2 d, d, a;\n\t"
      "mov.b64 {%0, %1}, d;}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}

// Keep flags (0/1) of 4 draws against thr, and their 4 mask bytes.
__device__ __forceinline__ uint32_t keep_bytes4(uint4 u, uint32_t thr) {
  const uint32_t k0 = u.x >= thr, k1 = u.y >= thr, k2 = u.z >= thr, k3 = u.w >= thr;
  return __byte_perm(__byte_perm(k0, k1, 0x3340), __byte_perm(k2, k3, 0x3340), 0x5410);
}

// The 8 keep flags of two keep_bytes4 words as one byte, element e in bit e.
// For w = b0 + b1 2^8 + b2 2^16 + b3 2^24 (each b 0 or 1), w * (2^21 + 2^14 +
// 2^7 + 1) holds b_i at bit 21 + i: the other partial products land at bits
// 0-16 (their sum stays below 2^17, so nothing carries into bit 21) or at
// bit 29 and above.
__device__ __forceinline__ uint32_t keep_bits8(uint2 kb) {
  constexpr uint32_t kGather = (1u << 21) | (1u << 14) | (1u << 7) | 1u;
  const uint32_t lo = (kb.x * kGather) >> 21 & 0xFu, hi = (kb.y * kGather) >> 21 & 0xFu;
  return lo | (hi << 4);
}




// ----------------------------------------------------- memory primitives --
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared asynchronous copy, L1 bypassed.
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src_gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(dst_smem)),
               "l"(src_gmem)
               : "memory");
}

// 8-byte global -> shared asynchronous copy.
// 4-byte global -> shared asynchronous copy (both addresses 4-byte aligned).
__device__ __forceinline__ void cp_async4(void* dst_smem, const void* src_gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_addr(dst_smem)),
               "l"(src_gmem)
               : "memory");
}

__device__ __forceinline__ void cp_async8(void* dst_smem, const void* src_gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_addr(dst_smem)),
               "l"(src_gmem)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Shared-memory loads as ordinary C++ loads, so the compiler may schedule them
// (the "memory" clobber of cp.async.wait_group still orders them after it).
__device__ __forceinline__ uint4 lds16(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ uint2 lds8(const void* p) {
  return *reinterpret_cast<const uint2*>(p);
}

// Read-only global load through the non-coherent path (small replicated
// parameters, re-read every row: kept in L1).
__device__ __forceinline__ uint4 ldg16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// Streamed (read-once) global load: evict-first.
__device__ __forceinline__ uint4 ldg16_stream(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

// Streaming (write-once) global stores: evict-first.
__device__ __forceinline__ void st16_stream(void* p, uint4 v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

__device__ __forceinline__ void st8_stream(void* p, uint2 v) {
  __stcs(reinterpret_cast<uint2*>(p), v);
}

// Streaming one-byte store (the low byte of v).
__device__ __forceinline__ void st1_stream(void* p, uint32_t v) {
  asm volatile("st.global.cs.u8 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ------------------------------------------ programmatic dependent launch --
// Every kernel of the library is launched with programmatic stream
// serialisation and never signals its dependents early, so the next kernel's
// blocks are placed as soon as every block of this one has exited, without
// the gap of a plain launch.  pdl_wait() returns once the previous kernel on
// the stream has completed and its memory operations are visible (at once for
// a plain launch); each kernel calls it, in every thread, before its first
// global memory access.  (Signalling earlier, so that the next kernel's
// blocks wait beside this kernel's last ones, measured slower.)
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------- bulk copies and mbarriers --
// The forward stages its inputs with bulk global -> shared copies issued by
// one producer warp and completed on mbarriers (transaction counts), the
// consumer warps releasing each stage through a second mbarrier.  Every wait
// is bounded: it gives up after kWaitLimitNs of %globaltimer and the caller
// reports SP_ERR_TIMEOUT instead of hanging.
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count)
               : "memory");
}

// Makes the initialised mbarriers visible to the copy engine and the block.
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}

// One arrival that also announces `bytes` of copies completing on b.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)),
               "r"(bytes)
               : "memory");
}

// A thread whose phase is still pending is suspended by the hardware for up
// to this long (or until the phase completes) before try_wait returns false,
// so a waiting thread takes no issue slots from the warps that compute.
constexpr uint32_t kTryWaitSuspendNs = 1000000;   // 1 ms

__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(b)), "r"(parity), "r"(kTryWaitSuspendNs)
      : "memory");
  return ok != 0;
}

// Wait until the phase of b with the given parity has completed; false if
// that takes longer than kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity) {
  if (mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(b, parity))
    if (global_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

// One contiguous global -> shared copy (16-byte aligned ends, a multiple of
// 16 bytes), completing on the mbarrier's transaction count.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst_smem)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Bulk shared -> global copies (the store direction of the same engine):
// issued by one thread, grouped by commit, waited for by group count.  The
// shared-memory source must have been made visible to the copy engine with
// fence_proxy_async_smem() by every thread that wrote it, before a barrier.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void bulk_s2g(void* dst, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_addr(src_smem)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Every committed bulk group has finished reading its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Every committed bulk group has completed (its global writes done).
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------------ clusters --
// A token row split over the CTAs of a thread-block cluster: each CTA
// publishes its part of the row sums in its own shared memory and arrives on
// the partner's mbarrier (release, cluster scope); the partner waits on its
// own mbarrier (acquire, cluster scope, bounded) and reads the value through
// distributed shared memory.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster arrives, then waits (a CTA may not
// exit while a partner can still reach its shared memory).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Address, in the cluster's shared window, of variable p of CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(b)), "r"(parity), "r"(kTryWaitSuspendNs)
      : "memory");
  return ok != 0;
}

// Bounded like mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* b, uint32_t parity) {
  if (mbar_try_wait_cluster(b, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait_cluster(b, parity))
    if (global_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

__device__ __forceinline__ float2 ld_cluster_f2(uint32_t cluster_addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y)
               : "r"(cluster_addr) : "memory");
  return v;
}

// ------------------------------------------------------ tensor memory --
// Tensor memory (TMEM, 128 lanes x 512 columns of 32 bits per SM) used as
// per-thread accumulator storage: warp w reaches lanes 32*(w % 4) .. +31, one
// lane per thread, and each thread keeps its values in a range of columns.
// Allocation, relinquish and dealloc are issued by one whole warp; the
// allocated base address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
               ::"r"(smem_addr(dst_smem)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n"
               ::"r"(taddr), "r"(ncols) : "memory");
}

// Block barrier that also orders this thread's tensor-memory accesses
// (and the allocation) against the other threads'.
__device__ __forceinline__ void tmem_sync_block() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// 8 / 16 consecutive columns of this thread's lane into registers; the wait
// for completion is in the same statement, so no value is read early.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float v[8]) {
  uint32_t r[8];
  __syncwarp();   // .sync.aligned: the whole warp, converged
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float v[16]) {
  uint32_t r[16];
  __syncwarp();   // .sync.aligned: the whole warp, converged
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Stores are asynchronous: tmem_wait_st() before the same columns are read again.
// Every helper first reconverges the warp (they follow per-thread branches).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float v[8]) {
  __syncwarp();   // .sync.aligned: the whole warp, converged
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n"
      ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
      "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])),
      "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float v[16]) {
  __syncwarp();   // .sync.aligned: the whole warp, converged
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};\n"
      ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
      "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])),
      "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  __syncwarp();   // .sync.aligned: the whole warp, converged
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// -------------------------------------------------------------- reductions --
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, m);
  return v;
}

// Two block-wide sums in a fixed order (deterministic): warp butterflies,
// one partial pair per warp in shared memory, then every warp runs the same
// butterfly over those partials, so all threads get the same bits.  `red` is
// a 32-entry shared slot; two consecutive calls must use different slots.
__device__ __forceinline__ float2 block_sum2(float a, float b, float2* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  a = warp_sum(a);
  b = warp_sum(b);
  if (lane == 0) red[warp] = make_float2(a, b);
  __syncthreads();
  const float2 p = lane < nw ? red[lane] : make_float2(0.f, 0.f);
  return make_float2(warp_sum(p.x), warp_sum(p.y));
}

// Block sums over the first NW warps only, synchronised on named barrier 1
// (a block whose last warp runs a copy producer that never joins them); same
// order and bits as block_sum2 over a block of NW warps.
template <int NW>
__device__ __forceinline__ void warps_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory");
}

template <int NW>
__device__ __forceinline__ float warps_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  if (lane == 0) red[warp] = v;
  warps_sync<NW>();
  return warp_sum(lane < NW ? red[lane] : 0.f);
}

template <int NW>
__device__ __forceinline__ float2 warps_sum2(float a, float b, float2* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = warp_sum(a);
  b = warp_sum(b);
  if (lane == 0) red[warp] = make_float2(a, b);
  warps_sync<NW>();
  const float2 p = lane < NW ? red[lane] : make_float2(0.f, 0.f);
  return make_float2(warp_sum(p.x), warp_sum(p.y));
}

// ------------------------------------------------------------- shard map --
// The rows of one block, walked as r0, r0 + step, r0 + 2 step, ... (step 1:
// a contiguous range; step = grid: every grid-th token): the row inside the
// shard moves by increments, and the shard lookup (a division and a search
// over the shard offsets) runs only when a step leaves the current shard or
// batch row.
struct RowWalk {
  int64_t row;     // token index in the (b, s) grid
  int64_t local;   // row index inside shard k's (b, s_k) tensor
  int64_t left;    // rows until the current shard ends in this batch row
  int k;

  __device__ __forceinline__ void locate(const ShardMap& m) {
    const int64_t bi = (m.b > 1 && m.s > 0) ? row / m.s : 0;
    const int64_t si = row - bi * m.s;
    k = 0;
    while (k + 1 < m.t && m.off[k + 1] <= si) ++k;   // skips empty shards
    local = bi * (m.off[k + 1] - m.off[k]) + (si - m.off[k]);
    left = m.off[k + 1] - si;
  }
  __device__ __forceinline__ void init(const ShardMap& m, int64_t r) {
    row = r;
    locate(m);
  }
  __device__ __forceinline__ void next(const ShardMap& m) {
    ++row;
    ++local;
    if (--left == 0) locate(m);
  }
  __device__ __forceinline__ void next(const ShardMap& m, int64_t step) {
    row += step;
    local += step;
    left -= step;
    if (left <= 0) locate(m);
  }
};

// First row and row count of block `blk` of `nblk` when `rows` rows are cut
// into contiguous ranges whose sizes differ by at most one.
__device__ __forceinline__ void block_rows(int64_t rows, int64_t blk, int64_t nblk, int64_t* r0,
                                           int64_t* n) {
  const int64_t a = rows * blk / nblk, b = rows * (blk + 1) / nblk;
  *r0 = a;
  *n = b - a;
}

// Device check of packed-sequence metadata: cu_seqlens[0] == 0, non-decreasing,
// cu_seqlens[n] == total.  Run by one warp; flags SP_ERR_DEVICE_CHECK.
__device__ __forceinline__ void check_cu_seqlens(const int32_t* cu, int32_t n, int64_t total,
                                                 int32_t* status) {
  if (cu == nullptr) return;
  bool bad = false;
  for (int i = threadIdx.x & 31; i <= n; i += 32) {
    const int32_t v = cu[i];
    if (i == 0 && v != 0) bad = true;
    if (i > 0 && v < cu[i - 1]) bad = true;
    if (i == n && static_cast<int64_t>(v) != total) bad = true;
  }
  if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0 && status != nullptr)
    *status = SP_ERR_DEVICE_CHECK;
}

}  // namespace spb
