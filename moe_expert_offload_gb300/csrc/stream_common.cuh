// Device helpers shared by the streaming decode kernels: mbarrier waits
// (bounded), bulk and tiled TMA copies, and the int4 -> bf16 fragment MMA
// building blocks (Edge0 §3.1 "math convention": w = s * q + b per 64-column
// group; the fragments carry 128 + q and the offset is removed on the fp32
// accumulator).
#pragma once
#include <cuda_bf16.h>

#include "moe_internal.cuh"

namespace moe {
namespace sc {

// A wait gives up after 1024 try_wait rounds plus kWaitCycles SM clock
// cycles (2^31: about one second at the 2.07 GHz maximum clock, longer at
// lower clocks), so a failure (a copy that never lands, a stage never
// released) ends the kernel with an error word instead of a hang.  One round
// may suspend the thread for a system-dependent time, so the bound is kept in
// cycles; kSpin rounds is a second cap.  The counter is read only once a wait
// has run 1024 rounds: the waits of the streaming kernels sit in their inner
// loops, where any extra work at the wait site (an early counter read, a
// second copy of the try_wait) measurably slowed them.
constexpr long long kWaitCycles = 1ll << 31;
constexpr uint32_t kSpin = 1u << 26;

__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void bar_init(uint32_t a, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(n) : "memory");
}

// Bounded wait for the completion of the phase with parity `parity`.
__device__ __forceinline__ bool bar_wait(uint32_t a, uint32_t parity) {
  long long t0 = 0;  // taken after the first 1024 rounds
  for (uint32_t i = 0; i < kSpin; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
    if ((i & 1023u) == 1023u) {
      const long long t = clock64();
      if (t0 == 0) t0 = t;
      else if (t - t0 > kWaitCycles) return false;
    }
  }
  return false;
}

// the whole warp waits; true only if every lane saw the phase complete
__device__ __forceinline__ bool warp_wait(uint32_t a, uint32_t parity) {
  return __all_sync(0xffffffffu, bar_wait(a, parity));
}

__device__ __forceinline__ void bar_arrive(uint32_t a) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(a)
               : "memory");
}

__device__ __forceinline__ void bar_expect(uint32_t a, uint32_t bytes) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(a),
      "r"(bytes)
      : "memory");
}

// global -> shared bulk copy (16-byte aligned, size a multiple of 16)
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint32_t nib_pair(uint32_t w, int i) {
  return ((w >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
}

// Not volatile: the MMA has no side effect, so the compiler may interleave
// independent accumulator chains (gate / up, several groups) to hide latency.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16 rows x one 64-column group: lo / hi are the lane's 8 code bytes of rows
// g and g + 8, b the group's 8 B-fragment registers (same k order as
// ffn_decode.cu: MMA jj takes nibble pairs (i, i+4), (i+1, i+5) of word jj/2).
__device__ __forceinline__ void group_mma(float (&d)[4], uint2 lo, uint2 hi,
                                          const uint32_t (&b)[8]) {
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const uint32_t wl = (jj < 2) ? lo.x : lo.y, wh = (jj < 2) ? hi.x : hi.y;
    const int i = 2 * (jj & 1);
    mma16816(d, nib_pair(wl, i), nib_pair(wh, i), nib_pair(wl, i + 1), nib_pair(wh, i + 1),
             b[2 * jj], b[2 * jj + 1]);
  }
}

// gate and up of one group, their MMAs interleaved (two independent chains)
__device__ __forceinline__ void group_mma2(float (&dg)[4], float (&du)[4], uint2 g0, uint2 g1,
                                           uint2 u0, uint2 u1, const uint32_t (&b)[8]) {
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const uint32_t gl = (jj < 2) ? g0.x : g0.y, gh = (jj < 2) ? g1.x : g1.y;
    const uint32_t ul = (jj < 2) ? u0.x : u0.y, uh = (jj < 2) ? u1.x : u1.y;
    const int i = 2 * (jj & 1);
    mma16816(dg, nib_pair(gl, i), nib_pair(gh, i), nib_pair(gl, i + 1), nib_pair(gh, i + 1),
             b[2 * jj], b[2 * jj + 1]);
    mma16816(du, nib_pair(ul, i), nib_pair(uh, i), nib_pair(ul, i + 1), nib_pair(uh, i + 1),
             b[2 * jj], b[2 * jj + 1]);
  }
}

__device__ __forceinline__ void frag_order(const uint32_t (&w)[8], uint4& o0, uint4& o1) {
  o0.x = __byte_perm(w[0], w[2], 0x5410);
  o0.y = __byte_perm(w[0], w[2], 0x7632);
  o0.z = __byte_perm(w[1], w[3], 0x5410);
  o0.w = __byte_perm(w[1], w[3], 0x7632);
  o1.x = __byte_perm(w[4], w[6], 0x5410);
  o1.y = __byte_perm(w[4], w[6], 0x7632);
  o1.z = __byte_perm(w[5], w[7], 0x5410);
  o1.w = __byte_perm(w[5], w[7], 0x7632);
}

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// shared -> global stores of a tile that arrived by TMA (the slot copy of an
// expert filled in this step).  Both sides are async-proxy operations; the
// proxy fence orders the issuing thread's view of the landed tile before the
// store reads it.  A thread that issued stores calls bulk_read_done() before
// the tile's buffer is handed back for reuse or the CTA exits.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// L2 policy for data read or written once per call (streamed weights): first
// in line for eviction, so that it does not push out what stays hot across
// calls (kernel code, cache tables, router weights).
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_load_4d_ef(uint32_t dst, const CUtensorMap* map, int x, int y,
                                               int z, int w, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_ef(uint32_t dst, const CUtensorMap* map, int x, int y,
                                               int z, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_store_4d_ef(const CUtensorMap* map, int x, int y, int z,
                                                int w, uint32_t src, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group.L2::cache_hint"
      " [%0, {%1, %2, %3, %4}], [%5], %6;" ::"l"(map),
      "r"(x), "r"(y), "r"(z), "r"(w), "r"(src), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_store_3d_ef(const CUtensorMap* map, int x, int y, int z,
                                                uint32_t src, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint"
      " [%0, {%1, %2, %3}], [%4], %5;" ::"l"(map),
      "r"(x), "r"(y), "r"(z), "r"(src), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, int x, int y, int z, int w,
                                             uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
          map),
      "r"(x), "r"(y), "r"(z), "r"(w), "r"(src)
      : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int x, int y, int z,
                                             uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(map),
      "r"(x), "r"(y), "r"(z), "r"(src)
      : "memory");
}

// (16-byte aligned, size a multiple of 16)
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// the shared-memory reads of every store this thread committed are done
__device__ __forceinline__ void bulk_read_done() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void load_frag(const unsigned char* p, bool valid, uint32_t (&b)[8]) {
  if (valid) {
    const uint4 v0 = reinterpret_cast<const uint4*>(p)[0];
    const uint4 v1 = reinterpret_cast<const uint4*>(p)[1];
    b[0] = v0.x; b[1] = v0.y; b[2] = v0.z; b[3] = v0.w;
    b[4] = v1.x; b[5] = v1.y; b[6] = v1.z; b[7] = v1.w;
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) b[e] = 0u;
  }
}

// One tensor map per blob array: bank, slot pool, shared expert.
struct CodeMaps {
  CUtensorMap m[3];
};


}  // namespace sc
}  // namespace moe
