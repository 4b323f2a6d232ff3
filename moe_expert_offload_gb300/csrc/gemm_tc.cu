// Prefill grouped expert GEMMs on the 5th-generation tensor cores.
//
// In prefill the routing union covers nearly every expert (FreeToken summary
// "background": prefill touches almost all experts, decode only a few), so
// the expert step is a dense contraction: per expert e, its T_e routed token
// rows times the dequantised int4 weights.  (Edge0 §3.1 "math convention":
// down(silu(gate(x)) * up(x)).)
//
//   GEMM1 (mode 1): [rows of e] x [Wg ; Wu]^T, K = H; epilogue SwiGLU
//                   h = silu(g) * u  -> h_perm (bf16)
//   GEMM2 (mode 2): [h rows of e] x Wd^T, K = I; epilogue weight w[t][j] ->
//                   y_assign[t][j] (bf16), summed later in j order.
//
// One CTA computes a 256 x 256 tile (BM x BN) with K in blocks of 64, as two
// M=128 MMAs per K step that share one dequantised B tile:
//   * Warp-specialised, stages handed over with mbarriers (no block-wide
//     barrier inside the K loop):
//       warps 0-3 gather A (256 rows x 64 bf16) row by row with cp.async into
//                 a 4-deep ring (each lane owns 16 fixed rows, addresses kept
//                 in registers); cp.async.mbarrier.arrive marks a stage full.
//                 Rows past the group's count are zero-filled, and a tile of at
//                 most 128 rows skips its second half entirely.
//       warps 5-12 one B row per thread: the int4 codes arrive by TMA (each
//                 warp a 3-deep ring of 32-row x 32-byte boxes), the group
//                 scales / biases 8 groups per 16-byte load; dequantised (one
//                 LOP3 per nibble pair gives (128+q) as bf16x2, then q = v - 128
//                 and w = s*q + b by bf16x2 fma) into a 2-deep B ring.
//       warp 4    one thread waits for both stages, issues the MMAs and frees
//                 the stages with tcgen05.commit.
//     Warps 5-12 then read the accumulators (tcgen05.ld) for the epilogue and
//     stage the bf16 output in shared memory, so that global stores cover whole
//     row segments.
//   * Both operands are K-major bf16 in the 128-byte swizzled layout; one
//     thread issues tcgen05.mma (M=128, N=256, K=16) into two TMEM
//     accumulators (512 columns) and tcgen05.commit signals an mbarrier when
//     the block's MMAs are done.
//   * K runs in a fixed within-8 permutation (columns 0,4,1,5,2,6,3,7 of
//     every 8) because that is the order one LOP3 yields nibble pairs; A is
//     stored in the same order (x is permuted once, GEMM1 writes h in it), so
//     every dot product is unchanged.
// FP4 experts (MXFP4, NVFP4) take the same path: each E2M1 code becomes its
// bf16 value through two byte-permute lookups (hi and lo bytes of the eight
// magnitudes) plus its sign bit, in the same (i, i + 4) column pairs, and is
// multiplied by its block scale in bf16 -- exact, as an E2M1 value times an
// E4M3 or power-of-two scale has at most six significant bits.  The NVFP4
// per-matrix fp32 scales multiply the fp32 accumulators in the epilogue.
// Every mbarrier wait is bounded: on time-out the CTA records MOE_DERR_WAIT,
// every role leaves its loop, the loader drains its own copies, and the CTA
// frees its TMEM and returns.
#include <cuda_bf16.h>

#include <cstring>

#include "moe_internal.cuh"
#include "stream_common.cuh"

namespace moe {
namespace {

constexpr int kBM = kPrefillTileRows;            // 256 rows: two M=128 accumulators
constexpr int kBK = 64;
// output columns of a tile (the N of each MMA): 256 (one CTA per SM) or 128
// (two co-resident CTAs per SM, so that one's fill and epilogue overlap the
// other's MMAs).  Measured on the 8192-token Qwen-shaped layer: gate/up 409 us
// at 256 vs 434 at 128; down (K = 512, short tiles) 299 us at 256 vs 291 at 128.
constexpr int kTileN1 = 256, kTileN2 = 128;
// warp roles: 0-3 gather A, 4 issues MMAs (one thread), 5-12 dequantise B and
// then drain the accumulators
constexpr int kLoadWarps = 4, kMmaWarp = 4, kDqWarp0 = 5;
constexpr int kHalfBytes = 128 * kBK * 2;        // 16 KB: one 128-row half of A
constexpr int kABytes = kBM * kBK * 2;           // 32 KB
// int4 codes reach shared memory by TMA: each dequant warp owns a ring of
// kCodeStages boxes of its 32 B rows x 32 bytes (one k-block), so the code
// loads leave the load/store pipe to the A gather and the bf16 stores
constexpr int kCodeStages = 3;
constexpr int kCodeBox = 32 * 32;

// ------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0: zero-fill the destination
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(count) : "memory");
}

// Bounded wait (about one second) for the completion of the phase with
// parity `parity`.
__device__ __forceinline__ bool mbar_wait(uint32_t addr, uint32_t parity) {
  return sc::bar_wait(addr, parity);
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// K-major operand in the 128-byte swizzled layout: rows of 128 bytes, groups
// of 8 rows 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;             // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset
  d |= (uint64_t)1 << 46;             // descriptor version
  d |= (uint64_t)2 << 61;             // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N = 256, M = 128 (one MMA covers one 128-row half of the tile;
// M = 128 is the largest shape a single CTA may issue).
constexpr int kMmaM = 128;
static_assert(kBM == 2 * kMmaM, "the tile is two M=128 halves");

// Per tile width BN: dequant warps (one B row per thread), threads, CTAs per
// SM, ring depths, TMEM columns (two M=128 accumulators of BN columns), the
// instruction descriptor and the dynamic shared memory.
template <int BN>
struct TileCfg {
  static constexpr int kDqWarps = BN / 32;
  static constexpr int kThreads = (kDqWarp0 + kDqWarps) * 32;
  static constexpr int kMinBlocks = BN == 256 ? 1 : 2;
  static constexpr int kStagesA = BN == 256 ? 4 : 2;  // A ring depth
  static constexpr int kStagesB = 2;                  // B operand ring depth
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                     ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kMmaM >> 4) << 24);
  static constexpr size_t kSmem = 1024 + (size_t)kStagesA * kABytes + (size_t)kStagesB * kBBytes +
                                  (size_t)kDqWarps * kCodeStages * kCodeBox;
};

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
      : "memory");
}

// 32 lanes x 32 consecutive fp32 columns of the accumulator.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// silu(g) = g / (1 + e^-g); the fast divide is far inside the bf16 rounding of h
// (the exponent is clamped so that the divisor stays finite)
__device__ __forceinline__ float silu(float g) {
  return __fdividef(g, 1.0f + __expf(fminf(-g, 80.0f)));
}

__device__ __forceinline__ uint32_t bf2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}


__device__ __forceinline__ void mbar_arrive(uint32_t addr) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(addr)
               : "memory");
}

__device__ __forceinline__ void cp_async_arrive(uint32_t addr) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(addr) : "memory");
}

// Tensor maps of one GEMM: m[0] over the layer's E blobs, m[1] over the shared
// expert's blob (int4 codes as u32 words [blob][B row][K / 8], boxes of 8 words
// x 32 rows); mode 2 only, m[2] over h_perm (u32 words [row][I / 2], boxes of
// 32 words x 256 rows, 128-byte swizzle: the A operand's layout).
struct GemmMaps {
  CUtensorMap m[3];
};

// bf16 of E2M1 codes: the high and low bytes of the eight magnitudes 0, 0.5,
// 1, 1.5, 2, 3, 4, 6 (index = the code's low three bits), as byte-permute tables
constexpr uint32_t kE2m1HiA = 0x3F3F3F00u, kE2m1HiB = 0x40404040u;
constexpr uint32_t kE2m1LoA = 0xC0800000u, kE2m1LoB = 0xC0804000u;

// One word of eight E2M1 codes (columns c0 .. c7, low nibble first) as the
// bf16x2 pairs (c_i, c_{i+4}), i = 0..3: the order the int4 path yields.
__device__ __forceinline__ void e2m1_pairs(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t sa = w & 0x7777u, sb = (w >> 16) & 0x7777u;
  const uint32_t hia = __byte_perm(kE2m1HiA, kE2m1HiB, sa), loa = __byte_perm(kE2m1LoA, kE2m1LoB, sa);
  const uint32_t hib = __byte_perm(kE2m1HiA, kE2m1HiB, sb), lob = __byte_perm(kE2m1LoA, kE2m1LoB, sb);
  const uint32_t u = __byte_perm(loa, hia, 0x5140), v = __byte_perm(loa, hia, 0x7362);
  const uint32_t ub = __byte_perm(lob, hib, 0x5140), vb = __byte_perm(lob, hib, 0x7362);
  o[0] = __byte_perm(u, ub, 0x5410) | ((w << 12) & 0x80008000u);
  o[1] = __byte_perm(u, ub, 0x7632) | ((w << 8) & 0x80008000u);
  o[2] = __byte_perm(v, vb, 0x5410) | ((w << 4) & 0x80008000u);
  o[3] = __byte_perm(v, vb, 0x7632) | (w & 0x80008000u);
}

// bf16 bits of one block scale byte: E4M3 (NVFP4; through fp16, both exact) or
// E8M0 2^(e-127) (MXFP4; 0 is 2^-127, a bf16 subnormal; 255 is NaN).
template <int FMT>
__device__ __forceinline__ uint32_t fp4_scale_bf16(uint32_t byte) {
  if constexpr (FMT == MOE_FORMAT_NVFP4) {
    uint32_t r;
    const uint16_t pair = (uint16_t)(byte | (byte << 8));  // both halves: e4m3(byte)
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(pair));
    const float f = __half2float(__ushort_as_half((unsigned short)(r & 0xFFFFu)));
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
  } else {
    return byte == 0u ? 0x0040u : byte == 255u ? 0x7FC0u : byte << 7;
  }
}

template <int MODE, int BN, int FMT>
__global__ void __launch_bounds__(TileCfg<BN>::kThreads, TileCfg<BN>::kMinBlocks)
    grouped_gemm_kernel(GemmArgs g, const __grid_constant__ GemmMaps maps) {
  using C = TileCfg<BN>;
  constexpr int kDqWarps = C::kDqWarps, kThreads = C::kThreads;
  constexpr int kStagesA = C::kStagesA, kStagesB = C::kStagesB, kBBytes = C::kBBytes;
  constexpr int kTmemCols = C::kTmemCols, kBN = BN;
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full_a[kStagesA], empty_a[kStagesA];
  __shared__ __align__(8) uint64_t full_b[kStagesB], empty_b[kStagesB], acc_full;
  __shared__ __align__(8) uint64_t code_full[kDqWarps][kCodeStages];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int s_fail;
  __shared__ const uint16_t* arow_s[kBM];
  const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
  // n-tiles run fastest: the CTAs sharing an m-tile's A rows are resident
  // together, so A comes from HBM once and from L2 for the other n-tiles
  const int nt = blockIdx.x, mt = blockIdx.y;
  if (mt >= *g.n_tiles) return;
  const int grp = g.tile_g[mt], row0 = g.tile_row0[mt], rows = g.tile_rows[mt];
  const int H = g.H, I = g.I;
  const int K = (MODE == 1) ? H : I, nk = K / kBK;
  const bool two = rows > 128;  // second 128-row half in use

  // shared memory: A ring | B ring (1024-aligned base)
  const uint32_t s0 = smem_u32(smem_raw);
  const uint32_t sbase = (s0 + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (sbase - s0);
  const uint32_t a_addr = sbase;
  const uint32_t b_addr = sbase + kStagesA * kABytes;
  unsigned char* b_ptr = gbase + kStagesA * kABytes;
  const uint32_t code_addr = b_addr + kStagesB * kBBytes;
  const unsigned char* code_ptr = b_ptr + kStagesB * kBBytes;

  // A source row of every tile row (null past the group's rows)
  for (int r = tid; r < kBM; r += kThreads) {
    const uint16_t* p = nullptr;
    if (r < rows) {
      int64_t src;
      if (MODE == 1) {
        const int a = g.perm[row0 + r];
        src = (a < g.T * g.k) ? a / g.k : a - g.T * g.k;
      } else {
        src = row0 + r;
      }
      p = g.a_src + src * K;
    }
    arow_s[r] = p;
  }
  if (wid == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int i = 0; i < kStagesA; ++i) {
      // mode 1: one cp.async arrive per loader lane; mode 2: the TMA issuer's expect_tx
      mbar_init(smem_u32(&full_a[i]), MODE == 1 ? 32 * kLoadWarps : 1);
      mbar_init(smem_u32(&empty_a[i]), 1);  // tcgen05.commit
    }
    for (int i = 0; i < kStagesB; ++i) {
      mbar_init(smem_u32(&full_b[i]), kDqWarps);  // one arrive per dequant warp
      mbar_init(smem_u32(&empty_b[i]), 1);
    }
    mbar_init(smem_u32(&acc_full), 1);
    for (int i = 0; i < kDqWarps * kCodeStages; ++i) mbar_init(smem_u32(&code_full[0][0] + i), 1);
    s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (MODE == 2 && wid < kLoadWarps) {
    // ----------------------------------------------- A loader, mode 2: TMA
    // the tile's h rows are contiguous (row0 ...): one 256-row x 64-column box
    // per block; rows past the group's count are computed and never stored
    if (wid == 0 && lane == 0) {
      const CUtensorMap* amap = &maps.m[2];
      sc::tma_prefetch_map(amap);
      int issued = 0;
      for (int kb = 0; kb < nk; ++kb) {
        const int st = kb % kStagesA, use = kb / kStagesA;
        if (use > 0 && !mbar_wait(smem_u32(&empty_a[st]), (use - 1) & 1)) s_fail = 1;
        if (s_fail) break;
        sc::bar_expect(smem_u32(&full_a[st]), kABytes);
        sc::tma_load_3d(a_addr + st * kABytes, amap, kb * (kBK / 2), row0, 0,
                        smem_u32(&full_a[st]));
        ++issued;
      }
      // after a failed wait: let the copies still in flight land (bounded)
      if (issued < nk)
        for (int j = issued > kStagesA ? issued - kStagesA : 0; j < issued; ++j)
          mbar_wait(smem_u32(&full_a[j % kStagesA]), (j / kStagesA) & 1);
    }
  } else if (wid < kLoadWarps) {
    // ---------------------------------------------------------- A loader
    // lane: rows wid*64 + lane/8 + 4j (j < 16), 16-byte chunk lane % 8
    constexpr int kRowsPerLane = kBM / (kLoadWarps * 4);
    const int c = lane & 7;
    const uint16_t* src[kRowsPerLane];
    uint32_t doff[kRowsPerLane];
    uint32_t vmask = 0;
#pragma unroll
    for (int j = 0; j < kRowsPerLane; ++j) {
      const int r = wid * (kBM / kLoadWarps) + (lane >> 3) + 4 * j;
      const uint16_t* p = arow_s[r];
      src[j] = p ? p + c * 8 : g.a_src;
      doff[j] = (r >> 7) * kHalfBytes + swz(r & 127, c);
      if (p) vmask |= 1u << j;
    }
    const bool active = two || wid * (kBM / kLoadWarps) < 128;
    for (int kb = 0; kb < nk; ++kb) {
      const int st = kb % kStagesA, use = kb / kStagesA;
      if (use > 0 && !mbar_wait(smem_u32(&empty_a[st]), (use - 1) & 1)) s_fail = 1;
      if (s_fail) break;
      const uint32_t ab = a_addr + st * kABytes;
      if (active) {
#pragma unroll
        for (int j = 0; j < kRowsPerLane; ++j)
          cp_async16(ab + doff[j], src[j] + kb * kBK, (vmask >> j) & 1u);
      }
      cp_async_arrive(smem_u32(&full_a[st]));
    }
    cp_async_wait<0>();
  } else if (wid == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int sa = kb % kStagesA, sb = kb % kStagesB;
        ok = mbar_wait(smem_u32(&full_a[sa]), (kb / kStagesA) & 1) &&
             mbar_wait(smem_u32(&full_b[sb]), (kb / kStagesB) & 1);
        if (!ok || s_fail) {
          ok = false;
          break;
        }
        fence_async_smem();
        tc_fence_after();
        const uint32_t ab = a_addr + sa * kABytes;
        const uint32_t bb = b_addr + sb * kBBytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint64_t bd = smem_desc(bb + kk * 32);
          mma_bf16(tmem, smem_desc(ab + kk * 32), bd, C::kIdesc, (kb | kk) != 0);
          if (two)
            mma_bf16(tmem + kBN, smem_desc(ab + kHalfBytes + kk * 32), bd, C::kIdesc,
                     (kb | kk) != 0);
        }
        mma_commit(smem_u32(&empty_a[sa]));
        mma_commit(smem_u32(&empty_b[sb]));
      }
      if (ok)
        mma_commit(smem_u32(&acc_full));
      else
        s_fail = 1;
    }
    __syncwarp();
  } else {
    // ------------------------------------------- B dequantisation (row t)
    const int t = tid - kDqWarp0 * 32, w = wid - kDqWarp0;  // warp w: B rows 32w .. 32w+31
    const uint8_t* blob = (grp < g.E) ? g.experts + (int64_t)grp * g.blob_bytes : g.shared;
    const BlobOffsets off = blob_offsets(H, I);
    const Fp4Offsets fo = fp4_offsets(H, I, FMT == MOE_FORMAT_INT4 ? MOE_FORMAT_NVFP4 : FMT);
    int64_t row, so, bo;
    int my;  // first row of this warp's code box in the map
    if (MODE == 1) {
      const bool up = t >= kBN / 2;
      row = (int64_t)nt * (kBN / 2) + (up ? t - kBN / 2 : t);
      so = FMT == MOE_FORMAT_INT4 ? (up ? off.us : off.gs) : (up ? fo.us : fo.gs);
      bo = up ? off.ub : off.gb;
      my = (up ? I : 0) + nt * (kBN / 2) + 32 * (w % (kDqWarps / 2));  // up rows follow the gate rows
    } else {
      row = (int64_t)nt * kBN + t;
      so = FMT == MOE_FORMAT_INT4 ? off.ds : fo.ds;
      bo = off.db;
      my = nt * kBN + 32 * w;
    }
    const int G = K / kGroup;
    const bool g8 = (G & 7) == 0;  // scales fetched 8 groups (16 bytes) at a time, else 2
    const int span = g8 ? 8 : 2;
    const uint8_t* srow = blob + so + row * G * 2;
    const uint8_t* brw = blob + bo + row * G * 2;
    const CUtensorMap* map = &maps.m[grp < g.E ? 0 : 1];
    const int mz = grp < g.E ? grp : 0;
    const uint32_t cbase = code_addr + (uint32_t)(w * kCodeStages * kCodeBox);
    const unsigned char* cptr = code_ptr + w * kCodeStages * kCodeBox;
    auto issue = [&](int kb) {  // lane 0: the codes of block kb into slot kb % kCodeStages
      const uint32_t bar = smem_u32(&code_full[w][kb % kCodeStages]);
      sc::bar_expect(bar, kCodeBox);
      sc::tma_load_3d(cbase + (kb % kCodeStages) * kCodeBox, map, kb * 8, my, mz, bar);
    };
    int issued = 0;
    if (lane == 0) {
      sc::tma_prefetch_map(map);
      for (; issued < nk && issued < kCodeStages; ++issued) issue(issued);
    }
    struct SB { uint32_t s0, s1, s2, s3, b0, b1, b2, b3; };
    auto load_sb = [&](int kb, SB& v) {
      if (g8) {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(srow + kb * 2));
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(brw + kb * 2));
        v = SB{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      } else {
        v.s0 = __ldg(reinterpret_cast<const uint32_t*>(srow + kb * 2));
        v.b0 = __ldg(reinterpret_cast<const uint32_t*>(brw + kb * 2));
      }
    };
    // FP4: this row's block scale bytes of k-block kb (4 of 16 columns, or 2 of 32)
    const uint8_t* frow = blob + so + row * (K / (FMT == MOE_FORMAT_NVFP4 ? 16 : 32));
    auto load_fs = [&](int kb) -> uint32_t {
      if constexpr (FMT == MOE_FORMAT_NVFP4)
        return __ldg(reinterpret_cast<const uint32_t*>(frow + kb * 4));
      else
        return __ldg(reinterpret_cast<const uint16_t*>(frow + kb * 2));
    };
    SB cur{}, nxt{};
    uint32_t fs_cur = 0, fs_nxt = 0;
    if constexpr (FMT == MOE_FORMAT_INT4) {
      load_sb(0, cur);
      if (span < nk) load_sb(span, nxt);
    } else {
      fs_cur = load_fs(0);
      if (nk > 1) fs_nxt = load_fs(1);
    }
    const __nv_bfloat162 k128 = __floats2bfloat162_rn(128.0f, 128.0f);
    int kb = 0, consumed = 0;
    bool failed = false;
    for (; kb < nk; ++kb) {
      const int sb = kb % kStagesB, use = kb / kStagesB, cs = kb % kCodeStages;
      if constexpr (FMT == MOE_FORMAT_INT4) {
        if (kb > 0 && kb % span == 0) {
          cur = nxt;
          if (kb + span < nk) load_sb(kb + span, nxt);
        }
      } else if (kb > 0) {
        fs_cur = fs_nxt;
        if (kb + 1 < nk) fs_nxt = load_fs(kb + 1);
      }
      // the stage's previous MMAs are done (lane 0), this block's codes have landed (all lanes)
      if (lane == 0 && use > 0 && !mbar_wait(smem_u32(&empty_b[sb]), (use - 1) & 1)) s_fail = 1;
      const bool cok = mbar_wait(smem_u32(&code_full[w][cs]), (kb / kCodeStages) & 1);
      if (!__all_sync(0xffffffffu, cok) && lane == 0) s_fail = 1;
      if (__shfl_sync(0xffffffffu, (int)s_fail, 0)) {
        failed = true;
        break;
      }
      const uint4 q0 = *reinterpret_cast<const uint4*>(cptr + cs * kCodeBox + lane * 32);
      const uint4 q1 = *reinterpret_cast<const uint4*>(cptr + cs * kCodeBox + lane * 32 + 16);
      // every lane's reads of the slot come before its refill through the async proxy
      fence_async_smem();
      __syncwarp();
      consumed = kb + 1;
      if (lane == 0 && issued < nk) issue(issued++);
      const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
      unsigned char* bb = b_ptr + sb * kBBytes;
      if constexpr (FMT == MOE_FORMAT_INT4) {
        const int gi = kb % span;  // group within the fetched span
        const uint32_t sw = gi < 2 ? cur.s0 : gi < 4 ? cur.s1 : gi < 6 ? cur.s2 : cur.s3;
        const uint32_t bw = gi < 2 ? cur.b0 : gi < 4 ? cur.b1 : gi < 6 ? cur.b2 : cur.b3;
        const uint32_t sh = (gi & 1) ? (sw >> 16) : (sw & 0xFFFFu);
        const uint32_t bh = (gi & 1) ? (bw >> 16) : (bw & 0xFFFFu);
        const uint32_t s2u = sh | (sh << 16), b2u = bh | (bh << 16);
        const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162*>(&s2u);
        const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&b2u);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t v = ((words[c] >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
            const __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v), k128);
            const __nv_bfloat162 wv = __hfma2(q, s2, b2);
            o[i] = *reinterpret_cast<const uint32_t*>(&wv);
          }
          *reinterpret_cast<uint4*>(bb + swz(t, c)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      } else {
        // word c holds columns 8c .. 8c + 7: block c / 2 (16 columns) or c / 4 (32)
        constexpr int kBlocks = FMT == MOE_FORMAT_NVFP4 ? 4 : 2;
        uint32_t sc2[kBlocks];
#pragma unroll
        for (int j = 0; j < kBlocks; ++j) {
          const uint32_t h = fp4_scale_bf16<FMT>((fs_cur >> (8 * j)) & 0xFFu);
          sc2[j] = h | (h << 16);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t o[4];
          e2m1_pairs(words[c], o);
          const __nv_bfloat162 s2 =
              *reinterpret_cast<const __nv_bfloat162*>(&sc2[c / (8 / kBlocks)]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 wv = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&o[i]), s2);
            o[i] = *reinterpret_cast<const uint32_t*>(&wv);
          }
          *reinterpret_cast<uint4*>(bb + swz(t, c)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&full_b[sb]));
    }
    // after a failed wait: let this warp's code copies still in flight land (bounded)
    if (failed && lane == 0)
      for (int j = consumed; j < issued; ++j)
        mbar_wait(smem_u32(&code_full[w][j % kCodeStages]), (j / kCodeStages) & 1);

    // ---------------------------------------------------------- epilogue
    int ok = 1;
    if (lane == 0) {
      if (!mbar_wait(smem_u32(&acc_full), 0)) s_fail = 1;
      ok = !s_fail;
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      tc_fence_after();
      // NVFP4: the fp32 matrix scales of gate, up and down multiply the sums
      float sg = 1.0f, su = 1.0f, sd = 1.0f;
      if constexpr (FMT == MOE_FORMAT_NVFP4) {
        const float* mat = reinterpret_cast<const float*>(blob + fo.mat);
        sg = __ldg(mat);
        su = __ldg(mat + 1);
        sd = __ldg(mat + 2);
      }
      const int q = wid & 3, ch = (wid - kDqWarp0) >> 2;  // TMEM lane quarter, column half
      // Each warp stages its 32 rows x kRowBytes of output (bf16) in the idle A
      // ring, 16-byte chunks XOR-swizzled by the row within each 128-byte segment
      // (conflict-free both ways), then writes whole row segments: a store
      // instruction covers 4 (or 2) rows x 128 (or 256) contiguous bytes instead
      // of 32 rows x 16 bytes.
      constexpr int kColsW = MODE == 1 ? 64 : 128;  // this warp's output columns (of a row)
      constexpr int kRowBytes = 2 * kColsW;
      constexpr int kLanesPerRow = kRowBytes / 16, kRowsPerStore = 32 / kLanesPerRow;
      unsigned char* stg = gbase + (wid - kDqWarp0) * 32 * kRowBytes;
      auto sidx = [](int rr, int c) {
        return rr * kRowBytes + ((c & ~7) << 4) + (((c & 7) ^ (rr & 7)) << 4);
      };
#pragma unroll
      for (int hm = 0; hm < 2; ++hm) {
        if (hm == 1 && !two) break;
        const int r = hm * 128 + 32 * q + lane;  // this lane's accumulator row
        const uint32_t trow = tmem + hm * kBN + ((uint32_t)(32 * q) << 16);
        int64_t dst_row = 0;
        if (MODE == 1) {
#pragma unroll
          for (int c = 0; c < 64; c += 32) {
            float gv[32], uv[32];
            tmem_ld32(trow + 64 * ch + c, gv);
            tmem_ld32(trow + kBN / 2 + 64 * ch + c, uv);
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              float h[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                if constexpr (FMT == MOE_FORMAT_NVFP4)
                  h[i] = silu(gv[e + i] * sg) * (uv[e + i] * su);
                else
                  h[i] = silu(gv[e + i]) * uv[e + i];
              }
              *reinterpret_cast<uint4*>(stg + sidx(lane, (c + e) >> 3)) = make_uint4(
                  bf2(h[0], h[4]), bf2(h[1], h[5]), bf2(h[2], h[6]), bf2(h[3], h[7]));
            }
          }
        } else {
          float wgt = 0.0f;
          if (r < rows) {
            const int a = g.perm[row0 + r];
            const int Tk = g.T * g.k;
            if (a < Tk) {
              dst_row = (int64_t)(a / g.k) * (g.k + 1) + a % g.k;
              wgt = g.weights[a];
            } else {
              dst_row = (int64_t)(a - Tk) * (g.k + 1) + g.k;
              wgt = 1.0f;
            }
            wgt *= sd;
          }
#pragma unroll
          for (int c = 0; c < kColsW; c += 32) {
            float v[32];
            tmem_ld32(trow + kColsW * ch + c, v);
#pragma unroll
            for (int e = 0; e < 32; e += 8)
              *reinterpret_cast<uint4*>(stg + sidx(lane, (c + e) >> 3)) = make_uint4(
                  bf2(wgt * v[e], wgt * v[e + 1]), bf2(wgt * v[e + 2], wgt * v[e + 3]),
                  bf2(wgt * v[e + 4], wgt * v[e + 5]), bf2(wgt * v[e + 6], wgt * v[e + 7]));
          }
        }
        __syncwarp();
#pragma unroll 4
        for (int i = 0; i < 32; i += kRowsPerStore) {
          const int rr = i + lane / kLanesPerRow, c = lane % kLanesPerRow;
          const int rt = hm * 128 + 32 * q + rr;  // tile row
          const int64_t drow = __shfl_sync(0xffffffffu, dst_row, rr);
          const uint4 v = *reinterpret_cast<const uint4*>(stg + sidx(rr, c));
          if (rt < rows) {
            uint16_t* dst = MODE == 1
                ? g.h_out + (int64_t)(row0 + rt) * I + nt * (kBN / 2) + 64 * ch + 8 * c
                : g.y_out + drow * H + nt * kBN + kColsW * ch + 8 * c;
            *reinterpret_cast<uint4*>(dst) = v;
          }
        }
        __syncwarp();  // the staging tile is refilled for the second half
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && s_fail && g.err) atomicOr(g.err, MOE_DERR_WAIT);
  if (wid == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
}

}  // namespace

// One (mode, tile width, format) instantiation: its shared-memory attribute once
// per device, then the launch (n-tiles along x, m-tiles along y).
template <int MODE, int BN, int FMT>
cudaError_t launch_mode(const GemmArgs& a, const GemmMaps& maps, int max_tiles, int d,
                        cudaStream_t st) {
  using C = TileCfg<BN>;
  static bool attr_done[64] = {};
  if (!attr_done[d]) {
    const cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<MODE, BN, FMT>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)C::kSmem);
    if (e != cudaSuccess) return e;
    attr_done[d] = true;
  }
  const dim3 grid(MODE == 1 ? a.I / (BN / 2) : a.H / BN, max_tiles);
  grouped_gemm_kernel<MODE, BN, FMT><<<grid, C::kThreads, C::kSmem, st>>>(a, maps);
  return cudaGetLastError();
}

cudaError_t launch_grouped_gemm(int mode, const GemmArgs& a, int max_tiles, cudaStream_t st) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= 64) return cudaErrorInvalidDevice;
  // code maps: mode 1 the gate rows then the up rows ([2I][H/2] bytes, contiguous
  // in the blob), mode 2 the down rows ([H][I/2] bytes)
  const BlobOffsets off = blob_offsets(a.H, a.I);
  const int64_t K = mode == 1 ? a.H : a.I;
  const uint64_t rows = mode == 1 ? 2 * (uint64_t)a.I : (uint64_t)a.H;
  const int64_t q0 = mode == 1 ? off.gq : off.dq;
  GemmMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (mode == 2) {  // A = h_perm rows as u32 words, 128-byte swizzle
    const uint64_t R = (uint64_t)a.T * a.k + a.T;
    const uint64_t dims[3] = {(uint64_t)a.I / 2, R, 1};
    const uint64_t strides[2] = {(uint64_t)a.I * 2, R * a.I * 2};
    const uint32_t box[3] = {kBK / 2, kBM, 1};
    if ((e = encode_tiled_u32(&maps.m[2], a.a_src, 3, dims, strides, box, true)) != cudaSuccess)
      return e;
  }
  const uint8_t* bases[2] = {a.experts, a.shared ? a.shared : a.experts};
  const uint64_t nblob[2] = {(uint64_t)a.E, 1};
  for (int i = 0; i < 2; ++i) {
    const uint64_t dims[3] = {(uint64_t)K / 8, rows, nblob[i]};
    const uint64_t strides[2] = {(uint64_t)K / 2, (uint64_t)a.blob_bytes};
    const uint32_t box[3] = {8, 32, 1};
    if ((e = encode_tiled_u32(&maps.m[i], bases[i] + q0, 3, dims, strides, box, false)) !=
        cudaSuccess)
      return e;
  }
  if (mode == 1) {
    if (a.format == MOE_FORMAT_MXFP4)
      return launch_mode<1, kTileN1, MOE_FORMAT_MXFP4>(a, maps, max_tiles, d, st);
    if (a.format == MOE_FORMAT_NVFP4)
      return launch_mode<1, kTileN1, MOE_FORMAT_NVFP4>(a, maps, max_tiles, d, st);
    return launch_mode<1, kTileN1, MOE_FORMAT_INT4>(a, maps, max_tiles, d, st);
  }
  if (a.format == MOE_FORMAT_MXFP4)
    return launch_mode<2, kTileN2, MOE_FORMAT_MXFP4>(a, maps, max_tiles, d, st);
  if (a.format == MOE_FORMAT_NVFP4)
    return launch_mode<2, kTileN2, MOE_FORMAT_NVFP4>(a, maps, max_tiles, d, st);
  return launch_mode<2, kTileN2, MOE_FORMAT_INT4>(a, maps, max_tiles, d, st);
}

}  // namespace moe
