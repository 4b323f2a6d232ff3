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
//   * A (256 rows x 64 bf16) is gathered row by row with cp.async into a
//     4-deep ring, two blocks ahead; rows past the expert's count are zero and
//     a tile of at most 128 rows skips its second half entirely.
//   * The raw int4 codes and group scales/biases of B (256 rows) are loaded
//     straight into registers, also two blocks ahead (three named register
//     sets in rotation); 16 warps dequantise them (one LOP3 per nibble pair
//     gives (128+q) as bf16x2, then q = v - 128 and w = s*q + b by bf16x2 fma)
//     into a double-buffered B operand.
//   * Both operands are K-major bf16 in the 128-byte swizzled layout; one
//     thread issues tcgen05.mma (M=128, N=256, K=16) into two TMEM
//     accumulators (512 columns) and tcgen05.commit signals an mbarrier when
//     the block's MMAs are done.
//   * K runs in a fixed within-8 permutation (columns 0,4,1,5,2,6,3,7 of
//     every 8) because that is the order one LOP3 yields nibble pairs; A is
//     stored in the same order (x is permuted once, GEMM1 writes h in it), so
//     every dot product is unchanged.
// Every mbarrier wait is bounded: on time-out the CTA records MOE_DERR_WAIT,
// drains its own copies, frees its TMEM and returns.
#include <cuda_bf16.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kBM = kPrefillTileRows;            // 256 rows: two M=128 accumulators
constexpr int kBN = 256, kBK = 64;
constexpr int kThreads = 512;
constexpr int kStages = 4;                       // A ring depth
constexpr int kAhead = 2;                        // blocks loaded ahead (A and B codes)
constexpr int kHalfBytes = 128 * kBK * 2;        // 16 KB: one 128-row half of A
constexpr int kABytes = kBM * kBK * 2;           // 32 KB
constexpr int kBBytes = kBN * kBK * 2;           // 32 KB
constexpr int kTmemCols = 512;
constexpr uint32_t kWaitIters = 1u << 20;

// ------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0: zero-fill the destination
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
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

// Bounded wait for the completion of the phase with parity `parity`.
__device__ __forceinline__ bool mbar_wait(uint32_t addr, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitIters; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
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
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kMmaM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
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

__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

__device__ __forceinline__ uint32_t bf2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}


template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(GemmArgs g) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t mbar[2];
  __shared__ uint32_t tmem_slot;
  __shared__ const uint16_t* arow_s[kBM];
  const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
  const int mt = blockIdx.x, nt = blockIdx.y;
  if (mt >= *g.n_tiles) return;
  const int grp = g.tile_g[mt], row0 = g.tile_row0[mt], rows = g.tile_rows[mt];
  const int H = g.H, I = g.I;
  const int K = (MODE == 1) ? H : I, nk = K / kBK;

  // shared memory: A ring | B double buffer | raw ring (1024-aligned base)
  const uint32_t s0 = smem_u32(smem_raw);
  const uint32_t sbase = (s0 + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (sbase - s0);
  const uint32_t a_addr = sbase;
  const uint32_t b_addr = sbase + kStages * kABytes;
  unsigned char* b_ptr = gbase + (b_addr - sbase);

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
    mbar_init(smem_u32(&mbar[0]), 1);
    mbar_init(smem_u32(&mbar[1]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // B row r of the tile -> its codes / scale / bias rows
  const uint8_t* blob = (grp < g.E) ? g.experts + (int64_t)grp * g.blob_bytes : g.shared;
  const BlobOffsets off = blob_offsets(H, I);
  auto brow = [&](int r, int which) -> const uint8_t* {  // which: 0 codes, 1 scale, 2 bias
    int64_t row, o;
    if (MODE == 1) {
      const bool up = r >= kBN / 2;
      row = (int64_t)nt * (kBN / 2) + (up ? r - kBN / 2 : r);
      o = which == 0 ? (up ? off.uq : off.gq) : which == 1 ? (up ? off.us : off.gs)
                                                           : (up ? off.ub : off.gb);
    } else {
      row = (int64_t)nt * kBN + r;
      o = which == 0 ? off.dq : which == 1 ? off.ds : off.db;
    }
    return which == 0 ? blob + o + row * (K / 2) : blob + o + row * (K / kGroup) * 2;
  };
  // this thread's B items: half a code row (16 bytes) plus the row's scale
  // and bias words (groups kb & ~1 and kb | 1)
  const int lr = tid >> 1, lh = tid & 1;
  const uint8_t* qsrc = brow(lr, 0) + lh * 16;
  const uint8_t* ssrc = brow(lr, 1);
  const uint8_t* bsrc = brow(lr, 2);
  const bool two = rows > 128;  // second 128-row half in use

  struct BRegs {
    uint4 q;
    uint32_t s, b;
  };
  auto load_b = [&](int kb, BRegs& r) {
    r.q = __ldg(reinterpret_cast<const uint4*>(qsrc + kb * 32));
    r.s = __ldg(reinterpret_cast<const uint32_t*>(ssrc + (kb & ~1) * 2));
    r.b = __ldg(reinterpret_cast<const uint32_t*>(bsrc + (kb & ~1) * 2));
  };
  auto load_a = [&](int kb) {
    const uint32_t ab = a_addr + (kb % kStages) * kABytes;
#pragma unroll
    for (int j = 0; j < (kBM * 8) / kThreads; ++j) {
      const int i = tid + j * kThreads, r = i >> 3, c = i & 7;
      if (r < 128 || two) {
        const uint16_t* p = arow_s[r];
        const uint32_t dst = ab + (r >> 7) * kHalfBytes + swz(r & 127, c);
        cp_async16(dst, p ? p + kb * kBK + c * 8 : g.a_src, p != nullptr);
      }
    }
  };
  // registers of block kb -> B operand buffer kb % 2 (chunks 4lh..4lh+3 of row lr)
  auto dequant = [&](int kb, const BRegs& r) {
    const uint32_t sh = (kb & 1) ? (r.s >> 16) : (r.s & 0xFFFFu);
    const uint32_t bh = (kb & 1) ? (r.b >> 16) : (r.b & 0xFFFFu);
    const uint32_t s2u = sh | (sh << 16), b2u = bh | (bh << 16);
    const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162*>(&s2u);
    const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&b2u);
    const __nv_bfloat162 k128 = __floats2bfloat162_rn(128.0f, 128.0f);
    const uint32_t words[4] = {r.q.x, r.q.y, r.q.z, r.q.w};
    unsigned char* bb = b_ptr + (kb & 1) * kBBytes;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t v = ((words[c] >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
        const __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v), k128);
        const __nv_bfloat162 w = __hfma2(q, s2, b2);
        o[i] = *reinterpret_cast<const uint32_t*>(&w);
      }
      *reinterpret_cast<uint4*>(bb + swz(lr, 4 * lh + c)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  };

  // ---- main loop: blocks kb+1, kb+2 load while block kb is dequantised and
  // block kb-1's MMAs run; buffers of block kb-2 are reused once its MMAs end.
  bool failed = false;
  BRegs r0, r1, r2;
  load_a(0);
  cp_async_commit();
  load_b(0, r0);
  if (nk > 1) {
    load_a(1);
    load_b(1, r1);
  }
  cp_async_commit();
  auto iteration = [&](int kb, const BRegs& cur, BRegs& nxt) -> bool {
    bool ok = true;
    if (kb >= 2) ok = mbar_wait(smem_u32(&mbar[kb & 1]), ((kb - 2) >> 1) & 1);
    if (__syncthreads_or(!ok)) return false;
    tc_fence_after();
    if (kb + kAhead < nk) {
      load_a(kb + kAhead);
      load_b(kb + kAhead, nxt);
    }
    cp_async_commit();
    cp_async_wait<kAhead>();
    __syncthreads();
    dequant(kb, cur);
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ab = a_addr + (kb % kStages) * kABytes;
      const uint32_t bb = b_addr + (kb & 1) * kBBytes;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        const uint64_t bd = smem_desc(bb + kk * 32);
        mma_bf16(tmem, smem_desc(ab + kk * 32), bd, (kb | kk) != 0);
        if (two) mma_bf16(tmem + kBN, smem_desc(ab + kHalfBytes + kk * 32), bd, (kb | kk) != 0);
      }
      mma_commit(smem_u32(&mbar[kb & 1]));
    }
    return true;
  };
  int kb = 0;
  for (; kb < nk; kb += 3) {
    if (!iteration(kb, r0, r2)) break;
    if (kb + 1 < nk && !iteration(kb + 1, r1, r0)) {
      kb += 1;
      break;
    }
    if (kb + 2 < nk && !iteration(kb + 2, r2, r1)) {
      kb += 2;
      break;
    }
  }
  failed = kb < nk;
  // the last block's commit covers every MMA issued before it
  const int last = failed ? kb - 1 : nk - 1;
  bool done = true;
  if (last >= 0) done = mbar_wait(smem_u32(&mbar[last & 1]), (last >> 1) & 1);
  cp_async_wait<0>();
  if (__syncthreads_or(!done)) failed = true;
  tc_fence_after();

  if (!failed) {
    // 16 warps: TMEM lane quarter q = warp % 4, column quarter cq = warp / 4
    const int q = wid & 3, cq = wid >> 2;
#pragma unroll
    for (int hm = 0; hm < 2; ++hm) {
      if (hm == 1 && !two) break;
      const int r = hm * 128 + 32 * q + lane;
      const uint32_t trow = tmem + hm * kBN + ((uint32_t)(32 * q) << 16);
      if (MODE == 1) {
        float gv[32], uv[32];
        tmem_ld32(trow + 32 * cq, gv);
        tmem_ld32(trow + kBN / 2 + 32 * cq, uv);
        if (r < rows) {
          uint16_t* dst = g.h_out + (int64_t)(row0 + r) * I + nt * (kBN / 2) + 32 * cq;
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            float h[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) h[i] = silu(gv[e + i]) * uv[e + i];
            *reinterpret_cast<uint4*>(dst + e) =
                make_uint4(bf2(h[0], h[4]), bf2(h[1], h[5]), bf2(h[2], h[6]), bf2(h[3], h[7]));
          }
        }
      } else {
        int64_t dst_row = 0;
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
        }
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          float v[32];
          tmem_ld32(trow + 64 * cq + c, v);
          if (r < rows) {
            uint16_t* dst = g.y_out + dst_row * H + nt * kBN + 64 * cq + c;
#pragma unroll
            for (int e = 0; e < 32; e += 8)
              *reinterpret_cast<uint4*>(dst + e) = make_uint4(
                  bf2(wgt * v[e], wgt * v[e + 1]), bf2(wgt * v[e + 2], wgt * v[e + 3]),
                  bf2(wgt * v[e + 4], wgt * v[e + 5]), bf2(wgt * v[e + 6], wgt * v[e + 7]));
          }
        }
      }
    }
  } else if (tid == 0 && g.err) {
    atomicOr(g.err, MOE_DERR_WAIT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (wid == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
}

}  // namespace

cudaError_t launch_grouped_gemm(int mode, const GemmArgs& a, int max_tiles, cudaStream_t st) {
  static bool attr_done[2][64] = {};
  const size_t smem = 1024 + (size_t)kStages * kABytes + 2 * (size_t)kBBytes;
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= 64) return cudaErrorInvalidDevice;
  if (mode == 1) {
    if (!attr_done[0][d]) {
      e = cudaFuncSetAttribute(grouped_gemm_kernel<1>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      attr_done[0][d] = true;
    }
    const dim3 grid(max_tiles, a.I / (kBN / 2));
    grouped_gemm_kernel<1><<<grid, kThreads, smem, st>>>(a);
  } else {
    if (!attr_done[1][d]) {
      e = cudaFuncSetAttribute(grouped_gemm_kernel<2>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      attr_done[1][d] = true;
    }
    const dim3 grid(max_tiles, a.H / kBN);
    grouped_gemm_kernel<2><<<grid, kThreads, smem, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace moe
