// Decode expert FFN as one persistent, cooperative kernel:
//   y[t] = sum_j w[t][j] * Wd_e (silu(Wg_e x_t) * (Wu_e x_t))  (+ shared(x_t))
// with int4 affine group-64 weights (Edge0 §3.1 "math convention") or MXFP4 /
// NVFP4 weights, every executed expert's term added once (FreeToken summary
// "core method": the partial sums of the cached and the direct sets merge
// exactly -- no term dropped or counted twice).  The same kernel, instantiated
// with FUSED, is the whole decode layer step: router logits, selection, the
// control step (CTA 0) and this FFN in one launch (below).
//
// Decode streams megabytes of packed weights against a few KB of
// activations; the kernel keeps HBM streaming and spends few SM
// instructions per weight:
//  * one CTA per SM for the whole call.  The CTA owns a balanced, contiguous
//    range of gate/up tiles (entry, 16 rows of I, all of H) and one of down
//    tiles (entry, RD rows of H, all of I).  A producer warp streams their
//    16 KB code stages and 2 KB scale blocks through a ring of shared-memory
//    slots with tiled TMA loads, gate/up first, then down, so the down
//    weights arrive while the gate/up tiles are still being computed;
//  * sixteen consumer warps each take one 64-column group of every stage
//    (two 16-row group tiles: gate and up of one row tile, or two down row
//    tiles) and run m16n8k16 fp16 MMAs with the tokens as the N columns.  A
//    code word (8 nibbles, columns c..c+7) becomes four fp16x2 A registers in
//    five integer instructions: an even column's nibble OR-ed under 0x6400
//    reads as 1024 + q, an odd column's nibble left in bits 4-7 under 0x5400
//    reads as 64 + q.  These offsets m_c are per-column constants, removed on
//    the fp32 accumulator together with the group's scale s and bias b:
//        sum_c (s q_c + b) x_c = s (D - O) + b X,
//        D = sum_c (m_c + q_c) x_c,  O = sum_c m_c x_c,  X = sum_c x_c;
//  * activations enter as fp16 B fragments, scaled by a power of two per
//    token (x) or per entry and token (h) so that |x'| < 1; for bf16 x the
//    scaled value is exact in fp16.  The scale is applied back in fp32;
//  * a gate/up tile's sixteen warp partials meet in shared memory and one
//    warp adds them in warp order and writes h = silu(g) * u for its rows;
//    once every CTA has written its h rows (a grid-wide count), each down tile
//    builds its entry's h fragments and every warp adds its rows' weighted
//    results into y with fp32 atomics: the routed terms of an output meet in
//    arrival order, so y repeats run to run within fp32 rounding, not bit for
//    bit (y is zeroed by the CTAs before that count);
//  * when the call carries the step's fill, a writer warp stores every landed
//    stage of an expert being filled into its new slot (TMA stores through the
//    slot pool's maps, the same boxes as the loads) before the stage goes back
//    to the producer.
// The CTAs wait on one another (a down tile on its entry's gate/up tiles), so
// the kernel is launched cooperatively and all CTAs are resident.  Every wait
// is bounded: after a time-out the CTA records the failure, its warps keep
// walking the same barriers without waiting or computing, and the last CTA to
// finish unmaps the experts filled in this step (their slots may hold a partial
// copy), so the cache never maps a slot whose blob was not written.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "control_common.cuh"
#include "moe_internal.cuh"
#include "route_select.cuh"
#include "stream_common.cuh"

namespace moe {
namespace {
using namespace sc;

constexpr int kCW = 16;                    // consumer warps
constexpr int kProdW = kCW;                // producer warp
constexpr int kFillW = kCW + 1;            // fill writer warp
constexpr int kThreads = (kCW + 2) * 32;
constexpr int kConsThreads = kCW * 32;
constexpr int kCodeBytes = 16384;          // int4 codes of one stage
constexpr int kScaleBytes = 2048;          // bf16 scales and biases of one stage
constexpr int kSlotBytes = kCodeBytes + kScaleBytes;  // 18 x 1024
constexpr int kMaxSt = 16;
constexpr int kMaxEnt = 128;
constexpr int kMaxTok = 8;
constexpr int kMaxIds = 512;
constexpr int kGuCols = 1024;              // H columns of one gate/up stage
constexpr size_t kDynBudget = 216 * 1024;  // + ~8 KB static, under the 227 KB per block

// Shared-memory plan and tile shapes of one launch.
struct CoopGeom {
  int nks;       // gate/up stages per tile: H / 1024
  int RD, KSD;   // down tile rows; down stage columns (of I)
  int nkd, ngs;  // down stages per tile; 64-column groups per down stage
  int nbd;       // TMA boxes per down stage: KSD / 256
  int nst;       // ring slots
  int frow;      // bytes per token row of B fragments: 2 max(H, I) + 16
  size_t o_frag, o_ox, o_red, smem;
};

CoopGeom coop_geom(int H, int I, int T) {
  CoopGeom g{};
  g.nks = H / kGuCols;
  if (I % 1024 == 0) {
    g.RD = 32;
    g.KSD = 1024;
  } else {
    g.RD = 64;
    g.KSD = 512;
  }
  g.nkd = I / g.KSD;
  g.ngs = g.KSD / 64;
  g.nbd = g.KSD / 256;
  const int mx = H > I ? H : I;
  g.frow = 2 * mx + 16;
  const size_t frag = (size_t)T * g.frow;
  const size_t ox = (size_t)(mx / 64) * kMaxTok * 8;
  // two partial-sum buffers: the ring between the consumer warps and a tile's reducer
  const size_t red = 2 * (size_t)kCW * 32 * T * 4;
  const size_t fixed = 1024 + frag + ox + red;
  const size_t left = kDynBudget > fixed ? kDynBudget - fixed : 0;
  int nst = (int)(left / kSlotBytes);
  if (nst > kMaxSt) nst = kMaxSt;
  if (nst >= 3) {
    g.nst = nst;
    g.o_frag = (size_t)nst * kSlotBytes;
    g.o_ox = g.o_frag + frag;
    g.o_red = g.o_ox + ox;
    g.smem = g.o_red + red + 1024;
    return g;
  }
  g.nst = 0;
  return g;
}

// Tensor maps per blob array (0 bank, 1 slot pool, 2 shared expert):
//   gu_code  u32 words [blob][gate/up][row of I][word of H/8], box 32 x 16 x 2
//            (4 KB), 128-byte swizzle
//   gu_scale u32 words [blob][gs,gb,us,ub][row of I][word of H/128], box 8 x 16 x 4
//   dn_code  u32 words [blob][row of H][word of I/8], box 32 x RD, swizzled
//   dn_scale u32 words [blob][ds,db][row of H][word of I/128], box KSD/128 x RD x 2
struct CoopMaps {
  CUtensorMap gu_code[3], gu_scale[3], dn_code[3], dn_scale[3];
};

// Masks and exponent words of the fp16 code conversion, held in registers
// (opaque to the compiler, so that it keeps them there across the loop):
// an even column's nibble OR-ed under 0x6400 reads as 1024 + q, an odd
// column's nibble, left in bits 4-7, under 0x5400 as 64 + q.
struct Cvt {
  uint32_t mev, kev, mod, kod;
};
__device__ __forceinline__ Cvt cvt_consts() {
  Cvt c;
  asm volatile("mov.b32 %0, 0x000F000F;" : "=r"(c.mev));
  asm volatile("mov.b32 %0, 0x64006400;" : "=r"(c.kev));
  asm volatile("mov.b32 %0, 0x00F000F0;" : "=r"(c.mod));
  asm volatile("mov.b32 %0, 0x54005400;" : "=r"(c.kod));
  return c;
}

// One m16n8k16 fp16 MMA whose A fragment is built from the lane's code words
// of rows g (wl) and g + 8 (wh): nibbles 0 and 4 (k slots 2t, 2t + 1) and
// nibbles 1 and 5 (k slots 2t + 8, 2t + 9), four LOP3s.  ZERO: D = A B, else
// D += A B.
template <bool ZERO>
__device__ __forceinline__ void mma_cvt(float (&d)[4], uint32_t wl, uint32_t wh, uint32_t b0,
                                        uint32_t b1, const Cvt& c) {
  if (ZERO) {
    asm("{\n .reg .b32 a0, a1, a2, a3;\n"
        " lop3.b32 a0, %4, %6, %7, 0xEA;\n lop3.b32 a1, %5, %6, %7, 0xEA;\n"
        " lop3.b32 a2, %4, %8, %9, 0xEA;\n lop3.b32 a3, %5, %8, %9, 0xEA;\n"
        " mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {a0,a1,a2,a3},"
        " {%10,%11}, {%12,%13,%14,%15};\n}"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(wl), "r"(wh), "r"(c.mev), "r"(c.kev), "r"(c.mod), "r"(c.kod), "r"(b0), "r"(b1),
          "f"(0.0f), "f"(0.0f), "f"(0.0f), "f"(0.0f));
  } else {
    asm("{\n .reg .b32 a0, a1, a2, a3;\n"
        " lop3.b32 a0, %4, %6, %7, 0xEA;\n lop3.b32 a1, %5, %6, %7, 0xEA;\n"
        " lop3.b32 a2, %4, %8, %9, 0xEA;\n lop3.b32 a3, %5, %8, %9, 0xEA;\n"
        " mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {a0,a1,a2,a3},"
        " {%10,%11}, {%0,%1,%2,%3};\n}"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(wl), "r"(wh), "r"(c.mev), "r"(c.kev), "r"(c.mod), "r"(c.kod), "r"(b0), "r"(b1));
  }
}

// Two 16-row x 64-column group tiles against one set of B registers:
// (l0, h0) and (l1, h1) are the lane's two code words of rows g and g + 8 of
// each tile; b holds [word j][half][b0, b1].  Word j, half 0 feeds nibbles
// (0, 4) and (1, 5), half 1 (after a shift by 8) nibbles (2, 6) and (3, 7),
// matching the B fragment built for the same columns.  d0, d1 are written.
__device__ __forceinline__ void group2(float (&d0)[4], float (&d1)[4], uint2 l0, uint2 h0,
                                       uint2 l1, uint2 h1, const uint32_t (&b)[8],
                                       const Cvt& c) {
  mma_cvt<true>(d0, l0.x, h0.x, b[0], b[1], c);
  mma_cvt<true>(d1, l1.x, h1.x, b[0], b[1], c);
  mma_cvt<false>(d0, l0.x >> 8, h0.x >> 8, b[2], b[3], c);
  mma_cvt<false>(d1, l1.x >> 8, h1.x >> 8, b[2], b[3], c);
  mma_cvt<false>(d0, l0.y, h0.y, b[4], b[5], c);
  mma_cvt<false>(d1, l1.y, h1.y, b[4], b[5], c);
  mma_cvt<false>(d0, l0.y >> 8, h0.y >> 8, b[6], b[7], c);
  mma_cvt<false>(d1, l1.y >> 8, h1.y >> 8, b[6], b[7], c);
}

// ------------------------------------------------------------ FP4 operands
// An FP4 weight is e2m1(code) * block scale.  Both factors are exact in fp16
// and so is their product for an NVFP4 block (|e2m1| <= 6, E4M3 in
// [2^-9, 448]); an MXFP4 block's E8M0 power of two enters as 2^(e - 127 + 8)
// (the 2^-8 is applied back in fp32), exact for E8M0 bytes 95..134.  The
// product goes into the MMA's A operand, so the fp32 accumulator sums
// dequantised weights times x with no per-block correction; the NVFP4 matrix
// scale is applied in fp32 after the sum.
constexpr int kMxBias = 8;

// fp16x2 {s, s} of one block scale byte.
template <int FMT>
__device__ __forceinline__ uint32_t fp4_scale2(uint32_t byte) {
  uint32_t r;
  if constexpr (FMT == MOE_FORMAT_NVFP4) {
    const uint16_t pair = (uint16_t)(byte | (byte << 8));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(pair));
  } else {
    const int e = (int)byte - 127 + kMxBias;  // 2^e in fp16
    uint32_t h;
    if (byte == 255u) h = 0x7E00u;           // NaN
    else if (e > 15) h = 0x7C00u;            // beyond fp16: inf
    else if (e >= -14) h = (uint32_t)(e + 15) << 10;
    else if (e >= -24) h = 1u << (e + 24);   // fp16 subnormal, still exact
    else h = 0u;
    r = h | (h << 16);
  }
  return r;
}

// D += A B (m16n8k16, fp16 in, fp32 accumulate) with A from E2M1 codes:
// word wl of row g and wh of row g + 8 (8 codes each, columns 8j .. 8j + 7 of
// the lane's 16), bytes 2 HB (columns +4HB, +4HB+1: k slots 2t, 2t+1) and
// 2 HB + 1 (+4HB+2, +4HB+3: k slots 2t+8, 2t+9), each times its row's block
// scale (sl, sh).
template <int HB>
__device__ __forceinline__ void mma_fp4(float (&d)[4], uint32_t wl, uint32_t wh, uint32_t sl,
                                        uint32_t sh, uint32_t b0, uint32_t b1) {
  if (HB == 0) {
    asm("{\n .reg .b8 l0, l1, l2, l3, h0, h1, h2, h3;\n .reg .b32 a0, a1, a2, a3;\n"
        " mov.b32 {l0, l1, l2, l3}, %4;\n mov.b32 {h0, h1, h2, h3}, %5;\n"
        " cvt.rn.f16x2.e2m1x2 a0, l0;\n cvt.rn.f16x2.e2m1x2 a1, h0;\n"
        " cvt.rn.f16x2.e2m1x2 a2, l1;\n cvt.rn.f16x2.e2m1x2 a3, h1;\n"
        " mul.rn.f16x2 a0, a0, %6;\n mul.rn.f16x2 a1, a1, %7;\n"
        " mul.rn.f16x2 a2, a2, %6;\n mul.rn.f16x2 a3, a3, %7;\n"
        " mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {a0,a1,a2,a3},"
        " {%8,%9}, {%0,%1,%2,%3};\n}"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(wl), "r"(wh), "r"(sl), "r"(sh), "r"(b0), "r"(b1));
  } else {
    asm("{\n .reg .b8 l0, l1, l2, l3, h0, h1, h2, h3;\n .reg .b32 a0, a1, a2, a3;\n"
        " mov.b32 {l0, l1, l2, l3}, %4;\n mov.b32 {h0, h1, h2, h3}, %5;\n"
        " cvt.rn.f16x2.e2m1x2 a0, l2;\n cvt.rn.f16x2.e2m1x2 a1, h2;\n"
        " cvt.rn.f16x2.e2m1x2 a2, l3;\n cvt.rn.f16x2.e2m1x2 a3, h3;\n"
        " mul.rn.f16x2 a0, a0, %6;\n mul.rn.f16x2 a1, a1, %7;\n"
        " mul.rn.f16x2 a2, a2, %6;\n mul.rn.f16x2 a3, a3, %7;\n"
        " mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {a0,a1,a2,a3},"
        " {%8,%9}, {%0,%1,%2,%3};\n}"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(wl), "r"(wh), "r"(sl), "r"(sh), "r"(b0), "r"(b1));
  }
}

// Two 16-row x 64-column FP4 group tiles against one set of B registers, added
// into d0, d1: (l0, h0) are the lane's codes of rows g and g + 8 of tile 0
// (16 columns, 8 bytes each) with scales (s0l, s0h), likewise tile 1; b holds
// the 16 x values of the lane's columns in order (MMA m: b[2m], b[2m + 1]).
__device__ __forceinline__ void group2_fp4(float (&d0)[4], float (&d1)[4], uint2 l0, uint2 h0,
                                           uint2 l1, uint2 h1, uint32_t s0l, uint32_t s0h,
                                           uint32_t s1l, uint32_t s1h, const uint32_t (&b)[8]) {
  mma_fp4<0>(d0, l0.x, h0.x, s0l, s0h, b[0], b[1]);
  mma_fp4<0>(d1, l1.x, h1.x, s1l, s1h, b[0], b[1]);
  mma_fp4<1>(d0, l0.x, h0.x, s0l, s0h, b[2], b[3]);
  mma_fp4<1>(d1, l1.x, h1.x, s1l, s1h, b[2], b[3]);
  mma_fp4<0>(d0, l0.y, h0.y, s0l, s0h, b[4], b[5]);
  mma_fp4<0>(d1, l1.y, h1.y, s1l, s1h, b[4], b[5]);
  mma_fp4<1>(d0, l0.y, h0.y, s0l, s0h, b[6], b[7]);
  mma_fp4<1>(d1, l1.y, h1.y, s1l, s1h, b[6], b[7]);
}

__device__ __forceinline__ uint32_t h2u(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 1 / P with P the smallest power of two above m (|v| / P < 1); 1 when m is
// zero, denormal or not finite.
__device__ __forceinline__ float inv_pow2_above(float m) {
  const uint32_t u = __float_as_uint(m);
  const int e = (int)((u >> 23) & 0xFFu);
  if (!(m > 0.0f) || e == 0 || e == 0xFF) return 1.0f;
  int ep = e + 1;  // biased exponent of P
  if (ep > 253) ep = 253;
  return __uint_as_float((uint32_t)(254 - ep) << 23);
}

// B fragment item: 16 columns (c0 .. c0 + 15, c0 = 64 G + 16 t4) of one token
// row, already scaled, rounded to fp16 and stored as [word j][half][b0, b1];
// returns their contributions to O (weights 1024 even / 64 odd columns) and X.
__device__ __forceinline__ void frag_item(const float (&v)[16], unsigned char* dst, float& o,
                                          float& x) {
  uint32_t r[8];
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = 8 * j + 2 * h;
      r[4 * j + 2 * h] = h2u(v[c], v[c + 4]);
      r[4 * j + 2 * h + 1] = h2u(v[c + 1], v[c + 5]);
    }
  reinterpret_cast<uint4*>(dst)[0] = make_uint4(r[0], r[1], r[2], r[3]);
  reinterpret_cast<uint4*>(dst)[1] = make_uint4(r[4], r[5], r[6], r[7]);
  o = 0.0f;
  x = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float q = __half2float(__float2half_rn(v[i]));
    o += ((i & 1) ? 64.0f : 1024.0f) * q;
    x += q;
  }
}

// B fragment item of the FP4 path: 16 columns of one token row, already
// scaled, rounded to fp16 and stored in column order.
__device__ __forceinline__ void frag_plain(const float (&v)[16], unsigned char* dst) {
  uint32_t r[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) r[j] = h2u(v[2 * j], v[2 * j + 1]);
  reinterpret_cast<uint4*>(dst)[0] = make_uint4(r[0], r[1], r[2], r[3]);
  reinterpret_cast<uint4*>(dst)[1] = make_uint4(r[4], r[5], r[6], r[7]);
}

__device__ __forceinline__ void cons_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsThreads) : "memory");
}

__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait (about one second of SM clock) until *p >= target, then an
// acquire fence.  One thread polls a grid-wide count with relaxed loads.
__device__ bool wait_count(const uint32_t* p, uint32_t target) {
  long long t0 = 0;
  for (uint32_t i = 0; i < kSpin; ++i) {
    if (ld_relaxed(p) >= target) {
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      return true;
    }
    if ((i & 255u) == 255u) {
      const long long t = clock64();
      if (t0 == 0) t0 = t;
      else if (t - t0 > kWaitCycles) return false;
    }
  }
  return false;
}

__device__ __forceinline__ void red_release_gpu_add(uint32_t* p) { red_release_add(p, 1u); }

struct ConsSync {
  __device__ void operator()() const { cons_sync(); }
};

// One-kernel layer step: CTA 0's consumer warps run the selection and the
// control step in the ring's shared memory (CTA 0 streams no weights).
constexpr int kCtlK = 8;  // victims per step (KMAX of the victim lists)
using CtlSh = ctl::CtlShared<kCtlK, kConsThreads>;
constexpr int kWideK = 8;  // the wide (one-token) selection's largest k
struct SelScratch {
  float a[kMaxTok][32 * 8];
  float b[kMaxTok][rsel::kMaxK], c[kMaxTok][rsel::kMaxK];
  float sum[kMaxTok];
  int32_t slot[256];  // slot_of_id of the layer's E experts before the step
  // the wide selection: each warp's k best (order key, expert id, value) at
  // position w k + r, and the group scores
  uint32_t ckey[kCW * kWideK];
  int32_t cid[kCW * kWideK];
  float cval[kCW * kWideK];
  float gs[kCW];
};
static_assert(sizeof(CtlSh) + sizeof(SelScratch) <= 3 * (size_t)kSlotBytes,
              "control step scratch must fit in the smallest ring");

// Router selection of a single token by E / 32 warps (E % 32 == 0, E <= 512,
// k <= 8): warp w holds experts 32 w + lane.  The same decisions and weights
// as rsel::softmax_token / rsel::sigmoid_group_token (the order of rsel::better
// everywhere): each warp takes its own k best, writes them at positions
// w k + r (ascending expert id among equal scores), and warp 0 takes the k best
// of those.  Sigmoid-group with one warp per group (E / n_groups == 32): the
// group scores (sum of the two largest selection scores) meet in shared memory
// first, and only the kept groups' warps put forward candidates.  All consumer
// threads call it; warp 0 writes ids / weights.
__device__ void select_wide(const LayerFuse& lf, int E, int k, int32_t* ids, float* wts,
                            SelScratch& ss) {
  const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
  const int NW = E >> 5;
  const bool sig = lf.router != MOE_ROUTER_SOFTMAX_TOPK;
  float v = 0.0f, sv = 0.0f;  // this lane's logit (softmax) or sigmoid score
  uint32_t key = 0u;
  if (wid < NW) {
    const int e = 32 * wid + lane;
    const float l = __ldcg(lf.logits + e);
    if (sig) {
      const float bias = lf.sel_bias ? __ldg(lf.sel_bias + e) : 0.0f;
      sv = rsel::moe_sigmoid(l);
      v = __fadd_rn(sv, bias);  // selection score
      // the group's two largest selection scores (t2 == t1 when it appears twice)
      float t1 = v, t2 = -FLT_MAX;
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) {
        const float b1 = __shfl_xor_sync(0xffffffffu, t1, d);
        const float b2 = __shfl_xor_sync(0xffffffffu, t2, d);
        t2 = fmaxf(fminf(t1, b1), fmaxf(t2, b2));
        t1 = fmaxf(t1, b1);
      }
      if (lane == 0) ss.gs[wid] = __fadd_rn(t1, t2);
    } else {
      v = l;
      sv = l;
    }
    key = rsel::ord_key(v);
  }
  if (sig) {
    cons_sync();
    // this warp's group kept: fewer than topk_groups groups ahead of it
    if (wid < NW) {
      const float mine = ss.gs[wid];
      int ahead = 0;
      for (int h = 0; h < NW; ++h) ahead += rsel::better(ss.gs[h], h, mine, wid) ? 1 : 0;
      if (ahead >= lf.topk_groups) key = 0u;
    }
  }
  if (wid < NW) {
    // the warp's k best: a winner lane drops out; rank r goes to position w k + r
    for (int r = 0; r < k; ++r) {
      const uint32_t M = __reduce_max_sync(0xffffffffu, key);
      const uint32_t me = (M != 0u && key == M) ? (uint32_t)lane : 0xffffffffu;
      const uint32_t wl = __reduce_min_sync(0xffffffffu, me);
      const float wv = __shfl_sync(0xffffffffu, sv, wl & 31);
      if (lane == 0) {
        ss.ckey[wid * kWideK + r] = M;
        ss.cid[wid * kWideK + r] = M != 0u ? 32 * wid + (int)wl : 0x7fffffff;
        ss.cval[wid * kWideK + r] = wv;
      }
      if ((uint32_t)lane == wl) key = 0u;
    }
  }
  cons_sync();
  if (wid == 0) {
    // up to 16 x 8 candidates, four per lane at positions lane + 32 i
    constexpr int CPL = kCW * kWideK / 32;
    uint32_t ck[CPL], cs[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int pos = lane + 32 * i, w = pos / kWideK, r = pos % kWideK;
      ck[i] = (w < NW && r < k) ? ss.ckey[w * kWideK + r] : 0u;
      cs[i] = (uint32_t)i;
    }
    rsel::lane_sort_desc<CPL>(ck, cs);
    int rid[2];
    rsel::warp_topk<CPL>(ck, cs, k, rid);  // positions w k' + r (k' = kWideK)
    const int pos = rid[0];
    const bool got = lane < k && pos != 0x7fffffff;
    const int e = got ? ss.cid[pos] : 0x7fffffff;
    const float val = got ? ss.cval[pos] : 0.0f;
    float S = 0.0f;
    if (sig) {
      for (int r = 0; r < k; ++r) S = __fadd_rn(S, __shfl_sync(0xffffffffu, val, r));
      if (lane < k) {
        ids[lane] = e;
        wts[lane] = __fmul_rn(__fdiv_rn(val, S), lf.scale);
      }
    } else {
      const float top = __shfl_sync(0xffffffffu, val, 0);
      const float ex = lane < k ? rsel::moe_exp(__fsub_rn(val, top)) : 0.0f;
      for (int r = 0; r < k; ++r) S = __fadd_rn(S, __shfl_sync(0xffffffffu, ex, r));
      if (lane < k) {
        ids[lane] = e;
        wts[lane] = __fdiv_rn(ex, S);
      }
    }
  }
}

// Every CTA of the one-kernel layer step, consumer threads (tid < 512), once
// every CTA's logits are stored: the router selection (one warp per token,
// into s_ids / s_wts), then the dedup, ranks and hit / miss of the routed ids
// against the slot table read before the logits count (FreeToken summary
// "method steps").  Every CTA takes the same decisions from the same data, so
// no CTA waits for another's plan; CTA 0 (ctl) also writes the routing
// outputs, moves the hits' recency stamps and keeps the misses for the
// victim scan.  Returns false when the logits never all arrived.
template <bool CTL>
__device__ bool layer_route_classify(const FfnArgs& a, const LayerFuse& lf, CtlSh& cs,
                                     SelScratch& ss, int32_t* s_ids, float* s_wts) {
  const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
  const int T = a.T, k = a.k, E = a.E, n = T * k;
  if (tid == 0) {
    cs.bad = 0;
    cs.nu = 0;
    cs.nh = 0;
    cs.nm = 0;
    cs.nu = wait_count(lf.sync + kSyncLogits, gridDim.x) ? 0 : -1;  // every CTA's logits
  }
  cons_sync();
  if (cs.nu < 0) return false;
  const bool wide = T == 1 && (E & 31) == 0 && E <= 32 * kCW && k <= kWideK &&
                    (lf.router == MOE_ROUTER_SOFTMAX_TOPK || E / lf.n_groups == 32);
  if (wide) {
    select_wide(lf, E, k, s_ids, s_wts, ss);
  } else if (wid < T) {
    if (lf.router == MOE_ROUTER_SOFTMAX_TOPK)
      rsel::softmax_token<8>(lf.logits, wid, E, k, s_ids, s_wts, ss.b[wid], ss.c[wid],
                             &ss.sum[wid]);
    else
      rsel::sigmoid_group_token<8>(lf.logits, lf.sel_bias, wid, E, lf.n_groups, lf.topk_groups, k,
                                   lf.scale, s_ids, s_wts, ss.a[wid], ss.b[wid], &ss.sum[wid]);
  }
  cons_sync();
  if (wid == 0) {
    const int32_t e = lane < n ? s_ids[lane] : 0;
    const int base = a.layer * E;
    ctl::ctl_classify_warp<CTL, kCtlK, kConsThreads>(
        lf.c, cs, n, e, cs.now, [&](int32_t u) { return ss.slot[u - base]; });
  } else if (CTL && wid == 1 && lane < n) {
    lf.ids_out[lane] = s_ids[lane];
    lf.wts_out[lane] = s_wts[lane];
  }
  cons_sync();
  return true;
}

// CTA 0 of the one-kernel layer step, after the classification: the victim
// scan and the slot-table update (every CTA has read the slot table before
// the logits count), then the fill set is published for the fill writers.
__device__ void layer_evict(const LayerFuse& lf, CtlSh& cs,
                            const uint32_t (&early)[CtlSh::NE],
                            const int32_t (&early_id)[CtlSh::NE]) {
  ctl::ctl_evict<kCtlK, kConsThreads>(lf.c, cs, cs.now, cs.nu, cs.nh, cs.nm, early, early_id,
                                      ConsSync{});
  cons_sync();
  if (threadIdx.x == 0) red_release_gpu_add(lf.sync + kSyncFill);  // the plan and the tables
}

template <bool FUSED, int FMT>
__global__ void __launch_bounds__(kThreads, 1)
    ffn_coop_kernel(FfnArgs a, CoopGeom geo, const __grid_constant__ CoopMaps maps, LayerFuse lf) {
  // bytes of scales per stage; FP4: elements per block scale
  constexpr int kSB = FMT == MOE_FORMAT_MXFP4 ? 1024 : 2048;
  constexpr int kBlk = FMT == MOE_FORMAT_NVFP4 ? 16 : 32;
  // FP4: per entry, the fp32 factors applied after the sums of gate, up and
  // down (the NVFP4 matrix scales; 2^-8 for MXFP4's shifted block scales)
  __shared__ float s_fac[FMT != MOE_FORMAT_INT4 ? kMaxEnt : 1][3];
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full[kMaxSt], empty[kMaxSt], rfull[2], rfree[2];
  __shared__ int s_map[kMaxEnt], s_bi[kMaxEnt], s_fs[kMaxEnt], s_uid[kMaxEnt];
  __shared__ int s_ntok[kMaxEnt];
  __shared__ int8_t s_tok[kMaxEnt][kMaxTok];
  __shared__ int32_t s_ids[kMaxIds];
  __shared__ float s_wts[kMaxIds];
  __shared__ uint32_t s_vmax[kMaxTok];  // max |x| (float bits) per token
  __shared__ float s_px[kMaxTok];       // power of two applied back per token (x)
  // per token slot of the current down entry: 1 / the power of two applied to
  // h, and routing weight times that power of two
  __shared__ float s_ih[kMaxTok], s_wp[kMaxTok];
  __shared__ int s_fail;
  __shared__ __align__(16) uint32_t s_zero[8];  // B fragment and (O, X) of an absent token
  __shared__ __align__(8) uint64_t s_lgbar;     // one-kernel step: the staged router rows
  // the first ring slot that generic-proxy code used in this launch (routing
  // scratch, staged rows): the producer fences once before its TMA reuses it
  __shared__ int s_gen_slot;
  const int H = a.H, I = a.I, T = a.T, k = a.k;
  const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
  const int nst = geo.nst;
  unsigned char* smem = smem_raw + ((1024u - (su32(smem_raw) & 1023u)) & 1023u);
  unsigned char* ring = smem;
  unsigned char* frag = smem + geo.o_frag;
  float2* ox = reinterpret_cast<float2*>(smem + geo.o_ox);
  float* red = reinterpret_cast<float*>(smem + geo.o_red);
  // counter words (zero at launch): CTAs past their gate/up range, (unused),
  // completed CTAs, failure flag, per (entry, token slot) max |h| (float bits)
  uint32_t* gu_cnt = a.ctr;
  uint32_t* done = a.ctr + 2;
  uint32_t* failw = a.ctr + 3;
  uint32_t* hmax = a.ctr + 4;

  if (tid == 0) {
    const int nrel = kCW + (a.fill_fused ? 1 : 0);  // warps that release a stage
    for (int i = 0; i < nst; ++i) {
      bar_init(su32(&full[i]), 1);
      bar_init(su32(&empty[i]), nrel);
    }
    for (int i = 0; i < 2; ++i) {
      bar_init(su32(&rfull[i]), kCW);  // every consumer warp's partial is written
      bar_init(su32(&rfree[i]), 1);    // the tile's reducer has read them
    }
    bar_init(su32(&s_lgbar), 1);
    s_gen_slot = FUSED ? nst - 3 : nst;
    s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the tensor maps are kernel parameters: fetch them before the wait
  if (wid == kProdW && lane < 12) {
    const CUtensorMap* mp = lane < 3   ? &maps.gu_code[lane]
                            : lane < 6 ? &maps.gu_scale[lane - 3]
                            : lane < 9 ? &maps.dn_code[lane - 6]
                                       : &maps.dn_scale[lane - 9];
    tma_prefetch_map(mp);
  }
  if (tid < kMaxTok) s_vmax[tid] = 0u;
  if (tid < 8) s_zero[tid] = 0u;
  // x as fp16 B fragments of this CTA (scaled by a power of two per token),
  // the per-group sums O and X of the scaled, rounded values, and y = 0 on
  // this CTA's slice of the NY CTAs that run tiles (consumer threads)
  auto zero_y = [&](unsigned yb, unsigned NY) {
    const unsigned ny = (unsigned)T * H;
    for (unsigned i = yb * ny / NY + tid; i < (yb + 1) * ny / NY; i += kConsThreads) a.y[i] = 0.0f;
  };
  auto prep_x = [&](unsigned yb, unsigned NY) {
    const int ctid = tid;
    // max |x| per token: a warp's lanes read 32 consecutive 8-element chunks of x
    // (one token: H / 8 is a multiple of 32), four chunks per lane in flight
    const int cpt = H / 8, nch = T * cpt;
    const uint4* xq = reinterpret_cast<const uint4*>(a.x);
    for (int i0 = ctid; i0 < nch; i0 += 4 * kConsThreads) {
      uint4 v4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int idx = i0 + u * kConsThreads;
        v4[u] = idx < nch ? __ldg(xq + idx) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int idx = i0 + u * kConsThreads;
        if (idx >= nch) break;  // (the same for every lane of the warp)
        const uint32_t w4[4] = {v4[u].x, v4[u].y, v4[u].z, v4[u].w};
        uint32_t m = 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          m = max(m, (w4[q] << 16) & 0x7FFFFFFFu);
          m = max(m, w4[q] & 0x7FFF0000u);
        }
        m = __reduce_max_sync(0xffffffffu, m);
        if (lane == 0) atomicMax(&s_vmax[idx / cpt], m);
      }
    }
    cons_sync();
    if (ctid < T) s_px[ctid] = 1.0f / inv_pow2_above(__uint_as_float(s_vmax[ctid]));
    // the fragments, two items per thread with both items' loads in flight
    const int ng = H / 64, n_items = T * ng * 4;
    for (int b0 = 0; b0 < n_items; b0 += 2 * kConsThreads) {
      uint4 pv[2][2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int it = b0 + u * kConsThreads + ctid;
        if (it < n_items) {
          const int t = it / (ng * 4), rem = it - t * ng * 4, G = rem >> 2, q4 = rem & 3;
          const uint4* px = reinterpret_cast<const uint4*>(a.x + (int64_t)t * H + G * 64 + q4 * 16);
          pv[u][0] = __ldg(px);
          pv[u][1] = __ldg(px + 1);
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int it = b0 + u * kConsThreads + ctid;
        const bool in = it < n_items;
        const int t = in ? it / (ng * 4) : 0, rem = it - t * ng * 4, G = rem >> 2, q4 = rem & 3;
        float v[16];
        float o = 0.0f, xs = 0.0f;
        if (in) {
          const float sc = inv_pow2_above(__uint_as_float(s_vmax[t]));
          const uint4 p0 = pv[u][0], p1 = pv[u][1];
          const uint32_t wv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            v[2 * i] = __uint_as_float(wv[i] << 16) * sc;
            v[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u) * sc;
          }
          if constexpr (FMT == MOE_FORMAT_INT4)
            frag_item(v, frag + (size_t)t * geo.frow + G * 128 + q4 * 32, o, xs);
          else
            frag_plain(v, frag + (size_t)t * geo.frow + G * 128 + q4 * 32);
        }
        o += __shfl_xor_sync(0xffffffffu, o, 1);
        o += __shfl_xor_sync(0xffffffffu, o, 2);
        xs += __shfl_xor_sync(0xffffffffu, xs, 1);
        xs += __shfl_xor_sync(0xffffffffu, xs, 2);
        if (in && q4 == 0) ox[G * kMaxTok + t] = make_float2(o, xs);
      }
    }
    // y starts at zero (ordered before the down tiles' adds by the grid-wide
    // gate/up count; the one-kernel step zeroes it before its logits count)
    if (!FUSED) zero_y(yb, NY);
    cons_sync();
  };

  // FP4: entry r's fp32 factors (map m, blob index bi)
  auto set_factors = [&](int r, int m, int bi) {
    if constexpr (FMT == MOE_FORMAT_NVFP4) {
      const uint8_t* base = m == 0 ? a.bank : m == 1 ? a.pool : a.shared;
      const float* mat = reinterpret_cast<const float*>(
          base + (int64_t)bi * a.blob_bytes + fp4_offsets(H, I, FMT).mat);
      s_fac[r][0] = __ldg(mat);
      s_fac[r][1] = __ldg(mat + 1);
      s_fac[r][2] = __ldg(mat + 2);
    } else if constexpr (FMT == MOE_FORMAT_MXFP4) {
      s_fac[r][0] = s_fac[r][1] = s_fac[r][2] = 1.0f / (float)(1 << kMxBias);
    }
  };

  const unsigned Gall = gridDim.x;
  // CTAs that run tiles: all of them, or all but CTA 0 in the one-kernel layer step
  const unsigned G = FUSED ? Gall - 1 : Gall, b = FUSED ? blockIdx.x - 1 : blockIdx.x;
  const bool ctl_cta = FUSED && blockIdx.x == 0;
  int n_uniq = 0, n_exec = 0;
  const int n_ids = T * k;
  if constexpr (FUSED) {
    // ------------------------------------------- one-kernel layer step
    uint32_t* sync = lf.sync;
    uint32_t early[CtlSh::NE];
    int32_t early_id[CtlSh::NE];
    // the routing scratch in the ring's last three slots: the stream fills the
    // first slots first, so its opening stages do not wait for a proxy fence
    unsigned char* scr = ring + (size_t)(nst - 3) * kSlotBytes;
    CtlSh& cs = *reinterpret_cast<CtlSh*>(scr);
    SelScratch& ss = *reinterpret_cast<SelScratch*>(scr + sizeof(CtlSh));
    griddep_wait();  // x, the cache tables and the pool of the previous kernels
    // the next kernel may be scheduled now: its CTAs start on SMs this grid
    // frees and wait for its completion before reading anything
    griddep_launch();
    if (wid < kCW) {
      const int E = a.E, np = T * E;
      if (ctl_cta) {
        // the victim scan's first stamps, and the step's clock
        ctl::ctl_early_loads<CtlSh::NE, kConsThreads>(lf.c, early, early_id);
        for (int i = tid; i < (int)(sizeof(cs.shit) / 4); i += kConsThreads) cs.shit[i] = 0u;
        if (tid == 0) {
          cs.now = lf.c.clock[0] + 1u;
          lf.c.clock[0] = cs.now;
        }
      }
      // the layer's slot table before the step (read before the logits count:
      // CTA 0 changes it only after every CTA has arrived there)
      for (int i = tid; i < E; i += kConsThreads) ss.slot[i] = lf.c.slot_of_id[a.layer * E + i];
      // router logits (the fixed order of every router path): pair p = (t, e)
      // on CTA p % Gall, warp p / Gall.  Past 256 chunks per row (a warp would
      // load its two rows in several rounds) the CTA's x rows and router rows
      // are first staged in the ring's free slots by bulk copies: one round trip.
      const int mine = np > (int)blockIdx.x ? (np - 1 - (int)blockIdx.x) / (int)Gall + 1 : 0;
      const uint32_t rowb = (uint32_t)H * 2u;
      const int nsl = (int)(((size_t)(T + mine) * rowb + kSlotBytes - 1) / kSlotBytes);
      const bool staged = H > 2048 && mine <= kCW && nsl <= nst - 3;
      unsigned char* stg = scr - (size_t)nsl * kSlotBytes;  // the slots before the scratch
      if (staged) {
        if (tid == 0) {
          s_gen_slot = nst - 3 - nsl;
          bar_expect(su32(&s_lgbar), (uint32_t)(T + mine) * rowb);
          for (int t = 0; t < T; ++t)
            bulk_g2s(su32(stg + (size_t)t * rowb), a.x + (size_t)t * H, rowb, su32(&s_lgbar));
          for (int i = 0; i < mine; ++i) {
            const int p = (int)blockIdx.x + (int)Gall * i, e = p % E;
            bulk_g2s(su32(stg + (size_t)(T + i) * rowb), lf.w_router + (size_t)e * H, rowb,
                     su32(&s_lgbar));
          }
        }
        const bool got = warp_wait(su32(&s_lgbar), 0);
        if (wid < mine && got) {
          const int p = (int)blockIdx.x + (int)Gall * wid, t = p / E;
          const float v = rsel::router_dot_smem(reinterpret_cast<const uint4*>(stg + (size_t)t * rowb),
                                                reinterpret_cast<const uint4*>(stg + (size_t)(T + wid) * rowb), H);
          if (lane == 0) lf.logits[p] = v;
        }
        if (!got && lane == 0) s_fail = 1;
      } else {
        for (int p = (int)blockIdx.x + (int)Gall * wid; p < np; p += (int)Gall * kCW) {
          const int t = p / E, e = p - t * E;
          const float v =
              rsel::router_dot_warp(a.x + (size_t)t * H, lf.w_router + (size_t)e * H, H);
          if (lane == 0) lf.logits[p] = v;
        }
      }
      // y starts at zero: ordered before every down tile's adds by the logits count,
      // which every CTA waits for before its first tile
      if (!ctl_cta) zero_y(b, G);
      cons_sync();
      if (tid == 0) red_release_gpu_add(sync + kSyncLogits);
      if (!ctl_cta) prep_x(b, G);
      const bool routed = ctl_cta ? layer_route_classify<true>(a, lf, cs, ss, s_ids, s_wts)
                                  : layer_route_classify<false>(a, lf, cs, ss, s_ids, s_wts);
      if (!routed) {
        if (tid == 0) s_fail = 1;
      } else if (!ctl_cta) {
        // the entries: ranked unique ids, read from their slot (hit) or the bank
        n_uniq = cs.nu;
        n_exec = n_uniq + a.has_shared;
        if (tid < n_exec) {
          const int r = tid;
          int mi = 2, bi = 0, uid = -1;
          if (r < n_uniq) {
            uid = cs.suniq[r];
            const int32_t slot = cs.sslot[r];
            mi = slot >= 0 ? 1 : 0;
            bi = slot >= 0 ? slot : uid;
          }
          s_map[r] = mi;
          s_bi[r] = bi;
          s_fs[r] = -1;  // an F entry's slot: learnt by the fill writer
          s_uid[r] = uid;
          set_factors(r, mi, bi);
        }
      } else {
        layer_evict(lf, cs, early, early_id);
      }
    }
    __syncthreads();
    if (!ctl_cta && !s_fail) {
      n_uniq = cs.nu;
      n_exec = n_uniq + a.has_shared;
    }
  } else {
    griddep_wait();  // the plan (and the cleared counters) of the previous kernels
    griddep_launch();
    n_uniq = a.counts[0];
    n_exec = n_uniq + a.has_shared;
    for (int i = tid; i < n_ids; i += kThreads) {
      s_ids[i] = a.ids[i];
      s_wts[i] = a.weights[i];
    }
    if (tid < n_exec) {
      // where entry r's weights are read and the slot an F entry is written to
      const int r = tid;
      int mi = 2, bi = 0, uid = -1;
      int32_t fs = -1;
      if (r < n_uniq) {
        uid = a.uniq[r];
        const int32_t slot = ffn_slot(a, uid, &fs);
        mi = slot >= 0 ? 1 : 0;
        bi = slot >= 0 ? slot : uid;
      }
      s_map[r] = mi;
      s_bi[r] = bi;
      s_fs[r] = fs;
      s_uid[r] = uid;
      set_factors(r, mi, bi);
    }
  }
  __syncthreads();

  const int tpe_gu = I / 16, tpe_dn = H / geo.RD;
  const int n_gu = ctl_cta ? 0 : n_exec * tpe_gu, n_dn = ctl_cta ? 0 : n_exec * tpe_dn;
  // balanced contiguous ranges (32-bit: tiles x CTAs stays below 2^32)
  const int gu_lo = (int)(b * (unsigned)n_gu / G), gu_hi = (int)((b + 1) * (unsigned)n_gu / G);
  const int dn_lo = (int)(b * (unsigned)n_dn / G), dn_hi = (int)((b + 1) * (unsigned)n_dn / G);
  const int nks = geo.nks, nkd = geo.nkd, RD = geo.RD, KSD = geo.KSD;
  const int base = a.layer * a.E;

  if (wid == kProdW) {
    // ------------------------------------------------------------ producer
    int n = 0, s = 0, rnd = 0;  // stages issued; ring slot and round of stage n
    // slots from gen_slot on held generic-proxy data (routing scratch, staged router
    // rows): one proxy fence orders those accesses before the first TMA write there
    const int gen_slot = s_gen_slot;
    bool fenced = false;
    bool ok = !a.inject_stall;  // test hook: no copies, every wait runs out
    const uint64_t pol = l2_evict_first();  // weights are read once per call
    auto slot_ready = [&]() {
      bool r = true;
      if (lane == 0) {
        r = rnd == 0 || bar_wait(su32(&empty[s]), (rnd - 1) & 1);
        if (r) bar_expect(su32(&full[s]), kCodeBytes + kSB);
      }
      if (!fenced && s >= gen_slot) {
        fence_proxy_async_smem();
        fenced = true;
      }
      return __shfl_sync(0xffffffffu, r, 0) != 0;
    };
    auto advance = [&]() {
      ++n;
      if (++s == nst) {
        s = 0;
        ++rnd;
      }
    };
    for (int tile = gu_lo; ok && tile < gu_hi; ++tile) {
      const int r = tile / tpe_gu, row0 = (tile % tpe_gu) * 16, m = s_map[r], bi = s_bi[r];
      for (int ks = 0; ks < nks; ++ks) {
        if (!(ok = slot_ready())) break;
        const uint32_t dst = su32(ring + (size_t)s * kSlotBytes);
        if (lane < 4)
          tma_load_4d_ef(dst + lane * 4096, &maps.gu_code[m], ks * 128 + 32 * lane, row0, 0, bi,
                         su32(&full[s]), pol);
        else if (lane == 4)
          tma_load_4d_ef(dst + kCodeBytes, &maps.gu_scale[m],
                         FMT == MOE_FORMAT_INT4 ? ks * 8 : ks * (kGuCols / kBlk / 4), row0, 0, bi,
                         su32(&full[s]), pol);
        advance();
      }
    }
    for (int tile = dn_lo; ok && tile < dn_hi; ++tile) {
      const int r = tile / tpe_dn, row0 = (tile % tpe_dn) * RD, m = s_map[r], bi = s_bi[r];
      for (int kd = 0; kd < nkd; ++kd) {
        if (!(ok = slot_ready())) break;
        const uint32_t dst = su32(ring + (size_t)s * kSlotBytes);
        if (lane < geo.nbd)
          tma_load_3d_ef(dst + lane * RD * 128, &maps.dn_code[m], kd * (KSD / 8) + 32 * lane,
                         row0, bi, su32(&full[s]), pol);
        else if (lane == geo.nbd) {
          if constexpr (FMT == MOE_FORMAT_INT4)
            tma_load_4d_ef(dst + kCodeBytes, &maps.dn_scale[m], kd * (KSD / 128), row0, 0, bi,
                           su32(&full[s]), pol);
          else
            tma_load_3d_ef(dst + kCodeBytes, &maps.dn_scale[m], kd * (KSD / kBlk / 4), row0, bi,
                           su32(&full[s]), pol);
        }
        advance();
      }
    }
    // wait (bounded) until every copy this warp issued has landed
    bool landed = true;
    if (lane == 0)
      for (int i = n > nst ? n - nst : 0; i < n; ++i)
        landed = bar_wait(su32(&full[i % nst]), (i / nst) & 1) && landed;
    if (lane == 0 && (!ok || !landed)) s_fail = 1;
  } else if (wid == kFillW) {
    // ---------------------------------------------------------- fill writer
    if (a.fill_fused) {
      int s = 0;
      uint32_t ph = 0;  // ring slot and phase parity of the next stage
      auto advance = [&]() {
        if (++s == nst) {
          s = 0;
          ph ^= 1u;
        }
      };
      bool ok = true;
      const uint64_t pol = l2_evict_first();  // the slot is not read again in this call
      // (one-kernel step) the F entries' slots are learnt at the first entry
      // read from the bank, once the control step has published its fills
      bool known = !FUSED;
      auto fill_slot = [&](int r) -> int {
        if (!known && r < n_uniq && s_map[r] == 0) {
          bool got = true;
          if (lane == 0) got = wait_count(lf.sync + kSyncFill, 1u);
          got = __shfl_sync(0xffffffffu, (int)got, 0) != 0;
          asm volatile("fence.acq_rel.gpu;" ::: "memory");
          if (got) {
            const int nf = __ldcg(a.counts + 4);
            for (int e = lane; e < n_uniq; e += 32) {
              int32_t fs = -1;
              if (s_map[e] == 0)
                for (int i = 0; i < nf; ++i)
                  if (__ldcg(a.fill_ids + i) == s_uid[e]) fs = __ldcg(a.fill_slots + i);
              s_fs[e] = fs;
            }
          } else {
            ok = false;
          }
          __syncwarp();
          known = true;
        }
        return s_fs[r];
      };
      // bytes of the blob past its tiled sections (FP4: the matrix scales, and
      // the padding to 256 bytes), copied by the CTA with the entry's first tile
      const int64_t tail_off = FMT == MOE_FORMAT_INT4
                                   ? blob_offsets(H, I).db + (int64_t)H * (I / kGroup) * 2
                                   : fp4_offsets(H, I, FMT).mat;
      const int tail16 = (int)((a.blob_bytes - tail_off) / 16);
      for (int tile = gu_lo; ok && tile < gu_hi; ++tile) {
        const int r = tile / tpe_gu, row0 = (tile % tpe_gu) * 16, fs = fill_slot(r);
        if (fs >= 0 && row0 == 0 && tail16 > 0) {
          const uint4* src =
              reinterpret_cast<const uint4*>(a.bank + (int64_t)s_bi[r] * a.blob_bytes + tail_off);
          uint4* dst = reinterpret_cast<uint4*>(a.pool_w + (int64_t)fs * a.blob_bytes + tail_off);
          for (int i = lane; i < tail16; i += 32) dst[i] = __ldg(src + i);
        }
        for (int ks = 0; ks < nks; ++ks, advance()) {
          if (!(ok = warp_wait(su32(&full[s]), ph))) break;
          if (fs >= 0 && lane <= 4) {
            const uint32_t src = su32(ring + (size_t)s * kSlotBytes);
            fence_proxy_async_smem();
            if (lane < 4)
              tma_store_4d_ef(&maps.gu_code[1], ks * 128 + 32 * lane, row0, 0, fs,
                              src + lane * 4096, pol);
            else
              tma_store_4d_ef(&maps.gu_scale[1],
                              FMT == MOE_FORMAT_INT4 ? ks * 8 : ks * (kGuCols / kBlk / 4), row0, 0,
                              fs, src + kCodeBytes, pol);
            bulk_commit();
            bulk_read_done();
          }
          __syncwarp();
          if (lane == 0) bar_arrive(su32(&empty[s]));
        }
      }
      for (int tile = dn_lo; ok && tile < dn_hi; ++tile) {
        const int r = tile / tpe_dn, row0 = (tile % tpe_dn) * RD, fs = fill_slot(r);
        for (int kd = 0; kd < nkd; ++kd, advance()) {
          if (!(ok = warp_wait(su32(&full[s]), ph))) break;
          if (fs >= 0 && lane <= geo.nbd) {
            const uint32_t src = su32(ring + (size_t)s * kSlotBytes);
            fence_proxy_async_smem();
            if (lane < geo.nbd)
              tma_store_3d_ef(&maps.dn_code[1], kd * (KSD / 8) + 32 * lane, row0, fs,
                              src + lane * RD * 128, pol);
            else if constexpr (FMT == MOE_FORMAT_INT4)
              tma_store_4d_ef(&maps.dn_scale[1], kd * (KSD / 128), row0, 0, fs,
                              src + kCodeBytes, pol);
            else
              tma_store_3d_ef(&maps.dn_scale[1], kd * (KSD / kBlk / 4), row0, fs,
                              src + kCodeBytes, pol);
            bulk_commit();
            bulk_read_done();
          }
          __syncwarp();
          if (lane == 0) bar_arrive(su32(&empty[s]));
        }
      }
      asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // the slot writes are done
      if (!ok && lane == 0) s_fail = 1;
    }
  } else {
    // ----------------------------------------------------------- consumers
    const int w = wid, g = lane >> 2, t4 = lane & 3, ctid = tid;
    // tokens routed to each entry (ascending)
    if (ctid < n_exec) {
      const int r = ctid, uid = s_uid[r];
      int nt = 0;
      for (int t = 0; t < T; ++t) {
        bool hit = r >= n_uniq;
        for (int j = 0; j < k && !hit; ++j) hit = base + s_ids[t * k + j] == uid;
        if (hit) s_tok[r][nt++] = (int8_t)t;
      }
      s_ntok[r] = nt;
    }
    if constexpr (!FUSED)
      prep_x(b, G);  // (ends with a consumer barrier)
    else
      cons_sync();
    bool ok = true;
    int n = 0, lt = 0;  // stages consumed; gate/up tiles finished (partial buffer ring)
    const unsigned char* zblk = reinterpret_cast<const unsigned char*>(s_zero);
    const float2* zq = reinterpret_cast<const float2*>(s_zero);
    const Cvt cv = cvt_consts();
    const size_t rsz = (size_t)kCW * 32 * T;  // floats per partial buffer
    // Hand this warp's partials of tile lt to the ring; the tile's reducer
    // (warp lt % kCW) waits for all of them.  Returns the buffer.
    auto put_partials = [&](const float (&p0)[4], const float (&p1)[4]) -> float* {
      const int p = lt & 1, u = lt >> 1;
      if (u > 0 && ok) ok = warp_wait(su32(&rfree[p]), (u - 1) & 1);
      float* rb = red + p * rsz;
      float* rw = rb + (size_t)w * 32 * T;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = g + 8 * (e >> 1), nn = 2 * t4 + (e & 1);
        if (nn < T) {
          rw[row * T + nn] = p0[e];
          rw[(16 + row) * T + nn] = p1[e];
        }
      }
      __syncwarp();
      if (lane == 0) bar_arrive(su32(&rfull[p]));
      return rb;
    };
    // ------------------------------------------------ gate/up tiles
    // Per-warp constant byte offsets inside a stage: the lane's code bytes of row g
    // (box w / 4, 16-byte chunk (2 (w % 4) + t4 / 2) ^ g; rows g + 8, 16 + g (up),
    // 24 + g follow at +1024, +2048, +3072) and its scales ([gs, gb, us, ub][16 rows]
    // [16 groups] bf16: group w of row g; row g + 8 at +256, the next array at +512).
    const int coff_gu =
        (w >> 2) * 4096 + (((((w & 3) << 1) | (t4 >> 1)) ^ g) << 4) + (t4 & 1) * 8 + g * 128;
    const int soff_gu = kCodeBytes + (g * 16 + w) * 2;
    // FP4: the lane's block scale byte of row g in a stage ([gate, up][16 rows]
    // [1024 / block bytes]); row g + 8 at +8 rows, up at +16 rows
    constexpr int kRowB = kGuCols / kBlk;
    const int fsoff_gu =
        kCodeBytes + g * kRowB + (FMT == MOE_FORMAT_NVFP4 ? 4 * w + t4 : 2 * w + (t4 >> 1));
    const unsigned char* st = ring;  // the ring slot of stage n
    int sidx = 0;
    uint32_t ph = 0;
    auto next_slot = [&]() {
      st += kSlotBytes;
      if (++sidx == nst) {
        sidx = 0;
        st = ring;
        ph ^= 1u;
      }
    };
    int cur = -1, ntok = 0, tb = -1, to0 = -1, to1 = -1;
    for (int tile = gu_lo; tile < gu_hi; ++tile) {
      const int r = tile / tpe_gu;
      if (r != cur) {
        cur = r;
        ntok = s_ntok[r];
        tb = g < ntok ? s_tok[r][g] : -1;
        to0 = 2 * t4 < ntok ? s_tok[r][2 * t4] : -1;
        to1 = 2 * t4 + 1 < ntok ? s_tok[r][2 * t4 + 1] : -1;
      }
      float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
      // this warp's group G = 16 ks + w of H: B fragments and (O, X) of the
      // tokens; a token slot the entry does not use reads the zero block
      const unsigned char* pb =
          tb >= 0 ? frag + (size_t)tb * geo.frow + w * 128 + t4 * 32 : zblk;
      const float2* pq0 = to0 >= 0 ? ox + w * kMaxTok + to0 : zq;
      const float2* pq1 = to1 >= 0 ? ox + w * kMaxTok + to1 : zq;
      const int sb = tb >= 0 ? 16 * 128 : 0, sq0 = to0 >= 0 ? 16 * kMaxTok : 0,
                sq1 = to1 >= 0 ? 16 * kMaxTok : 0;
      for (int ks = 0; ks < nks; ++ks, ++n) {
        if (ok) ok = warp_wait(su32(&full[sidx]), ph);
        // the stage's codes and scales into registers, then the slot goes back
        // to the producer at once: its refill overlaps this warp's math
        uint2 gl, gh, ul, uh;
        uint16_t sv[8];
        uint32_t fsc[4];  // FP4: scale bytes of gate rows g, g + 8, up rows g, g + 8
        if (ok) {
          const unsigned char* cb = st + coff_gu;
          gl = *reinterpret_cast<const uint2*>(cb);
          gh = *reinterpret_cast<const uint2*>(cb + 1024);
          ul = *reinterpret_cast<const uint2*>(cb + 2048);
          uh = *reinterpret_cast<const uint2*>(cb + 3072);
          if constexpr (FMT == MOE_FORMAT_INT4) {
            const unsigned char* sc = st + soff_gu;
#pragma unroll
            for (int e = 0; e < 8; ++e) sv[e] = *reinterpret_cast<const uint16_t*>(sc + 256 * e);
          } else {
            const unsigned char* sc = st + fsoff_gu;
            fsc[0] = sc[0];
            fsc[1] = sc[8 * kRowB];
            fsc[2] = sc[16 * kRowB];
            fsc[3] = sc[24 * kRowB];
          }
        }
        __syncwarp();
        if (lane == 0) bar_arrive(su32(&empty[sidx]));
        next_slot();
        if (ok) {
          const uint4 v0 = reinterpret_cast<const uint4*>(pb)[0];
          const uint4 v1 = reinterpret_cast<const uint4*>(pb)[1];
          const uint32_t b[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          if constexpr (FMT == MOE_FORMAT_INT4) {
            const float2 q0 = *pq0, q1 = *pq1;
            // sv: gs, gb, us, ub of rows g and g + 8 ([array][row] order, rows 8 apart)
            const float sg0 = bf(sv[0]), sg1 = bf(sv[1]), bg0 = bf(sv[2]), bg1 = bf(sv[3]);
            const float su0 = bf(sv[4]), su1 = bf(sv[5]), bu0 = bf(sv[6]), bu1 = bf(sv[7]);
            float dg[4], du[4];
            group2(dg, du, gl, gh, ul, uh, b, cv);
            ag[0] = fmaf(sg0, dg[0] - q0.x, fmaf(bg0, q0.y, ag[0]));
            ag[1] = fmaf(sg0, dg[1] - q1.x, fmaf(bg0, q1.y, ag[1]));
            ag[2] = fmaf(sg1, dg[2] - q0.x, fmaf(bg1, q0.y, ag[2]));
            ag[3] = fmaf(sg1, dg[3] - q1.x, fmaf(bg1, q1.y, ag[3]));
            au[0] = fmaf(su0, du[0] - q0.x, fmaf(bu0, q0.y, au[0]));
            au[1] = fmaf(su0, du[1] - q1.x, fmaf(bu0, q1.y, au[1]));
            au[2] = fmaf(su1, du[2] - q0.x, fmaf(bu1, q0.y, au[2]));
            au[3] = fmaf(su1, du[3] - q1.x, fmaf(bu1, q1.y, au[3]));
          } else {
            group2_fp4(ag, au, gl, gh, ul, uh, fp4_scale2<FMT>(fsc[0]), fp4_scale2<FMT>(fsc[1]),
                       fp4_scale2<FMT>(fsc[2]), fp4_scale2<FMT>(fsc[3]), b);
          }
        }
        pb += sb;
        pq0 += sq0;
        pq1 += sq1;
      }
      const float* rb = put_partials(ag, au);
      if (w == lt % kCW) {
        // reducer: sum the warps' partials in warp order, h = silu(g) * u for the
        // tile's 16 rows, max |h| per token slot, then free the partial buffer
        const int p = lt & 1;
        if (ok) ok = warp_wait(su32(&rfull[p]), (lt >> 1) & 1);
        const int row0 = (tile % tpe_gu) * 16;
        for (int nn = 0; nn < ntok; ++nn) {
          float v = 0.0f;
          if (lane < 16) {
            float gs = 0.0f, us = 0.0f;
#pragma unroll
            for (int ww = 0; ww < kCW; ++ww) {
              gs += rb[((size_t)ww * 32 + lane) * T + nn];
              us += rb[((size_t)ww * 32 + 16 + lane) * T + nn];
            }
            const float P = s_px[s_tok[r][nn]];
            if constexpr (FMT == MOE_FORMAT_INT4) {
              gs *= P;
              us *= P;
            } else {
              gs *= P * s_fac[r][0];
              us *= P * s_fac[r][1];
            }
            v = __fdividef(gs, 1.0f + __expf(fminf(-gs, 80.0f))) * us;
            a.h[((int64_t)r * T + nn) * I + row0 + lane] = v;
          }
          const uint32_t mb = __reduce_max_sync(0xffffffffu, __float_as_uint(v) & 0x7FFFFFFFu);
          if (lane == 0) atomicMax(&hmax[r * kMaxTok + nn], mb);
        }
        __syncwarp();
        if (lane == 0) bar_arrive(su32(&rfree[p]));
      }
      ++lt;
    }
    // this CTA's h rows are written: one arrival on the grid-wide count
    cons_sync();
    if (ctid == 0) red_release_add(gu_cnt, 1u);  // release: this CTA's h rows and maxima

    // --------------------------------------------------- down tiles
    const int ngs = geo.ngs, gi = w % ngs, p = w / ngs;
    // per-warp constant offsets inside a down stage: the lane's code bytes of row
    // 32 p + g (box gi / 4 of RD rows x 128 B; rows + 8, + 16, + 24 at +1024, +2048,
    // +3072) and its scales ([ds, db][RD rows][ngs groups] bf16; db at +sbo)
    const int coff_dn = (gi >> 2) * (RD * 128) + (((((gi & 3) << 1) | (t4 >> 1)) ^ g) << 4) +
                        (t4 & 1) * 8 + (32 * p + g) * 128;
    const int soff_dn = kCodeBytes + ((32 * p + g) * ngs + gi) * 2;
    // FP4: the lane's block scale byte of row 32 p + g ([RD rows][KSD / block
    // bytes]); rows + 8, + 16, + 24 follow at 8 row strides
    const int kRowD = KSD / kBlk;
    const int fsoff_dn = kCodeBytes + (32 * p + g) * kRowD +
                         (FMT == MOE_FORMAT_NVFP4 ? 4 * gi + t4 : 2 * gi + (t4 >> 1));
    const int sbo = RD * ngs * 2;
    cur = -1;
    for (int tile = dn_lo; tile < dn_hi; ++tile) {
      const int r = tile / tpe_dn, rb = tile % tpe_dn, row0 = rb * RD;
      if (r != cur) {
        // before the first down tile: every CTA's gate/up rows written (grid-wide
        // count); then entry r's h as B fragments, replacing the previous ones
        ntok = s_ntok[r];
        cons_sync();
        if (ctid == 0 && ok && cur < 0 && !wait_count(gu_cnt, Gall)) s_fail = 1;
        cur = r;
        cons_sync();
        // h, its per-token maxima and the routing weights in one round of loads
        if (ctid < ntok) {
          const int nn = ctid;
          const float inv = inv_pow2_above(__uint_as_float(__ldcg(hmax + r * kMaxTok + nn)));
          s_ih[nn] = inv;
          // routing weight of this entry for the slot's token: the sum over the
          // ranks j naming it (a token may list an expert twice); 1 for the
          // shared expert
          float wsum = 1.0f;
          if (r < n_uniq) {
            const int t = s_tok[r][nn], uid = s_uid[r];
            wsum = 0.0f;
            for (int j = 0; j < k; ++j)
              if (base + s_ids[t * k + j] == uid) wsum += s_wts[t * k + j];
          }
          if constexpr (FMT != MOE_FORMAT_INT4) wsum *= s_fac[r][2];
          s_wp[nn] = wsum / inv;
        }
        const float* hr = a.h + (int64_t)r * T * I;
        const int ngi = I / 64, n_items = ntok * ngi * 4;
        for (int b0 = 0; b0 < n_items; b0 += kConsThreads) {
          const int it = b0 + ctid;
          const bool in = it < n_items;
          const int nn = in ? it / (ngi * 4) : 0, rem = it - nn * ngi * 4, G = rem >> 2,
                    q4 = rem & 3;
          float v[16];
          float o = 0.0f, xs = 0.0f;
          if (in) {
            const float4* ph =
                reinterpret_cast<const float4*>(hr + (int64_t)nn * I + G * 64 + q4 * 16);
            float4 f[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) f[e] = __ldcg(ph + e);
            const float sc =
                inv_pow2_above(__uint_as_float(__ldcg(hmax + r * kMaxTok + nn)));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              v[4 * e] = f[e].x * sc;
              v[4 * e + 1] = f[e].y * sc;
              v[4 * e + 2] = f[e].z * sc;
              v[4 * e + 3] = f[e].w * sc;
            }
            if constexpr (FMT == MOE_FORMAT_INT4)
              frag_item(v, frag + (size_t)nn * geo.frow + G * 128 + q4 * 32, o, xs);
            else
              frag_plain(v, frag + (size_t)nn * geo.frow + G * 128 + q4 * 32);
          }
          o += __shfl_xor_sync(0xffffffffu, o, 1);
          o += __shfl_xor_sync(0xffffffffu, o, 2);
          xs += __shfl_xor_sync(0xffffffffu, xs, 1);
          xs += __shfl_xor_sync(0xffffffffu, xs, 2);
          if (in && q4 == 0) ox[G * kMaxTok + nn] = make_float2(o, xs);
        }
        cons_sync();
        if (s_fail) ok = false;
      }
      float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
      const int n0 = 2 * t4, n1 = 2 * t4 + 1;
      // this warp's group G = kd ngs + gi of I: h fragments of token slot g and
      // (O, X) of slots n0, n1; slots past the entry's tokens read the zero block
      const unsigned char* pb =
          g < ntok ? frag + (size_t)g * geo.frow + gi * 128 + t4 * 32 : zblk;
      const float2* pq0 = n0 < ntok ? ox + gi * kMaxTok + n0 : zq;
      const float2* pq1 = n1 < ntok ? ox + gi * kMaxTok + n1 : zq;
      const int sb = g < ntok ? ngs * 128 : 0, sq0 = n0 < ntok ? ngs * kMaxTok : 0,
                sq1 = n1 < ntok ? ngs * kMaxTok : 0;
      for (int kd = 0; kd < nkd; ++kd, ++n) {
        if (ok) ok = warp_wait(su32(&full[sidx]), ph);
        // codes and scales into registers, then the slot goes back at once
        uint2 l0, h0, l1, h1;
        uint16_t sv[8];
        uint32_t fsc[4];  // FP4: scale bytes of rows g, g + 8, g + 16, g + 24 (of 32 p ..)
        if (ok) {
          const unsigned char* cb = st + coff_dn;
          l0 = *reinterpret_cast<const uint2*>(cb);
          h0 = *reinterpret_cast<const uint2*>(cb + 1024);
          l1 = *reinterpret_cast<const uint2*>(cb + 2048);
          h1 = *reinterpret_cast<const uint2*>(cb + 3072);
          if constexpr (FMT == MOE_FORMAT_INT4) {
            const unsigned char* sc = st + soff_dn;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              sv[e] = *reinterpret_cast<const uint16_t*>(sc + 16 * ngs * e);
              sv[4 + e] = *reinterpret_cast<const uint16_t*>(sc + sbo + 16 * ngs * e);
            }
          } else {
            const unsigned char* sc = st + fsoff_dn;
#pragma unroll
            for (int e = 0; e < 4; ++e) fsc[e] = sc[8 * e * kRowD];
          }
        }
        __syncwarp();
        if (lane == 0) bar_arrive(su32(&empty[sidx]));
        next_slot();
        if (ok) {
          const uint4 v0 = reinterpret_cast<const uint4*>(pb)[0];
          const uint4 v1 = reinterpret_cast<const uint4*>(pb)[1];
          const uint32_t b[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          if constexpr (FMT == MOE_FORMAT_INT4) {
            const float2 q0 = *pq0, q1 = *pq1;
            // sv: ds of rows g, g + 8, g + 16, g + 24 (of the warp's 32), then db
            const float s00 = bf(sv[0]), s01 = bf(sv[1]), s10 = bf(sv[2]), s11 = bf(sv[3]);
            const float b00 = bf(sv[4]), b01 = bf(sv[5]), b10 = bf(sv[6]), b11 = bf(sv[7]);
            float d0[4], d1[4];
            group2(d0, d1, l0, h0, l1, h1, b, cv);
            a0[0] = fmaf(s00, d0[0] - q0.x, fmaf(b00, q0.y, a0[0]));
            a0[1] = fmaf(s00, d0[1] - q1.x, fmaf(b00, q1.y, a0[1]));
            a0[2] = fmaf(s01, d0[2] - q0.x, fmaf(b01, q0.y, a0[2]));
            a0[3] = fmaf(s01, d0[3] - q1.x, fmaf(b01, q1.y, a0[3]));
            a1[0] = fmaf(s10, d1[0] - q0.x, fmaf(b10, q0.y, a1[0]));
            a1[1] = fmaf(s10, d1[1] - q1.x, fmaf(b10, q1.y, a1[1]));
            a1[2] = fmaf(s11, d1[2] - q0.x, fmaf(b11, q0.y, a1[2]));
            a1[3] = fmaf(s11, d1[3] - q1.x, fmaf(b11, q1.y, a1[3]));
          } else {
            group2_fp4(a0, a1, l0, h0, l1, h1, fp4_scale2<FMT>(fsc[0]), fp4_scale2<FMT>(fsc[1]),
                       fp4_scale2<FMT>(fsc[2]), fp4_scale2<FMT>(fsc[3]), b);
          }
        }
        pb += sb;
        pq0 += sq0;
        pq1 += sq1;
      }
      // this warp's rows of the tile (32 p + {g, g + 8}, 32 p + 16 + {g, g + 8}) for
      // token slots 2 t4, 2 t4 + 1, times the entry's routing weight of the token,
      // added into y (fp32 atomics: the routed terms meet in y in arrival order)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int nn = 2 * t4 + (e & 1);
        if (ok && nn < ntok) {
          const int t = s_tok[r][nn];
          const float wp = s_wp[nn];
          float* yo = a.y + (int64_t)t * H + row0 + 32 * p + g + 8 * (e >> 1);
          atomicAdd(yo, wp * a0[e]);
          atomicAdd(yo + 16, wp * a1[e]);
        }
      }
    }
    if (!ok && lane == 0) s_fail = 1;
  }

  __syncthreads();
  __shared__ int s_last;
  if (tid == 0) {
    const bool f = s_fail != 0;
    if (f) {
      if (a.err) atomicOr(a.err, MOE_DERR_WAIT);
      atomicExch(failw, 1u);
    }
    __threadfence();
    s_last = atomicAdd(done, 1u) == gridDim.x - 1;
    if (s_last) {
      // last CTA: when any CTA gave up while this call carried the step's
      // fills, an F slot may hold a partial copy -- unmap every F entry
      __threadfence();
      if (a.fill_fused && atomicAdd(failw, 0u) != 0u) {
        const int nf = __ldcg(a.counts + 4);
        for (int i = 0; i < nf; ++i) {
          const int32_t f = __ldcg(a.fill_ids + i), v = __ldcg(a.fill_slots + i);
          a.tab_slot_of_id[f] = -1;
          a.tab_id_of_slot[v] = -1;
          a.tab_ts[v] = 0u;
        }
      }
    }
  }
  if constexpr (FUSED) {
    // last CTA: every other CTA is past its last use of the sync words, which
    // are left zero for the next step
    __syncthreads();
    if (s_last)
      for (int i = tid; i < kSyncCtr + 4 + 8 * kMaxEnt; i += kThreads) lf.sync[i] = 0u;
  }
}

static_assert(kSyncCtr + 4 + 8 * kMaxEnt <= MOE_CACHE_SYNC_WORDS, "sync words");

template <bool FUSED, int FMT>
bool coop_attr_set(size_t smem) {
  static size_t done[64];
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return false;
  if (done[d] >= smem) return true;
  if (cudaFuncSetAttribute(ffn_coop_kernel<FUSED, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return false;
  done[d] = smem;
  return true;
}

}  // namespace

bool ffn_coop_supported(int H, int I, int k, int T, int has_shared) {
  if (H % kGuCols != 0 || I % 512 != 0 || T < 1 || T > kMaxTok) return false;
  if ((long)T * k > kMaxIds || (long)T * k + has_shared > kMaxEnt) return false;
  return coop_geom(H, I, T).nst > 0;
}

namespace {

template <bool FUSED, int FMT>
cudaError_t launch_coop_fmt(const FfnArgs& a, const LayerFuse& lf, cudaStream_t st) {
  static int sms[64];
  if (!ffn_coop_supported(a.H, a.I, a.k, a.T, a.has_shared) || a.max_entries > kMaxEnt ||
      a.n_ctr < ffn_ctr_words(a.H, a.max_entries))
    return cudaErrorInvalidValue;
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= 64) return cudaErrorInvalidDevice;
  if (!sms[d]) {
    e = cudaDeviceGetAttribute(&sms[d], cudaDevAttrMultiProcessorCount, d);
    if (e != cudaSuccess) return e;
  }
  const CoopGeom geo = coop_geom(a.H, a.I, a.T);
  CoopMaps maps;
  memset(&maps, 0, sizeof(maps));
  const BlobOffsets off = blob_offsets(a.H, a.I);
  const Fp4Offsets foff = fp4_offsets(a.H, a.I, FMT);
  const uint64_t blk = (uint64_t)foff.block;
  const uint8_t* bases[3] = {a.bank, a.pool, a.shared ? a.shared : a.bank};
  const uint64_t nblob[3] = {(uint64_t)a.n_bank, (uint64_t)a.n_pool,
                             a.shared ? 1ull : (uint64_t)a.n_bank};
  const uint64_t H = a.H, I = a.I, B = a.blob_bytes;
  for (int i = 0; i < 3; ++i) {
    {
      const uint64_t dims[4] = {H / 8, I, 2, nblob[i]};
      const uint64_t strides[3] = {H / 2, I * H / 2, B};
      const uint32_t box[4] = {32, 16, 2, 1};
      if ((e = encode_tiled_u32(&maps.gu_code[i], bases[i] + off.gq, 4, dims, strides, box,
                                true)) != cudaSuccess)
        return e;
    }
    if (FMT == MOE_FORMAT_INT4) {
      const uint64_t dims[4] = {H / 128, I, 4, nblob[i]};
      const uint64_t strides[3] = {H / 32, I * H / 32, B};
      const uint32_t box[4] = {8, 16, 4, 1};
      if ((e = encode_tiled_u32(&maps.gu_scale[i], bases[i] + off.gs, 4, dims, strides, box,
                                false)) != cudaSuccess)
        return e;
    } else {
      // one scale byte per block: [gate, up][row of I][H / block bytes]
      const uint64_t dims[4] = {H / blk / 4, I, 2, nblob[i]};
      const uint64_t strides[3] = {H / blk, I * H / blk, B};
      const uint32_t box[4] = {(uint32_t)(kGuCols / blk / 4), 16, 2, 1};
      if ((e = encode_tiled_u32(&maps.gu_scale[i], bases[i] + foff.gs, 4, dims, strides, box,
                                false)) != cudaSuccess)
        return e;
    }
    {
      const uint64_t dims[3] = {I / 8, H, nblob[i]};
      const uint64_t strides[2] = {I / 2, B};
      const uint32_t box[3] = {32, (uint32_t)geo.RD, 1};
      if ((e = encode_tiled_u32(&maps.dn_code[i], bases[i] + off.dq, 3, dims, strides, box,
                                true)) != cudaSuccess)
        return e;
    }
    if (FMT == MOE_FORMAT_INT4) {
      const uint64_t dims[4] = {I / 128, H, 2, nblob[i]};
      const uint64_t strides[3] = {I / 32, H * I / 32, B};
      const uint32_t box[4] = {(uint32_t)(geo.KSD / 128), (uint32_t)geo.RD, 2, 1};
      if ((e = encode_tiled_u32(&maps.dn_scale[i], bases[i] + off.ds, 4, dims, strides, box,
                                false)) != cudaSuccess)
        return e;
    } else {
      // [row of H][I / block bytes]
      const uint64_t dims[3] = {I / blk / 4, H, nblob[i]};
      const uint64_t strides[2] = {I / blk, B};
      const uint32_t box[3] = {(uint32_t)(geo.KSD / blk / 4), (uint32_t)geo.RD, 1};
      if ((e = encode_tiled_u32(&maps.dn_scale[i], bases[i] + foff.ds, 3, dims, strides, box,
                                false)) != cudaSuccess)
        return e;
    }
  }
  if (!coop_attr_set<FUSED, FMT>(geo.smem)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(sms[d]);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = geo.smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, ffn_coop_kernel<FUSED, FMT>, a, geo, maps, lf);
  if (e == cudaErrorInvalidValue || e == cudaErrorNotSupported) {
    // a runtime that does not take both attributes together: launch it
    // cooperatively, after the previous kernel has completed
    (void)cudaGetLastError();
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, ffn_coop_kernel<FUSED, FMT>, a, geo, maps, lf);
  }
  return e;
}

template <bool FUSED>
cudaError_t launch_coop(const FfnArgs& a, const LayerFuse& lf, cudaStream_t st) {
  switch (a.format) {
    case MOE_FORMAT_INT4:
      return launch_coop_fmt<FUSED, MOE_FORMAT_INT4>(a, lf, st);
    case MOE_FORMAT_MXFP4:
      return launch_coop_fmt<FUSED, MOE_FORMAT_MXFP4>(a, lf, st);
    case MOE_FORMAT_NVFP4:
      return launch_coop_fmt<FUSED, MOE_FORMAT_NVFP4>(a, lf, st);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_ffn_coop(const FfnArgs& a, cudaStream_t st) {
  return launch_coop<false>(a, LayerFuse{}, st);
}

bool layer_fused_supported(int H, int I, int E, int k, int T, int has_shared, int K, int router,
                           int n_groups) {
  if (!ffn_coop_supported(H, I, k, T, has_shared)) return false;
  if (T * k > 32 || K < 1 || K > kCtlK || E < 1 || E > 256 || k > rsel::kMaxK) return false;
  if (router != MOE_ROUTER_SOFTMAX_TOPK && (n_groups < 1 || n_groups > 32)) return false;
  return true;
}

cudaError_t launch_layer_fused(const FfnArgs& a, const LayerFuse& lf, cudaStream_t st) {
  if (!layer_fused_supported(a.H, a.I, a.E, a.k, a.T, a.has_shared, lf.c.K, lf.router,
                             lf.n_groups) ||
      !lf.sync || !lf.logits || !lf.w_router || !lf.ids_out || !lf.wts_out || !a.fill_fused ||
      a.ids != lf.ids_out || a.weights != lf.wts_out || lf.c.ids != lf.ids_out ||
      a.ctr != lf.sync + kSyncCtr)
    return cudaErrorInvalidValue;
  return launch_coop<true>(a, lf, st);
}

}  // namespace moe
