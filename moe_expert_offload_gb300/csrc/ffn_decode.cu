// Decode expert FFN: int4 affine group-64 SwiGLU experts
// y_e = Wd (silu(Wg x) * (Wu x)) (Edge0 §3.1 "math convention"), executed
// for every routed id of the step -- H and F from their slots, C in place
// from the bank -- plus the always-on shared expert, and the exact weighted
// merge of the per-expert partial outputs (FreeToken summary "core method").
//
// Decode streams MBs of packed weights against a few KB of activations, so
// the kernels are built to keep HBM busy with few instructions per weight:
//
//  * Each lane loads 8 code bytes (16 columns of one 64-column group) of two
//    rows 8 apart, straight into registers.  One LOP3 turns a nibble pair
//    into a bf16x2 holding (128 + q_a, 128 + q_b) (exponent bits 0x43), which
//    is fed as the A fragment of a warp-level m16n8k16 bf16 MMA.  The lane's
//    16 columns are consumed in the permuted order the fragment layout
//    implies, and the activations are stored in shared memory in that same
//    order (any consistent permutation of k leaves the dot product intact).
//  * Four MMAs cover one group for 16 rows; the group's scale and bias are
//    applied to the fp32 accumulator:  s * A + (b - 128 s) * X with
//    X = sum of the group's activations, i.e. sum_j (s q_j + b) x_j.
//  * The MMA's N columns carry the tokens: phase A one token per column,
//    phase B a hi/lo bf16 split of each fp32 h value in a column pair, so the
//    down projection keeps ~2^-17 relative precision in h.
//
// Phase A (gate/up): CTA = (entry, 16 rows of I); its 8 warps split the K
//   (= H) groups, the CTA sums the warps' partials and writes
//   h[entry][t][i] = silu(g) * u into the workspace.
// Phase B (down): CTA = (entry, 64 rows of H), one 16-row tile per warp; it
//   writes the weighted partial  w[t][j] * (Wd h)[o]  into partial[t][j][o]
//   (j = this expert's rank in token t's routing, k for the shared expert).
//   The last CTA to finish a row block (arrival counter) adds partial[t][0..k]
//   in j order into y: a fixed order, no data atomics, deterministic.
#include <cuda_bf16.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kWarpsA = 8;   // K slices per 16-row tile (phase A)
constexpr int kWarpsB = 4;   // 16-row tiles per CTA (phase B)
constexpr int kRowsBlkB = 16 * kWarpsB;
constexpr int kBatchA = 4;   // groups in flight per warp (phase A)
constexpr int kBatchB = 8;   // groups in flight per warp (phase B)
constexpr int kTokA = 8;     // tokens per MMA N tile, phase A (one per column)
constexpr int kTokB = 4;     // tokens per MMA N tile, phase B (hi/lo column pairs)

__device__ __forceinline__ uint2 ld_stream8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

// bf16x2 (128 + nibble i, 128 + nibble i+4) of an 8-nibble word.
__device__ __forceinline__ uint32_t nib_pair(uint32_t w, int i) {
  return ((w >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 64-column group for 16 rows.  lo / hi: the lane's 8 code bytes (16
// columns) of rows g and g + 8; b: the group's 8 B-fragment registers.
// MMA jj takes nibble pairs (i, i+4) and (i+1, i+5), i = 2 (jj & 1), of word
// jj / 2, so k slot 2t, 2t+1 of MMA jj is column 16t + 8(jj/2) + i (+4) and
// slot 2t+8, 2t+9 is column 16t + 8(jj/2) + i + 1 (+4).
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

// 16 consecutive bf16 columns (8 words w[0..7], low half = even column) into
// the B-fragment order 0,4,1,5, 2,6,3,7, 8,12,9,13, 10,14,11,15.
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

struct EntryInfo {
  const uint8_t* blob;
  int ntok;
};

// Entry r of the step (the r-th unique routed id, or the shared expert after
// them): its weights and the tokens routed to it (ascending), with the rank j
// of the expert in each token's routing and its weight.
__device__ bool resolve_entry(const FfnArgs& a, int r, int* stok, int* sj, float* sw,
                              EntryInfo* out) {
  __shared__ int s_cnt;
  const int n_uniq = a.counts[0];
  const int n_exec = n_uniq + a.has_shared;
  if (r >= n_exec) return false;
  const int tid = threadIdx.x, lane = tid & 31;
  if (r < n_uniq) {
    const int32_t id = a.uniq[r];
    if (tid == 0) {
      const int32_t slot = ffn_slot(a, id);
      out->blob = slot >= 0 ? a.pool + (int64_t)slot * a.blob_bytes
                            : a.bank + (int64_t)id * a.blob_bytes;
    }
    if (tid < 32) {
      const int base = a.layer * a.E, n = a.T * a.k;
      int cnt = 0;
      for (int n0 = 0; n0 < n; n0 += 32) {
        const int i = n0 + lane;
        const bool m = i < n && base + a.ids[i] == id;
        const unsigned b = __ballot_sync(0xffffffffu, m);
        const int p = cnt + __popc(b & ((1u << lane) - 1u));
        if (m && p < kMaxDecodeT) {  // more only if a token repeats an id
          stok[p] = i / a.k;
          sj[p] = i % a.k;
          sw[p] = a.weights[i];
        }
        cnt += __popc(b);
      }
      if (lane == 0) s_cnt = cnt < kMaxDecodeT ? cnt : kMaxDecodeT;
    }
  } else {
    if (tid == 0) {
      out->blob = a.shared;
      s_cnt = a.T;
    }
    for (int t = tid; t < a.T; t += blockDim.x) {
      stok[t] = t;
      sj[t] = a.k;
      sw[t] = 1.0f;
    }
  }
  __syncthreads();
  out->ntok = s_cnt;
  return true;
}

// (s, b - 128 s) per (row, group) of `rows` rows from row0 into shared memory
// (row-major [rows][ng + 1]: the pad keeps the 8 rows a warp reads at once in
// distinct banks; rows past nrows get zeros).  The block is contiguous
// in the blob, so it moves in 16-byte vectors with all loads issued first.
__device__ void stage_scales(const uint16_t* s, const uint16_t* b, int row0, int rows, int nrows,
                             int ng, float2* dst) {
  constexpr int kU = 4;
  const int64_t begin = (int64_t)row0 * ng;
  const int valid = (min(row0 + rows, nrows) - row0) * ng;
  const int nvec = rows * ng / 8;
  const uint4* sv4 = reinterpret_cast<const uint4*>(s + begin);
  const uint4* bv4 = reinterpret_cast<const uint4*>(b + begin);
  for (int base = 0; base < nvec; base += kU * blockDim.x) {
    uint4 sv[kU], bv[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = base + u * blockDim.x + threadIdx.x;
      if (v < nvec && 8 * v < valid) {
        sv[u] = __ldg(sv4 + v);
        bv[u] = __ldg(bv4 + v);
      } else {
        sv[u] = bv[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = base + u * blockDim.x + threadIdx.x;
      if (v < nvec) {
        const uint32_t sw4[4] = {sv[u].x, sv[u].y, sv[u].z, sv[u].w};
        const uint32_t bw4[4] = {bv[u].x, bv[u].y, bv[u].z, bv[u].w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int e = 8 * v + j, rr = e / ng, g = e - rr * ng;
          const uint32_t w = (j & 1) ? (sw4[j >> 1] & 0xFFFF0000u) : (sw4[j >> 1] << 16);
          const uint32_t c = (j & 1) ? (bw4[j >> 1] & 0xFFFF0000u) : (bw4[j >> 1] << 16);
          const float sv_f = __uint_as_float(w);
          dst[rr * (ng + 1) + g] = make_float2(sv_f, fmaf(-128.0f, sv_f, __uint_as_float(c)));
        }
      }
    }
  }
}

// ------------------------------------------------------------------ phase A
// smem: xf [tok_rows][2H+16] bytes (bf16 x in fragment order), xsum
// [ng][kTokA*NT] fp32, sbg / sbu [16][ng+1] (s, b'), red [kWarpsA][2][16][kTokA*NT].
template <int NT>
__global__ void __launch_bounds__(kWarpsA * 32) ffn_gate_up_kernel(FfnArgs a, int n_tick,
                                                                   int tok_rows) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int stok[kMaxDecodeT], sj[kMaxDecodeT];
  __shared__ float sw[kMaxDecodeT];
  __shared__ EntryInfo ent;
  constexpr int NTOK = kTokA * NT;
  const int H = a.H, I = a.I, ng = H / kGroup;
  const int xstride = 2 * H + 16;
  unsigned char* xf = smem;
  float* xsum = reinterpret_cast<float*>(smem + (size_t)tok_rows * xstride);
  float2* sbg = reinterpret_cast<float2*>(xsum + ng * NTOK);
  float2* sbu = sbg + 16 * (ng + 1);
  float* red = reinterpret_cast<float*>(sbu + 16 * (ng + 1));

  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_tick; i += blockDim.x) a.tick[i] = 0u;
  const int tiles = I / 16;
  const int r = blockIdx.x / tiles, row0 = (blockIdx.x - r * tiles) * 16;
  if (!resolve_entry(a, r, stok, sj, sw, &ent)) return;

  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, t4 = lane & 3;
  const BlobOffsets off = blob_offsets(H, I);
  const uint8_t* blob = ent.blob;
  const int64_t crow = H / 2;
  const uint8_t* gq = blob + off.gq + (row0 + gid) * crow + t4 * 8;
  const uint8_t* uq = blob + off.uq + (row0 + gid) * crow + t4 * 8;
  stage_scales(reinterpret_cast<const uint16_t*>(blob + off.gs),
               reinterpret_cast<const uint16_t*>(blob + off.gb), row0, 16, I, ng, sbg);
  stage_scales(reinterpret_cast<const uint16_t*>(blob + off.us),
               reinterpret_cast<const uint16_t*>(blob + off.ub), row0, 16, I, ng, sbu);
  const int g_lo = wid * ng / kWarpsA, g_hi = (wid + 1) * ng / kWarpsA;
  // codes of one batch of groups: [group][gate lo, gate hi, up lo, up hi]
  auto load_batch = [&](int gb, uint2 (&c)[kBatchA][4]) {
#pragma unroll
    for (int i = 0; i < kBatchA; ++i) {
      if (gb + i < g_hi) {
        const int64_t o = (int64_t)(gb + i) * 32;
        c[i][0] = ld_stream8(gq + o);
        c[i][1] = ld_stream8(gq + 8 * crow + o);
        c[i][2] = ld_stream8(uq + o);
        c[i][3] = ld_stream8(uq + 8 * crow + o);
      }
    }
  };
  uint2 cur[kBatchA][4], nxt[kBatchA][4];
  load_batch(g_lo, cur);  // first weights in flight before the activations are staged
  bool have = true;

  for (int t0 = 0; t0 < ent.ntok; t0 += tok_rows) {
    const int nt = min(tok_rows, ent.ntok - t0);
    __syncthreads();
    // x of tokens t0.. into fragment order, plus per-group sums; the 4
    // quarters of a group sit on 4 consecutive lanes, whole warps take part
    const int n_stage = (nt * ng * 4 + 31) / 32 * 32;
    for (int it = threadIdx.x; it < n_stage; it += blockDim.x) {
      const bool in = it < nt * ng * 4;
      const int n = in ? it / (ng * 4) : 0, rem = it - n * ng * 4, g = rem >> 2, q = rem & 3;
      uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
      float s = 0.0f;
      if (in) {
        const uint4* p = reinterpret_cast<const uint4*>(a.x + (int64_t)stok[t0 + n] * H +
                                                        g * 64 + q * 16);
        const uint4 u0 = __ldg(p), u1 = __ldg(p + 1);
        const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j)
          s += __uint_as_float(w[j] << 16) + __uint_as_float(w[j] & 0xFFFF0000u);
        frag_order(w, o0, o1);
      }
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (in) {
        uint4* d = reinterpret_cast<uint4*>(xf + (size_t)n * xstride + g * 128 + q * 32);
        d[0] = o0;
        d[1] = o1;
        if (q == 0) xsum[g * NTOK + n] = s;
      }
    }
    __syncthreads();

    float acc[NT][2][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][m][e] = 0.0f;

    for (int gb = g_lo; gb < g_hi; gb += kBatchA) {
      if (!have) load_batch(gb, cur);
      have = false;
      if (gb + kBatchA < g_hi) {  // next batch in flight while this one computes
        load_batch(gb + kBatchA, nxt);
        have = true;
      }
#pragma unroll
      for (int i = 0; i < kBatchA; ++i) {
        const int g = gb + i;
        if (g >= g_hi) break;
        const float2 sg0 = sbg[gid * (ng + 1) + g], sg1 = sbg[(gid + 8) * (ng + 1) + g];
        const float2 su0 = sbu[gid * (ng + 1) + g], su1 = sbu[(gid + 8) * (ng + 1) + g];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const int n = j * kTokA + gid;
          uint32_t bf[8];
          load_frag(xf + (size_t)n * xstride + g * 128 + t4 * 32, n < nt, bf);
          float dg[4] = {0.f, 0.f, 0.f, 0.f}, du[4] = {0.f, 0.f, 0.f, 0.f};
          group_mma(dg, cur[i][0], cur[i][1], bf);
          group_mma(du, cur[i][2], cur[i][3], bf);
          const float2 X =
              *reinterpret_cast<const float2*>(xsum + g * NTOK + j * kTokA + 2 * t4);
          acc[j][0][0] = fmaf(sg0.x, dg[0], fmaf(sg0.y, X.x, acc[j][0][0]));
          acc[j][0][1] = fmaf(sg0.x, dg[1], fmaf(sg0.y, X.y, acc[j][0][1]));
          acc[j][0][2] = fmaf(sg1.x, dg[2], fmaf(sg1.y, X.x, acc[j][0][2]));
          acc[j][0][3] = fmaf(sg1.x, dg[3], fmaf(sg1.y, X.y, acc[j][0][3]));
          acc[j][1][0] = fmaf(su0.x, du[0], fmaf(su0.y, X.x, acc[j][1][0]));
          acc[j][1][1] = fmaf(su0.x, du[1], fmaf(su0.y, X.y, acc[j][1][1]));
          acc[j][1][2] = fmaf(su1.x, du[2], fmaf(su1.y, X.x, acc[j][1][2]));
          acc[j][1][3] = fmaf(su1.x, du[3], fmaf(su1.y, X.y, acc[j][1][3]));
        }
      }
      if (have) {
#pragma unroll
        for (int i = 0; i < kBatchA; ++i)
#pragma unroll
          for (int e = 0; e < 4; ++e) cur[i][e] = nxt[i][e];
      }
    }
    // sum the K slices of the 8 warps, then h = silu(g) * u
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = gid + 8 * (e >> 1), n = j * kTokA + 2 * t4 + (e & 1);
          red[((wid * 2 + m) * 16 + row) * NTOK + n] = acc[j][m][e];
        }
    __syncthreads();
    for (int it = threadIdx.x; it < 16 * nt; it += blockDim.x) {
      const int row = it / nt, n = it - row * nt;
      float g = 0.0f, u = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarpsA; ++w) {
        g += red[((w * 2 + 0) * 16 + row) * NTOK + n];
        u += red[((w * 2 + 1) * 16 + row) * NTOK + n];
      }
      const float silu = g / (1.0f + __expf(-g));
      a.h[((int64_t)r * a.T + stok[t0 + n]) * I + row0 + row] = silu * u;
    }
  }
}

// ------------------------------------------------------------------ phase B
// smem: hf [2*kTokB*NT columns][2I+16] bytes (hi/lo bf16 h in fragment order),
// hsum [ngi][kTokB*NT] fp32, sb [64][ngi+1] (s, b').
template <int NT>
__global__ void __launch_bounds__(kWarpsB * 32) ffn_down_kernel(FfnArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int stok[kMaxDecodeT], sj[kMaxDecodeT];
  __shared__ float sw[kMaxDecodeT];
  __shared__ EntryInfo ent;
  __shared__ int s_last;
  constexpr int NTOK = kTokB * NT;
  const int H = a.H, I = a.I, ngi = I / kGroup;
  const int nslot = a.k + a.has_shared;
  const int hstride = 2 * I + 16;
  unsigned char* hf = smem;
  float* hsum = reinterpret_cast<float*>(smem + (size_t)(2 * NTOK) * hstride);
  float2* sb = reinterpret_cast<float2*>(hsum + ngi * NTOK);
  const int nblk = (H + kRowsBlkB - 1) / kRowsBlkB;
  const int r = blockIdx.x / nblk, blk = blockIdx.x - r * nblk;
  if (a.counts[0] + a.has_shared == 0) {  // nothing routed to a valid expert: y = 0
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.T * H; i += gridDim.x * blockDim.x)
      a.y[i] = 0.0f;
    return;
  }
  if (!resolve_entry(a, r, stok, sj, sw, &ent)) return;

  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, t4 = lane & 3;
  const int o0 = blk * kRowsBlkB, orow = o0 + wid * 16 + gid;
  const BlobOffsets off = blob_offsets(H, I);
  const uint8_t* blob = ent.blob;
  const int64_t crow = I / 2;
  const uint8_t* dq_lo = blob + off.dq + min(orow, H - 1) * crow + t4 * 8;
  const uint8_t* dq_hi = blob + off.dq + min(orow + 8, H - 1) * crow + t4 * 8;
  stage_scales(reinterpret_cast<const uint16_t*>(blob + off.ds),
               reinterpret_cast<const uint16_t*>(blob + off.db), o0, kRowsBlkB, H, ngi, sb);
  const float2* sbw = sb + (wid * 16) * (ngi + 1);
  auto load_batch = [&](int gb, uint2 (&c)[kBatchB][2]) {
#pragma unroll
    for (int i = 0; i < kBatchB; ++i) {
      if (gb + i < ngi) {
        const int64_t o = (int64_t)(gb + i) * 32;
        c[i][0] = ld_stream8(dq_lo + o);
        c[i][1] = ld_stream8(dq_hi + o);
      }
    }
  };
  uint2 cur[kBatchB][2], nxt[kBatchB][2];
  load_batch(0, cur);  // first weights in flight before h is staged
  bool have = true;

  for (int t0 = 0; t0 < ent.ntok; t0 += NTOK) {
    const int nt = min(NTOK, ent.ntok - t0);
    __syncthreads();
    // h of tokens t0.. as hi/lo bf16 column pairs (column 2n hi, 2n+1 lo)
    const int n_stage = (nt * ngi * 4 + 31) / 32 * 32;  // whole warps reach the shuffles
    for (int it = threadIdx.x; it < n_stage; it += blockDim.x) {
      const bool in = it < nt * ngi * 4;
      const int n = in ? it / (ngi * 4) : 0, rem = it - n * ngi * 4;
      const int g = rem >> 2, q = rem & 3;
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0.0f;
      if (in) {
        const float4* p = reinterpret_cast<const float4*>(
            a.h + ((int64_t)r * a.T + stok[t0 + n]) * I + g * 64 + q * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 f = __ldcg(p + i);
          v[4 * i] = f.x;
          v[4 * i + 1] = f.y;
          v[4 * i + 2] = f.z;
          v[4 * i + 3] = f.w;
        }
      }
      uint32_t whi[8], wlo[8];
      float s = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float h0 = v[2 * j], h1 = v[2 * j + 1];
        s += h0 + h1;
        const __nv_bfloat162 hi = __floats2bfloat162_rn(h0, h1);
        const float2 hb = __bfloat1622float2(hi);
        whi[j] = *reinterpret_cast<const uint32_t*>(&hi);
        wlo[j] = pack_bf16(h0 - hb.x, h1 - hb.y);
      }
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (in) {
        uint4 o0h, o1h, o0l, o1l;
        frag_order(whi, o0h, o1h);
        frag_order(wlo, o0l, o1l);
        uint4* dh = reinterpret_cast<uint4*>(hf + (size_t)(2 * n) * hstride + g * 128 + q * 32);
        uint4* dl =
            reinterpret_cast<uint4*>(hf + (size_t)(2 * n + 1) * hstride + g * 128 + q * 32);
        dh[0] = o0h;
        dh[1] = o1h;
        dl[0] = o0l;
        dl[1] = o1l;
        if (q == 0) hsum[g * NTOK + n] = s;
      }
    }
    __syncthreads();

    float acc[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = 0.0f;
    for (int gb = 0; gb < ngi; gb += kBatchB) {
      if (!have) load_batch(gb, cur);
      have = false;
      if (gb + kBatchB < ngi) {  // next batch in flight while this one computes
        load_batch(gb + kBatchB, nxt);
        have = true;
      }
#pragma unroll
      for (int i = 0; i < kBatchB; ++i) {
        const int g = gb + i;
        if (g >= ngi) break;
        const float2 s0 = sbw[gid * (ngi + 1) + g], s1 = sbw[(gid + 8) * (ngi + 1) + g];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const int col = j * 2 * kTokB + gid;  // = 2 * token + (0 hi / 1 lo)
          uint32_t bf[8];
          load_frag(hf + (size_t)col * hstride + g * 128 + t4 * 32, (col >> 1) < nt, bf);
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          group_mma(d, cur[i][0], cur[i][1], bf);
          const float X = hsum[g * NTOK + j * kTokB + t4];
          acc[j][0] = fmaf(s0.x, d[0] + d[1], fmaf(s0.y, X, acc[j][0]));
          acc[j][1] = fmaf(s1.x, d[2] + d[3], fmaf(s1.y, X, acc[j][1]));
        }
      }
      if (have) {
#pragma unroll
        for (int i = 0; i < kBatchB; ++i) {
          cur[i][0] = nxt[i][0];
          cur[i][1] = nxt[i][1];
        }
      }
    }
    // lane (gid, t4) holds rows orow and orow + 8 for token t0 + j*kTokB + t4
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int n = j * kTokB + t4;
      if (n < nt) {
        const int p = t0 + n;
        float* dst = a.partial + ((int64_t)stok[p] * nslot + sj[p]) * H;
        if (orow < H) dst[orow] = sw[p] * acc[j][0];
        if (orow + 8 < H) dst[orow + 8] = sw[p] * acc[j][1];
      }
    }
  }

  // arrival: the last entry to finish this row block combines it
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int n_exec = a.counts[0] + a.has_shared;
    const unsigned prev = atomicAdd(&a.tick[blk], 1u);
    s_last = (prev == (unsigned)(n_exec - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int nrow = min(kRowsBlkB, H - o0);
  for (int it = threadIdx.x; it < a.T * nrow; it += blockDim.x) {
    const int t = it / nrow, o = o0 + (it - t * nrow);
    float yv = 0.0f;
    for (int j = 0; j < nslot; ++j) {
      if (j < a.k) {
        const int32_t e = a.ids[t * a.k + j];
        if (e < 0 || e >= a.E) continue;  // skipped by the control step as well
      }
      yv += __ldcg(a.partial + ((int64_t)t * nslot + j) * H + o);
    }
    a.y[(int64_t)t * H + o] = yv;
  }
  if (threadIdx.x == 0) a.tick[blk] = 0u;
}

size_t smem_a(int H, int NT, int tok_rows) {
  const size_t ng = H / kGroup, ntok = kTokA * NT;
  return (size_t)tok_rows * (2 * H + 16) + ng * ntok * 4 + 2 * 16 * (ng + 1) * 8 +
         (size_t)kWarpsA * 2 * 16 * ntok * 4;
}

size_t smem_b(int I, int NT) {
  const size_t ngi = I / kGroup, ntok = kTokB * NT;
  return 2 * ntok * (2 * I + 16) + ngi * ntok * 4 + (size_t)kRowsBlkB * (ngi + 1) * 8;
}

// Opt a kernel into more than 48 KB of dynamic shared memory, once per device
// and size (a host-side function attribute, not a stream operation).
template <typename Kern>
cudaError_t raise_smem(Kern kernel, size_t bytes, size_t (&done)[64]) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d >= 0 && d < 64 && done[d] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && d >= 0 && d < 64) done[d] = bytes;
  return e;
}

}  // namespace

size_t ffn_workspace_bytes(int H, int I, int k, int T, int has_shared) {
  auto al = [](size_t b) { return (b + 255) / 256 * 256; };
  const size_t max_entries = (size_t)T * k + has_shared;
  const size_t nctr = (size_t)ffn_ctr_words(H, (int)max_entries);
  return al(max_entries * T * I * 4) + al((size_t)T * (k + has_shared) * H * 4) + al(nctr * 4);
}

void ffn_carve_workspace(FfnArgs& a, void* ws) {
  auto al = [](size_t b) { return (b + 255) / 256 * 256; };
  const size_t max_entries = (size_t)a.T * a.k + a.has_shared;
  uint8_t* p = static_cast<uint8_t*>(ws);
  a.h = reinterpret_cast<float*>(p);
  p += al(max_entries * a.T * a.I * 4);
  a.partial = reinterpret_cast<float*>(p);
  p += al((size_t)a.T * (a.k + a.has_shared) * a.H * 4);
  a.tick = reinterpret_cast<uint32_t*>(p);
  a.max_entries = (int)max_entries;
  a.ctr = a.tick;
  a.n_ctr = ffn_ctr_words(a.H, a.max_entries);
}

bool ffn_fill_fusable(int H, int I, int k, int T, int has_shared) {
  const long max_entries = (long)T * k + has_shared;  // as ffn_carve_workspace
  if (ffn_coop_supported(H, I, k, T, has_shared)) return true;
  return max_entries <= 128 && ffn_stream_smem(H, T) != SIZE_MAX &&
         ffn_down_stream_smem(H, I, T) != SIZE_MAX;
}

cudaError_t launch_ffn_decode(const FfnArgs& a, cudaStream_t st, bool ctr_zeroed) {
  if (ffn_coop_supported(a.H, a.I, a.k, a.T, a.has_shared)) {
    // the cooperative kernel needs its counters at zero
    if (!ctr_zeroed) {
      const cudaError_t e = cudaMemsetAsync(a.ctr, 0, (size_t)a.n_ctr * 4, st);
      if (e != cudaSuccess) return e;
    }
    return launch_ffn_coop(a, st);
  }
  if (a.format != MOE_FORMAT_INT4) return cudaErrorNotSupported;  // FP4: the cooperative kernel only
  static size_t done_a1[64], done_a2[64], done_b1[64], done_b2[64];
  const int nblk = (a.H + kRowsBlkB - 1) / kRowsBlkB;
  const int grid_a = a.max_entries * (a.I / 16);
  const int grid_b = a.max_entries * nblk;
  cudaError_t e;
  // phase A: tokens staged per pass, bounded so shared memory stays near 100 KB
  const int ntile_a = a.T <= kTokA ? 1 : 2;
  const size_t fixed_a = smem_a(a.H, ntile_a, 0);
  const size_t row_a = (size_t)(2 * a.H + 16);
  int tok_rows = a.T < kTokA * ntile_a ? a.T : kTokA * ntile_a;
  while (tok_rows > 1 && fixed_a + tok_rows * row_a > 100 * 1024) --tok_rows;
  const size_t sa = fixed_a + tok_rows * row_a;
  const int ntick = (a.H + 15) / 16;
  if (a.max_entries <= 128 && ffn_stream_smem(a.H, a.T) != SIZE_MAX) {
    if ((e = launch_ffn_gate_up_stream(a, ntick, st)) != cudaSuccess) return e;
  } else if (ntile_a == 1) {
    if ((e = raise_smem(ffn_gate_up_kernel<1>, sa, done_a1)) != cudaSuccess) return e;
    ffn_gate_up_kernel<1><<<grid_a, kWarpsA * 32, sa, st>>>(a, ntick, tok_rows);
  } else {
    if ((e = raise_smem(ffn_gate_up_kernel<2>, sa, done_a2)) != cudaSuccess) return e;
    ffn_gate_up_kernel<2><<<grid_a, kWarpsA * 32, sa, st>>>(a, ntick, tok_rows);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.max_entries <= 128 && ffn_down_stream_smem(a.H, a.I, a.T) != SIZE_MAX) {
    return launch_ffn_down_stream(a, st);
  } else if (a.T <= kTokB) {
    const size_t sb = smem_b(a.I, 1);
    if ((e = raise_smem(ffn_down_kernel<1>, sb, done_b1)) != cudaSuccess) return e;
    ffn_down_kernel<1><<<grid_b, kWarpsB * 32, sb, st>>>(a);
  } else {
    const size_t sb = smem_b(a.I, 2);
    if ((e = raise_smem(ffn_down_kernel<2>, sb, done_b2)) != cudaSuccess) return e;
    ffn_down_kernel<2><<<grid_b, kWarpsB * 32, sb, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace moe
