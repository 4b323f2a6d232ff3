// Router scoring and selection shared by the router kernels, the fused decode
// control step and the fused decode layer kernel (Edge0 §2 "MoE routing"):
// one logit per warp in a fixed order, the library's exp and sigmoid, the
// top-k order, and the per-token softmax-top-k and sigmoid-group selections,
// each run by one warp.  Logits are read through L2 (they may have been
// written by other CTAs of the same grid).  Every floating-point step is an explicitly rounded IEEE
// operation, so a plain CPU program reproduces the decisions bit for bit.
#pragma once
#include <float.h>

#include "moe_internal.cuh"

namespace moe {
namespace rsel {

constexpr int kMaxK = 64;

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// One router logit x . w (bf16 rows of H, 16-byte aligned) by one warp, in
// the fixed order every router path uses: lane j accumulates the 8-element
// chunks c = j, j+32, ... in ascending order with fma from 0, then the lane
// sums go through an xor butterfly 16, 8, 4, 2, 1.  Every lane returns the
// logit.
__device__ __forceinline__ float router_dot_warp(const uint16_t* __restrict__ x,
                                                 const uint16_t* __restrict__ w, int H) {
  const int lane = threadIdx.x & 31;
  const uint4* xr = reinterpret_cast<const uint4*>(x);
  const uint4* wr = reinterpret_cast<const uint4*>(w);
  const int chunks = H >> 3;
  float acc = 0.0f;
  // eight chunks' loads in flight at a time, then their fmas in chunk order
  for (int c0 = lane; c0 < chunks; c0 += 32 * 8) {
    uint4 xv[8], wv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int c = c0 + 32 * u;
      if (c < chunks) {
        xv[u] = __ldg(xr + c);
        wv[u] = __ldg(wr + c);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (c0 + 32 * u >= chunks) break;
      acc = __fmaf_rn(bf_lo(xv[u].x), bf_lo(wv[u].x), acc);
      acc = __fmaf_rn(bf_hi(xv[u].x), bf_hi(wv[u].x), acc);
      acc = __fmaf_rn(bf_lo(xv[u].y), bf_lo(wv[u].y), acc);
      acc = __fmaf_rn(bf_hi(xv[u].y), bf_hi(wv[u].y), acc);
      acc = __fmaf_rn(bf_lo(xv[u].z), bf_lo(wv[u].z), acc);
      acc = __fmaf_rn(bf_hi(xv[u].z), bf_hi(wv[u].z), acc);
      acc = __fmaf_rn(bf_lo(xv[u].w), bf_lo(wv[u].w), acc);
      acc = __fmaf_rn(bf_hi(xv[u].w), bf_hi(wv[u].w), acc);
    }
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, d));
  return acc;
}

// router_dot_warp on rows staged in shared memory (the same chunk-to-lane
// assignment, the same fma order and butterfly): bit-identical logits.
__device__ __forceinline__ float router_dot_smem(const uint4* xr, const uint4* wr, int H) {
  const int lane = threadIdx.x & 31;
  const int chunks = H >> 3;
  float acc = 0.0f;
  for (int c = lane; c < chunks; c += 32) {
    const uint4 xv = xr[c], wv = wr[c];
    acc = __fmaf_rn(bf_lo(xv.x), bf_lo(wv.x), acc);
    acc = __fmaf_rn(bf_hi(xv.x), bf_hi(wv.x), acc);
    acc = __fmaf_rn(bf_lo(xv.y), bf_lo(wv.y), acc);
    acc = __fmaf_rn(bf_hi(xv.y), bf_hi(wv.y), acc);
    acc = __fmaf_rn(bf_lo(xv.z), bf_lo(wv.z), acc);
    acc = __fmaf_rn(bf_hi(xv.z), bf_hi(wv.z), acc);
    acc = __fmaf_rn(bf_lo(xv.w), bf_lo(wv.w), acc);
    acc = __fmaf_rn(bf_hi(xv.w), bf_hi(wv.w), acc);
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, d));
  return acc;
}

// exp(x) in fp32: Cody-Waite reduction x = n ln2 + r (ln2 = 0x1.62e4p-1 +
// 0x1.7f7d1cp-20, the high part short enough that n * hi is exact), the
// degree-7 Taylor polynomial of e^r (coefficients 1/7! .. 1/0!) in Horner
// form with fused multiply-adds, and an exact 2^n scale from exponent bits.
// x is clamped to [-87, 88], so n is in [-126, 127] and 2^n is normal.
__device__ __forceinline__ float moe_exp(float x) {
  x = fminf(fmaxf(x, -87.0f), 88.0f);
  const float n = rintf(__fmul_rn(x, 0x1.715476p+0f));
  float r = __fmaf_rn(n, -0x1.62e4p-1f, x);
  r = __fmaf_rn(n, -0x1.7f7d1cp-20f, r);
  float p = 0x1.a01a02p-13f;           // 1/5040
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);  // 1/720
  p = __fmaf_rn(p, r, 0x1.111112p-7f);   // 1/120
  p = __fmaf_rn(p, r, 0x1.555556p-5f);   // 1/24
  p = __fmaf_rn(p, r, 0x1.555556p-3f);   // 1/6
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const int ni = (int)n;
  return __fmul_rn(p, __int_as_float((ni + 127) << 23));
}

// 1 / (1 + exp(-z)), the reciprocal correctly rounded (the same bits as the
// IEEE division 1 / d).
__device__ __forceinline__ float moe_sigmoid(float z) {
  const float d = __fadd_rn(1.0f, moe_exp(-z));
  return __frcp_rn(d);
}

// (value, index) order used for every top-k: larger value first, lower
// index first among equal values.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, d);
    const int oi = __shfl_xor_sync(0xffffffffu, i, d);
    if (better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

// Unsigned key with the order of the fp32 values (larger value <=> larger
// key; -0 and +0 share a key, so equal values tie); a NaN gets key 1, below
// every number.  Key 0 marks an entry that is out of the race.  Branch-free,
// so that the loads feeding it stay in flight together.
__device__ __forceinline__ uint32_t ord_key(float v) {
  const uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));  // -0 -> +0
  const uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (v != v) ? 1u : k;
}

// Compare-exchange of (key, slot) pairs into descending order of `better`:
// larger key first, the lower slot first among equal keys.
__device__ __forceinline__ void cex_desc(uint32_t& ka, uint32_t& ia, uint32_t& kb, uint32_t& ib) {
  const bool sw = kb > ka || (kb == ka && ib < ia);
  const uint32_t k0 = sw ? kb : ka, i0 = sw ? ib : ia, k1 = sw ? ka : kb, i1 = sw ? ia : ib;
  ka = k0;
  ia = i0;
  kb = k1;
  ib = i1;
}

// The lane's N (a power of two) candidates sorted into descending order by
// Batcher's odd-even merge sort (a fixed network: every index is a constant).
template <int N>
__device__ __forceinline__ void lane_sort_desc(uint32_t (&key)[N], uint32_t (&slot)[N]) {
#pragma unroll
  for (int p = 1; p < N; p <<= 1)
#pragma unroll
    for (int q = p; q >= 1; q >>= 1)
#pragma unroll
      for (int j = q % p; j + q < N; j += 2 * q)
#pragma unroll
        for (int i = 0; i < q; ++i)
          if (i + j + q < N && (i + j) / (2 * p) == (i + j + q) / (2 * p))
            cex_desc(key[i + j], slot[i + j], key[i + j + q], slot[i + j + q]);
}

// The warp's k best candidates in the order of `better`: lane j holds
// candidates e = j + 32 slot, sorted per lane (key 0: out).  Each round the
// warp takes the largest head key, the lowest index among the lanes holding
// it, and that lane pops its head.  Rank r's index goes to lane r % 32
// (rid[r / 32]); with no candidate left, 0x7fffffff.
template <int N>
__device__ __forceinline__ void warp_topk(uint32_t (&key)[N], uint32_t (&slot)[N], int k,
                                          int (&rid)[2]) {
  const int lane = threadIdx.x & 31;
  rid[0] = rid[1] = 0x7fffffff;
  for (int r = 0; r < k; ++r) {
    const uint32_t M = __reduce_max_sync(0xffffffffu, key[0]);
    const uint32_t mine = (M != 0u && key[0] == M) ? (uint32_t)(lane + 32 * slot[0]) : 0xffffffffu;
    const uint32_t emin = __reduce_min_sync(0xffffffffu, mine);
    if (mine == emin) {
#pragma unroll
      for (int i = 0; i < N - 1; ++i) {
        key[i] = key[i + 1];
        slot[i] = slot[i + 1];
      }
      key[N - 1] = 0u;
    }
    const int id = M != 0u ? (int)emin : 0x7fffffff;
    if (r == lane) rid[0] = id;
    if (r == lane + 32) rid[1] = id;
  }
}

// v[id / 32] of lane id % 32, for the id each lane asks for (0 for 0x7fffffff).
template <int N>
__device__ __forceinline__ float warp_fetch(const float (&v)[N], int id) {
  float r = 0.0f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float x = __shfl_sync(0xffffffffu, v[i], id & 31);
    if ((id >> 5) == i) r = x;
  }
  return r;
}

// Softmax-top-k of token t, one warp; lane j holds experts j + 32 i.  The k
// winners in the order of `better` (larger logit first, lower index among
// equal logits); weights exp(l_r - l_0) / S with S the fixed-order sum
// r = 0, 1, ..., k-1 from 0 (k <= kMaxK).  The trailing scratch pointers are
// unused (kept for the callers' layout).
template <int EPL>
__device__ __forceinline__ void softmax_token(const float* __restrict__ logits, int t, int E,
                                              int k, int32_t* __restrict__ ids,
                                              float* __restrict__ wts, float*, float*, float*) {
  const int lane = threadIdx.x & 31;
  float v[EPL];
  uint32_t key[EPL], slot[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    v[i] = (lane + 32 * i < E) ? __ldcg(logits + (size_t)t * E + lane + 32 * i) : 0.0f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    key[i] = (lane + 32 * i < E) ? ord_key(v[i]) : 0u;
    slot[i] = (uint32_t)i;
  }
  lane_sort_desc<EPL>(key, slot);
  int rid[2];
  warp_topk<EPL>(key, slot, k, rid);
  const float top = warp_fetch<EPL>(v, __shfl_sync(0xffffffffu, rid[0], 0));
  float ex[2] = {0.0f, 0.0f};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float lv = warp_fetch<EPL>(v, rid[h]);
    if (lane + 32 * h < k) ex[h] = moe_exp(__fsub_rn(lv, top));
  }
  float S = 0.0f;
  for (int r = 0; r < k; ++r)
    S = __fadd_rn(S, __shfl_sync(0xffffffffu, r < 32 ? ex[0] : ex[1], r & 31));
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = lane + 32 * h;
    if (r < k) {
      ids[(size_t)t * k + r] = rid[h];
      wts[(size_t)t * k + r] = __fdiv_rn(ex[h], S);
    }
  }
}

// Sigmoid-group selection of token t, one warp (n_groups <= 32, E <= 32 * EPL):
// s = sigmoid(logit), selection score s + bias; group score = the sum of the
// two largest selection scores of the group; the topk_groups best groups
// (order of `better`) are kept and the k best selection scores among their
// experts win; weights s_r / S * scale, S the fixed-order sum of the winners'
// s.  Scratch in shared memory (groups narrower than 32 experts only): ssel
// [32 * EPL]; the other scratch pointers are unused.
template <int EPL>
__device__ __forceinline__ void sigmoid_group_token(const float* __restrict__ logits,
                                                    const float* __restrict__ bias, int t, int E,
                                                    int n_groups, int topk_groups, int k,
                                                    float scale, int32_t* __restrict__ ids,
                                                    float* __restrict__ wts, float* ssel, float*,
                                                    float*) {
  const int lane = threadIdx.x & 31;
  const int gsz = E / n_groups;
  float s[EPL], sel[EPL], bv[EPL];
  uint32_t key[EPL], slot[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const bool in = lane + 32 * i < E;
    s[i] = in ? __ldcg(logits + (size_t)t * E + lane + 32 * i) : 0.0f;
    bv[i] = (in && bias) ? bias[lane + 32 * i] : 0.0f;
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const bool in = lane + 32 * i < E;
    s[i] = in ? moe_sigmoid(s[i]) : 0.0f;
    sel[i] = in ? __fadd_rn(s[i], bv[i]) : -FLT_MAX;
  }
  // group score: sum of the two largest selection scores of the group; t1 >= t2
  // (t2 == t1 when the largest appears twice)
  uint32_t kept = 0;  // bit g: group g kept
  if (gsz % 32 == 0) {
    // group g = register rows i in [g gsz/32, (g+1) gsz/32) of every lane: the
    // lane's two largest of each group, then an xor butterfly merging the
    // lanes' pairs, all groups at once; every lane ends with every score
    const int rows = gsz >> 5;
    float t1[EPL], t2[EPL];  // n_groups <= EPL here
    if (rows == 1) {
#pragma unroll
      for (int g = 0; g < EPL; ++g) {
        t1[g] = g < n_groups ? sel[g] : -FLT_MAX;
        t2[g] = -FLT_MAX;
      }
    } else {
#pragma unroll
      for (int g = 0; g < EPL; ++g) {
        t1[g] = -FLT_MAX;
        t2[g] = -FLT_MAX;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
          if (g < n_groups && i >= g * rows && i < (g + 1) * rows) {
            const float z = sel[i];
            t2[g] = fmaxf(t2[g], fminf(t1[g], z));
            t1[g] = fmaxf(t1[g], z);
          }
      }
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1)
#pragma unroll
      for (int g = 0; g < EPL; ++g) {
        const float b1 = __shfl_xor_sync(0xffffffffu, t1[g], d);
        const float b2 = __shfl_xor_sync(0xffffffffu, t2[g], d);
        t2[g] = fmaxf(fminf(t1[g], b1), fmaxf(t2[g], b2));
        t1[g] = fmaxf(t1[g], b1);
      }
    // the topk_groups best groups, computed alike by every lane: each group's
    // rank is the number of groups ahead of it in the order of `better`
#pragma unroll
    for (int g = 0; g < EPL; ++g) t1[g] = __fadd_rn(t1[g], t2[g]);
#pragma unroll
    for (int g = 0; g < EPL; ++g) {
      int ahead = 0;
#pragma unroll
      for (int h = 0; h < EPL; ++h)
        ahead += (h < n_groups && better(t1[h], h, t1[g], g)) ? 1 : 0;
      if (g < n_groups && ahead < topk_groups) kept |= 1u << g;
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i < E) ssel[lane + 32 * i] = sel[i];
    __syncwarp();
    float gscore = -FLT_MAX;
    if (lane < n_groups) {
      float t1 = -FLT_MAX, t2 = -FLT_MAX;
      for (int e = lane * gsz; e < (lane + 1) * gsz; ++e) {
        const float z = ssel[e];
        if (z > t1) {
          t2 = t1;
          t1 = z;
        } else if (z > t2) {
          t2 = z;
        }
      }
      gscore = __fadd_rn(t1, t2);
    }
    uint32_t gtaken = (lane < n_groups) ? 0u : 1u;
    for (int r = 0; r < topk_groups; ++r) {
      float bvg = gtaken ? -FLT_MAX : gscore;
      int bi = gtaken ? 0x7fffffff : lane;
      warp_argmax(bvg, bi);
      if (bi == lane) gtaken = 1;
      kept |= 1u << bi;
    }
    __syncwarp();
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    key[i] = (e < E && ((kept >> (e / gsz)) & 1u)) ? ord_key(sel[i]) : 0u;
    slot[i] = (uint32_t)i;
  }
  lane_sort_desc<EPL>(key, slot);
  int rid[2];
  warp_topk<EPL>(key, slot, k, rid);
  float rs[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) rs[h] = warp_fetch<EPL>(s, rid[h]);
  float S = 0.0f;
  for (int r = 0; r < k; ++r)
    S = __fadd_rn(S, __shfl_sync(0xffffffffu, r < 32 ? rs[0] : rs[1], r & 31));
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = lane + 32 * h;
    if (r < k) {
      ids[(size_t)t * k + r] = rid[h];
      wts[(size_t)t * k + r] = __fmul_rn(__fdiv_rn(rs[h], S), scale);
    }
  }
}

}  // namespace rsel
}  // namespace moe
