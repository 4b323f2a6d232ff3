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

__device__ __forceinline__ float moe_sigmoid(float z) {
  const float d = __fadd_rn(1.0f, moe_exp(-z));
  return __fdiv_rn(1.0f, d);
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

// Softmax-top-k of token t, one warp; lane j holds experts j + 32 i.  Scratch
// in shared memory: sv, sex [kMaxK], ssum [1].
template <int EPL>
__device__ __forceinline__ void softmax_token(const float* __restrict__ logits, int t, int E,
                                              int k, int32_t* __restrict__ ids,
                                              float* __restrict__ wts, float* sv, float* sex,
                                              float* ssum) {
  const int lane = threadIdx.x & 31;
  float v[EPL];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldcg(logits + (size_t)t * E + e) : -FLT_MAX;
    if (e >= E) taken |= 1u << i;
  }
  for (int r = 0; r < k; ++r) {
    float bv = -FLT_MAX;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (!(taken >> i & 1u) && better(v[i], e, bv, bi)) {
        bv = v[i];
        bi = e;
      }
    }
    warp_argmax(bv, bi);
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == 0) {
      sv[r] = bv;
      ids[(size_t)t * k + r] = bi;
    }
  }
  __syncwarp();
  if (lane == 0) {
    const float top = sv[0];
    float S = 0.0f;
    for (int r = 0; r < k; ++r) {
      const float ex = moe_exp(__fsub_rn(sv[r], top));
      sex[r] = ex;
      S = __fadd_rn(S, ex);
    }
    ssum[0] = S;
  }
  __syncwarp();
  for (int r = lane; r < k; r += 32) wts[(size_t)t * k + r] = __fdiv_rn(sex[r], ssum[0]);
}

// Sigmoid-group selection of token t, one warp (n_groups <= 32, E <= 32 * EPL).
// Scratch in shared memory: ssel [32 * EPL], ss [kMaxK], ssum [1].
template <int EPL>
__device__ __forceinline__ void sigmoid_group_token(const float* __restrict__ logits,
                                                    const float* __restrict__ bias, int t, int E,
                                                    int n_groups, int topk_groups, int k,
                                                    float scale, int32_t* __restrict__ ids,
                                                    float* __restrict__ wts, float* ssel,
                                                    float* ss, float* ssum) {
  const int lane = threadIdx.x & 31;
  const int gsz = E / n_groups;
  float s[EPL], sel[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      s[i] = moe_sigmoid(__ldcg(logits + (size_t)t * E + e));
      sel[i] = __fadd_rn(s[i], bias ? bias[e] : 0.0f);
      ssel[e] = sel[i];
    } else {
      s[i] = 0.0f;
      sel[i] = -FLT_MAX;
    }
  }
  __syncwarp();
  // group score: sum of the two largest selection scores of the group
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
  uint32_t kept = 0;  // bit g: group g kept
  uint32_t gtaken = (lane < n_groups) ? 0u : 1u;
  for (int r = 0; r < topk_groups; ++r) {
    float bv = gtaken ? -FLT_MAX : gscore;
    int bi = gtaken ? 0x7fffffff : lane;
    warp_argmax(bv, bi);
    if (bi == lane) gtaken = 1;
    kept |= 1u << bi;
  }
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e >= E || !((kept >> (e / gsz)) & 1u)) taken |= 1u << i;
  }
  for (int r = 0; r < k; ++r) {
    float bv = -FLT_MAX;
    int bi = 0x7fffffff;
    float bs = 0.0f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (!(taken >> i & 1u) && better(sel[i], e, bv, bi)) {
        bv = sel[i];
        bi = e;
        bs = s[i];
      }
    }
    const int mine = bi;
    warp_argmax(bv, bi);
    const bool win = (bi == mine) && ((bi & 31) == lane);
    if (win) {
      taken |= 1u << (bi >> 5);
      ss[r] = bs;
      ids[(size_t)t * k + r] = bi;
    }
  }
  __syncwarp();
  if (lane == 0) {
    float S = 0.0f;
    for (int r = 0; r < k; ++r) S = __fadd_rn(S, ss[r]);
    ssum[0] = S;
  }
  __syncwarp();
  for (int r = lane; r < k; r += 32)
    wts[(size_t)t * k + r] = __fmul_rn(__fdiv_rn(ss[r], ssum[0]), scale);
}

}  // namespace rsel
}  // namespace moe
