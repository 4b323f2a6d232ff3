// Router scoring (Edge0 §2 "MoE routing"): logits x . W_r^T in a fixed fp32
// order, then softmax-top-k or sigmoid-group selection, one warp per token.
//
// Routing decisions must be reproducible bit for bit by a plain CPU program,
// so every floating-point step here is an explicitly rounded IEEE operation
// (__fmaf_rn, __fadd_rn, __fmul_rn, __fdiv_rn: nothing for the compiler to
// contract) and exp is the library's own function below, not CUDA's.
#include <float.h>

#include "moe_internal.cuh"
#include "route_select.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// One warp per (token, expert).  Lane j accumulates 8-element chunks
// c = j, j+32, ... in order with fma from 0; the lane sums then go through an
// xor butterfly 16, 8, 4, 2, 1.  x rows and W rows are 16-byte aligned.
__global__ void __launch_bounds__(128) router_logits_kernel(const uint16_t* __restrict__ x,
                                                            const uint16_t* __restrict__ w, int T,
                                                            int E, int H,
                                                            float* __restrict__ logits) {
  griddep_launch();
  griddep_wait();  // x may come from the previous kernel
  const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (warp >= T * E) return;
  const int t = warp / E, e = warp - t * E;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  const uint4* wr = reinterpret_cast<const uint4*>(w + (size_t)e * H);
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
  if (lane == 0) logits[(size_t)t * E + e] = acc;
}

// Tiled logits for many tokens, same order as router_logits_kernel: CTA =
// 16 tokens x 16 experts, 8 warps of 4 tokens x 8 experts.  H goes through
// shared memory in 256-column slices; in slice s lane j owns chunk 32 s + j,
// so each lane still accumulates chunks j, j+32, ... in ascending order with
// fma from 0.  The 32 sums of a lane are then combined by a reduce-scatter
// over the same xor partners 16, 8, 4, 2, 1 (each add pairs the same two
// lane partials as the butterfly, and fp addition is commutative, so every
// logit is bit-identical); lane j ends with pair j.  Needs H % 256 == 0.
constexpr int kTileTok = 16, kTileExp = 16;

__global__ void __launch_bounds__(256) router_logits_tiled_kernel(const uint16_t* __restrict__ x,
                                                                  const uint16_t* __restrict__ w,
                                                                  int T, int E, int H,
                                                                  float* __restrict__ logits) {
  __shared__ __align__(16) uint4 xs[kTileTok][32];  // 16 rows x 256 bf16
  griddep_launch();
  griddep_wait();
  __shared__ __align__(16) uint4 ws[kTileExp][32];
  const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kTileTok, e0 = blockIdx.y * kTileExp;
  const int tw = (wid >> 1) * 4, ew = (wid & 1) * 8;
  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
  // staging: 32 rows (16 x, 16 W) x 32 chunks = 1024 uint4, 4 per thread
  uint4 nx[4];
  auto fetch = [&](int s) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = tid + 256 * j, row = i >> 5, c = i & 31;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (row < kTileTok) {
        if (t0 + row < T)
          v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + row) * H + s * 256) + c);
      } else if (e0 + row - kTileTok < E) {
        v = __ldg(reinterpret_cast<const uint4*>(w + (size_t)(e0 + row - kTileTok) * H +
                                                 s * 256) + c);
      }
      nx[j] = v;
    }
  };
  const int ns = H / 256;
  fetch(0);
  for (int s = 0; s < ns; ++s) {
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = tid + 256 * j, row = i >> 5, c = i & 31;
      if (row < kTileTok)
        xs[row][c] = nx[j];
      else
        ws[row - kTileTok][c] = nx[j];
    }
    __syncthreads();
    if (s + 1 < ns) fetch(s + 1);
    // widen once per slice (x) and once per expert row (W), not per product
    float xf[4][8];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const uint4 v = xs[tw + a][lane];
      xf[a][0] = bf_lo(v.x); xf[a][1] = bf_hi(v.x); xf[a][2] = bf_lo(v.y); xf[a][3] = bf_hi(v.y);
      xf[a][4] = bf_lo(v.z); xf[a][5] = bf_hi(v.z); xf[a][6] = bf_lo(v.w); xf[a][7] = bf_hi(v.w);
    }
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const uint4 v = ws[ew + b][lane];
      const float wf[8] = {bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y),
                           bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w)};
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        float& r = acc[a * 8 + b];
#pragma unroll
        for (int e = 0; e < 8; ++e) r = __fmaf_rn(xf[a][e], wf[e], r);
      }
    }
  }
  // reduce-scatter: after the step of width d the lane keeps the half of its
  // values selected by (lane & d); finally lane j holds pair j = a*8 + b
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
#pragma unroll
    for (int i = 0; i < d; ++i) {
      const bool upper = lane & d;
      const float send = upper ? acc[i] : acc[i + d];
      const float keep = upper ? acc[i + d] : acc[i];
      acc[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, d));
    }
  }
  const int t = t0 + tw + (lane >> 3), e = e0 + ew + (lane & 7);
  if (t < T && e < E) logits[(size_t)t * E + e] = acc[0];
}

constexpr int kSelWarps = 4;

// Softmax-top-k, one warp per token.
template <int EPL>
__global__ void __launch_bounds__(kSelWarps * 32)
    select_softmax_kernel(const float* __restrict__ logits, int T, int E, int k,
                          int32_t* __restrict__ ids, float* __restrict__ wts) {
  __shared__ float sv[kSelWarps][rsel::kMaxK];
  __shared__ float sex[kSelWarps][rsel::kMaxK];
  __shared__ float ssum[kSelWarps];
  griddep_launch();
  griddep_wait();  // logits from the previous kernel
  const int wid = threadIdx.x >> 5;
  const int t = blockIdx.x * kSelWarps + wid;
  if (t >= T) return;
  rsel::softmax_token<EPL>(logits, t, E, k, ids, wts, sv[wid], sex[wid], &ssum[wid]);
}

// Sigmoid-group, one warp per token (n_groups <= 32, E <= 32 * EPL).
template <int EPL>
__global__ void __launch_bounds__(kSelWarps * 32)
    select_sigmoid_group_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                                int T, int E, int n_groups, int topk_groups, int k, float scale,
                                int32_t* __restrict__ ids, float* __restrict__ wts) {
  __shared__ float ssel[kSelWarps][32 * EPL];
  __shared__ float ss[kSelWarps][rsel::kMaxK];
  __shared__ float ssum[kSelWarps];
  griddep_launch();
  griddep_wait();  // logits from the previous kernel
  const int wid = threadIdx.x >> 5;
  const int t = blockIdx.x * kSelWarps + wid;
  if (t >= T) return;
  rsel::sigmoid_group_token<EPL>(logits, bias, t, E, n_groups, topk_groups, k, scale, ids, wts,
                                 ssel[wid], ss[wid], &ssum[wid]);
}

template <int EPL>
cudaError_t launch_select(const moe_spec& sp, const float* logits, const float* bias, int T,
                          int32_t* ids, float* weights, cudaStream_t st) {
  const int grid = (T + kSelWarps - 1) / kSelWarps;
  if (sp.router == MOE_ROUTER_SOFTMAX_TOPK)
    return launch_pdl(select_softmax_kernel<EPL>, dim3(grid), dim3(kSelWarps * 32), 0, st, logits,
                      T, sp.num_experts, sp.top_k, ids, weights);
  return launch_pdl(select_sigmoid_group_kernel<EPL>, dim3(grid), dim3(kSelWarps * 32), 0, st,
                    logits, bias, T, sp.num_experts, sp.n_groups, sp.topk_groups, sp.top_k,
                    sp.routed_scale, ids, weights);
}

}  // namespace

cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* w, int T, int E, int H,
                                 float* logits, cudaStream_t st) {
  if (H % 256 == 0 && T >= kTileTok) {
    const dim3 grid((T + kTileTok - 1) / kTileTok, (E + kTileExp - 1) / kTileExp);
    return launch_pdl(router_logits_tiled_kernel, grid, dim3(256), 0, st, x, w, T, E, H, logits);
  }
  const long warps = (long)T * E;
  const int grid = (int)((warps + 3) / 4);
  return launch_pdl(router_logits_kernel, dim3(grid), dim3(128), 0, st, x, w, T, E, H, logits);
}

cudaError_t launch_router_select(const moe_spec& sp, const float* logits, const float* bias,
                                 int T, int32_t* ids, float* weights, cudaStream_t st) {
  const int E = sp.num_experts;
  if (E <= 32) return launch_select<1>(sp, logits, bias, T, ids, weights, st);
  if (E <= 64) return launch_select<2>(sp, logits, bias, T, ids, weights, st);
  if (E <= 128) return launch_select<4>(sp, logits, bias, T, ids, weights, st);
  if (E <= 256) return launch_select<8>(sp, logits, bias, T, ids, weights, st);
  if (E <= 512) return launch_select<16>(sp, logits, bias, T, ids, weights, st);
  return launch_select<32>(sp, logits, bias, T, ids, weights, st);
}

}  // namespace moe
