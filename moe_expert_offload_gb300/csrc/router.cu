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

using rsel::bf_hi;
using rsel::bf_lo;

// One warp per (token, expert): rsel::router_dot_warp.
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
  const float acc = rsel::router_dot_warp(x + (size_t)t * H, w + (size_t)e * H, H);
  if (lane == 0) logits[(size_t)t * E + e] = acc;
}

// Tiled logits for many tokens, same order as router_logits_kernel: CTA =
// 32 tokens x 16 experts, 8 warps of 8 tokens x 8 experts.  H goes through
// shared memory in 256-column slices (cp.async into a ring of kTileStages
// slices, kTileStages - 1 of them in flight while one is used); in
// slice s lane j owns chunk 32 s + j, so each lane still accumulates chunks
// j, j+32, ... in ascending order with fma from 0.  A lane holds its chunk of
// the warp's 8 expert rows widened to fp32 and streams the 8 token rows
// through them: 64 partial sums per lane.  These are combined by a
// reduce-scatter over the same xor partners 16, 8, 4, 2, 1 (each add pairs
// the same two lane partials as the butterfly, and fp addition is
// commutative, so every logit is bit-identical), separately for pairs 0..31
// and 32..63; lane j ends with pairs j and 32 + j.  Needs H % 256 == 0.
constexpr int kTileTok = 32, kTileExp = 16, kTileMinT = 16, kTileStages = 4;
constexpr int kTileRows = kTileTok + kTileExp;                          // rows per slice
constexpr size_t kTileSmem = (size_t)kTileStages * kTileRows * 32 * 16;  // 96 KB

__device__ __forceinline__ void cp16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}

__global__ void __launch_bounds__(256, 1) router_logits_tiled_kernel(const uint16_t* __restrict__ x,
                                                                     const uint16_t* __restrict__ w,
                                                                     int T, int E, int H,
                                                                     float* __restrict__ logits) {
  // ring of slices: 32 token rows then 16 expert rows of 256 bf16 (32 x 16 B) each
  extern __shared__ __align__(16) uint4 ring[];  // [kTileStages][kTileRows][32]
  griddep_launch();
  griddep_wait();
  const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kTileTok, e0 = blockIdx.y * kTileExp;
  const int tw = (wid >> 1) * 8, ew = (wid & 1) * 8;
  const int ns = H / 256;
  // slice s into ring slot s % kTileStages: 48 rows x 32 chunks = 1536 16-byte
  // copies, 6 per thread; rows past T or E are zero-filled (source size 0,
  // address kept in bounds).  A group is committed even when s >= ns, so the
  // wait below always counts kTileStages - 1 groups.
  auto issue = [&](int s) {
    if (s < ns) {
      uint4* slot = ring + (size_t)(s % kTileStages) * kTileRows * 32;
#pragma unroll
      for (int j = 0; j < 6; ++j) {
        const int i = tid + 256 * j, row = i >> 5, c = i & 31;
        const bool ok = row < kTileTok ? t0 + row < T : e0 + row - kTileTok < E;
        const size_t grow = row < kTileTok ? (size_t)(t0 + row) : (size_t)(e0 + row - kTileTok);
        const uint16_t* base = row < kTileTok ? x : w;
        const uint16_t* src = base + (ok ? grow * H + (size_t)s * 256 + c * 8 : 0);
        cp16((uint32_t)__cvta_generic_to_shared(slot + row * 32 + c), src, ok);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  float acc[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
#pragma unroll
  for (int s = 0; s < kTileStages - 1; ++s) issue(s);
  for (int s = 0; s < ns; ++s) {
    issue(s + kTileStages - 1);  // into the slot freed at the end of slice s - 1
    asm volatile("cp.async.wait_group %0;" ::"n"(kTileStages - 1) : "memory");
    __syncthreads();
    const uint4* xs = ring + (size_t)(s % kTileStages) * kTileRows * 32;
    const uint4* ws = xs + kTileTok * 32;
    float wf[8][8];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const uint4 v = ws[(ew + b) * 32 + lane];
      wf[b][0] = bf_lo(v.x); wf[b][1] = bf_hi(v.x); wf[b][2] = bf_lo(v.y); wf[b][3] = bf_hi(v.y);
      wf[b][4] = bf_lo(v.z); wf[b][5] = bf_hi(v.z); wf[b][6] = bf_lo(v.w); wf[b][7] = bf_hi(v.w);
    }
#pragma unroll
    for (int a = 0; a < 8; ++a) {
      const uint4 v = xs[(tw + a) * 32 + lane];
      const float xf[8] = {bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y),
                           bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w)};
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        float& r = acc[a * 8 + b];
#pragma unroll
        for (int e = 0; e < 8; ++e) r = __fmaf_rn(xf[e], wf[b][e], r);
      }
    }
    __syncthreads();  // slot s % kTileStages is refilled by the issue of slice s + kTileStages
  }
  // reduce-scatter of each half: after the step of width d the lane keeps the
  // half of its values selected by (lane & d); lane j ends with pair h*32 + j
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float* v = acc + 32 * h;
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
#pragma unroll
      for (int i = 0; i < d; ++i) {
        const bool upper = lane & d;
        const float send = upper ? v[i] : v[i + d];
        const float keep = upper ? v[i + d] : v[i];
        v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, d));
      }
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int pr = 32 * h + lane;  // pair a * 8 + b
    const int t = t0 + tw + (pr >> 3), e = e0 + ew + (pr & 7);
    if (t < T && e < E) logits[(size_t)t * E + e] = acc[32 * h];
  }
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
  if (H % 256 == 0 && T >= kTileMinT) {
    const dim3 grid((T + kTileTok - 1) / kTileTok, (E + kTileExp - 1) / kTileExp);
    static bool attr_set[64];
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return e;
    if (d >= 0 && d < 64 && !attr_set[d]) {
      e = cudaFuncSetAttribute(router_logits_tiled_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTileSmem);
      if (e != cudaSuccess) return e;
      attr_set[d] = true;
    }
    return launch_pdl(router_logits_tiled_kernel, grid, dim3(256), kTileSmem, st, x, w, T, E, H,
                      logits);
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
