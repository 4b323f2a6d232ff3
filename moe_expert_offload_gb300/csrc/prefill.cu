// Prefill path around the grouped GEMMs (FreeToken summary "method steps":
// prefill computes layer l from one whole-layer buffer while the next layer
// streams into the other; reader "System Architecture" ping-pong buffers).
//
//   1. x -> x_perm: each 8-element chunk reordered 0,4,1,5,2,6,3,7 (the K
//      order of the GEMM operands).
//   2. routing permute: a stable counting sort of the T*k (token, rank)
//      assignments by expert, in chunks of 2048 ids; the shared expert (if any) is one more group
//      holding every token in order.  Offsets, and 256-row m-tiles per group.
//   3. GEMM1 (gate/up + SwiGLU) and GEMM2 (down, weighted per assignment).
//   4. combine: y[t] = sum over j = 0..k of y_assign[t][j], in j order.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kTileRows = kPrefillTileRows;

__global__ void permute_x_kernel(const uint4* __restrict__ x, uint4* __restrict__ xp, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 v = __ldg(x + i);
    uint4 o;
    o.x = __byte_perm(v.x, v.z, 0x5410);
    o.y = __byte_perm(v.x, v.z, 0x7632);
    o.z = __byte_perm(v.y, v.w, 0x5410);
    o.w = __byte_perm(v.y, v.w, 0x7632);
    xp[i] = o;
  }
}

// Assignments are permuted in chunks of kChunk ids (8 warps x 256): the
// chunk's per-expert counts, then every chunk's base in each group, then each
// warp places its ids in order.  The result is the stable counting sort.
constexpr int kChunk = 2048;
constexpr int kChunkWarps = 8;
constexpr int kWarpIds = kChunk / kChunkWarps;

// chunk c: per-expert counts cnt[c][e] (ids outside [0, E) are flagged and skipped)
__global__ void __launch_bounds__(256) chunk_count_kernel(const int32_t* __restrict__ ids, int n,
                                                          int E, int32_t* __restrict__ cnt,
                                                          int32_t* err) {
  extern __shared__ int32_t h[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  bool bad = false;
  const int i0 = blockIdx.x * kChunk, i1 = min(n, i0 + kChunk);
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    const int e = ids[i];
    if (e >= 0 && e < E)
      atomicAdd(&h[e], 1);
    else
      bad = true;
  }
  if (bad && err) atomicOr(err, MOE_DERR_BAD_ID);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[(int64_t)blockIdx.x * E + e] = h[e];
}

// One CTA: group offsets (exclusive scan of counts, group E = shared expert
// with T rows) and the m-tile table (256 rows per tile, ragged last tile).
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ cnt, int nch,
                                                    int32_t* __restrict__ cbase,
                                                    int32_t* counts, int E, int T,
                                                    int has_shared, int32_t* offsets,
                                                    int32_t* tile_g, int32_t* tile_row0,
                                                    int32_t* tile_rows, int32_t* n_tiles,
                                                    int max_tiles) {
  __shared__ int s_wr[32], s_wt[32];
  const int G = E + 1;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // each thread owns one group (G = E + 1 <= 1024); routed group totals from the chunk counts
  int c = 0, t = 0;
  if (tid < E)
    for (int ch = 0; ch < nch; ++ch) c += cnt[(int64_t)ch * E + tid];
  else if (tid == E)
    c = has_shared ? T : 0;
  if (tid < G) {
    counts[tid] = c;
    t = (c + kTileRows - 1) / kTileRows;
  }
  // block exclusive scans of rows and tiles
  int ir = c, it = t;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int vr = __shfl_up_sync(0xffffffffu, ir, d), vt = __shfl_up_sync(0xffffffffu, it, d);
    if (lane >= d) {
      ir += vr;
      it += vt;
    }
  }
  if (lane == 31) {
    s_wr[wid] = ir;
    s_wt[wid] = it;
  }
  __syncthreads();
  if (wid == 0) {
    int wr = s_wr[lane], wt = s_wt[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int vr = __shfl_up_sync(0xffffffffu, wr, d), vt = __shfl_up_sync(0xffffffffu, wt, d);
      if (lane >= d) {
        wr += vr;
        wt += vt;
      }
    }
    s_wr[lane] = wr;
    s_wt[lane] = wt;
  }
  __syncthreads();
  const int base_r = (wid > 0 ? s_wr[wid - 1] : 0) + ir - c;
  const int base_t = (wid > 0 ? s_wt[wid - 1] : 0) + it - t;
  if (tid < E) {  // where each chunk's ids of group tid start
    int run = base_r;
    for (int ch = 0; ch < nch; ++ch) {
      cbase[(int64_t)ch * E + tid] = run;
      run += cnt[(int64_t)ch * E + tid];
    }
  }
  if (tid < G) {
    offsets[tid] = base_r;
    for (int j = 0; j < t; ++j) {
      const int m = base_t + j;
      if (m < max_tiles) {
        tile_g[m] = tid;
        tile_row0[m] = base_r + j * kTileRows;
        tile_rows[m] = min(kTileRows, c - j * kTileRows);
      }
    }
  }
  if (tid == G - 1) {
    offsets[G] = base_r + c;
    *n_tiles = min(base_t + t, max_tiles);
  }
}

// CTA c < nch: chunk c's ids to perm in ascending order within each group.
// Each warp counts its 256 ids per expert, the warps' starts follow from the
// chunk base, then each warp walks its ids 32 at a time (lanes of equal
// expert ranked by lane).  CTA nch (shared expert) writes T*k + t for every t.
__global__ void __launch_bounds__(kChunkWarps * 32) scatter_kernel(
    const int32_t* __restrict__ ids, int n, int T, int E, int nch,
    const int32_t* __restrict__ cbase, const int32_t* __restrict__ offsets,
    int32_t* __restrict__ perm) {
  extern __shared__ int32_t wb[];  // [kChunkWarps][E]: per-warp counts, then starts
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (blockIdx.x == nch) {
    const int base = offsets[E];
    for (int t = tid; t < T; t += blockDim.x) perm[base + t] = n + t;
    return;
  }
  for (int i = tid; i < kChunkWarps * E; i += blockDim.x) wb[i] = 0;
  __syncthreads();
  const int i0 = blockIdx.x * kChunk + w * kWarpIds, i1 = min(n, i0 + kWarpIds);
  for (int b = i0; b < i1; b += 32) {
    const int i = b + lane;
    int e = i < i1 ? ids[i] : -1;
    if (e < 0 || e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) wb[w * E + e] += __popc(peers);
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int run = cbase[(int64_t)blockIdx.x * E + e];
    for (int v = 0; v < kChunkWarps; ++v) {
      const int c = wb[v * E + e];
      wb[v * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int b = i0; b < i1; b += 32) {
    const int i = b + lane;
    int e = i < i1 ? ids[i] : -1;
    if (e < 0 || e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int start = wb[w * E + e];
      perm[start + __popc(peers & ((1u << lane) - 1u))] = i;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) wb[w * E + e] += __popc(peers);
    __syncwarp();
  }
}

// y[t][o] = sum_{j=0..k} y_assign[t][j][o] (bf16 terms, fp32 sum, j order);
// routed terms whose id was invalid are skipped.
__global__ void combine_kernel(const uint16_t* __restrict__ ya, const int32_t* __restrict__ ids,
                               int T, int k, int E, int H, int has_shared, float* __restrict__ y) {
  const int nslot = k + 1;
  const int64_t n = (int64_t)T * H / 8;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = (i * 8) / H, o = (i * 8) % H;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < nslot; ++j) {
      if (j < k) {
        const int e = ids[t * k + j];
        if (e < 0 || e >= E) continue;
      } else if (!has_shared) {
        continue;
      }
      const uint4 v = __ldcs(reinterpret_cast<const uint4*>(ya + (t * nslot + j) * H + o));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] += __uint_as_float(w[q] << 16);
        acc[2 * q + 1] += __uint_as_float(w[q] & 0xFFFF0000u);
      }
    }
    float4* dst = reinterpret_cast<float4*>(y + t * H + o);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// The double buffer's whole-layer copy (bank -> layer buffer), n 16-byte words:
// one CTA of 256 threads per SM, each thread with eight streaming loads in
// flight before its eight stores (L2 evict-first on both sides: the layer
// passes through once).  It holds no shared memory and few registers, so it
// shares every SM with the routing kernels it runs beside (their CTAs leave
// room for it) instead of taking SMs from them.
__global__ void __launch_bounds__(256) layer_copy_kernel(const uint4* __restrict__ src,
                                                         uint4* __restrict__ dst, int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 7 * stride < n; i += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldcs(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < 8; ++u) __stcs(dst + i + u * stride, v[u]);
  }
  for (; i < n; i += stride) __stcs(dst + i, __ldcs(src + i));
}

size_t al256(size_t b) { return (b + 255) / 256 * 256; }

int max_tiles_for(int E, int k, int T) {
  return (int)(((int64_t)T * k + T + kTileRows - 1) / kTileRows) + E + 1;
}

}  // namespace

size_t prefill_workspace_bytes(int H, int I, int E, int k, int T) {
  const size_t R = (size_t)T * k + T;
  const size_t mt = max_tiles_for(E, k, T);
  const size_t nch = ((size_t)T * k + kChunk - 1) / kChunk;
  return al256((size_t)T * H * 2) + al256((size_t)(E + 1) * 4) + al256((size_t)(E + 2) * 4) +
         al256(R * 4) + 3 * al256(mt * 4) + al256(4) + al256(R * I * 2) +
         al256((size_t)T * (k + 1) * H * 2) + 2 * al256(nch * E * 4);
}

void prefill_carve(PrefillBufs& b, void* ws, int H, int I, int E, int k, int T) {
  const size_t R = (size_t)T * k + T;
  const size_t mt = max_tiles_for(E, k, T);
  uint8_t* p = static_cast<uint8_t*>(ws);
  auto take = [&](size_t n) {
    uint8_t* q = p;
    p += al256(n);
    return q;
  };
  b.x_perm = reinterpret_cast<uint16_t*>(take((size_t)T * H * 2));
  b.counts = reinterpret_cast<int32_t*>(take((size_t)(E + 1) * 4));
  b.offsets = reinterpret_cast<int32_t*>(take((size_t)(E + 2) * 4));
  b.perm = reinterpret_cast<int32_t*>(take(R * 4));
  b.tile_g = reinterpret_cast<int32_t*>(take(mt * 4));
  b.tile_row0 = reinterpret_cast<int32_t*>(take(mt * 4));
  b.tile_rows = reinterpret_cast<int32_t*>(take(mt * 4));
  b.n_tiles = reinterpret_cast<int32_t*>(take(4));
  b.h_perm = reinterpret_cast<uint16_t*>(take(R * I * 2));
  b.y_assign = reinterpret_cast<uint16_t*>(take((size_t)T * (k + 1) * H * 2));
  b.nch = (int)(((size_t)T * k + kChunk - 1) / kChunk);
  b.chunk_cnt = reinterpret_cast<int32_t*>(take((size_t)b.nch * E * 4));
  b.chunk_base = reinterpret_cast<int32_t*>(take((size_t)b.nch * E * 4));
  b.max_tiles = (int)mt;
}

cudaError_t launch_prefill_ffn(const GemmArgs& base, const PrefillBufs& b, const uint16_t* x,
                               const int32_t* ids, int has_shared, float* y, cudaStream_t st) {
  const int H = base.H, E = base.E, k = base.k, T = base.T;
  const int n = T * k;
  cudaError_t e;
  const int64_t nx = (int64_t)T * H / 8;
  permute_x_kernel<<<(int)((nx + 255) / 256 < 4096 ? (nx + 255) / 256 : 4096), 256, 0, st>>>(
      reinterpret_cast<const uint4*>(x), reinterpret_cast<uint4*>(b.x_perm), nx);
  chunk_count_kernel<<<b.nch, 256, E * 4, st>>>(ids, n, E, b.chunk_cnt, base.err);
  plan_kernel<<<1, 1024, 0, st>>>(b.chunk_cnt, b.nch, b.chunk_base, b.counts, E, T, has_shared,
                                  b.offsets, b.tile_g, b.tile_row0, b.tile_rows, b.n_tiles,
                                  b.max_tiles);
  scatter_kernel<<<b.nch + (has_shared ? 1 : 0), kChunkWarps * 32, kChunkWarps * E * 4, st>>>(
      ids, n, T, E, b.nch, b.chunk_base, b.offsets, b.perm);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  GemmArgs a = base;
  a.perm = b.perm;
  a.tile_g = b.tile_g;
  a.tile_row0 = b.tile_row0;
  a.tile_rows = b.tile_rows;
  a.n_tiles = b.n_tiles;
  a.a_src = b.x_perm;
  a.h_out = b.h_perm;
  a.y_out = b.y_assign;
  if ((e = launch_grouped_gemm(1, a, b.max_tiles, st)) != cudaSuccess) return e;
  a.a_src = b.h_perm;
  if ((e = launch_grouped_gemm(2, a, b.max_tiles, st)) != cudaSuccess) return e;
  const int64_t nc = (int64_t)T * H / 8;
  combine_kernel<<<(int)((nc + 255) / 256 < 8192 ? (nc + 255) / 256 : 8192), 256, 0, st>>>(
      b.y_assign, ids, T, k, E, H, has_shared, y);
  return cudaGetLastError();
}

cudaError_t launch_layer_copy(const void* src, void* dst, size_t bytes, cudaStream_t st) {
  if (bytes == 0) return cudaSuccess;
  if (((uintptr_t)src | (uintptr_t)dst | bytes) & 15u)
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st);
  int d = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d);
  if (e != cudaSuccess) return e;
  layer_copy_kernel<<<sms, 256, 0, st>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                         (int64_t)(bytes / 16));
  return cudaGetLastError();
}

}  // namespace moe
