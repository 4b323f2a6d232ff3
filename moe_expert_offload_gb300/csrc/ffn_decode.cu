// Decode expert FFN: int4 affine group-64 SwiGLU experts
// y_e = Wd (silu(Wg x) * (Wu x)) (Edge0 §3.1 "math convention"), executed
// for every routed id of the step -- H and F from their slots, C in place
// from the bank -- plus the always-on shared expert, and the exact weighted
// merge of the per-expert partial outputs (FreeToken summary "core method").
//
// Decode moves a few KB of activations against MBs of packed weights, so it
// is bound by HBM bandwidth.  Each warp streams 16-byte code vectors
// straight into registers and dequantises there:
//   a byte pair of nibbles is spread into a bf16x2 holding 128 + q with one
//   LOP3 (0x4300 | q), each half widened to fp32 by a shift or a mask, and a
//   32-column chunk is reduced as A = sum (128 + q_j) x_j.  With
//   X = sum x_j over the chunk (precomputed once per token), the chunk's
//   contribution is  s * A + (b - 128 s) * X  = sum (s q_j + b) x_j.
// Activations live in shared memory as fp32, rotated per chunk so that the
// 16-byte loads of the eight lanes of a quarter warp hit distinct banks.
//
// Phase A (gate/up): CTA = (entry, 32 rows of I): 8 warps x 4 gate/up row
//   pairs, h[entry][t][i] = silu(g) * u into the workspace.
// Phase B (down): CTA = (entry, block of H rows); it writes the weighted
//   partial  w[t][j] * (Wd h)[o]  into partial[t][j][o], where j is the rank
//   of this expert in token t's routing (j = k for the shared expert).  The
//   last CTA to finish a row block (arrival counter) sums partial[t][0..k]
//   in j order into y: a fixed order, no atomics on data, deterministic.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsA = 4;  // gate/up row pairs per warp (phase A)
constexpr int kRowsB = 4;  // down rows per lane (phase B)
constexpr int kTT = 2;     // tokens staged per pass

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// sum_j (128 + q_j) x_j over one 8-column word (nibble j = column j).
__device__ __forceinline__ float word_dot(uint32_t w, float4 lo, float4 hi, float acc) {
  const float xl[4] = {lo.x, lo.y, lo.z, lo.w};
  const float xh[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t p = ((w >> (4 * k)) & 0x000F000Fu) | 0x43004300u;
    acc = fmaf(__uint_as_float(p << 16), xl[k], acc);
    acc = fmaf(__uint_as_float(p & 0xFFFF0000u), xh[k], acc);
  }
  return acc;
}

__device__ __forceinline__ float chunk_dot(uint4 q, const float4 (&xv)[8]) {
  float a = word_dot(q.x, xv[0], xv[1], 0.0f);
  a = word_dot(q.y, xv[2], xv[3], a);
  a = word_dot(q.z, xv[4], xv[5], a);
  return word_dot(q.w, xv[6], xv[7], a);
}

// Entry r of the step: its blob and the tokens routed to it.
struct EntryInfo {
  const uint8_t* blob;
  int ntok;
};

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
      const int32_t slot = a.slot_of_id[id];
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

// Stage `nt` fp32 vectors of length n (from bf16 x rows or fp32 h rows) into
// shared memory: chunk c (32 values) holds its eight float4 slots rotated by
// c, and xsum[c] = sum of the chunk's 32 values.
template <bool kBf16>
__device__ void stage_vectors(const void* src, int64_t row_stride, const int* rows, int nt, int n,
                              float* xs, float* xsum) {
  const int nc = n / 32;
  for (int it = threadIdx.x; it < nt * nc; it += blockDim.x) {
    const int tt = it / nc, c = it - tt * nc;
    float v[32];
    if (kBf16) {
      const uint4* p = reinterpret_cast<const uint4*>(
          static_cast<const uint16_t*>(src) + (int64_t)rows[tt] * row_stride + c * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 u = __ldg(p + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
          v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
      }
    } else {
      const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) +
                                                        (int64_t)rows[tt] * row_stride + c * 32);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 f = __ldcg(p + i);
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
      }
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) s += v[i];
    float4* dst = reinterpret_cast<float4*>(xs + (int64_t)tt * n + c * 32);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      dst[(q + c) & 7] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    xsum[tt * nc + c] = s;
  }
}

__device__ __forceinline__ void load_chunk(const float* xs, int c, float4 (&xv)[8]) {
  const float4* p = reinterpret_cast<const float4*>(xs + c * 32);
#pragma unroll
  for (int q = 0; q < 8; ++q) xv[q] = p[(q + c) & 7];
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// ------------------------------------------------------------------ phase A
__global__ void __launch_bounds__(kThreads, 2) ffn_gate_up_kernel(FfnArgs a, int n_tick) {
  extern __shared__ __align__(16) float smem[];
  __shared__ int stok[kMaxDecodeT], sj[kMaxDecodeT];
  __shared__ float sw[kMaxDecodeT];
  __shared__ EntryInfo ent;
  const int H = a.H, I = a.I, nch = H / 32;
  float* xs = smem;                  // [kTT][H]
  float* xsum = smem + kTT * H;      // [kTT][H/32]
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_tick; i += kThreads) a.tick[i] = 0u;

  const int tasks = I / (kWarps * kRowsA);
  const int r = blockIdx.x / tasks, rb = blockIdx.x - r * tasks;
  if (!resolve_entry(a, r, stok, sj, sw, &ent)) return;
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i0 = (rb * kWarps + wid) * kRowsA;
  const BlobOffsets off = blob_offsets(H, I);
  const uint8_t* blob = ent.blob;
  const int64_t crow = H / 2, srow = H / kGroup;
  const uint8_t* gq = blob + off.gq + i0 * crow;
  const uint8_t* uq = blob + off.uq + i0 * crow;
  const uint16_t* gs = reinterpret_cast<const uint16_t*>(blob + off.gs) + i0 * srow;
  const uint16_t* gb = reinterpret_cast<const uint16_t*>(blob + off.gb) + i0 * srow;
  const uint16_t* us = reinterpret_cast<const uint16_t*>(blob + off.us) + i0 * srow;
  const uint16_t* ub = reinterpret_cast<const uint16_t*>(blob + off.ub) + i0 * srow;

  for (int t0 = 0; t0 < ent.ntok; t0 += kTT) {
    const int nt = min(kTT, ent.ntok - t0);
    __syncthreads();
    stage_vectors<true>(a.x, H, stok + t0, nt, H, xs, xsum);
    __syncthreads();
    float accg[kRowsA][kTT], accu[kRowsA][kTT];
#pragma unroll
    for (int j = 0; j < kRowsA; ++j)
#pragma unroll
      for (int tt = 0; tt < kTT; ++tt) accg[j][tt] = accu[j][tt] = 0.0f;

    for (int c = lane; c < nch; c += 32) {
      uint4 qg[kRowsA], qu[kRowsA];
#pragma unroll
      for (int j = 0; j < kRowsA; ++j) {
        qg[j] = ld_stream(gq + j * crow + c * 16);
        qu[j] = ld_stream(uq + j * crow + c * 16);
      }
      float sg[kRowsA], bg[kRowsA], su[kRowsA], bu[kRowsA];
#pragma unroll
      for (int j = 0; j < kRowsA; ++j) {
        const int gi = j * (int)srow + (c >> 1);
        sg[j] = bf16f(__ldg(gs + gi));
        bg[j] = fmaf(-128.0f, sg[j], bf16f(__ldg(gb + gi)));
        su[j] = bf16f(__ldg(us + gi));
        bu[j] = fmaf(-128.0f, su[j], bf16f(__ldg(ub + gi)));
      }
#pragma unroll
      for (int tt = 0; tt < kTT; ++tt) {
        if (tt < nt) {
          float4 xv[8];
          load_chunk(xs + tt * H, c, xv);
          const float X = xsum[tt * nch + c];
#pragma unroll
          for (int j = 0; j < kRowsA; ++j) {
            accg[j][tt] = fmaf(sg[j], chunk_dot(qg[j], xv), fmaf(bg[j], X, accg[j][tt]));
            accu[j][tt] = fmaf(su[j], chunk_dot(qu[j], xv), fmaf(bu[j], X, accu[j][tt]));
          }
        }
      }
    }
#pragma unroll
    for (int tt = 0; tt < kTT; ++tt) {
#pragma unroll
      for (int j = 0; j < kRowsA; ++j) {
        const float g = warp_sum(accg[j][tt]);
        const float u = warp_sum(accu[j][tt]);
        if (lane == j && tt < nt) {
          const float silu = g / (1.0f + __expf(-g));
          a.h[((int64_t)r * a.T + stok[t0 + tt]) * I + i0 + j] = silu * u;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ phase B
// lanes_per_row lanes (a power of two <= 32) share one down row; a warp
// covers rows_per_warp = (32 / lanes_per_row) * kRowsB rows.
__global__ void __launch_bounds__(kThreads, 2) ffn_down_kernel(FfnArgs a, int lanes_per_row,
                                                               int rows_per_cta) {
  extern __shared__ __align__(16) float smem[];
  __shared__ int stok[kMaxDecodeT], sj[kMaxDecodeT];
  __shared__ float sw[kMaxDecodeT];
  __shared__ EntryInfo ent;
  __shared__ int s_last;
  const int H = a.H, I = a.I, nch = I / 32;
  const int nslot = a.k + a.has_shared;
  float* hs = smem;              // [kTT][I]
  float* hsum = smem + kTT * I;  // [kTT][I/32]
  const int nblk = (H + rows_per_cta - 1) / rows_per_cta;
  const int r = blockIdx.x / nblk, blk = blockIdx.x - r * nblk;
  if (!resolve_entry(a, r, stok, sj, sw, &ent)) return;

  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lpr = lanes_per_row, rpi = 32 / lpr;
  const int rsub = lane / lpr, cl = lane - rsub * lpr;
  const int o_warp = blk * rows_per_cta + wid * rpi * kRowsB;
  const BlobOffsets off = blob_offsets(H, I);
  const uint8_t* blob = ent.blob;
  const int64_t crow = I / 2, srow = I / kGroup;
  const uint8_t* dq = blob + off.dq;
  const uint16_t* ds = reinterpret_cast<const uint16_t*>(blob + off.ds);
  const uint16_t* db = reinterpret_cast<const uint16_t*>(blob + off.db);
  int orow[kRowsB];
#pragma unroll
  for (int j = 0; j < kRowsB; ++j) orow[j] = o_warp + rsub + rpi * j;

  for (int t0 = 0; t0 < ent.ntok; t0 += kTT) {
    const int nt = min(kTT, ent.ntok - t0);
    __syncthreads();
    {
      int hrow[kTT];
      for (int tt = 0; tt < nt; ++tt) hrow[tt] = r * a.T + stok[t0 + tt];
      stage_vectors<false>(a.h, I, hrow, nt, I, hs, hsum);
    }
    __syncthreads();
    float acc[kRowsB][kTT];
#pragma unroll
    for (int j = 0; j < kRowsB; ++j)
#pragma unroll
      for (int tt = 0; tt < kTT; ++tt) acc[j][tt] = 0.0f;
    for (int c = cl; c < nch; c += lpr) {
      uint4 qd[kRowsB];
      float s[kRowsB], b[kRowsB];
#pragma unroll
      for (int j = 0; j < kRowsB; ++j) {
        const int o = orow[j] < H ? orow[j] : H - 1;
        qd[j] = ld_stream(dq + o * crow + c * 16);
        const int gi = o * (int)srow + (c >> 1);
        s[j] = bf16f(__ldg(ds + gi));
        b[j] = fmaf(-128.0f, s[j], bf16f(__ldg(db + gi)));
      }
#pragma unroll
      for (int tt = 0; tt < kTT; ++tt) {
        if (tt < nt) {
          float4 xv[8];
          load_chunk(hs + tt * I, c, xv);
          const float X = hsum[tt * nch + c];
#pragma unroll
          for (int j = 0; j < kRowsB; ++j)
            acc[j][tt] = fmaf(s[j], chunk_dot(qd[j], xv), fmaf(b[j], X, acc[j][tt]));
        }
      }
    }
#pragma unroll
    for (int tt = 0; tt < kTT; ++tt) {
#pragma unroll
      for (int j = 0; j < kRowsB; ++j) {
        float v = acc[j][tt];
        for (int d = lpr >> 1; d >= 1; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
        if (cl == 0 && tt < nt && orow[j] < H) {
          const int p = t0 + tt;
          a.partial[((int64_t)stok[p] * nslot + sj[p]) * H + orow[j]] = sw[p] * v;
        }
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
  const int o0 = blk * rows_per_cta;
  const int nrow = min(rows_per_cta, H - o0);
  for (int it = threadIdx.x; it < a.T * nrow; it += kThreads) {
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

int lanes_per_row_for(int I) {
  int nch = I / 32, l = 1;
  while (l * 2 <= nch && l * 2 <= 32) l *= 2;
  return l;
}

}  // namespace

// Opt the two kernels into more than 48 KB of dynamic shared memory, once
// per device and size (a host-side setting, not a stream operation).
static cudaError_t raise_smem_limit(size_t bytes) {
  constexpr int kMaxDev = 64;
  static size_t done[kMaxDev] = {};
  if (bytes <= 48 * 1024) return cudaSuccess;
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d >= 0 && d < kMaxDev && done[d] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(ffn_gate_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(ffn_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)bytes);
  if (e == cudaSuccess && d >= 0 && d < kMaxDev) done[d] = bytes;
  return e;
}

static int down_rows_per_cta(int I) { return kWarps * (32 / lanes_per_row_for(I)) * kRowsB; }

size_t ffn_workspace_bytes(int H, int I, int k, int T, int has_shared) {
  auto al = [](size_t b) { return (b + 255) / 256 * 256; };
  const size_t max_entries = (size_t)T * k + has_shared;
  const size_t nblk = (H + down_rows_per_cta(I) - 1) / down_rows_per_cta(I);
  return al(max_entries * T * I * 4) + al((size_t)T * (k + has_shared) * H * 4) + al(nblk * 4);
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
}

cudaError_t launch_ffn_decode(const FfnArgs& a, cudaStream_t st) {
  const int lpr = lanes_per_row_for(a.I);
  const int rows_b = down_rows_per_cta(a.I);
  const int nblk = (a.H + rows_b - 1) / rows_b;
  const size_t smem_a = (size_t)kTT * a.H * 4 + (size_t)kTT * (a.H / 32) * 4;
  const size_t smem_b = (size_t)kTT * a.I * 4 + (size_t)kTT * (a.I / 32) * 4;
  cudaError_t e = raise_smem_limit(smem_a > smem_b ? smem_a : smem_b);
  if (e != cudaSuccess) return e;
  const int grid_a = a.max_entries * (a.I / (kWarps * kRowsA));
  ffn_gate_up_kernel<<<grid_a, kThreads, smem_a, st>>>(a, nblk);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ffn_down_kernel<<<a.max_entries * nblk, kThreads, smem_b, st>>>(a, lpr, rows_b);
  return cudaGetLastError();
}

}  // namespace moe
