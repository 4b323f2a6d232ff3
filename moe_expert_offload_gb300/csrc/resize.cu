// Elastic re-division of the shared slot pool at a safe point between steps
// (FreeToken reader, "Elastic Memory Management": the number of slots follows
// the free memory -- floor(free / slot size) -- the excess slots are evicted
// on a shrink, new empty slots appear on a growth, and neither the bank nor
// the routing changes).
//
// On a shrink from S to S' slots the cache keeps its S' most recently routed
// experts: the occupied slots with the smallest keys (ts, slot) -- the order
// of the victim scan -- are evicted until at most S' remain, and the kept
// experts that sit in slots >= S' move (tables and blob) to the free slots
// below S', pairing both in ascending slot order.  Slots past the smaller of
// the two sizes are left empty (id -1, ts 0), so a later growth starts from
// empty slots.  The clock does not move.
//
// Two kernels: one CTA plans and updates the tables (a radix select over the
// 64-bit keys finds the eviction threshold in eight counting passes, then
// block scans place the moves), and a grid copies the moved blobs.
#include <cstdint>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRzThreads = 1024;
constexpr int kRzWarps = kRzThreads / 32;

struct RzShared {
  uint32_t warp[kRzWarps];
  uint32_t total;
  int bad;
  uint32_t hist[256];  // radix select: keys per digit value
  uint32_t digit, below;
};

// Sum of v over the block (all threads call it; two barriers).
__device__ uint32_t block_sum(uint32_t v, RzShared& sh) {
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  v = __reduce_add_sync(0xffffffffu, v);
  if (lane == 0) sh.warp[wid] = v;
  __syncthreads();
  if (wid == 0) {
    uint32_t w = lane < kRzWarps ? sh.warp[lane] : 0u;
    w = __reduce_add_sync(0xffffffffu, w);
    if (lane == 0) sh.total = w;
  }
  __syncthreads();
  const uint32_t t = sh.total;
  __syncthreads();  // sh is reused by the next call
  return t;
}

// Exclusive prefix of the 0/1 flag f over the block in thread order, plus the
// block's total (all threads call it).
__device__ uint32_t block_scan(uint32_t f, uint32_t& total, RzShared& sh) {
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bal = __ballot_sync(0xffffffffu, f != 0u);
  const uint32_t below = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) sh.warp[wid] = __popc(bal);
  __syncthreads();
  if (wid == 0) {
    const uint32_t c = lane < kRzWarps ? sh.warp[lane] : 0u;
    uint32_t incl = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    if (lane < kRzWarps) sh.warp[lane] = incl - c;  // exclusive
    if (lane == 31) sh.total = incl;
  }
  __syncthreads();
  const uint32_t r = sh.warp[wid] + below;
  total = sh.total;
  __syncthreads();
  return r;
}

__device__ __forceinline__ uint64_t slot_key(const uint32_t* ts, int v) {
  return ((uint64_t)ts[v] << 32) | (uint32_t)v;
}

// ws: [0] evicted, [1] moved, [2] occupied after, [3] error bits (MOE_DERR_RANGE:
// the tables were not a bijection and nothing was changed), then the move
// sources, the move destinations and the evicted ids (cap entries each).
__global__ void __launch_bounds__(kRzThreads, 1)
    resize_plan_kernel(int32_t* slot_of_id, int n_ids, int32_t* id_of_slot, uint32_t* ts, int S,
                       int S_new, int cap, int32_t* ws) {
  __shared__ RzShared sh;
  const int tid = threadIdx.x;
  int32_t* from = ws + 8;
  int32_t* to = from + cap;
  int32_t* evicted = to + cap;
  if (tid == 0) sh.bad = 0;
  __syncthreads();
  // the tables must be a bijection on the occupied slots
  uint32_t occ = 0;
  for (int v = tid; v < S; v += kRzThreads) {
    const int32_t u = id_of_slot[v];
    if (u >= n_ids || (u >= 0 && slot_of_id[u] != v)) sh.bad = 1;
    occ += u >= 0 ? 1u : 0u;
  }
  const uint32_t n_occ = block_sum(occ, sh);
  if (sh.bad) {
    if (tid == 0) {
      ws[0] = ws[1] = 0;
      ws[2] = (int32_t)n_occ;
      ws[3] = MOE_DERR_RANGE;
    }
    return;
  }
  const uint32_t n_ev = n_occ > (uint32_t)S_new ? n_occ - (uint32_t)S_new : 0u;

  // the eviction threshold: the n_ev-th smallest occupied key (keys are distinct,
  // so exactly n_ev keys lie at or below it), by a radix select over the 64-bit
  // keys, 8 bits per pass from the top: each pass counts the keys that share
  // the digits found so far by their next digit and keeps the digit whose
  // cumulative count first reaches the remaining rank
  uint64_t thr = 0;
  if (n_ev > 0) {
    uint64_t prefix = 0, pmask = 0;
    uint32_t rank = n_ev;  // 1-based rank among the keys that match prefix
    for (int shift = 56; shift >= 0; shift -= 8) {
      if (tid < 256) sh.hist[tid] = 0u;
      __syncthreads();
      for (int v = tid; v < S; v += kRzThreads) {
        if (id_of_slot[v] < 0) continue;
        const uint64_t key = slot_key(ts, v);
        if ((key & pmask) == prefix) atomicAdd(&sh.hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid < 32) {
        // lane l holds digits 8 l .. 8 l + 7; an exclusive scan over the lanes
        uint32_t c[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = sh.hist[8 * tid + j];
          sum += c[j];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const uint32_t o = __shfl_up_sync(0xffffffffu, incl, d);
          if (tid >= d) incl += o;
        }
        uint32_t run = incl - sum;  // keys with a smaller digit than 8 l
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run < rank && rank <= run + c[j]) {
            sh.digit = 8u * tid + j;
            sh.below = run;
          }
          run += c[j];
        }
      }
      __syncthreads();
      prefix |= (uint64_t)sh.digit << shift;
      pmask |= (uint64_t)255u << shift;
      rank -= sh.below;
      __syncthreads();  // hist, digit and below are rewritten by the next pass
    }
    thr = prefix;
  }
  // evict (the list in ascending slot order)
  uint32_t base = 0;
  for (int v0 = 0; v0 < S; v0 += kRzThreads) {
    const int v = v0 + tid;
    const bool e = n_ev > 0 && v < S && id_of_slot[v] >= 0 && slot_key(ts, v) <= thr;
    uint32_t tot;
    const uint32_t r = block_scan(e ? 1u : 0u, tot, sh);
    if (e) {
      const int32_t u = id_of_slot[v];
      evicted[base + r] = u;
      slot_of_id[u] = -1;
      id_of_slot[v] = -1;
      ts[v] = 0;
    }
    base += tot;
  }
  __syncthreads();
  // sources: the kept experts at or past S_new, ascending
  uint32_t n_mv = 0;
  for (int v0 = S_new; v0 < S; v0 += kRzThreads) {
    const int v = v0 + tid;
    const bool f = v < S && id_of_slot[v] >= 0;
    uint32_t tot;
    const uint32_t r = block_scan(f ? 1u : 0u, tot, sh);
    if (f) from[n_mv + r] = v;
    n_mv += tot;
  }
  // destinations: the first n_mv free slots below S_new, ascending
  uint32_t n_to = 0;
  const int lim = S_new < S ? S_new : S;
  for (int v0 = 0; v0 < lim && n_to < n_mv; v0 += kRzThreads) {
    const int v = v0 + tid;
    const bool f = v < lim && id_of_slot[v] < 0;
    uint32_t tot;
    const uint32_t r = block_scan(f ? 1u : 0u, tot, sh);
    if (f && n_to + r < n_mv) to[n_to + r] = v;
    n_to += tot;
  }
  __syncthreads();
  // the moves (distinct slots on both sides), then the slots past the smaller size
  for (uint32_t i = tid; i < n_mv; i += kRzThreads) {
    const int a = from[i], b = to[i];
    const int32_t u = id_of_slot[a];
    id_of_slot[b] = u;
    ts[b] = ts[a];
    slot_of_id[u] = b;
  }
  __syncthreads();
  const int lo_v = S < S_new ? S : S_new, hi_v = S < S_new ? S_new : S;
  for (int v = lo_v + tid; v < hi_v; v += kRzThreads) {
    id_of_slot[v] = -1;
    ts[v] = 0;
  }
  if (tid == 0) {
    ws[0] = (int32_t)n_ev;
    ws[1] = (int32_t)n_mv;
    ws[2] = (int32_t)(n_occ - n_ev);
    ws[3] = 0;
  }
}

// The moved blobs: pool[from[i]] -> pool[to[i]] for i < ws[1] (the sources lie
// at or past S_new, the destinations below it: no copy overlaps another).
__global__ void __launch_bounds__(256) resize_move_kernel(const int32_t* __restrict__ ws, int cap,
                                                          uint8_t* __restrict__ pool,
                                                          int64_t blob_bytes) {
  const int n = ws[1];
  const int32_t* from = ws + 8;
  const int32_t* to = from + cap;
  const int64_t n16 = blob_bytes / 16;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int i = blockIdx.y; i < n; i += gridDim.y) {
    const uint4* src = reinterpret_cast<const uint4*>(pool + (int64_t)from[i] * blob_bytes);
    uint4* dst = reinterpret_cast<uint4*>(pool + (int64_t)to[i] * blob_bytes);
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n16; j += stride)
      dst[j] = __ldcs(src + j);
  }
}

}  // namespace

size_t resize_workspace_bytes(int S, int S_new) {
  const int cap = S > S_new ? S : S_new;
  return sizeof(int32_t) * (8 + 3 * (size_t)cap);
}

cudaError_t launch_cache_resize(int32_t* slot_of_id, int n_ids, int32_t* id_of_slot, uint32_t* ts,
                                int S, int S_new, uint8_t* pool, int64_t blob_bytes, int32_t* ws,
                                cudaStream_t st) {
  const int cap = S > S_new ? S : S_new;
  resize_plan_kernel<<<1, kRzThreads, 0, st>>>(slot_of_id, n_ids, id_of_slot, ts, S, S_new, cap,
                                               ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !pool || S_new >= S) return e;  // a growth moves nothing
  const int max_moves = S - S_new < S_new ? S - S_new : S_new;
  const int64_t n16 = blob_bytes / 16;
  int gx = (int)((n16 + 255) / 256);
  if (gx > 64) gx = 64;
  if (gx < 1) gx = 1;
  const int gy = max_moves < 1024 ? max_moves : 1024;
  resize_move_kernel<<<dim3(gx, gy), 256, 0, st>>>(ws, cap, pool, blob_bytes);
  return cudaGetLastError();
}

}  // namespace moe
