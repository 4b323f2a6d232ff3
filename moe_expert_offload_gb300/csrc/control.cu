// Device control step of the shared expert cache, one CTA per call
// (FreeToken summary "core method", "method steps", "novelty"; FreeToken
// reader "Semantic-Aware Expert Caching", "Elastic Memory Management"):
// dedup of the routed ids lE+e, hit/miss classification, the q* split of the
// misses into a fill set F and a direct set C, a single pass over the slots
// for the K least recently used victims, and the slot-table update.  Then the
// fill copies bank -> slot pool, sized by the device-side fill count.
//
// All routing-dependent sizes stay in device memory (plan->counts), so the
// step needs no host decision and can sit inside a captured graph.
#include <limits.h>

#include "moe_internal.cuh"
#include "route_select.cuh"

namespace moe {
namespace {

constexpr int kCtlThreads = 512;
constexpr int kCtlWarps = kCtlThreads / 32;
constexpr unsigned long long kNoKey = ~0ull;
constexpr int kEarlyTs = 8;  // recency stamps per thread loaded before the routed ids
constexpr int kEarlySlots = kEarlyTs * kCtlThreads;

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Insert `key` into the ascending list best[0..KMAX), dropping the largest.
template <int KMAX>
__device__ __forceinline__ void insert_key(unsigned long long (&best)[KMAX],
                                           unsigned long long key) {
  if (key >= best[KMAX - 1]) return;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    const unsigned long long lo = best[j] < key ? best[j] : key;
    key = best[j] < key ? key : best[j];
    best[j] = lo;
  }
}

// K rounds of warp-wide minimum over the heads of the per-lane ascending
// lists; round r's minimum is written to out[r] (keys unique).  A round is two
// warp reductions of 32-bit halves: the least recency stamp, then the least
// slot among the lanes holding that stamp.  The winning lane scanned that slot
// itself: if it is one of its NE early slots it also writes the slot's id from
// early_id to out_id[r], else -2 (not known).
template <int KMAX, int NE>
__device__ __forceinline__ void warp_k_smallest(unsigned long long (&best)[KMAX], int K,
                                                unsigned long long* out, int32_t* out_id,
                                                const int32_t (&early_id)[NE > 0 ? NE : 1]) {
  const int lane = threadIdx.x & 31;
  for (int r = 0; r < K; ++r) {
    const uint32_t hi = (uint32_t)(best[0] >> 32), lo = (uint32_t)best[0];
    const uint32_t mhi = __reduce_min_sync(0xffffffffu, hi);
    const uint32_t mlo = __reduce_min_sync(0xffffffffu, hi == mhi ? lo : 0xffffffffu);
    const unsigned long long m = ((unsigned long long)mhi << 32) | mlo;
    if (m != kNoKey && best[0] == m) {
      int32_t id = -2;
#pragma unroll
      for (int j = 0; j < NE; ++j)
        if ((int)mlo == (int)threadIdx.x + j * kCtlThreads) id = early_id[j];
      out_id[r] = id;
#pragma unroll
      for (int j = 0; j < KMAX - 1; ++j) best[j] = best[j + 1];
      best[KMAX - 1] = kNoKey;
    }
    if (lane == 0) out[r] = m;
  }
}

template <int KMAX, bool SEL>
__global__ void __launch_bounds__(kCtlThreads) cache_step_kernel(CacheArgs a, SelArgs sa) {
  __shared__ int32_t su[kMaxRouted];
  __shared__ int32_t suniq[kMaxRouted];
  __shared__ int32_t smiss[kMaxRouted];
  __shared__ uint8_t sfirst[kMaxRouted];
  __shared__ int swh[kCtlWarps], swm[kCtlWarps];
  __shared__ unsigned long long scand[kCtlWarps * KMAX];
  __shared__ int32_t scand_id[kCtlWarps * KMAX];
  __shared__ unsigned long long svict[KMAX];
  __shared__ int32_t sold[KMAX];
  __shared__ int s_nu, s_nh, s_nm, s_bad;
  __shared__ uint32_t s_now;
  __shared__ uint32_t shit[kEarlySlots / 32];  // slots hit this step (those < kEarlySlots)
  griddep_launch();
  griddep_wait();  // routed ids from the previous kernel

  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // the counters of the decode FFN that follows (its kernel reads them only
  // after this grid has completed)
  for (int i = tid; i < a.n_zero; i += kCtlThreads) a.zero_words[i] = 0u;
  const int n = a.n_ids, E = a.E;

  // The victim scan does not depend on the routed ids: the recency stamps of
  // this thread's first kEarlyTs slots are loaded now, alongside the ids, and
  // the slots hit this step are left out through a bitmap (their stamps
  // become `now`, which the scan excludes).
  constexpr int NE = KMAX <= 16 ? kEarlyTs : 0;  // (the K <= 32 list needs the registers)
  // keys hold the slot's place v in the scanned range [S0, S0 + S); the
  // victims written out are S0 + v (the order of (ts, v) and (ts, slot) agree)
  uint32_t early[NE > 0 ? NE : 1];
  int32_t early_id[NE > 0 ? NE : 1];  // the same slots' ids: a victim's is read from here
#pragma unroll
  for (int j = 0; j < NE; ++j) {
    const int v = tid + j * kCtlThreads;
    early[j] = v < a.S ? a.ts[a.S0 + v] : 0u;
    early_id[j] = v < a.S ? a.id_of_slot[a.S0 + v] : -1;
  }
  if constexpr (SEL) {
    // the router's selection for the step's tokens, one warp per token; the
    // ids are then read back below like those of a separate select kernel
    __shared__ float sel_a[kCtlWarps][32 * 8];
    __shared__ float sel_b[kCtlWarps][rsel::kMaxK], sel_c[kCtlWarps][rsel::kMaxK];
    __shared__ float sel_sum[kCtlWarps];
    if (wid < sa.T) {
      if (sa.router == MOE_ROUTER_SOFTMAX_TOPK)
        rsel::softmax_token<8>(sa.logits, wid, E, sa.k, sa.ids, sa.wts, sel_b[wid], sel_c[wid],
                               &sel_sum[wid]);
      else
        rsel::sigmoid_group_token<8>(sa.logits, sa.bias, wid, E, sa.n_groups, sa.topk_groups,
                                     sa.k, sa.scale, sa.ids, sa.wts, sel_a[wid], sel_b[wid],
                                     &sel_sum[wid]);
    }
    __syncthreads();
  }
  // (small steps) the routed ids, also independent of everything above
  int32_t e_early = 0;
  if (n <= 32 && wid == 0 && lane < n) e_early = a.ids[lane];
  for (int i = tid; i < kEarlySlots / 32; i += kCtlThreads) shit[i] = 0u;
  if (tid == 0) {
    s_now = a.clock[0] + 1u;
    a.clock[0] = s_now;
    s_bad = 0;
    s_nu = 0;
  }
  __syncthreads();
  const uint32_t now = s_now;

  int n_uniq, n_hit, m;
  if (n <= 32) {
    // up to 32 routed ids: one warp deduplicates, ranks and classifies them in
    // registers (one block barrier instead of five)
    if (wid == 0) {
      int32_t v = INT_MAX;  // bank id l*E + e; INT_MAX marks an id outside [0, E)
      if (lane < n) {
        const int32_t e = e_early;
        if (e < 0 || e >= E)
          s_bad = 1;
        else
          v = a.layer * E + e;
      }
      // first occurrences; a unique id's rank is the number of smaller unique ids
      const unsigned peers = __match_any_sync(0xffffffffu, v);
      const bool first = v != INT_MAX && (peers & lanemask_lt()) == 0;
      int rank = 0;
      for (int jj = 0; jj < n; ++jj) {
        const int32_t vj = __shfl_sync(0xffffffffu, v, jj);
        const int fj = __shfl_sync(0xffffffffu, (int)first, jj);
        rank += (fj && vj < v);
      }
      const int nu = __popc(__ballot_sync(0xffffffffu, first));
      if (first) suniq[rank] = v;
      __syncwarp();
      // hit / miss in rank order, order-preserving compaction
      const bool valid = lane < nu;
      const int32_t u = valid ? suniq[lane] : 0;
      const int32_t slot = valid ? a.slot_of_id[u] : -1;
      const bool hit = valid && slot >= 0, miss = valid && slot < 0;
      const unsigned hb = __ballot_sync(0xffffffffu, hit), mb = __ballot_sync(0xffffffffu, miss);
      if (hit) {
        const int p = __popc(hb & lanemask_lt());
        a.plan.hit_ids[p] = u;
        a.plan.hit_slots[p] = slot;
        a.ts[slot] = now;  // recency moves only when the router selects the expert
        const unsigned r = (unsigned)(slot - a.S0);  // the slot's place in the scanned range
        if (r < (unsigned)kEarlySlots) atomicOr(&shit[r >> 5], 1u << (r & 31));
      }
      if (miss) smiss[__popc(mb & lanemask_lt())] = u;
      if (lane == 0) {
        s_nu = nu;
        s_nh = __popc(hb);
        s_nm = __popc(mb);
      }
    }
    __syncthreads();
    n_uniq = s_nu;
    n_hit = s_nh;
    m = s_nm;
  } else {
    // routed ids -> bank ids l*E + e (INT_MAX marks an id outside [0, E))
    for (int i = tid; i < n; i += kCtlThreads) {
      const int32_t e = a.ids[i];
      if (e < 0 || e >= E) {
        su[i] = INT_MAX;
        s_bad = 1;
      } else {
        su[i] = a.layer * E + e;
      }
    }
    __syncthreads();

    // dedup: keep first occurrences; an entry's rank among the unique ids is
    // the number of smaller unique ids.
    for (int i = tid; i < n; i += kCtlThreads) {
      const int32_t v = su[i];
      uint8_t first = v != INT_MAX;
      for (int j = 0; j < i && first; ++j) first = su[j] != v;
      sfirst[i] = first;
    }
    __syncthreads();
    for (int i = tid; i < n; i += kCtlThreads) {
      if (!sfirst[i]) continue;
      const int32_t v = su[i];
      int r = 0;
      for (int j = 0; j < n; ++j) r += (sfirst[j] && su[j] < v);
      suniq[r] = v;
      atomicAdd(&s_nu, 1);
    }
    __syncthreads();
    n_uniq = s_nu;

    // hit / miss, order-preserving compaction in rounds of kCtlThreads
    int base_h = 0, base_m = 0;
    for (int base = 0; base < n_uniq; base += kCtlThreads) {
      const int r = base + tid;
      const bool valid = r < n_uniq;
      const int32_t u = valid ? suniq[r] : 0;
      const int32_t slot = valid ? a.slot_of_id[u] : -1;
      const bool hit = valid && slot >= 0, miss = valid && slot < 0;
      const unsigned hb = __ballot_sync(0xffffffffu, hit), mb = __ballot_sync(0xffffffffu, miss);
      if (lane == 0) {
        swh[wid] = __popc(hb);
        swm[wid] = __popc(mb);
      }
      __syncthreads();
      int oh = base_h, om = base_m, th = 0, tm = 0;
      for (int w = 0; w < kCtlWarps; ++w) {
        if (w < wid) {
          oh += swh[w];
          om += swm[w];
        }
        th += swh[w];
        tm += swm[w];
      }
      if (hit) {
        const int p = oh + __popc(hb & lanemask_lt());
        a.plan.hit_ids[p] = u;
        a.plan.hit_slots[p] = slot;
        a.ts[slot] = now;  // recency moves only when the router selects the expert
        const unsigned r = (unsigned)(slot - a.S0);  // the slot's place in the scanned range
        if (r < (unsigned)kEarlySlots) atomicOr(&shit[r >> 5], 1u << (r & 31));
      }
      if (miss) smiss[om + __popc(mb & lanemask_lt())] = u;
      base_h += th;
      base_m += tm;
      __syncthreads();
    }
    n_hit = base_h;
    m = base_m;
  }

  // q = round half up of m * B_P / B_H; pure fill when B_H <= B_P
  int q;
  if (m <= 0 || a.no_fill) {
    q = 0;
  } else if (a.bh <= a.bp) {
    q = m;
  } else {
    long long qq = (2LL * m * a.bp + a.bh) / (2LL * a.bh);
    q = (int)(qq < 0 ? 0 : (qq > m ? m : qq));
  }

  // one pass over the slots: K smallest keys (ts << 32 | slot), ts != now
  const int K = a.K;
  unsigned long long best[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) best[j] = kNoKey;
#pragma unroll
  for (int j = 0; j < NE; ++j) {
    const int v = tid + j * kCtlThreads;
    if (v < a.S && !(shit[v >> 5] >> (v & 31) & 1u))
      insert_key<KMAX>(best, ((unsigned long long)early[j] << 32) | (uint32_t)v);
  }
  const uint32_t* ts_r = a.ts + a.S0;
  for (int v = tid + NE * kCtlThreads; v < a.S; v += kCtlThreads) {  // read after the hit updates
    const uint32_t t = ts_r[v];
    if (t != now) insert_key<KMAX>(best, ((unsigned long long)t << 32) | (uint32_t)v);
  }
  warp_k_smallest<KMAX, NE>(best, K, &scand[wid * KMAX], &scand_id[wid * KMAX], early_id);
  __syncthreads();
  if (wid == 0) {
    // merge the warps' ascending lists: lane w < kCtlWarps holds the head of
    // warp w's list; each round takes the least head (keys unique)
    int pos = 0;
    for (int r = 0; r < K; ++r) {
      const unsigned long long h =
          (lane < kCtlWarps && pos < K) ? scand[lane * KMAX + pos] : kNoKey;
      const uint32_t hi = (uint32_t)(h >> 32), lo = (uint32_t)h;
      const uint32_t mhi = __reduce_min_sync(0xffffffffu, hi);
      const uint32_t mlo = __reduce_min_sync(0xffffffffu, hi == mhi ? lo : 0xffffffffu);
      const unsigned long long mk = ((unsigned long long)mhi << 32) | mlo;
      if (mk != kNoKey && h == mk) {
        sold[r] = scand_id[lane * KMAX + pos];
        ++pos;
      }
      if (lane == 0) svict[r] = mk;
    }
  }
  __syncthreads();

  int nv = 0;
  for (int r = 0; r < K; ++r) nv += svict[r] != kNoKey;
  const int n_fill = min(q, nv);

  for (int i = tid; i < K; i += kCtlThreads)
    a.plan.victims[i] = (i < nv) ? a.S0 + (int32_t)(svict[i] & 0xffffffffu) : -1;
  if (tid < n_fill) {
    const int32_t v = a.S0 + (int32_t)(svict[tid] & 0xffffffffu);
    const int32_t f = smiss[tid];
    const int32_t known = sold[tid];  // -2: the slot's id was not prefetched
    const int32_t old = known != -2 ? known : a.id_of_slot[v];
    if (old >= 0) a.slot_of_id[old] = -1;  // an evicted id is never one of F
    a.id_of_slot[v] = f;
    a.slot_of_id[f] = v;
    a.ts[v] = now;
    a.plan.fill_ids[tid] = f;
    a.plan.fill_slots[tid] = v;
    a.plan.evicted_ids[tid] = old;
  }
  for (int i = tid; i < m - n_fill; i += kCtlThreads) a.plan.direct_ids[i] = smiss[n_fill + i];
  for (int i = tid; i < n_uniq; i += kCtlThreads) a.plan.uniq[i] = suniq[i];
  if (tid == 0) {
    int32_t* c = a.plan.counts;
    c[0] = n_uniq;
    c[1] = n_hit;
    c[2] = m;
    c[3] = q;
    c[4] = n_fill;
    c[5] = m - n_fill;
    c[6] = nv;
    c[7] = (int32_t)now;
    if (s_bad) atomicOr(a.plan.err, MOE_DERR_BAD_ID);
  }
}

// bank[F_i] -> slot_pool[victim_i]; blockIdx.y = i; blocks past the device
// fill count return at once.  16-byte vectors, 4 in flight per thread.
__global__ void __launch_bounds__(256) fill_copy_kernel(const int32_t* __restrict__ counts,
                                                        const int32_t* __restrict__ fill_ids,
                                                        const int32_t* __restrict__ fill_slots,
                                                        const uint8_t* __restrict__ bank,
                                                        uint8_t* __restrict__ pool,
                                                        int64_t blob_bytes) {
  griddep_launch();
  griddep_wait();  // the plan from the control step
  const int i = blockIdx.y;
  if (i >= counts[4]) return;
  const uint4* src = reinterpret_cast<const uint4*>(bank + (int64_t)fill_ids[i] * blob_bytes);
  uint4* dst = reinterpret_cast<uint4*>(pool + (int64_t)fill_slots[i] * blob_bytes);
  const int64_t n16 = blob_bytes / 16;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; j + 3 * stride < n16; j += 4 * stride) {
    const uint4 v0 = __ldcs(src + j), v1 = __ldcs(src + j + stride);
    const uint4 v2 = __ldcs(src + j + 2 * stride), v3 = __ldcs(src + j + 3 * stride);
    dst[j] = v0;
    dst[j + stride] = v1;
    dst[j + 2 * stride] = v2;
    dst[j + 3 * stride] = v3;
  }
  for (; j < n16; j += stride) dst[j] = __ldcs(src + j);
}

__global__ void cache_reset_kernel(int32_t* slot_of_id, int n_ids, int32_t* id_of_slot,
                                   uint32_t* ts, int S, uint32_t* clock) {
  const int stride = gridDim.x * blockDim.x;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_ids; i += stride) slot_of_id[i] = -1;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < S; i += stride) {
    id_of_slot[i] = -1;
    ts[i] = 0;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) clock[0] = 0;
}

}  // namespace

cudaError_t launch_cache_step(const CacheArgs& a, cudaStream_t st) {
  const SelArgs none{};
  if (a.K <= 8)
    return launch_pdl(cache_step_kernel<8, false>, dim3(1), dim3(kCtlThreads), 0, st, a, none);
  if (a.K <= 16)
    return launch_pdl(cache_step_kernel<16, false>, dim3(1), dim3(kCtlThreads), 0, st, a, none);
  return launch_pdl(cache_step_kernel<32, false>, dim3(1), dim3(kCtlThreads), 0, st, a, none);
}

cudaError_t launch_cache_step_sel(const CacheArgs& a, const SelArgs& s, cudaStream_t st) {
  if (s.T < 1 || s.T > kSelFusedMaxT || s.T > kCtlWarps || a.E > kSelFusedMaxE ||
      s.k > rsel::kMaxK)
    return cudaErrorInvalidValue;
  if (a.K <= 8)
    return launch_pdl(cache_step_kernel<8, true>, dim3(1), dim3(kCtlThreads), 0, st, a, s);
  if (a.K <= 16)
    return launch_pdl(cache_step_kernel<16, true>, dim3(1), dim3(kCtlThreads), 0, st, a, s);
  return launch_pdl(cache_step_kernel<32, true>, dim3(1), dim3(kCtlThreads), 0, st, a, s);
}

cudaError_t launch_fill_copy(const moe_plan& plan, int K, const uint8_t* bank, uint8_t* pool,
                             int64_t blob_bytes, cudaStream_t st) {
  const int64_t n16 = blob_bytes / 16;
  int gx = (int)((n16 + 256 * 4 - 1) / (256 * 4));
  if (gx > 128) gx = 128;
  if (gx < 1) gx = 1;
  return launch_pdl(fill_copy_kernel, dim3(gx, K), dim3(256), 0, st, plan.counts, plan.fill_ids,
                    plan.fill_slots, bank, pool, blob_bytes);
}

cudaError_t launch_cache_reset(int32_t* slot_of_id, int n_ids, int32_t* id_of_slot, uint32_t* ts,
                               int S, uint32_t* clock, cudaStream_t st) {
  int n = n_ids > S ? n_ids : S;
  int grid = (n + 255) / 256;
  if (grid > 1024) grid = 1024;
  if (grid < 1) grid = 1;
  cache_reset_kernel<<<grid, 256, 0, st>>>(slot_of_id, n_ids, id_of_slot, ts, S, clock);
  return cudaGetLastError();
}

}  // namespace moe
