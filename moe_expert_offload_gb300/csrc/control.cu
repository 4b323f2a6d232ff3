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
#include "control_common.cuh"
#include "moe_internal.cuh"
#include "route_select.cuh"

namespace moe {
namespace {
using namespace ctl;

constexpr int kCtlThreads = 512;
constexpr int kCtlWarps = kCtlThreads / 32;

struct BlockSync {
  __device__ void operator()() const { __syncthreads(); }
};

template <int KMAX, bool SEL>
__global__ void __launch_bounds__(kCtlThreads) cache_step_kernel(CacheArgs a, SelArgs sa) {
  using Sh = CtlShared<KMAX, kCtlThreads>;
  constexpr int NE = Sh::NE;
  __shared__ Sh s;
  griddep_launch();
  griddep_wait();  // routed ids from the previous kernel

  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // the counters of the decode FFN that follows (its kernel reads them only
  // after this grid has completed)
  for (int i = tid; i < a.n_zero; i += kCtlThreads) a.zero_words[i] = 0u;
  const int n = a.n_ids, E = a.E;

  uint32_t early[NE > 0 ? NE : 1];
  int32_t early_id[NE > 0 ? NE : 1];  // the same slots' ids: a victim's is read from here
  ctl_early_loads<NE, kCtlThreads>(a, early, early_id);
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
  for (int i = tid; i < (int)(sizeof(s.shit) / 4); i += kCtlThreads) s.shit[i] = 0u;
  if (tid == 0) {
    s.now = a.clock[0] + 1u;
    a.clock[0] = s.now;
    s.bad = 0;
    s.nu = 0;
  }
  __syncthreads();
  const uint32_t now = s.now;

  int n_uniq, n_hit, m;
  if (n <= 32) {
    // up to 32 routed ids: one warp deduplicates, ranks and classifies them in
    // registers (one block barrier instead of five)
    if (wid == 0)
      ctl_classify_warp<true, KMAX, kCtlThreads>(a, s, n, e_early, now,
                                                 [&](int32_t u) { return a.slot_of_id[u]; });
    __syncthreads();
    n_uniq = s.nu;
    n_hit = s.nh;
    m = s.nm;
  } else {
    // routed ids -> bank ids l*E + e (INT_MAX marks an id outside [0, E))
    for (int i = tid; i < n; i += kCtlThreads) {
      const int32_t e = a.ids[i];
      if (e < 0 || e >= E) {
        s.su[i] = INT_MAX;
        s.bad = 1;
      } else {
        s.su[i] = a.layer * E + e;
      }
    }
    __syncthreads();

    // dedup: keep first occurrences; an entry's rank among the unique ids is
    // the number of smaller unique ids.
    for (int i = tid; i < n; i += kCtlThreads) {
      const int32_t v = s.su[i];
      uint8_t first = v != INT_MAX;
      for (int j = 0; j < i && first; ++j) first = s.su[j] != v;
      s.sfirst[i] = first;
    }
    __syncthreads();
    for (int i = tid; i < n; i += kCtlThreads) {
      if (!s.sfirst[i]) continue;
      const int32_t v = s.su[i];
      int r = 0;
      for (int j = 0; j < n; ++j) r += (s.sfirst[j] && s.su[j] < v);
      s.suniq[r] = v;
      atomicAdd(&s.nu, 1);
    }
    __syncthreads();
    n_uniq = s.nu;

    // hit / miss, order-preserving compaction in rounds of kCtlThreads
    int base_h = 0, base_m = 0;
    for (int base = 0; base < n_uniq; base += kCtlThreads) {
      const int r = base + tid;
      const bool valid = r < n_uniq;
      const int32_t u = valid ? s.suniq[r] : 0;
      int32_t slot = valid ? a.slot_of_id[u] : -1;
      if (valid && !checked_ok(slot >= -1 && slot < a.n_slots, a.plan.err)) slot = -1;
      const bool hit = valid && slot >= 0, miss = valid && slot < 0;
      const unsigned hb = __ballot_sync(0xffffffffu, hit), mb = __ballot_sync(0xffffffffu, miss);
      if (lane == 0) {
        s.swh[wid] = __popc(hb);
        s.swm[wid] = __popc(mb);
      }
      __syncthreads();
      int oh = base_h, om = base_m, th = 0, tm = 0;
      for (int w = 0; w < kCtlWarps; ++w) {
        if (w < wid) {
          oh += s.swh[w];
          om += s.swm[w];
        }
        th += s.swh[w];
        tm += s.swm[w];
      }
      if (hit) {
        const int p = oh + __popc(hb & lanemask_lt());
        a.plan.hit_ids[p] = u;
        a.plan.hit_slots[p] = slot;
        a.ts[slot] = now;  // recency moves only when the router selects the expert
        const unsigned rr = (unsigned)(slot - a.S0);  // the slot's place in the scanned range
        if (rr < (unsigned)Sh::kEarlySlots) atomicOr(&s.shit[rr >> 5], 1u << (rr & 31));
      }
      if (miss) s.smiss[om + __popc(mb & lanemask_lt())] = u;
      base_h += th;
      base_m += tm;
      __syncthreads();
    }
    n_hit = base_h;
    m = base_m;
  }
  ctl_evict<KMAX, kCtlThreads>(a, s, now, n_uniq, n_hit, m, early, early_id, BlockSync{});
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
                                   uint32_t* ts, int S, uint32_t* clock, uint32_t* sync) {
  const int stride = gridDim.x * blockDim.x;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_ids; i += stride) slot_of_id[i] = -1;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < S; i += stride) {
    id_of_slot[i] = -1;
    ts[i] = 0;
  }
  if (sync)
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < MOE_CACHE_SYNC_WORDS; i += stride)
      sync[i] = 0u;
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
                               int S, uint32_t* clock, uint32_t* sync, cudaStream_t st) {
  int n = n_ids > S ? n_ids : S;
  int grid = (n + 255) / 256;
  if (grid > 1024) grid = 1024;
  if (grid < 1) grid = 1;
  cache_reset_kernel<<<grid, 256, 0, st>>>(slot_of_id, n_ids, id_of_slot, ts, S, clock, sync);
  return cudaGetLastError();
}

}  // namespace moe
