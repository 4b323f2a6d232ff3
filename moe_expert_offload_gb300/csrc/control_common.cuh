// The control step of the shared expert cache as device functions, shared by
// the standalone control kernel (control.cu) and the fused decode layer kernel
// (ffn_coop.cu), so that both take the same decisions with the same code
// (FreeToken summary "core method", "method steps"; FreeToken reader
// "Semantic-Aware Expert Caching", "Elastic Memory Management"):
//   * ctl_classify_warp: dedup of up to 32 routed ids lE+e, their ranks,
//     hit / miss, the hits' recency stamps moved to `now`;
//   * ctl_evict: the q* split of the misses, one pass over the slots for the
//     K least recently used victims (keys (ts, slot) are unique), the slot
//     table update for the fill set F and the plan's remaining lists.
// The functions run on NTH threads (threadIdx.x < NTH) of one CTA and meet at
// `sync` (a functor: __syncthreads, or a named barrier when the CTA has other
// warps doing other work).
#pragma once
#include <limits.h>
#include <stdint.h>

#include "moe_internal.cuh"

namespace moe {
namespace ctl {

constexpr unsigned long long kNoKey = ~0ull;
constexpr int kEarlyTs = 8;  // recency stamps per thread loaded before the routed ids

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
// itself: if it is one of its NE early slots (slot threadIdx.x + j * NTH) it
// also writes the slot's id from early_id to out_id[r], else -2 (not known).
template <int KMAX, int NE, int NTH>
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
        if ((int)mlo == (int)threadIdx.x + j * NTH) id = early_id[j];
      out_id[r] = id;
#pragma unroll
      for (int j = 0; j < KMAX - 1; ++j) best[j] = best[j + 1];
      best[KMAX - 1] = kNoKey;
    }
    if (lane == 0) out[r] = m;
  }
}

// Shared state of one control step on NTH threads.
template <int KMAX, int NTH>
struct CtlShared {
  static constexpr int NW = NTH / 32;
  static constexpr int NE = KMAX <= 16 ? kEarlyTs : 0;  // (the K <= 32 list needs the registers)
  static constexpr int kEarlySlots = NE * NTH;
  int32_t su[kMaxRouted];
  int32_t suniq[kMaxRouted];
  int32_t smiss[kMaxRouted];
  int32_t sslot[32];  // (up to 32 routed ids) slot of each unique id before the step, or -1
  uint8_t sfirst[kMaxRouted];
  int swh[NW], swm[NW];
  unsigned long long scand[NW * KMAX];
  int32_t scand_id[NW * KMAX];
  unsigned long long svict[KMAX];
  int32_t sold[KMAX];
  int nu, nh, nm, bad;
  uint32_t now;
  uint32_t shit[kEarlySlots / 32 > 0 ? kEarlySlots / 32 : 1];  // slots hit (those < kEarlySlots)
};

// The recency stamps and ids of this thread's first NE slots of the scanned
// range (slot S0 + threadIdx.x + j NTH), loaded ahead of everything else: the
// victim scan does not depend on the routed ids, and the slots hit this step
// are left out through the shit bitmap (their stamps become `now`).
template <int NE, int NTH>
__device__ __forceinline__ void ctl_early_loads(const CacheArgs& a, uint32_t (&early)[NE > 0 ? NE : 1],
                                                int32_t (&early_id)[NE > 0 ? NE : 1]) {
#pragma unroll
  for (int j = 0; j < NE; ++j) {
    const int v = (int)threadIdx.x + j * NTH;
    early[j] = v < a.S ? a.ts[a.S0 + v] : 0u;
    early_id[j] = v < a.S ? a.id_of_slot[a.S0 + v] : -1;
  }
}

// Up to 32 routed ids (n <= 32, lane < n holds its expert id e): one warp
// deduplicates, ranks and classifies them in registers.  Unique bank ids
// l*E + e go to s.suniq in ascending order (with their slots before the step,
// slot_of(u), in s.sslot); counts to s.nu, s.nh, s.nm; an id outside [0, E)
// sets s.bad and is skipped.  With TABLES, also the hits to the plan in rank
// order with ts[slot] = now and the misses to s.smiss in rank order.  The
// caller syncs after it.
template <bool TABLES, int KMAX, int NTH, class SlotOf>
__device__ __forceinline__ void ctl_classify_warp(const CacheArgs& a, CtlShared<KMAX, NTH>& s,
                                                  int n, int32_t e, uint32_t now, SlotOf slot_of) {
  constexpr int kEarlySlots = CtlShared<KMAX, NTH>::kEarlySlots;
  const int lane = threadIdx.x & 31;
  int32_t v = INT_MAX;  // bank id l*E + e; INT_MAX marks an id outside [0, E)
  if (lane < n) {
    if (e < 0 || e >= a.E)
      s.bad = 1;
    else
      v = a.layer * a.E + e;
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
  if (first) s.suniq[rank] = v;
  __syncwarp();
  // hit / miss in rank order, order-preserving compaction
  const bool valid = lane < nu;
  const int32_t u = valid ? s.suniq[lane] : 0;
  int32_t slot = valid ? slot_of(u) : -1;
  if (valid && !checked_ok(slot >= -1 && slot < a.n_slots, a.plan.err)) slot = -1;
  const bool hit = valid && slot >= 0, miss = valid && slot < 0;
  const unsigned hb = __ballot_sync(0xffffffffu, hit), mb = __ballot_sync(0xffffffffu, miss);
  if (valid) s.sslot[lane] = slot;
  if (TABLES && hit) {
    const int p = __popc(hb & lanemask_lt());
    a.plan.hit_ids[p] = u;
    a.plan.hit_slots[p] = slot;
    a.ts[slot] = now;  // recency moves only when the router selects the expert
    const unsigned r = (unsigned)(slot - a.S0);  // the slot's place in the scanned range
    if (r < (unsigned)kEarlySlots) atomicOr(&s.shit[r >> 5], 1u << (r & 31));
  }
  if (TABLES && miss) s.smiss[__popc(mb & lanemask_lt())] = u;
  if (lane == 0) {
    s.nu = nu;
    s.nh = __popc(hb);
    s.nm = __popc(mb);
  }
}

// q = round half up of m * B_P / B_H, in [0, m]; all of m when B_H <= B_P;
// 0 with no fill (static policy) or no miss.
__device__ __forceinline__ int ctl_fill_quota(const CacheArgs& a, int m) {
  if (m <= 0 || a.no_fill) return 0;
  if (a.bh <= a.bp) return m;
  const long long qq = (2LL * m * a.bp + a.bh) / (2LL * a.bh);
  return (int)(qq < 0 ? 0 : (qq > m ? m : qq));
}

// The rest of the step once the routed ids are classified (n_uniq unique, m
// misses in s.smiss): q, the K least recently used slots of the scanned range
// whose stamp is not `now` (one pass), F = the first min(q, victims) misses
// into the victims in (ts, slot) order with the slot tables updated, C = the
// other misses, and the plan's lists and counts.
template <int KMAX, int NTH, class Sync>
__device__ __forceinline__ void ctl_evict(const CacheArgs& a, CtlShared<KMAX, NTH>& s,
                                          uint32_t now, int n_uniq, int n_hit, int m,
                                          const uint32_t (&early)[CtlShared<KMAX, NTH>::NE > 0
                                                                      ? CtlShared<KMAX, NTH>::NE
                                                                      : 1],
                                          const int32_t (&early_id)[CtlShared<KMAX, NTH>::NE > 0
                                                                        ? CtlShared<KMAX, NTH>::NE
                                                                        : 1],
                                          Sync sync) {
  constexpr int NE = CtlShared<KMAX, NTH>::NE, NW = CtlShared<KMAX, NTH>::NW;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int q = ctl_fill_quota(a, m);
  // one pass over the slots: K smallest keys (ts << 32 | v), ts != now; keys
  // hold the slot's place v in the scanned range [S0, S0 + S) (the order of
  // (ts, v) and (ts, slot) agree) and the victims written out are S0 + v
  const int K = a.K;
  unsigned long long best[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) best[j] = kNoKey;
#pragma unroll
  for (int j = 0; j < NE; ++j) {
    const int v = tid + j * NTH;
    if (v < a.S && !(s.shit[v >> 5] >> (v & 31) & 1u))
      insert_key<KMAX>(best, ((unsigned long long)early[j] << 32) | (uint32_t)v);
  }
  const uint32_t* ts_r = a.ts + a.S0;
  for (int v = tid + NE * NTH; v < a.S; v += NTH) {  // read after the hit updates
    const uint32_t t = ts_r[v];
    if (t != now) insert_key<KMAX>(best, ((unsigned long long)t << 32) | (uint32_t)v);
  }
  warp_k_smallest<KMAX, NE, NTH>(best, K, &s.scand[wid * KMAX], &s.scand_id[wid * KMAX],
                                 early_id);
  sync();
  if (wid == 0) {
    // merge the warps' ascending lists: lane w < NW holds the head of warp
    // w's list; each round takes the least head (keys unique)
    int pos = 0;
    for (int r = 0; r < K; ++r) {
      const unsigned long long h = (lane < NW && pos < K) ? s.scand[lane * KMAX + pos] : kNoKey;
      const uint32_t hi = (uint32_t)(h >> 32), lo = (uint32_t)h;
      const uint32_t mhi = __reduce_min_sync(0xffffffffu, hi);
      const uint32_t mlo = __reduce_min_sync(0xffffffffu, hi == mhi ? lo : 0xffffffffu);
      const unsigned long long mk = ((unsigned long long)mhi << 32) | mlo;
      if (mk != kNoKey && h == mk) {
        s.sold[r] = s.scand_id[lane * KMAX + pos];
        ++pos;
      }
      if (lane == 0) s.svict[r] = mk;
    }
  }
  sync();

  int nv = 0;
  for (int r = 0; r < K; ++r) nv += s.svict[r] != kNoKey;
  const int n_fill = min(q, nv);

  for (int i = tid; i < K; i += NTH)
    a.plan.victims[i] = (i < nv) ? a.S0 + (int32_t)(s.svict[i] & 0xffffffffu) : -1;
  if (tid < n_fill) {
    const int32_t v = a.S0 + (int32_t)(s.svict[tid] & 0xffffffffu);
    const int32_t f = s.smiss[tid];
    const int32_t known = s.sold[tid];  // -2: the slot's id was not prefetched
    int32_t old = known != -2 ? known : a.id_of_slot[v];
    if (!checked_ok(old >= -1 && old < a.n_bank, a.plan.err)) old = -1;
    if (old >= 0) a.slot_of_id[old] = -1;  // an evicted id is never one of F
    a.id_of_slot[v] = f;
    a.slot_of_id[f] = v;
    a.ts[v] = now;
    a.plan.fill_ids[tid] = f;
    a.plan.fill_slots[tid] = v;
    a.plan.evicted_ids[tid] = old;
  }
  for (int i = tid; i < m - n_fill; i += NTH) a.plan.direct_ids[i] = s.smiss[n_fill + i];
  for (int i = tid; i < n_uniq; i += NTH) a.plan.uniq[i] = s.suniq[i];
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
    if (s.bad) atomicOr(a.plan.err, MOE_DERR_BAD_ID);
  }
}

}  // namespace ctl
}  // namespace moe
