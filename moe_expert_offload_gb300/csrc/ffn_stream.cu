// Decode expert FFN, streaming gate/up phase: the same math as ffn_decode.cu
// (Edge0 §3.1 "math convention"; int4 affine group-64 weights, register-built
// (128+q) bf16 fragments into mma.sync m16n8k16, group scale and bias applied
// to the fp32 accumulator), organised so that HBM never waits on the SMs:
//
//  * one persistent CTA per SM owns a contiguous range of (entry, 16-row tile)
//    units of all executed experts;
//  * a producer warp streams each unit's gate and up code tiles through a
//    ring of shared-memory stages with tiled TMA loads (a few 4 KB boxes per
//    stage, completion counted in bytes on the stage's mbarrier), and the
//    unit's four scale / bias blocks into a separate buffer with bulk copies;
//  * each of the eight consumer warps owns a fixed K slice (GPW 64-column
//    groups of every stage): it stages the activations and converts the
//    scales of its own slice only, so no CTA-wide barrier sits on the path --
//    warps meet only at the stage mbarriers;
//  * the warps' partial sums go to a two-deep ring in shared memory and one
//    designated warp per unit (rotating) adds them in warp order and writes
//    h = silu(g) * u: the sum order is fixed, the result deterministic;
//  * when the call carries the step's fill copy, a writer warp follows the
//    same stages and, for an expert being filled (read from the bank), stores
//    each landed tile and scale block into the expert's new slot before the
//    stage goes back to the producer (one more arrival on the empty barriers).
// Every wait is bounded; on a time-out the kernel sets MOE_DERR_WAIT in the
// plan's error word, the producer still waits (bounded) for the copies it
// issued, and every warp returns.
#include "stream_common.cuh"

namespace moe {
namespace {
using namespace sc;

constexpr int kCW = 8;                     // consumer warps
constexpr int kFillW = kCW + 1;            // fill writer warp (after the producer, warp kCW)
constexpr int kSThreads = (kCW + 2) * 32;
constexpr int kTokS = 8;                   // tokens per MMA N tile (one per column)
constexpr int kRing = 2;                   // partial-sum ring depth
constexpr int kMaxStages = 8;
constexpr int kStreamMaxEntries = 128;
constexpr size_t kStreamSmemBudget = 220 * 1024;

// Gate / up code tiles arrive through a 4-D tensor map per blob array (bank,
// slot pool, shared expert): u32 words [blob][gate/up][row of I][word of H/8],
// box = 32 words (128 B) x 16 rows x both matrices = one 4 KB sub-tile,
// 128-byte swizzled: 16-byte chunk c of line L lands at chunk c ^ (L & 7), so
// the eight rows a warp reads at once fall in distinct banks.
//
// Shared-memory plan of one CTA.  GPW 64-column groups per consumer warp per
// stage, so a stage spans KC = 8 * GPW * 64 columns of H (KC / 256 sub-tiles);
// each warp owns gtot = H / 512 groups of a unit (its slice of every stage).
struct StreamGeom {
  int gpw, KC, nch, gtot, nsub;
  int stage;     // bytes: 32 rows (16 gate + 16 up) x KC / 2
  int nst;       // stages in the ring
  int tr;        // token rows staged per warp (min(T, 8))
  int xrow;      // bytes per staged token row of one warp: gtot * 128 + 16
  size_t o_raw, o_sbt, o_x, o_xsum, o_red, smem;
};

__host__ __device__ inline StreamGeom stream_geom(int H, int T, int nst) {
  StreamGeom g;
  const int ng = H / kGroup;
  g.gpw = (H % 1024 == 0) ? 2 : 1;
  g.KC = kCW * g.gpw * kGroup;
  g.nch = H / g.KC;
  g.gtot = ng / kCW;
  g.nsub = g.KC / 256;
  g.stage = 16 * g.KC;
  g.tr = T < kTokS ? T : kTokS;
  g.xrow = g.gtot * 128 + 16;
  g.nst = nst;
  g.o_raw = (size_t)nst * g.stage;                       // 4 blocks [16][ng] bf16
  g.o_sbt = g.o_raw + (size_t)4 * 16 * ng * 2;           // per warp [gtot][32] float2
  g.o_x = g.o_sbt + (size_t)kCW * g.gtot * 32 * 8;       // per warp [tr][xrow]
  g.o_xsum = g.o_x + (size_t)kCW * g.tr * g.xrow;        // per warp [gtot][8] fp32
  g.o_red = g.o_xsum + (size_t)kCW * g.gtot * kTokS * 4; // [ring][warp][32 rows][tr] fp32
  g.smem = g.o_red + (size_t)kRing * kCW * 32 * g.tr * 4 + 1024;  // + base alignment
  return g;
}

// Deepest ring that fits the budget (0 if not even two stages fit).
inline StreamGeom stream_plan(int H, int T) {
  StreamGeom g = stream_geom(H, T, 0);
  int nst = (int)((kStreamSmemBudget - (g.smem < kStreamSmemBudget ? g.smem : kStreamSmemBudget)) /
                  g.stage);
  if (nst > kMaxStages) nst = kMaxStages;
  if (nst < 2) nst = 0;
  return stream_geom(H, T, nst);
}

template <int GPW>
__global__ void __launch_bounds__(kSThreads, 1)
    ffn_gate_up_stream_kernel(FfnArgs a, int n_tick, StreamGeom geo,
                              const __grid_constant__ CodeMaps maps) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], sfull, sempty;
  __shared__ __align__(8) uint64_t rfull[kRing], rfree[kRing];
  __shared__ const uint8_t* sblob[kStreamMaxEntries];
  __shared__ int smap[kStreamMaxEntries], sbi[kStreamMaxEntries];
  __shared__ int sfs[kStreamMaxEntries];  // slot an F entry's blob is written to, else -1
  __shared__ int wtok[kCW][kTokS];
  __shared__ int s_fail;
  const int H = a.H, I = a.I, ng = H / kGroup;
  const int nst = geo.nst, nch = geo.nch, gtot = geo.gtot;
  // swizzled tiles need a 1024-byte aligned base
  unsigned char* smem = smem_raw + ((1024u - (su32(smem_raw) & 1023u)) & 1023u);
  constexpr int G = kCW * GPW;  // groups per stage
  const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    const int nrel = kCW + (a.fill_fused ? 1 : 0);  // warps that release a stage
    for (int i = 0; i < nst; ++i) {
      bar_init(su32(&full[i]), 1);
      bar_init(su32(&empty[i]), nrel);
    }
    bar_init(su32(&sfull), 1);
    bar_init(su32(&sempty), nrel);
    for (int i = 0; i < kRing; ++i) {
      bar_init(su32(&rfull[i]), kCW);
      bar_init(su32(&rfree[i]), 1);
    }
    s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  griddep_wait();  // the plan and the filled slots from the previous kernels
  if (blockIdx.x == 0)
    for (int i = tid; i < n_tick; i += blockDim.x) a.tick[i] = 0u;
  const int n_uniq = a.counts[0];
  // the producer's first unique ids, read alongside the count (rows past the
  // count exist: the plan holds T*k of them)
  const int32_t u_first = (wid == kCW && lane < a.T * a.k) ? a.uniq[lane] : 0;
  const int n_exec = n_uniq + a.has_shared;
  if (wid == kCW) {
    if (lane < 3) tma_prefetch_map(&maps.m[lane]);
    for (int r = lane; r < n_exec; r += 32) {
      // blob pointer (scale copies) and (tensor map, blob index) of entry r
      int mi = 2, bi = 0;
      int32_t fs = -1;
      if (r < n_uniq) {
        const int32_t id = r == lane ? u_first : a.uniq[r];
        const int32_t slot = ffn_slot(a, id, &fs);
        mi = slot >= 0 ? 1 : 0;
        bi = slot >= 0 ? slot : id;
      }
      smap[r] = mi;
      sbi[r] = bi;
      sblob[r] = (mi == 2 ? a.shared : mi == 1 ? a.pool : a.bank) + (int64_t)bi * a.blob_bytes;
      sfs[r] = fs;
    }
  }
  __syncthreads();
  // the down kernel may now take SMs as this grid's CTAs retire
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int tpe = I / 16;
  const int n_units = n_exec * tpe;
  // (32-bit: units x CTAs stays far below 2^32 for every shape the stream path takes)
  const int u_lo = (int)(blockIdx.x * (unsigned)n_units / gridDim.x);
  const int u_hi = (int)((blockIdx.x + 1) * (unsigned)n_units / gridDim.x);
  const BlobOffsets off = blob_offsets(H, I);
  unsigned char* stages = smem;
  unsigned char* sraw = smem + geo.o_raw;
  const int sblk = 16 * ng * 2;

  if (wid == kCW) {
    // -------------------------------------------------------- producer
    if (a.inject_stall) return;  // test hook: the other warps' waits run out
    int s = 0, rnd = 0, nq = 0, nu = 0;
    bool ok = true;
    for (int u = u_lo; ok && u < u_hi; ++u) {
      const int i = u - u_lo;
      const uint8_t* blob = sblob[u / tpe];
      const CUtensorMap* map = &maps.m[smap[u / tpe]];
      const int bidx = sbi[u / tpe];
      const int row0 = (u % tpe) * 16;
      // scales: single buffer, refilled once every warp converted the last unit
      if (lane == 0) {
        ok = i == 0 || bar_wait(su32(&sempty), (i - 1) & 1);
        if (ok) bar_expect(su32(&sfull), 4 * sblk);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ++nu;
      if (lane < 4) {
        const int64_t so = lane == 0 ? off.gs : lane == 1 ? off.gb : lane == 2 ? off.us : off.ub;
        bulk_g2s(su32(sraw + lane * sblk), blob + so + (int64_t)row0 * ng * 2, sblk,
                 su32(&sfull));
      }
      for (int kc = 0; kc < nch; ++kc) {
        if (lane == 0) {
          ok = rnd == 0 || bar_wait(su32(&empty[s]), (rnd - 1) & 1);
          if (ok) bar_expect(su32(&full[s]), geo.stage);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        // sub-tile c: words [kc * KC/8 + 32c, +32) of the 16 gate and 16 up rows
        if (lane < geo.nsub)
          tma_load_4d(su32(stages + s * geo.stage + lane * 4096), map,
                      kc * (geo.KC / 8) + 32 * lane, row0, 0, bidx, su32(&full[s]));
        ++nq;
        if (++s == nst) {
          s = 0;
          ++rnd;
        }
      }
    }
    // wait (bounded) until every copy this warp issued has landed
    if (lane < nst) {
      const int uses = nq > lane ? (nq - lane + nst - 1) / nst : 0;
      if (uses > 0 && !bar_wait(su32(&full[lane]), (uses - 1) & 1)) ok = false;
    }
    if (lane == 31 && nu > 0 && !bar_wait(su32(&sfull), (nu - 1) & 1)) ok = false;
    if (!__all_sync(0xffffffffu, ok)) s_fail = 1;
    if (lane == 0 && s_fail && a.err) atomicOr(a.err, MOE_DERR_WAIT);
    return;
  }
  if (wid == kFillW) {
    // ---------------------------------------------------- fill writer
    if (!a.fill_fused) return;
    int s = 0, rnd = 0;
    bool ok = true;
    for (int u = u_lo; ok && u < u_hi; ++u) {
      const int i = u - u_lo, row0 = (u % tpe) * 16, fs = sfs[u / tpe];
      ok = warp_wait(su32(&sfull), i & 1);
      if (!ok) break;
      if (fs >= 0 && lane < 4) {  // the unit's gate / up scale and bias rows
        const int64_t so = lane == 0 ? off.gs : lane == 1 ? off.gb : lane == 2 ? off.us : off.ub;
        fence_proxy_async_smem();
        bulk_s2g(a.pool_w + (int64_t)fs * a.blob_bytes + so + (int64_t)row0 * ng * 2,
                 su32(sraw + lane * sblk), sblk);
        bulk_commit();
        bulk_read_done();
      }
      __syncwarp();
      if (lane == 0) bar_arrive(su32(&sempty));
      for (int kc = 0; kc < nch; ++kc) {
        ok = warp_wait(su32(&full[s]), rnd & 1);
        if (!ok) break;
        if (fs >= 0 && lane < geo.nsub) {  // the stage's sub-tiles, same boxes as the loads
          fence_proxy_async_smem();
          tma_store_4d(&maps.m[1], kc * (geo.KC / 8) + 32 * lane, row0, 0, fs,
                       su32(stages + s * geo.stage + lane * 4096));
          bulk_commit();
          bulk_read_done();
        }
        __syncwarp();
        if (lane == 0) bar_arrive(su32(&empty[s]));
        if (++s == nst) {
          s = 0;
          ++rnd;
        }
      }
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // the slot writes are done
    if (!__all_sync(0xffffffffu, ok)) s_fail = 1;
    if (lane == 0 && s_fail && a.err) atomicOr(a.err, MOE_DERR_WAIT);
    return;
  }

  // ---------------------------------------------------------- consumers
  const int w = wid, gid = lane >> 2, t4 = lane & 3;
  float2* sbt = reinterpret_cast<float2*>(smem + geo.o_sbt) + (size_t)w * gtot * 32;
  unsigned char* xw = smem + geo.o_x + (size_t)w * geo.tr * geo.xrow;
  float* xsum = reinterpret_cast<float*>(smem + geo.o_xsum) + (size_t)w * gtot * kTokS;
  float* red = reinterpret_cast<float*>(smem + geo.o_red);
  const int tr = geo.tr;
  const uint16_t* raw = reinterpret_cast<const uint16_t*>(sraw);
  int prev_r = -1, ntok = 0, s = 0, rnd = 0;
  bool ok = true;
  for (int u = u_lo; ok && u < u_hi; ++u) {
    const int i = u - u_lo, r = u / tpe, row0 = (u % tpe) * 16;
    if (r != prev_r) {
      // tokens routed to entry r (ascending; this warp's own copy of the list)
      int cnt;
      if (r < n_uniq) {
        const int32_t id = a.uniq[r];
        const int base = a.layer * a.E, n = a.T * a.k;
        cnt = 0;
        for (int n0 = 0; n0 < n; n0 += 32) {
          const int ii = n0 + lane;
          bool mt = ii < n && base + a.ids[ii] == id;
          // a token listing the id twice is staged once (h is per token)
          for (int jj = mt ? ii - ii % a.k : ii; jj < ii; ++jj)
            if (base + a.ids[jj] == id) mt = false;
          const unsigned b = __ballot_sync(0xffffffffu, mt);
          const int pos = cnt + __popc(b & ((1u << lane) - 1u));
          if (mt && pos < kTokS) wtok[w][pos] = ii / a.k;
          cnt += __popc(b);
        }
      } else {
        if (lane < a.T && lane < kTokS) wtok[w][lane] = lane;
        cnt = a.T;
      }
      ntok = cnt < tr ? cnt : tr;
      __syncwarp();
      // x of those tokens on this warp's groups, in fragment order, + group sums
      const int per_tok = gtot * 4;
      const int n_items = ntok * per_tok;
      // two items per lane at a time: both loads in flight before either is used
      for (int it0 = 0; it0 < n_items; it0 += 64) {
        uint4 v[2][2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int it = it0 + 32 * h + lane;
          v[h][0] = v[h][1] = make_uint4(0u, 0u, 0u, 0u);
          if (it < n_items) {
            const int n = it / per_tok, rem = it - n * per_tok, gi = rem >> 2, qq = rem & 3;
            const int g = (gi / GPW) * G + w * GPW + (gi % GPW);
            const uint4* px =
                reinterpret_cast<const uint4*>(a.x + (int64_t)wtok[w][n] * H + g * 64 + qq * 16);
            v[h][0] = __ldg(px);
            v[h][1] = __ldg(px + 1);
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int it = it0 + 32 * h + lane;
          const bool in = it < n_items;
          const int n = in ? it / per_tok : 0, rem = it - n * per_tok, gi = rem >> 2, qq = rem & 3;
          uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
          float sx = 0.0f;
          if (in) {
            const uint32_t wv[8] = {v[h][0].x, v[h][0].y, v[h][0].z, v[h][0].w,
                                    v[h][1].x, v[h][1].y, v[h][1].z, v[h][1].w};
#pragma unroll
            for (int j = 0; j < 8; ++j)
              sx += __uint_as_float(wv[j] << 16) + __uint_as_float(wv[j] & 0xFFFF0000u);
            frag_order(wv, o0, o1);
          }
          sx += __shfl_xor_sync(0xffffffffu, sx, 1);
          sx += __shfl_xor_sync(0xffffffffu, sx, 2);
          if (in) {
            uint4* d = reinterpret_cast<uint4*>(xw + (size_t)n * geo.xrow + gi * 128 + qq * 32);
            d[0] = o0;
            d[1] = o1;
            if (qq == 0) xsum[gi * kTokS + n] = sx;
          }
        }
      }
      __syncwarp();
      prev_r = r;
    }

    // this warp's groups of the unit's scales -> (s, b - 128 s), lane = row
    if (!warp_wait(su32(&sfull), i & 1)) {
      ok = false;
      break;
    }
    {
      const int m = lane >> 4, row = lane & 15;
      const uint16_t* rs = raw + (2 * m) * 16 * ng + row * ng;
      const uint16_t* rb = raw + (2 * m + 1) * 16 * ng + row * ng;
      for (int kc = 0; kc < nch; ++kc) {
#pragma unroll
        for (int j = 0; j < GPW; ++j) {
          const int g = kc * G + w * GPW + j;
          const float sv = bf(rs[g]);
          sbt[(kc * GPW + j) * 32 + lane] = make_float2(sv, fmaf(-128.0f, sv, bf(rb[g])));
        }
      }
    }
    __syncwarp();
    if (lane == 0) bar_arrive(su32(&sempty));

    float acc[2][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[m][e] = 0.0f;
    const unsigned char* xg = xw + (size_t)gid * geo.xrow + t4 * 32;
    const bool has_tok = gid < ntok;
    for (int kc = 0; kc < nch; ++kc) {
      if (!warp_wait(su32(&full[s]), rnd & 1)) {
        ok = false;
        break;
      }
      const unsigned char* st = stages + s * geo.stage + gid * 128 + (t4 & 1) * 8;
#pragma unroll
      for (int j = 0; j < GPW; ++j) {
        const int gl = w * GPW + j, gi = kc * GPW + j;
        // group gl = 32 bytes of sub-tile gl / 4; the lane's 8 bytes sit in
        // 16-byte chunk 2 (gl % 4) + t4 / 2, swizzled by the row (gid)
        const unsigned char* cg =
            st + (gl >> 2) * 4096 + ((((gl & 3) << 1) | (t4 >> 1)) ^ gid) * 16;
        const uint2 g0 = *reinterpret_cast<const uint2*>(cg);
        const uint2 g1 = *reinterpret_cast<const uint2*>(cg + 8 * 128);
        const uint2 u0 = *reinterpret_cast<const uint2*>(cg + 16 * 128);
        const uint2 u1 = *reinterpret_cast<const uint2*>(cg + 24 * 128);
        uint32_t bfr[8];
        if (has_tok) {
          const uint4* px = reinterpret_cast<const uint4*>(xg + gi * 128);
          const uint4 v0 = px[0], v1 = px[1];
          bfr[0] = v0.x; bfr[1] = v0.y; bfr[2] = v0.z; bfr[3] = v0.w;
          bfr[4] = v1.x; bfr[5] = v1.y; bfr[6] = v1.z; bfr[7] = v1.w;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) bfr[e] = 0u;
        }
        float dg[4] = {0.f, 0.f, 0.f, 0.f}, du[4] = {0.f, 0.f, 0.f, 0.f};
        group_mma2(dg, du, g0, g1, u0, u1, bfr);
        const float2 X = *reinterpret_cast<const float2*>(xsum + gi * kTokS + 2 * t4);
        const float2* sb = sbt + gi * 32;
        const float2 sg0 = sb[gid], sg1 = sb[8 + gid], su0 = sb[16 + gid], su1 = sb[24 + gid];
        acc[0][0] = fmaf(sg0.x, dg[0], fmaf(sg0.y, X.x, acc[0][0]));
        acc[0][1] = fmaf(sg0.x, dg[1], fmaf(sg0.y, X.y, acc[0][1]));
        acc[0][2] = fmaf(sg1.x, dg[2], fmaf(sg1.y, X.x, acc[0][2]));
        acc[0][3] = fmaf(sg1.x, dg[3], fmaf(sg1.y, X.y, acc[0][3]));
        acc[1][0] = fmaf(su0.x, du[0], fmaf(su0.y, X.x, acc[1][0]));
        acc[1][1] = fmaf(su0.x, du[1], fmaf(su0.y, X.y, acc[1][1]));
        acc[1][2] = fmaf(su1.x, du[2], fmaf(su1.y, X.x, acc[1][2]));
        acc[1][3] = fmaf(su1.x, du[3], fmaf(su1.y, X.y, acc[1][3]));
      }
      __syncwarp();
      if (lane == 0) bar_arrive(su32(&empty[s]));
      if (++s == nst) {
        s = 0;
        ++rnd;
      }
    }
    if (!ok) break;

    // partial sums -> ring slot p; the unit's designated warp adds them
    const int p = i % kRing, pr = i / kRing;
    if (pr > 0 && !warp_wait(su32(&rfree[p]), (pr - 1) & 1)) {
      ok = false;
      break;
    }
    float* rp = red + (size_t)p * kCW * 32 * tr;
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = m * 16 + gid + 8 * (e >> 1), n = 2 * t4 + (e & 1);
        if (n < ntok) rp[((size_t)w * 32 + row) * tr + n] = acc[m][e];
      }
    __syncwarp();
    if (lane == 0) bar_arrive(su32(&rfull[p]));
    if (w == i % kCW) {
      if (!warp_wait(su32(&rfull[p]), pr & 1)) {
        ok = false;
        break;
      }
      for (int it = lane; it < 16 * ntok; it += 32) {
        const int row = it / ntok, n = it - row * ntok;
        float gs = 0.0f, us = 0.0f;
#pragma unroll
        for (int ww = 0; ww < kCW; ++ww) {
          gs += rp[((size_t)ww * 32 + row) * tr + n];
          us += rp[((size_t)ww * 32 + 16 + row) * tr + n];
        }
        const float silu = gs / (1.0f + __expf(-gs));
        a.h[((int64_t)r * a.T + wtok[w][n]) * I + row0 + row] = silu * us;
      }
      __syncwarp();
      if (lane == 0) bar_arrive(su32(&rfree[p]));
    }
  }
  if (!ok && lane == 0) {
    s_fail = 1;
    if (a.err) atomicOr(a.err, MOE_DERR_WAIT);
  }
}

// ------------------------------------------------------------------ phase B
// Down projection, streamed the same way.  Unit = (entry, 128 output rows);
// warp w owns rows 16w..16w+15 over the whole K = I, so a unit needs no
// cross-warp sum.  A stage is one 128-row x 256-column tile of Wd codes (a
// 16 KB TMA box of a 3-D map [blob][row of H][word of I/8], 128-byte
// swizzled).  The B operand is h of the entry's tokens, each fp32 value split
// into a bf16 hi / lo column pair (~2^-17 relative), four tokens per MMA.
// Each warp writes  w[t][j] * (Wd h)  into partial[t][j][rows]; the last entry
// to finish a 16-row tile (arrival counter) adds partial[t][0..k] in j order
// into y.  The kernel is launched as a programmatic dependent of the gate/up
// kernel: its producer starts streaming weights while that kernel drains and
// its consumers wait for it (griddepcontrol.wait) before reading h.
constexpr int kTokB = 4;     // tokens per MMA N tile (hi / lo column pairs)
constexpr int kRowsB = 128;  // output rows per unit (kCW warps x 16)
constexpr int kStageB = kRowsB * 128;
constexpr int kMaxMatch = 4;  // routing slots of one token listed per entry

struct DownGeom {
  int ngi, nch;  // 64-column groups of I, stages per unit (I / 256)
  int nst;
  int tr;        // distinct tokens staged (min(T, 8))
  int hrow;      // bytes per staged h row (one bf16 half of one token): 2 I + 16
  size_t o_raw, o_sbt, o_h, o_hsum, smem;
};

__host__ __device__ inline DownGeom down_geom(int I, int T, int nst) {
  DownGeom g;
  g.ngi = I / kGroup;
  g.nch = I / 256;
  g.nst = nst;
  g.tr = T < kTokS ? T : kTokS;
  const int nt = (g.tr + kTokB - 1) / kTokB;
  g.hrow = 2 * I + 16;
  g.o_raw = (size_t)nst * kStageB;                      // ds, db blocks [128][ngi] bf16
  g.o_sbt = g.o_raw + (size_t)2 * kRowsB * g.ngi * 2;   // per warp [16][ngi + 1] float2
  g.o_h = g.o_sbt + (size_t)kCW * 16 * (g.ngi + 1) * 8; // [8 nt][hrow]
  g.o_hsum = g.o_h + (size_t)8 * nt * g.hrow;           // [ngi][4 nt] fp32
  g.smem = g.o_hsum + (size_t)g.ngi * kTokB * nt * 4 + 1024;
  return g;
}

inline DownGeom down_plan(int I, int T) {
  DownGeom g = down_geom(I, T, 0);
  int nst = (int)((kStreamSmemBudget - (g.smem < kStreamSmemBudget ? g.smem : kStreamSmemBudget)) /
                  kStageB);
  if (nst > kMaxStages) nst = kMaxStages;
  if (nst < 2) nst = 0;
  return down_geom(I, T, nst);
}

// named barrier over the consumer warps only
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCW * 32) : "memory");
}

// One warp's arrival on a 16-row tile of y after storing its partial rows:
// the last of the n_exec entries to arrive adds partial[t][0..k] in j order.
__device__ void arrive_tile(const FfnArgs& a, int tile, int n_exec, int nslot) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  __threadfence();
  unsigned prev = 0;
  if (lane == 0) prev = atomicAdd(&a.tick[tile], 1u);
  prev = __shfl_sync(0xffffffffu, prev, 0);
  if (prev != (unsigned)(n_exec - 1)) return;
  __threadfence();
  for (int it = lane; it < 16 * a.T; it += 32) {
    const int t = it >> 4, o = tile * 16 + (it & 15);
    float yv = 0.0f;
    // eight slots at a time: every load is issued before the first add, the adds
    // stay in j order; an invalid routed id (skipped by the control step as
    // well) contributes nothing
    for (int j0 = 0; j0 < nslot; j0 += 8) {
      float p[8];
      bool v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int j = j0 + q;
        v[q] = j < nslot;
        if (v[q] && j < a.k) {
          const int32_t e = a.ids[t * a.k + j];
          v[q] = e >= 0 && e < a.E;
        }
        p[q] = v[q] ? __ldcg(a.partial + ((int64_t)t * nslot + j) * a.H + o) : 0.0f;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (v[q]) yv += p[q];
    }
    a.y[(int64_t)t * a.H + o] = yv;
  }
  __syncwarp();
  if (lane == 0) a.tick[tile] = 0u;
}

template <int NT>
__global__ void __launch_bounds__(kSThreads, 1)
    ffn_down_stream_kernel(FfnArgs a, DownGeom geo, const __grid_constant__ CodeMaps maps) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], sfull, sempty;
  __shared__ const uint8_t* sblob[kStreamMaxEntries];
  __shared__ int smap[kStreamMaxEntries], sbi[kStreamMaxEntries];
  __shared__ int sfs[kStreamMaxEntries];  // slot an F entry's blob is written to, else -1
  __shared__ int utok[kTokS], s_ntok;
  // routing slots j (and weights) of each staged token that name the entry
  __shared__ int mj[kTokS][kMaxMatch], mcnt[kTokS];
  __shared__ float mw[kTokS][kMaxMatch];
  constexpr int NTOK = kTokB * NT;
  const int H = a.H, I = a.I, ngi = geo.ngi, nst = geo.nst, nch = geo.nch;
  unsigned char* smem = smem_raw + ((1024u - (su32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    const int nrel = kCW + (a.fill_fused ? 1 : 0);  // warps that release a stage
    for (int i = 0; i < nst; ++i) {
      bar_init(su32(&full[i]), 1);
      bar_init(su32(&empty[i]), nrel);
    }
    bar_init(su32(&sfull), 1);
    bar_init(su32(&sempty), nrel);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the routing plan is complete before the gate/up kernel starts; only h
  // (and the arrival counters it resets) need that kernel to finish
  const int n_uniq = a.counts[0];
  const int n_exec = n_uniq + a.has_shared;
  if (n_exec == 0) {  // nothing routed to a valid expert: y = 0
    for (int i = blockIdx.x * blockDim.x + tid; i < a.T * H; i += gridDim.x * blockDim.x)
      a.y[i] = 0.0f;
    return;
  }
  if (wid == kCW) {
    if (lane < 3) tma_prefetch_map(&maps.m[lane]);
    for (int r = lane; r < n_exec; r += 32) {
      int mi = 2, bi = 0;
      int32_t fs = -1;
      if (r < n_uniq) {
        const int32_t id = a.uniq[r];
        const int32_t slot = ffn_slot(a, id, &fs);
        mi = slot >= 0 ? 1 : 0;
        bi = slot >= 0 ? slot : id;
      }
      smap[r] = mi;
      sbi[r] = bi;
      sblob[r] = (mi == 2 ? a.shared : mi == 1 ? a.pool : a.bank) + (int64_t)bi * a.blob_bytes;
      sfs[r] = fs;
    }
  }
  __syncthreads();

  const int upe = H / kRowsB;
  const int n_units = n_exec * upe;
  // (32-bit: units x CTAs stays far below 2^32 for every shape the stream path takes)
  const int u_lo = (int)(blockIdx.x * (unsigned)n_units / gridDim.x);
  const int u_hi = (int)((blockIdx.x + 1) * (unsigned)n_units / gridDim.x);
  const BlobOffsets off = blob_offsets(H, I);
  unsigned char* stages = smem;
  unsigned char* sraw = smem + geo.o_raw;
  const int rblk = kRowsB * ngi * 2;

  if (wid == kCW) {
    // -------------------------------------------------------- producer
    int s = 0, rnd = 0, nq = 0, nu = 0;
    bool ok = true;
    for (int u = u_lo; ok && u < u_hi; ++u) {
      const int i = u - u_lo, r = u / upe, o0 = (u % upe) * kRowsB;
      const uint8_t* blob = sblob[r];
      const CUtensorMap* map = &maps.m[smap[r]];
      if (lane == 0) {
        ok = i == 0 || bar_wait(su32(&sempty), (i - 1) & 1);
        if (ok) bar_expect(su32(&sfull), 2 * rblk);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ++nu;
      if (lane < 2)
        bulk_g2s(su32(sraw + lane * rblk), blob + (lane ? off.db : off.ds) + (int64_t)o0 * ngi * 2,
                 rblk, su32(&sfull));
      for (int kc = 0; kc < nch; ++kc) {
        if (lane == 0) {
          ok = rnd == 0 || bar_wait(su32(&empty[s]), (rnd - 1) & 1);
          if (ok) {
            bar_expect(su32(&full[s]), kStageB);
            tma_load_3d(su32(stages + s * kStageB), map, kc * 32, o0, sbi[r], su32(&full[s]));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        ++nq;
        if (++s == nst) {
          s = 0;
          ++rnd;
        }
      }
    }
    if (lane < nst) {
      const int uses = nq > lane ? (nq - lane + nst - 1) / nst : 0;
      if (uses > 0 && !bar_wait(su32(&full[lane]), (uses - 1) & 1)) ok = false;
    }
    if (lane == 31 && nu > 0 && !bar_wait(su32(&sfull), (nu - 1) & 1)) ok = false;
    if (!__all_sync(0xffffffffu, ok) && lane == 0 && a.err) atomicOr(a.err, MOE_DERR_WAIT);
    return;
  }
  if (wid == kFillW) {
    // ---------------------------------------------------- fill writer
    if (!a.fill_fused) return;
    int s = 0, rnd = 0;
    bool ok = true;
    for (int u = u_lo; ok && u < u_hi; ++u) {
      const int i = u - u_lo, o0 = (u % upe) * kRowsB, fs = sfs[u / upe];
      ok = warp_wait(su32(&sfull), i & 1);
      if (!ok) break;
      if (fs >= 0 && lane < 2) {  // the unit's down scale and bias rows
        fence_proxy_async_smem();
        bulk_s2g(a.pool_w + (int64_t)fs * a.blob_bytes + (lane ? off.db : off.ds) +
                     (int64_t)o0 * ngi * 2,
                 su32(sraw + lane * rblk), rblk);
        bulk_commit();
        bulk_read_done();
      }
      __syncwarp();
      if (lane == 0) bar_arrive(su32(&sempty));
      for (int kc = 0; kc < nch; ++kc) {
        ok = warp_wait(su32(&full[s]), rnd & 1);
        if (!ok) break;
        if (fs >= 0 && lane == 0) {  // the stage: one 128-row box, as loaded
          fence_proxy_async_smem();
          tma_store_3d(&maps.m[1], kc * 32, o0, fs, su32(stages + s * kStageB));
          bulk_commit();
          bulk_read_done();
        }
        __syncwarp();
        if (lane == 0) bar_arrive(su32(&empty[s]));
        if (++s == nst) {
          s = 0;
          ++rnd;
        }
      }
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // the slot writes are done
    if (!__all_sync(0xffffffffu, ok) && lane == 0 && a.err) atomicOr(a.err, MOE_DERR_WAIT);
    return;
  }

  // ---------------------------------------------------------- consumers
  const int w = wid, gid = lane >> 2, t4 = lane & 3;
  const int ctid = tid;  // 0 .. kCW * 32 - 1
  float2* sbt = reinterpret_cast<float2*>(smem + geo.o_sbt) + (size_t)w * 16 * (ngi + 1);
  unsigned char* hf = smem + geo.o_h;
  float* hsum = reinterpret_cast<float*>(smem + geo.o_hsum);
  const uint16_t* raw = reinterpret_cast<const uint16_t*>(sraw);
  const int nslot = a.k + a.has_shared, hrow = geo.hrow;
  // warp 0: the tokens routed to entry r and their routing slots and weights
  auto lists = [&](int r) {
    if (w == 0) {
      // distinct tokens routed to entry r, ascending
      int cnt;
      if (r < n_uniq) {
        const int32_t id = a.uniq[r];
        const int base = a.layer * a.E, n = a.T * a.k;
        cnt = 0;
        for (int n0 = 0; n0 < n; n0 += 32) {
          const int ii = n0 + lane;
          bool mt = ii < n && base + a.ids[ii] == id;
          for (int jj = mt ? ii - ii % a.k : ii; jj < ii; ++jj)
            if (base + a.ids[jj] == id) mt = false;
          const unsigned b = __ballot_sync(0xffffffffu, mt);
          const int pos = cnt + __popc(b & ((1u << lane) - 1u));
          if (mt && pos < kTokS) utok[pos] = ii / a.k;
          cnt += __popc(b);
        }
      } else {
        if (lane < a.T && lane < kTokS) utok[lane] = lane;
        cnt = a.T;
      }
      const int nt = cnt < geo.tr ? cnt : geo.tr;
      if (lane == 0) s_ntok = nt;
      __syncwarp();
      if (lane < nt) {
        const int t = utok[lane];
        int c = 0;
        if (r < n_uniq) {
          const int32_t id = a.uniq[r];
          for (int jj = 0; jj < a.k; ++jj)
            if (a.layer * a.E + a.ids[t * a.k + jj] == id) {
              if (c < kMaxMatch) {
                mj[lane][c] = jj;
                mw[lane][c] = a.weights[t * a.k + jj];
              }
              ++c;
            }
        } else {
          mj[lane][0] = a.k;
          mw[lane][0] = 1.0f;
          c = 1;
        }
        mcnt[lane] = c;
      }
    }
  };
  // the first entry's lists need only the routing plan: built before the wait
  int listed = -1;
  if (u_lo < u_hi) {
    listed = u_lo / upe;
    lists(listed);
  }
  // h is written by the gate/up kernel: wait for it to complete
  griddep_wait();
  griddep_launch();  // the next kernel may be scheduled (it waits for this one)
  int prev_r = -1, ntok = 0, s = 0, rnd = 0, pend = -1;
  bool ok = true;  // after a failed wait the warp keeps walking the loop (no waits,
                   // no math) so that every consumer warp meets the same barriers
  for (int u = u_lo; u < u_hi; ++u) {
    const int i = u - u_lo, r = u / upe, o0 = (u % upe) * kRowsB;
    if (r != prev_r) {
      // every warp is done with the previous entry's h and lists (and sees the
      // first entry's lists, built before the wait)
      consumers_sync();
      if (r != listed) {
        lists(r);
        listed = r;
        consumers_sync();
      }
      ntok = s_ntok;
      // h of those tokens as hi / lo bf16 column pairs in fragment order
      const int n_items = ntok * ngi * 4;
      for (int it0 = 0; it0 < n_items; it0 += kCW * 32) {
        const int it = it0 + ctid;
        const bool in = it < n_items;
        const int n = in ? it / (ngi * 4) : 0, rem = it - n * ngi * 4, g = rem >> 2, qq = rem & 3;
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = 0.0f;
        if (in) {
          const float4* p =
              reinterpret_cast<const float4*>(a.h + ((int64_t)r * a.T + utok[n]) * I + g * 64 + qq * 16);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 f = __ldcg(p + e);
            v[4 * e] = f.x;
            v[4 * e + 1] = f.y;
            v[4 * e + 2] = f.z;
            v[4 * e + 3] = f.w;
          }
        }
        uint32_t whi[8], wlo[8];
        float sx = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float h0 = v[2 * j], h1 = v[2 * j + 1];
          sx += h0 + h1;
          const __nv_bfloat162 hi = __floats2bfloat162_rn(h0, h1);
          const float2 hb = __bfloat1622float2(hi);
          whi[j] = *reinterpret_cast<const uint32_t*>(&hi);
          wlo[j] = pack_bf16(h0 - hb.x, h1 - hb.y);
        }
        sx += __shfl_xor_sync(0xffffffffu, sx, 1);
        sx += __shfl_xor_sync(0xffffffffu, sx, 2);
        if (in) {
          uint4 o0h, o1h, o0l, o1l;
          frag_order(whi, o0h, o1h);
          frag_order(wlo, o0l, o1l);
          uint4* dh = reinterpret_cast<uint4*>(hf + (size_t)(2 * n) * hrow + g * 128 + qq * 32);
          uint4* dl = reinterpret_cast<uint4*>(hf + (size_t)(2 * n + 1) * hrow + g * 128 + qq * 32);
          dh[0] = o0h;
          dh[1] = o1h;
          dl[0] = o0l;
          dl[1] = o1l;
          if (qq == 0) hsum[g * NTOK + n] = sx;
        }
      }
      consumers_sync();
      prev_r = r;
    }

    // this warp's 16 rows of the unit's scales -> (s, b - 128 s), lane = group
    ok = ok && warp_wait(su32(&sfull), i & 1);
    if (ok) {
      const uint16_t* rs = raw + (size_t)(16 * w) * ngi;
      const uint16_t* rb = rs + kRowsB * ngi;
      for (int row = 0; row < 16; ++row)
        for (int g = lane; g < ngi; g += 32) {
          const float sv = bf(rs[row * ngi + g]);
          sbt[row * (ngi + 1) + g] = make_float2(sv, fmaf(-128.0f, sv, bf(rb[row * ngi + g])));
        }
      __syncwarp();
      if (lane == 0) bar_arrive(su32(&sempty));
    }

    float acc[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = 0.0f;
    for (int kc = 0; ok && kc < nch; ++kc) {
      ok = warp_wait(su32(&full[s]), rnd & 1);
      if (!ok) break;
      const unsigned char* st = stages + s * kStageB + (16 * w + gid) * 128 + (t4 & 1) * 8;
#pragma unroll
      for (int gs = 0; gs < 4; ++gs) {
        const int g = kc * 4 + gs;
        const unsigned char* cg = st + ((((gs << 1) | (t4 >> 1)) ^ gid) * 16);
        const uint2 lo = *reinterpret_cast<const uint2*>(cg);
        const uint2 hi = *reinterpret_cast<const uint2*>(cg + 8 * 128);
        const float2 s0 = sbt[gid * (ngi + 1) + g], s1 = sbt[(gid + 8) * (ngi + 1) + g];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const int col = j * 2 * kTokB + gid;  // = 2 * token + (0 hi / 1 lo)
          uint32_t bfr[8];
          load_frag(hf + (size_t)col * hrow + g * 128 + t4 * 32, (col >> 1) < ntok, bfr);
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          group_mma(d, lo, hi, bfr);
          const float X = hsum[g * NTOK + j * kTokB + t4];
          acc[j][0] = fmaf(s0.x, d[0] + d[1], fmaf(s0.y, X, acc[j][0]));
          acc[j][1] = fmaf(s1.x, d[2] + d[3], fmaf(s1.y, X, acc[j][1]));
        }
      }
      __syncwarp();
      if (lane == 0) bar_arrive(su32(&empty[s]));
      if (++s == nst) {
        s = 0;
        ++rnd;
      }
    }
    if (!ok) continue;

    // the previous unit's partials were stored long ago: its arrival (fence +
    // counter) is cheap here and stays off the path of this unit's math
    if (pend >= 0) arrive_tile(a, pend, n_exec, nslot);
    // lane (gid, t4) holds rows orow, orow + 8 of token utok[j * 4 + t4]:
    // weighted into every routing slot of that token that names this expert
    const int orow = o0 + 16 * w + gid;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int n = j * kTokB + t4;
      if (n < ntok) {
        const int t = utok[n], c = mcnt[n];
        for (int m = 0; m < c && m < kMaxMatch; ++m) {
          float* dst = a.partial + ((int64_t)t * nslot + mj[n][m]) * H;
          dst[orow] = mw[n][m] * acc[j][0];
          dst[orow + 8] = mw[n][m] * acc[j][1];
        }
        if (c > kMaxMatch) {  // a token naming this expert more than kMaxMatch times
          const int32_t id = a.uniq[r];
          for (int jj = 0, m = 0; jj < a.k; ++jj) {
            if (a.layer * a.E + a.ids[t * a.k + jj] != id || m++ < kMaxMatch) continue;
            float* dst = a.partial + ((int64_t)t * nslot + jj) * H;
            dst[orow] = a.weights[t * a.k + jj] * acc[j][0];
            dst[orow + 8] = a.weights[t * a.k + jj] * acc[j][1];
          }
        }
      }
    }
    pend = (o0 >> 4) + w;
  }
  if (ok && pend >= 0) arrive_tile(a, pend, n_exec, nslot);
  if (!ok && lane == 0 && a.err) atomicOr(a.err, MOE_DERR_WAIT);
}
}  // namespace

size_t ffn_stream_smem(int H, int T) {
  if (H % 512 != 0 || T < 1 || T > kTokS) return SIZE_MAX;
  const StreamGeom g = stream_plan(H, T);
  return g.nst ? g.smem : SIZE_MAX;
}

cudaError_t launch_ffn_gate_up_stream(const FfnArgs& a, int n_tick, cudaStream_t st) {
  static size_t done1[64], done2[64];
  static int sms[64];
  if (a.max_entries > kStreamMaxEntries) return cudaErrorInvalidValue;
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= 64) return cudaErrorInvalidDevice;
  if (!sms[d]) {
    e = cudaDeviceGetAttribute(&sms[d], cudaDevAttrMultiProcessorCount, d);
    if (e != cudaSuccess) return e;
  }
  const StreamGeom geo = stream_plan(a.H, a.T);
  if (!geo.nst) return cudaErrorInvalidValue;
  // gate and up code matrices of every blob: [blob][matrix][row][word]
  CodeMaps maps;
  const uint64_t strides[3] = {(uint64_t)a.H / 2, (uint64_t)a.I * a.H / 2,
                               (uint64_t)a.blob_bytes};
  const uint32_t box[4] = {32, 16, 2, 1};
  const uint8_t* bases[3] = {a.bank, a.pool, a.shared ? a.shared : a.bank};
  const int nblob[3] = {a.n_bank, a.n_pool, a.shared ? 1 : a.n_bank};
  for (int i = 0; i < 3; ++i) {
    const uint64_t dims[4] = {(uint64_t)a.H / 8, (uint64_t)a.I, 2, (uint64_t)nblob[i]};
    if ((e = encode_tiled_u32(&maps.m[i], bases[i], 4, dims, strides, box)) != cudaSuccess)
      return e;
  }
  const int units = a.max_entries * (a.I / 16);
  const int grid = units < sms[d] ? units : sms[d];
  if (geo.gpw == 2) {
    if (done2[d] < geo.smem) {
      e = cudaFuncSetAttribute(ffn_gate_up_stream_kernel<2>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.smem);
      if (e != cudaSuccess) return e;
      done2[d] = geo.smem;
    }
    return launch_pdl(ffn_gate_up_stream_kernel<2>, dim3(grid), dim3(kSThreads), geo.smem, st, a,
                      n_tick, geo, maps);
  } else {
    if (done1[d] < geo.smem) {
      e = cudaFuncSetAttribute(ffn_gate_up_stream_kernel<1>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.smem);
      if (e != cudaSuccess) return e;
      done1[d] = geo.smem;
    }
    return launch_pdl(ffn_gate_up_stream_kernel<1>, dim3(grid), dim3(kSThreads), geo.smem, st, a,
                      n_tick, geo, maps);
  }
}

size_t ffn_down_stream_smem(int H, int I, int T) {
  if (I % 256 != 0 || H % kRowsB != 0 || T < 1 || T > kTokS) return SIZE_MAX;
  const DownGeom g = down_plan(I, T);
  return g.nst ? g.smem : SIZE_MAX;
}

cudaError_t launch_ffn_down_stream(const FfnArgs& a, cudaStream_t st) {
  static size_t done1[64], done2[64];
  static int sms[64];
  if (a.max_entries > kStreamMaxEntries) return cudaErrorInvalidValue;
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= 64) return cudaErrorInvalidDevice;
  if (!sms[d]) {
    e = cudaDeviceGetAttribute(&sms[d], cudaDevAttrMultiProcessorCount, d);
    if (e != cudaSuccess) return e;
  }
  const DownGeom geo = down_plan(a.I, a.T);
  if (!geo.nst) return cudaErrorInvalidValue;
  // down code matrix of every blob: [blob][row of H][word of I/8]
  CodeMaps maps;
  const BlobOffsets off = blob_offsets(a.H, a.I);
  const uint64_t strides[2] = {(uint64_t)a.I / 2, (uint64_t)a.blob_bytes};
  const uint32_t box[3] = {32, kRowsB, 1};
  const uint8_t* bases[3] = {a.bank, a.pool, a.shared ? a.shared : a.bank};
  const int nblob[3] = {a.n_bank, a.n_pool, a.shared ? 1 : a.n_bank};
  for (int i = 0; i < 3; ++i) {
    const uint64_t dims[3] = {(uint64_t)a.I / 8, (uint64_t)a.H, (uint64_t)nblob[i]};
    if ((e = encode_tiled_u32(&maps.m[i], bases[i] + off.dq, 3, dims, strides, box)) !=
        cudaSuccess)
      return e;
  }
  const int units = a.max_entries * (a.H / kRowsB);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(units < sms[d] ? units : sms[d]);
  cfg.blockDim = dim3(kSThreads);
  cfg.dynamicSmemBytes = geo.smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (geo.tr <= kTokB) {
    if (done1[d] < geo.smem) {
      e = cudaFuncSetAttribute(ffn_down_stream_kernel<1>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.smem);
      if (e != cudaSuccess) return e;
      done1[d] = geo.smem;
    }
    return cudaLaunchKernelEx(&cfg, ffn_down_stream_kernel<1>, a, geo, maps);
  }
  if (done2[d] < geo.smem) {
    e = cudaFuncSetAttribute(ffn_down_stream_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)geo.smem);
    if (e != cudaSuccess) return e;
    done2[d] = geo.smem;
  }
  return cudaLaunchKernelEx(&cfg, ffn_down_stream_kernel<2>, a, geo, maps);
}

}  // namespace moe
