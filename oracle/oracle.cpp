// CPU oracle for the per-layer MoE expert step.  TEST INFRASTRUCTURE ONLY.
//
// This file is a plain, slow, scalar restatement of what the step computes.
// It exists so the CUDA path can be checked against an independent program:
// it shares no code, header, table or constant generator with the CUDA
// library, and only the test suite, the smoke check and the timed CPU
// baseline of the benchmark may load it.  The product never calls it.
//
// Sources (FreeToken paper summary "paper.rainbus.top/paper/2608.16157",
// FreeToken reader "paperglide.net ... freetoken", Edge0 translation
// "bittide.aicompass.dev ... arXiv 2609.18063"):
//   * routing families          - Edge0 §2 "MoE routing"
//   * int4 affine group-64      - Edge0 §2 "Quantisation", §3.1 "executor paths"
//   * expert math               - Edge0 §3.1 "math convention":
//                                 down(silu(gate(x)) * up(x))
//   * lE+e bank ids, dedup, hit classification, q* split, single-pass
//     K-victim choice           - FreeToken "core method", "method steps",
//                                 "novelty"; reader "Semantic-Aware Expert
//                                 Caching" and "Elastic Memory Management"
//   * exact merge of partials   - FreeToken "core method"
//
// Readings where the pages are silent (each is listed in the design notes):
//   * blob byte layout and nibble order (low nibble = even column)
//   * dequant w = s*q + b with q unsigned 0..15 (additive "bias")
//   * router dot product order (CANON-DOT below), own exp (ORACLE-EXP below)
//   * softmax-top-k weights computed over the selected k only
//   * sigmoid-group tie rules and normalise-then-scale order
//   * q rounding half-up, F = lowest-id misses, q capped by K
//   * clock advanced once per control call; victims exclude slots hit now
//   * replacement policies compared with the shared LRU: per-layer LRU on an
//     equal split of the slots (floor(S / L) each, the rest unused); static
//     placement fills nothing (q = 0); a placed slot starts with ts 0
//   * shared expert added with weight 1
//
// Parity status: every function below is pinned by the not-gpu tests
// (worked examples from the pages, closed forms, brute force, float64).
//
// Threads: or_set_threads(n) lets the row loops of the dequantisation and of
// the float64 expert run on n host threads (OpenMP when built with -fopenmp).
// Each output row is computed by one thread in the same order as with one
// thread, so the results are identical bit for bit; the default is one thread.
//
// Build: g++ -std=c++17 -O2 -ffp-contract=off -fPIC -shared [-fopenmp]
// (no -ffast-math).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

const int kGroup = 64;
int g_threads = 1;  // host threads for the row loops (or_set_threads)

float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

float bits_to_float(uint32_t u) {
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Byte offsets of the nine sections of an expert blob (the layout reading).
struct BlobLayout {
  int64_t gq, uq, dq, gs, gb, us, ub, ds, db, total;
};

BlobLayout layout_of(int64_t H, int64_t I) {
  BlobLayout L;
  int64_t codes_gu = I * H / 2;       // [I][H] nibbles
  int64_t codes_d = H * I / 2;        // [H][I] nibbles
  int64_t sb_gu = I * (H / kGroup) * 2;  // bf16 [I][H/64]
  int64_t sb_d = H * (I / kGroup) * 2;   // bf16 [H][I/64]
  L.gq = 0;
  L.uq = L.gq + codes_gu;
  L.dq = L.uq + codes_gu;
  L.gs = L.dq + codes_d;
  L.gb = L.gs + sb_gu;
  L.us = L.gb + sb_gu;
  L.ub = L.us + sb_gu;
  L.ds = L.ub + sb_gu;
  L.db = L.ds + sb_d;
  int64_t end = L.db + sb_d;
  L.total = (end + 255) / 256 * 256;
  return L;
}

// Code of column c in a packed row: two codes per byte, low nibble = even c.
int code_at(const uint8_t* row, int64_t c) {
  uint8_t byte = row[c / 2];
  return (c % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
}

// Dequantised weight of a [rows][cols] matrix: w = s*q + b in fp32, with s
// and b the bf16 scale and bias of the 64-column group holding column c.
float weight_at(const uint8_t* codes, const uint16_t* s, const uint16_t* b, int64_t cols,
                int64_t r, int64_t c) {
  int q = code_at(codes + r * (cols / 2), c);
  int64_t g = r * (cols / kGroup) + c / kGroup;
  float sf = bf16_to_float(s[g]);
  float bf = bf16_to_float(b[g]);
  float prod = sf * (float)q;  // exact: 8-bit x 4-bit significands
  return prod + bf;
}

}  // namespace

extern "C" {

// Host threads for the row loops (n >= 1); returns the count now in effect
// (1 when the library was built without OpenMP).
int or_set_threads(int n) {
#ifdef _OPENMP
  g_threads = n < 1 ? 1 : n;
#else
  (void)n;
  g_threads = 1;
#endif
  return g_threads;
}

// ------------------------------------------------------------------ layout
int64_t or_expert_bytes(int H, int I) {
  if (H <= 0 || I <= 0 || H % kGroup || I % kGroup) return -1;
  return layout_of(H, I).total;
}

// off[0..9] = gq uq dq gs gb us ub ds db total
void or_blob_offsets(int H, int I, int64_t* off) {
  BlobLayout L = layout_of(H, I);
  int64_t v[10] = {L.gq, L.uq, L.dq, L.gs, L.gb, L.us, L.ub, L.ds, L.db, L.total};
  for (int i = 0; i < 10; ++i) off[i] = v[i];
}

// ----------------------------------------------------------------- dequant
// Edge0 §2 "Quantisation" / §3.1: int4 affine group-64 weights with a scale
// and a bias per group.  out[r][c] = s[r][c/64] * q[r][c] + b[r][c/64].
void or_dequant(const uint8_t* codes, const uint16_t* s, const uint16_t* b, int rows, int cols,
                float* out) {
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) out[r * cols + c] = weight_at(codes, s, b, cols, r, c);
}

// Dequantise matrix `which` (0 = gate [I][H], 1 = up [I][H], 2 = down [H][I])
// straight out of an expert blob.
void or_blob_matrix(const uint8_t* blob, int H, int I, int which, float* out) {
  BlobLayout L = layout_of(H, I);
  const uint8_t* q;
  const uint16_t *s, *b;
  int rows, cols;
  if (which == 0) {
    q = blob + L.gq; s = (const uint16_t*)(blob + L.gs); b = (const uint16_t*)(blob + L.gb);
    rows = I; cols = H;
  } else if (which == 1) {
    q = blob + L.uq; s = (const uint16_t*)(blob + L.us); b = (const uint16_t*)(blob + L.ub);
    rows = I; cols = H;
  } else {
    q = blob + L.dq; s = (const uint16_t*)(blob + L.ds); b = (const uint16_t*)(blob + L.db);
    rows = H; cols = I;
  }
  or_dequant(q, s, b, rows, cols, out);
}

// --------------------------------------------------------------- ORACLE-EXP
// Own single-precision exp (not any library's): Cody-Waite reduction
// x = n*ln2 + r with ln2 split into a short high part and a low part,
// |r| <= ln2/2, then the degree-7 Taylor polynomial of e^r in Horner form with
// fused multiply-adds, then exact scaling by 2^n built from exponent bits.
// x is clamped to [-87, 88] so 2^n stays a normal number.
float or_exp(float x) {
  const float kLog2e = 1.44269504088896341f;
  const float kLn2Hi = 0.693145751953125f;        // 0x3F317200, 15 significant bits
  const float kLn2Lo = 1.42860682030941723e-06f;  // ln2 - kLn2Hi
  if (x < -87.0f) x = -87.0f;
  if (x > 88.0f) x = 88.0f;
  float t = x * kLog2e;
  float n = std::nearbyint(t);  // round half to even (default rounding mode)
  float r = std::fma(n, -kLn2Hi, x);
  r = std::fma(n, -kLn2Lo, r);
  // Taylor coefficients 1/j! for j = 7 .. 0.
  float p = 1.0f / 5040.0f;
  p = std::fma(p, r, 1.0f / 720.0f);
  p = std::fma(p, r, 1.0f / 120.0f);
  p = std::fma(p, r, 1.0f / 24.0f);
  p = std::fma(p, r, 1.0f / 6.0f);
  p = std::fma(p, r, 0.5f);
  p = std::fma(p, r, 1.0f);
  p = std::fma(p, r, 1.0f);
  int ni = (int)n;
  float scale = bits_to_float((uint32_t)(ni + 127) << 23);
  return p * scale;
}

// Logistic sigmoid 1 / (1 + exp(-z)) with the exp above and IEEE division.
float or_sigmoid(float z) {
  float e = or_exp(-z);
  float d = 1.0f + e;
  return 1.0f / d;
}

// -------------------------------------------------------------- CANON-DOT
// Router logits l[t][e] = sum_h x[t][h] * W[e][h] in fp32, in one fixed order:
// H is cut into 8-element chunks; lane j (0..31) accumulates chunks
// c = j, j+32, j+64, ... in ascending order, elements in order, with fma from
// 0; then the 32 lane sums are combined by a butterfly: for d = 16, 8, 4, 2, 1
// every lane adds the value of lane (j xor d).  The result is lane 0's value.
// Requires H % 8 == 0.  Edge0 §2 "MoE routing" (logits feed both families).
int or_router_logits(const uint16_t* x, const uint16_t* w, int T, int E, int H, float* logits) {
  if (H % 8) return -1;
  const int chunks = H / 8;
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      float lane[32];
      for (int j = 0; j < 32; ++j) {
        float acc = 0.0f;
        for (int c = j; c < chunks; c += 32)
          for (int i = 0; i < 8; ++i) {
            int64_t h = (int64_t)c * 8 + i;
            acc = std::fma(bf16_to_float(x[(int64_t)t * H + h]),
                           bf16_to_float(w[(int64_t)e * H + h]), acc);
          }
        lane[j] = acc;
      }
      for (int d = 16; d >= 1; d /= 2) {
        float nxt[32];
        for (int j = 0; j < 32; ++j) nxt[j] = lane[j] + lane[j ^ d];
        std::memcpy(lane, nxt, sizeof(lane));
      }
      logits[(int64_t)t * E + e] = lane[0];
    }
  }
  return 0;
}

// ------------------------------------------------------------ routing
// Softmax-top-k (Edge0 §2, Qwen family): softmax over the logits, keep the
// top k, renormalise.  The full softmax denominator cancels in the
// renormalisation, so the weights are w_i = e_i / S with
// e_i = exp(l_i - l_max) over the selected experts and S their sum taken in
// rank order.  Rank order: logit descending, lower expert index first on ties.
int or_route_softmax_topk(const float* logits, int T, int E, int k, int32_t* ids, float* wts) {
  if (k <= 0 || k > E) return -1;
  std::vector<int> idx(E);
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (int64_t)t * E;
    for (int e = 0; e < E; ++e) idx[e] = e;
    std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) {
      if (l[a] != l[b]) return l[a] > l[b];
      return a < b;
    });
    float top = l[idx[0]];
    std::vector<float> ex(k);
    float S = 0.0f;
    for (int i = 0; i < k; ++i) {
      ex[i] = or_exp(l[idx[i]] - top);
      S = S + ex[i];
    }
    for (int i = 0; i < k; ++i) {
      ids[(int64_t)t * k + i] = idx[i];
      wts[(int64_t)t * k + i] = ex[i] / S;
    }
  }
  return 0;
}

// Sigmoid-group (Edge0 §2, DeepSeek-V3 / Ling family): s = sigmoid(logit);
// selection score sel = s + bias (bias steers selection only); each of the
// n_groups contiguous expert groups is scored by the sum of its two largest
// sel values; the topk_groups best groups are kept (lower group index first on
// ties); inside them the k best sel are taken (lower expert index first on
// ties); weights are the raw sigmoid values renormalised over the k, then
// multiplied by `scale`:  w_i = (s_i / S) * scale, S summed in rank order.
int or_route_sigmoid_group(const float* logits, const float* bias, int T, int E, int n_groups,
                           int topk_groups, int k, float scale, int32_t* ids, float* wts) {
  if (n_groups <= 0 || E % n_groups) return -1;
  const int gsz = E / n_groups;
  if (gsz < 2 || topk_groups <= 0 || topk_groups > n_groups) return -1;
  if (k <= 0 || k > topk_groups * gsz) return -1;
  std::vector<float> s(E), sel(E), gscore(n_groups);
  std::vector<int> gidx(n_groups), cand;
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (int64_t)t * E;
    for (int e = 0; e < E; ++e) {
      s[e] = or_sigmoid(l[e]);
      sel[e] = s[e] + (bias ? bias[e] : 0.0f);
    }
    for (int g = 0; g < n_groups; ++g) {
      std::vector<float> v(sel.begin() + g * gsz, sel.begin() + (g + 1) * gsz);
      std::sort(v.begin(), v.end(), [](float a, float b) { return a > b; });
      gscore[g] = v[0] + v[1];
      gidx[g] = g;
    }
    std::stable_sort(gidx.begin(), gidx.end(), [&](int a, int b) {
      if (gscore[a] != gscore[b]) return gscore[a] > gscore[b];
      return a < b;
    });
    cand.clear();
    for (int i = 0; i < topk_groups; ++i)
      for (int e = gidx[i] * gsz; e < (gidx[i] + 1) * gsz; ++e) cand.push_back(e);
    std::stable_sort(cand.begin(), cand.end(), [&](int a, int b) {
      if (sel[a] != sel[b]) return sel[a] > sel[b];
      return a < b;
    });
    float S = 0.0f;
    for (int i = 0; i < k; ++i) S = S + s[cand[i]];
    for (int i = 0; i < k; ++i) {
      ids[(int64_t)t * k + i] = cand[i];
      float r = s[cand[i]] / S;
      wts[(int64_t)t * k + i] = r * scale;
    }
  }
  return 0;
}

// ------------------------------------------------------------------ q*
// FreeToken "core method": equating T_fill(q) = qS/B_P with
// T_cpu(m-q) = (m-q)S/(B_H-B_P) gives q* ~= m*B_P/B_H; as B_H -> B_P the split
// degenerates to pure fill, and with B_H < B_P (no residual host bandwidth)
// it stays pure fill.  Integer form with bandwidths in MB/s and round half up:
// q = floor((2*m*bp + bh) / (2*bh)), clamped to [0, m].
int or_q_star(int m, int bp, int bh) {
  if (m <= 0) return 0;
  if (bh <= bp) return m;
  int64_t num = 2 * (int64_t)m * bp + bh;
  int64_t q = num / (2 * (int64_t)bh);
  if (q < 0) q = 0;
  if (q > m) q = m;
  return (int)q;
}

// ------------------------------------------------------------ control step
// One decode control step for one MoE layer (FreeToken "method steps",
// "novelty"; reader "Semantic-Aware Expert Caching", "Elastic Memory
// Management"):
//   1. now = ++clock
//   2. U = ascending unique {layer*E + id} over the n routed ids
//   3. H = members of U with a slot; their slot gets ts = now (recency moves
//      only when the router selects an expert)
//   4. M = U \ H ascending, m = |M|, q from or_q_star
//   5. victims = the K smallest keys (ts, slot) over slots with ts != now
//      (empty slots have ts 0 and come first), one pass, ascending
//   6. n_fill = min(q, K, #victims); F = M[0:n_fill]; C = M[n_fill:]
//   7. for i < n_fill: slot v = victims[i] drops its old id and takes F[i]
//      with ts = now.
// counts = {n_uniq, n_hit, n_miss, q, n_fill, n_direct, n_victims, now}.
//
// Replacement policy (`policy`), for the miss-rate comparison of FreeToken
// summary "core method" and reader Figure 4(b), and Edge0 §3.1 "hot" path:
//   0  shared LRU: one pool for all layers, as above (FreeToken)
//   1  per-layer LRU: layer l owns the fixed slot range [l*S_l, (l+1)*S_l)
//      with S_l = floor(S / L); step 5 scans only that range, so each layer
//      runs its own LRU (Edge0 "hot" path: a fixed per-layer resident set);
//      the S - L*S_l slots past the last range stay unused
//   2  static placement: the slots hold what or_cache_place put there and
//      nothing is ever filled (q = 0, every miss goes to C); the pages'
//      baselines pin "hot" experts or whole layers at load time
// Returns 0, or -1 on an id outside [0, E), an unknown policy, or policy 1
// with S < L.
int or_cache_step(int E, int layer, const int32_t* ids, int n_ids, int S, int K, int bp, int bh,
                  int policy, int L, int32_t* slot_of_id, int32_t* id_of_slot, uint32_t* ts,
                  uint32_t* clock, int32_t* uniq, int32_t* hit_ids, int32_t* hit_slots,
                  int32_t* fill_ids, int32_t* fill_slots, int32_t* evicted_ids,
                  int32_t* direct_ids, int32_t* victims, int32_t* counts) {
  for (int i = 0; i < n_ids; ++i)
    if (ids[i] < 0 || ids[i] >= E) return -1;
  if (policy < 0 || policy > 2) return -1;
  if (policy == 1 && (L < 1 || S < L)) return -1;
  int s_lo = 0, s_hi = S;  // the slots this step may take victims from
  if (policy == 1) {
    s_lo = layer * (S / L);
    s_hi = s_lo + S / L;
  }
  uint32_t now = *clock + 1;
  *clock = now;

  std::vector<int32_t> U;
  for (int i = 0; i < n_ids; ++i) U.push_back(layer * E + ids[i]);
  std::sort(U.begin(), U.end());
  U.erase(std::unique(U.begin(), U.end()), U.end());

  std::vector<int32_t> H, Hs, M;
  for (int32_t u : U) {
    int32_t s = slot_of_id[u];
    if (s >= 0) {
      H.push_back(u);
      Hs.push_back(s);
      ts[s] = now;
    } else {
      M.push_back(u);
    }
  }
  int m = (int)M.size();
  int q = policy == 2 ? 0 : or_q_star(m, bp, bh);

  std::vector<std::pair<uint32_t, int32_t>> keys;
  for (int32_t v = s_lo; v < s_hi; ++v)
    if (ts[v] != now) keys.push_back({ts[v], v});
  std::sort(keys.begin(), keys.end());
  int nv = std::min<int>(K, (int)keys.size());

  int n_fill = std::min(q, nv);
  for (int i = 0; i < K; ++i) victims[i] = (i < nv) ? keys[i].second : -1;

  for (int i = 0; i < n_fill; ++i) {
    int32_t v = keys[i].second;
    int32_t old = id_of_slot[v];
    if (old >= 0) slot_of_id[old] = -1;
    id_of_slot[v] = M[i];
    slot_of_id[M[i]] = v;
    ts[v] = now;
    fill_ids[i] = M[i];
    fill_slots[i] = v;
    evicted_ids[i] = old;
  }
  int n_direct = m - n_fill;
  for (int i = 0; i < n_direct; ++i) direct_ids[i] = M[n_fill + i];
  for (size_t i = 0; i < U.size(); ++i) uniq[i] = U[i];
  for (size_t i = 0; i < H.size(); ++i) {
    hit_ids[i] = H[i];
    hit_slots[i] = Hs[i];
  }
  counts[0] = (int32_t)U.size();
  counts[1] = (int32_t)H.size();
  counts[2] = m;
  counts[3] = q;
  counts[4] = n_fill;
  counts[5] = n_direct;
  counts[6] = nv;
  counts[7] = (int32_t)now;
  return 0;
}

// Preload of a chosen set of bank ids (the static placements the pages
// compare against: KTransformers-style "hot" experts, llama.cpp-style whole
// layers; also a warm start for the LRU policies).  The tables are emptied,
// then ids[i] (= l*E + e) goes to
//   policy 0, 2: slot i
//   policy 1:    slot l*S_l + (number of ids of layer l before it in the list)
// with ts = 0 (placed, not yet used) and clock = 0.  Returns 0, or -1 on an
// id outside [0, L*E), a repeated id, more ids than slots (per layer range
// for policy 1), an unknown policy, or policy 1 with S < L.
int or_cache_place(int E, int L, int S, int policy, const int32_t* ids, int n,
                   int32_t* slot_of_id, int32_t* id_of_slot, uint32_t* ts, uint32_t* clock) {
  if (policy < 0 || policy > 2 || n < 0 || L < 1 || S < 1) return -1;
  if (policy == 1 && S < L) return -1;
  const int n_ids = L * E;
  std::vector<int32_t> slot(n_ids, -1), owner(S, -1), used(L, 0);
  for (int i = 0; i < n; ++i) {
    const int32_t u = ids[i];
    if (u < 0 || u >= n_ids || slot[u] >= 0) return -1;
    int v = i;
    if (policy == 1) {
      const int l = u / E;
      if (used[l] >= S / L) return -1;
      v = l * (S / L) + used[l]++;
    }
    if (v >= S) return -1;
    slot[u] = v;
    owner[v] = u;
  }
  for (int u = 0; u < n_ids; ++u) slot_of_id[u] = slot[u];
  for (int v = 0; v < S; ++v) {
    id_of_slot[v] = owner[v];
    ts[v] = 0;
  }
  *clock = 0;
  return 0;
}

// ------------------------------------------------------ elastic slot pool
// Slots a memory budget holds (reader "Elastic Memory Management": 10 slots
// of 0.5 GB in 5 GB, 8 in 4 GB, 12 in 6 GB): floor(free_bytes / slot_bytes).
// Returns -1 for slot_bytes <= 0 or free_bytes < 0.
int64_t or_slots_for_budget(int64_t free_bytes, int64_t slot_bytes) {
  if (slot_bytes <= 0 || free_bytes < 0) return -1;
  return free_bytes / slot_bytes;
}

// Re-division of the shared slot pool from S to S_new slots at a safe point
// between steps (reader "Elastic Memory Management": the excess slots are
// evicted on a shrink, freed memory becomes new slots on a growth, and the
// bank and the routing never change).  Readings where the page is silent:
//   * which experts go on a shrink: the occupied slots past S_new can only
//     stay if the most useful experts are kept, so the cache's own recency
//     decides: the n_occ - S_new occupied slots with the smallest keys
//     (ts, slot) -- the order of the victim scan -- are evicted;
//   * where the kept experts past S_new go: in ascending slot order, to the
//     free slots below S_new in ascending order, with their ts (their blob
//     is copied there);
//   * slots [S_new, S) are emptied (id -1, ts 0), and on a growth the new
//     slots [S, S_new) start empty; the clock does not move.
// Writes evicted ids in (ts, slot) order, the moves as (from, to) pairs and
// counts = {n_evicted, n_moved, n_occupied after}.  Returns 0, or -1 for
// S < 1, S_new < 1, or a table that is not a bijection.
int or_cache_resize(int n_ids, int S, int S_new, int32_t* slot_of_id, int32_t* id_of_slot,
                    uint32_t* ts, int32_t* evicted_ids, int32_t* move_from, int32_t* move_to,
                    int32_t* counts) {
  if (S < 1 || S_new < 1 || n_ids < 0) return -1;
  for (int v = 0; v < S; ++v) {
    const int32_t u = id_of_slot[v];
    if (u >= n_ids || (u >= 0 && slot_of_id[u] != v)) return -1;
  }
  // 1. evict the oldest occupied slots until at most S_new remain
  std::vector<std::pair<uint32_t, int32_t>> occ;
  for (int v = 0; v < S; ++v)
    if (id_of_slot[v] >= 0) occ.push_back({ts[v], v});
  std::sort(occ.begin(), occ.end());
  const int n_ev = std::max(0, (int)occ.size() - S_new);
  for (int i = 0; i < n_ev; ++i) {
    const int32_t v = occ[i].second;
    evicted_ids[i] = id_of_slot[v];
    slot_of_id[id_of_slot[v]] = -1;
    id_of_slot[v] = -1;
    ts[v] = 0;
  }
  // 2. the kept experts past S_new move to the free slots below it
  std::vector<int32_t> from, to;
  for (int v = S_new; v < S; ++v)
    if (id_of_slot[v] >= 0) from.push_back(v);
  for (int v = 0; v < S_new && v < S && to.size() < from.size(); ++v)
    if (id_of_slot[v] < 0) to.push_back(v);
  if (to.size() != from.size()) return -1;  // cannot happen: at most S_new kept
  for (size_t i = 0; i < from.size(); ++i) {
    const int32_t a = from[i], b = to[i], u = id_of_slot[a];
    id_of_slot[b] = u;
    ts[b] = ts[a];
    slot_of_id[u] = b;
    id_of_slot[a] = -1;
    ts[a] = 0;
    move_from[i] = a;
    move_to[i] = b;
  }
  // 3. slots past both sizes' common part start (or are left) empty
  for (int v = std::min(S, S_new); v < std::max(S, S_new); ++v) {
    id_of_slot[v] = -1;
    ts[v] = 0;
  }
  int n_occ = 0;
  for (int v = 0; v < S_new; ++v) n_occ += id_of_slot[v] >= 0 ? 1 : 0;
  counts[0] = n_ev;
  counts[1] = (int32_t)from.size();
  counts[2] = n_occ;
  return 0;
}

// -------------------------------------------------------------- expert FFN
}  // extern "C"

namespace {

struct DenseExpert {
  int H = 0, I = 0;
  std::vector<float> wg, wu, wd;  // dequantised fp32 [I][H], [I][H], [H][I]
};

DenseExpert dense_of(const uint8_t* blob, int H, int I) {
  DenseExpert d;
  d.H = H;
  d.I = I;
  d.wg.resize((size_t)I * H);
  d.wu.resize((size_t)I * H);
  d.wd.resize((size_t)H * I);
  or_blob_matrix(blob, H, I, 0, d.wg.data());
  or_blob_matrix(blob, H, I, 1, d.wu.data());
  or_blob_matrix(blob, H, I, 2, d.wd.data());
  return d;
}

// g = Wg x, u = Wu x, h = silu(g) * u, y = Wd h in float64 for one token.
void dense_forward(const DenseExpert& d, const uint16_t* x, double* y) {
  const int H = d.H, I = d.I;
  std::vector<double> xv(H), h(I);
  for (int c = 0; c < H; ++c) xv[c] = bf16_to_float(x[c]);
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1)
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int c = 0; c < H; ++c) {
      g += (double)d.wg[(size_t)i * H + c] * xv[c];
      u += (double)d.wu[(size_t)i * H + c] * xv[c];
    }
    double silu = g / (1.0 + std::exp(-g));
    h[i] = silu * u;
  }
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1)
  for (int o = 0; o < H; ++o) {
    double acc = 0.0;
    for (int i = 0; i < I; ++i) acc += (double)d.wd[(size_t)o * I + i] * h[i];
    y[o] = acc;
  }
}

}  // namespace

extern "C" {

// One expert on T tokens in float64 (Edge0 §3.1 "math convention"):
//   g = Wg x, u = Wu x, h = silu(g) * u, y = Wd h, silu(z) = z / (1 + e^-z),
// weights dequantised in fp32 (w = s*q + b) and widened, x widened from bf16.
// x is [T][H] bf16 bits, y is [T][H].
void or_expert_forward(const uint8_t* blob, int H, int I, const uint16_t* x, int T, double* y) {
  DenseExpert d = dense_of(blob, H, I);
  for (int t = 0; t < T; ++t) dense_forward(d, x + (int64_t)t * H, y + (int64_t)t * H);
}

// Whole-layer expert output (FreeToken "core method": the partial sums of the
// cached set G and the direct set C merge exactly, so the layer output is the
// plain routed sum):  y[t] = sum_j w[t][j] * expert_{ids[t][j]}(x[t])
//                            + shared(x[t])   (shared expert weight 1),
// the routed terms added in rank order j = 0..k-1, then the shared term.
// blobs[e] points at expert e's blob for this layer; shared_blob may be null.
// Each distinct expert is dequantised once and reused for all its tokens.
void or_moe_ffn(const uint8_t* const* blobs, int E, int H, int I, const uint16_t* x, int T,
                const int32_t* ids, const float* wts, int k, const uint8_t* shared_blob,
                int shared_I, double* y) {
  std::vector<DenseExpert> cache(E);
  std::vector<char> have(E, 0);
  DenseExpert shared;
  if (shared_blob) shared = dense_of(shared_blob, H, shared_I);
  std::vector<double> ye(H);
  for (int t = 0; t < T; ++t) {
    double* yt = y + (int64_t)t * H;
    const uint16_t* xt = x + (int64_t)t * H;
    for (int o = 0; o < H; ++o) yt[o] = 0.0;
    for (int j = 0; j < k; ++j) {
      int e = ids[(int64_t)t * k + j];
      if (!have[e]) {
        cache[e] = dense_of(blobs[e], H, I);
        have[e] = 1;
      }
      dense_forward(cache[e], xt, ye.data());
      double w = wts[(int64_t)t * k + j];
      for (int o = 0; o < H; ++o) yt[o] += w * ye[o];
    }
    if (shared_blob) {
      dense_forward(shared, xt, ye.data());
      for (int o = 0; o < H; ++o) yt[o] += ye[o];
    }
  }
}


// ------------------------------------------------------ FP4 expert formats
// The pages' deployed models keep their experts in NVFP4 (Qwen3.6 on the
// laptop, GLM-5.2) or MXFP4 (DeepSeek-V4-Flash) (FreeToken summary "Key
// results" table).  Both store FP4 E2M1 elements -- 1 sign, 2 exponent and 1
// mantissa bit, exponent bias 1, no infinity or NaN -- with one scale per
// block of consecutive elements of a row:
//   MXFP4  blocks of 32; scale E8M0 = 2^(e - 127), e = 255 is NaN
//   NVFP4  blocks of 16; scale FP8 E4M3 (bias 7, no infinity, S.1111.111 is
//          NaN), times one fp32 scale per matrix
// (the OCP Microscaling Formats specification for E2M1, E8M0 and E4M3;
// NVFP4 is NVIDIA's 16-element variant with E4M3 block scales).
// Expert blob (a reading: the pages give no layout): Wg codes [I][H/2], Wu
// codes [I][H/2], Wd codes [H][I/2] (low nibble = even column, as for int4),
// then one scale byte per block: Wg [I][H/B], Wu [I][H/B], Wd [H][I/B]; for
// NVFP4 then the fp32 matrix scales of Wg, Wu, Wd; the total rounded up to
// 256 bytes.  fmt: 0 = MXFP4 (B = 32), 1 = NVFP4 (B = 16).

double or_e2m1(int code) {
  const int sgn = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  const double mag = e == 0 ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return sgn ? -mag : mag;
}

double or_e4m3(int byte) {
  const int sgn = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
  if (e == 15 && m == 7) return std::nan("");
  const double mag = e == 0 ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return sgn ? -mag : mag;
}

double or_e8m0(int byte) { return byte == 255 ? std::nan("") : std::ldexp(1.0, byte - 127); }

// off[8]: gate codes, up codes, down codes, gate scales, up scales, down
// scales, matrix scales (NVFP4), total bytes.  Returns 0, or -1 on a bad
// format or shape (H, I multiples of 64).
int or_fp4_blob_offsets(int H, int I, int fmt, int64_t* off) {
  if ((fmt != 0 && fmt != 1) || H <= 0 || I <= 0 || H % 64 || I % 64) return -1;
  const int64_t B = fmt == 1 ? 16 : 32, hi = (int64_t)H * I;
  off[0] = 0;
  off[1] = hi / 2;
  off[2] = hi;
  off[3] = hi / 2 * 3;
  off[4] = off[3] + hi / B;
  off[5] = off[4] + hi / B;
  off[6] = off[5] + hi / B;
  const int64_t end = off[6] + (fmt == 1 ? 12 : 0);
  off[7] = (end + 255) / 256 * 256;
  return 0;
}

// Dequantised matrix `which` (0 gate [I][H], 1 up [I][H], 2 down [H][I]) in
// float64: w[r][c] = e2m1(code) * block scale (* the matrix scale, NVFP4).
int or_fp4_blob_matrix(const uint8_t* blob, int H, int I, int which, int fmt, double* out) {
  int64_t off[8];
  if (or_fp4_blob_offsets(H, I, fmt, off) || which < 0 || which > 2) return -1;
  const int rows = which == 2 ? H : I, cols = which == 2 ? I : H;
  const int B = fmt == 1 ? 16 : 32;
  const uint8_t* q = blob + off[which];
  const uint8_t* sc = blob + off[3 + which];
  double mat = 1.0;
  if (fmt == 1) {
    float f;
    std::memcpy(&f, blob + off[6] + 4 * which, 4);
    mat = f;
  }
  for (int r = 0; r < rows; ++r)
    for (int c = 0; c < cols; ++c) {
      const uint8_t byte = q[(int64_t)r * (cols / 2) + c / 2];
      const int code = (c & 1) ? (byte >> 4) : (byte & 15);
      const int sb = sc[(int64_t)r * (cols / B) + c / B];
      const double scale = fmt == 1 ? or_e4m3(sb) * mat : or_e8m0(sb);
      out[(int64_t)r * cols + c] = or_e2m1(code) * scale;
    }
  return 0;
}

// One FP4 expert on T tokens in float64, the same math as or_expert_forward:
// g = Wg x, u = Wu x, h = silu(g) * u, y = Wd h, x widened from bf16.
int or_fp4_expert_forward(const uint8_t* blob, int H, int I, int fmt, const uint16_t* x, int T,
                          double* y) {
  std::vector<double> wg((size_t)I * H), wu((size_t)I * H), wd((size_t)H * I);
  if (or_fp4_blob_matrix(blob, H, I, 0, fmt, wg.data()) ||
      or_fp4_blob_matrix(blob, H, I, 1, fmt, wu.data()) ||
      or_fp4_blob_matrix(blob, H, I, 2, fmt, wd.data()))
    return -1;
  std::vector<double> xv(H), h(I);
  for (int t = 0; t < T; ++t) {
    for (int c = 0; c < H; ++c) xv[c] = bf16_to_float(x[(int64_t)t * H + c]);
    for (int i = 0; i < I; ++i) {
      double g = 0.0, u = 0.0;
      for (int c = 0; c < H; ++c) {
        g += wg[(size_t)i * H + c] * xv[c];
        u += wu[(size_t)i * H + c] * xv[c];
      }
      h[i] = g / (1.0 + std::exp(-g)) * u;
    }
    for (int o = 0; o < H; ++o) {
      double acc = 0.0;
      for (int i = 0; i < I; ++i) acc += wd[(size_t)o * I + i] * h[i];
      y[(int64_t)t * H + o] = acc;
    }
  }
  return 0;
}

}  // extern "C"
