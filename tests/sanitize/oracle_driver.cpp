// Host sanitizer run of the CPU oracle (test infrastructure): every exported
// oracle function on small inputs, valid and invalid, built with
// AddressSanitizer and UndefinedBehaviorSanitizer by tests/test_sanitize_cpu.py.
// Exits 0 when every call returned what its contract says.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <random>
#include <vector>

extern "C" {
void or_blob_offsets(int H, int I, int64_t* off);
void or_blob_matrix(const uint8_t* blob, int H, int I, int which, float* out);
float or_exp(float x);
float or_sigmoid(float z);
int or_router_logits(const uint16_t* x, const uint16_t* w, int T, int E, int H, float* logits);
int or_route_softmax_topk(const float* logits, int T, int E, int k, int32_t* ids, float* wts);
int or_route_sigmoid_group(const float* logits, const float* bias, int T, int E, int n_groups,
                           int topk_groups, int k, float scale, int32_t* ids, float* wts);
int or_q_star(int m, int bp, int bh);
int or_cache_step(int E, int layer, const int32_t* ids, int n_ids, int S, int K, int bp, int bh,
                  int policy, int L, int32_t* slot_of_id, int32_t* id_of_slot, uint32_t* ts,
                  uint32_t* clock, int32_t* uniq, int32_t* hit_ids, int32_t* hit_slots,
                  int32_t* fill_ids, int32_t* fill_slots, int32_t* evicted_ids,
                  int32_t* direct_ids, int32_t* victims, int32_t* counts);
int or_cache_place(int E, int L, int S, int policy, const int32_t* ids, int n,
                   int32_t* slot_of_id, int32_t* id_of_slot, uint32_t* ts, uint32_t* clock);
void or_expert_forward(const uint8_t* blob, int H, int I, const uint16_t* x, int T, double* y);
void or_moe_ffn(const uint8_t* const* blobs, int E, int H, int I, const uint16_t* x, int T,
                const int32_t* ids, const float* wts, int k, const uint8_t* shared_blob,
                int shared_I, double* y);
double or_e2m1(int code);
double or_e4m3(int byte);
double or_e8m0(int byte);
int or_fp4_blob_offsets(int H, int I, int fmt, int64_t* off);
int or_fp4_blob_matrix(const uint8_t* blob, int H, int I, int which, int fmt, double* out);
int or_fp4_expert_forward(const uint8_t* blob, int H, int I, int fmt, const uint16_t* x, int T,
                          double* y);
}

static int g_fail = 0;
#define CHECK(c)                                                    \
  do {                                                              \
    if (!(c)) {                                                     \
      std::fprintf(stderr, "check failed line %d: %s\n", __LINE__, #c); \
      g_fail = 1;                                                   \
    }                                                               \
  } while (0)

static uint16_t bf16_of(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

int main() {
  std::mt19937 rng(7);
  const int H = 64, I = 64, E = 8, L = 2, T = 3, k = 2;
  // int4 blob: random codes, small positive bf16 scales, small bf16 biases
  int64_t off[10];
  or_blob_offsets(H, I, off);
  const int64_t total = off[9];
  std::vector<std::vector<uint8_t>> blobs(E, std::vector<uint8_t>((size_t)total));
  for (auto& b : blobs) {
    for (int64_t i = 0; i < off[3]; ++i) b[i] = (uint8_t)rng();
    for (int64_t i = off[3]; i + 1 < total; i += 2) {
      const uint16_t v = bf16_of(0.01f * (float)(rng() % 17) / 16.0f + 0.001f);
      std::memcpy(&b[i], &v, 2);
    }
  }
  std::vector<float> w((size_t)I * H);
  for (int which = 0; which < 3; ++which) {
    or_blob_matrix(blobs[0].data(), H, I, which, w.data());
    for (float v : w) CHECK(std::isfinite(v));
  }
  // exp / sigmoid over a sweep, including the clamps and non-finite inputs
  for (int i = -2000; i <= 2000; ++i) {
    const float x = 0.05f * (float)i;
    CHECK(std::isfinite(or_exp(x)) || x > 88.0f);
    const float s = or_sigmoid(x);
    CHECK(s >= 0.0f && s <= 1.0f);
  }
  (void)or_exp(INFINITY);
  (void)or_exp(-INFINITY);
  (void)or_sigmoid(NAN);
  // router and both selections
  std::vector<uint16_t> x((size_t)T * H), wr((size_t)E * H);
  std::normal_distribution<float> nd(0.0f, 1.0f);
  for (auto& v : x) v = bf16_of(nd(rng));
  for (auto& v : wr) v = bf16_of(0.02f * nd(rng));
  std::vector<float> logits((size_t)T * E), wts((size_t)T * 3), bias(E, 0.001f);
  std::vector<int32_t> ids((size_t)T * 3);
  CHECK(or_router_logits(x.data(), wr.data(), T, E, H, logits.data()) == 0);
  CHECK(or_route_softmax_topk(logits.data(), T, E, k, ids.data(), wts.data()) == 0);
  CHECK(or_route_softmax_topk(logits.data(), T, E, E + 1, ids.data(), wts.data()) != 0);
  CHECK(or_route_sigmoid_group(logits.data(), bias.data(), T, E, 4, 2, 3, 2.5f, ids.data(),
                               wts.data()) == 0);
  CHECK(or_route_sigmoid_group(logits.data(), nullptr, T, E, 3, 2, 3, 1.0f, ids.data(),
                               wts.data()) != 0);
  for (int m = 0; m < 40; ++m) CHECK(or_q_star(m, 52700, 77300) <= m);
  // control step over random traces under the three policies, then placement
  const int S = 6, K = 3;
  for (int policy = 0; policy < 3; ++policy) {
    std::vector<int32_t> slot_of_id(L * E, -1), id_of_slot(S, -1);
    std::vector<uint32_t> ts(S, 0);
    uint32_t clock = 0;
    std::vector<int32_t> uniq(T * k), hi(T * k), hs(T * k), fi(T * k), fs(T * k), ev(T * k),
        di(T * k), vi(K), cnt(8);
    if (policy == 2) {
      const int32_t place[3] = {0, 5, 9};
      CHECK(or_cache_place(E, L, S, policy, place, 3, slot_of_id.data(), id_of_slot.data(),
                           ts.data(), &clock) == 0);
    }
    for (int step = 0; step < 50; ++step) {
      std::vector<int32_t> r(T * k);
      for (auto& v : r) v = (int32_t)(rng() % E);
      CHECK(or_cache_step(E, step % L, r.data(), T * k, S, K, 52700, 77300, policy, L,
                          slot_of_id.data(), id_of_slot.data(), ts.data(), &clock, uniq.data(),
                          hi.data(), hs.data(), fi.data(), fs.data(), ev.data(), di.data(),
                          vi.data(), cnt.data()) == 0);
    }
    std::vector<int32_t> bad(T * k, E);
    CHECK(or_cache_step(E, 0, bad.data(), T * k, S, K, 52700, 77300, policy, L,
                        slot_of_id.data(), id_of_slot.data(), ts.data(), &clock, uniq.data(),
                        hi.data(), hs.data(), fi.data(), fs.data(), ev.data(), di.data(),
                        vi.data(), cnt.data()) != 0);
  }
  {
    std::vector<int32_t> slot_of_id(L * E), id_of_slot(S);
    std::vector<uint32_t> ts(S);
    uint32_t clock = 0;
    const int32_t rep[2] = {3, 3};
    CHECK(or_cache_place(E, L, S, 0, rep, 2, slot_of_id.data(), id_of_slot.data(), ts.data(),
                         &clock) != 0);
  }
  // int4 expert and layer FFN
  std::vector<double> y((size_t)T * H);
  or_expert_forward(blobs[1].data(), H, I, x.data(), T, y.data());
  for (double v : y) CHECK(std::isfinite(v));
  std::vector<const uint8_t*> ptrs(E);
  for (int e = 0; e < E; ++e) ptrs[e] = blobs[e].data();
  CHECK(or_route_softmax_topk(logits.data(), T, E, k, ids.data(), wts.data()) == 0);
  or_moe_ffn(ptrs.data(), E, H, I, x.data(), T, ids.data(), wts.data(), k, blobs[2].data(), I,
             y.data());
  for (double v : y) CHECK(std::isfinite(v));
  // FP4 decoders, layouts and experts
  for (int c = 0; c < 16; ++c) (void)or_e2m1(c);
  for (int b = 0; b < 256; ++b) {
    (void)or_e4m3(b);
    (void)or_e8m0(b);
  }
  for (int fmt = 0; fmt < 2; ++fmt) {
    int64_t fo[8];
    CHECK(or_fp4_blob_offsets(H, I, fmt, fo) == 0);
    std::vector<uint8_t> fb((size_t)fo[7], 0);
    for (int64_t i = 0; i < fo[3]; ++i) fb[i] = (uint8_t)rng();
    for (int64_t i = fo[3]; i < fo[6]; ++i) fb[i] = fmt == 0 ? (uint8_t)(120 + rng() % 4) : 0x30;
    if (fmt == 1) {
      const float mat[3] = {1.0f, 0.5f, 2.0f};
      std::memcpy(&fb[fo[6]], mat, 12);
    }
    std::vector<double> dm((size_t)I * H);
    for (int which = 0; which < 3; ++which)
      CHECK(or_fp4_blob_matrix(fb.data(), H, I, which, fmt, dm.data()) == 0);
    CHECK(or_fp4_expert_forward(fb.data(), H, I, fmt, x.data(), T, y.data()) == 0);
    for (double v : y) CHECK(std::isfinite(v));
  }
  int64_t fo[8];
  CHECK(or_fp4_blob_offsets(H, I, 2, fo) != 0);
  CHECK(or_fp4_blob_offsets(100, I, 0, fo) != 0);
  if (g_fail) return 1;
  std::printf("oracle sanitizer run: ok\n");
  return 0;
}
