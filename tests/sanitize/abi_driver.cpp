// Host sanitizer run of the C ABI's host-side paths (test infrastructure):
// spec, cache, plan and argument validation, sizes and launch accounting,
// each refusal before any device work, built with AddressSanitizer and
// UndefinedBehaviorSanitizer by tests/test_sanitize_cpu.py.  Needs no GPU:
// every call here either returns from host checks or is a pure size query.
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "moe.h"

static int g_fail = 0;
#define CHECK(c)                                                         \
  do {                                                                   \
    if (!(c)) {                                                          \
      std::fprintf(stderr, "check failed line %d: %s (%s)\n", __LINE__, #c, \
                   moe_last_error());                                    \
      g_fail = 1;                                                        \
    }                                                                    \
  } while (0)

static moe_spec spec(int L, int H, int I, int E, int k, int fmt = MOE_FORMAT_INT4) {
  moe_spec s;
  std::memset(&s, 0, sizeof(s));
  s.num_layers = L;
  s.hidden = H;
  s.inter = I;
  s.num_experts = E;
  s.top_k = k;
  s.router = MOE_ROUTER_SOFTMAX_TOPK;
  s.n_groups = 1;
  s.topk_groups = 1;
  s.routed_scale = 1.0f;
  s.group_size = 64;
  s.has_shared = 0;
  s.shared_inter = I;
  s.format = fmt;
  return s;
}

int main() {
  CHECK(std::strstr(moe_version(), "sm_103a") != nullptr);
  CHECK(moe_last_error() != nullptr);
  const moe_spec q = spec(40, 2048, 512, 256, 8);
  CHECK(moe_expert_bytes(&q) == 1769472);
  CHECK(moe_expert_bytes(nullptr) == 0);
  moe_spec bad = q;
  bad.hidden = 100;
  CHECK(moe_expert_bytes(&bad) == 0);
  bad = q;
  bad.format = 7;
  CHECK(moe_expert_bytes(&bad) == 0);
  bad = q;
  bad.router = MOE_ROUTER_SIGMOID_GROUP;
  bad.n_groups = 3;
  CHECK(moe_expert_bytes(&bad) == 0);
  const moe_spec nv = spec(40, 2048, 512, 256, 8, MOE_FORMAT_NVFP4);
  const moe_spec mx = spec(40, 2048, 512, 256, 8, MOE_FORMAT_MXFP4);
  CHECK(moe_expert_bytes(&nv) == 1769728);
  CHECK(moe_expert_bytes(&mx) == 1671168);
  // size queries
  CHECK(moe_ffn_workspace_bytes(&q, 1) > 0);
  CHECK(moe_layer_workspace_bytes(&q, 8) > moe_layer_workspace_bytes(&q, 1));
  CHECK(moe_prefill_workspace_bytes(&q, 8192) > 0);
  // launch accounting with and without the cache's sync words
  uint32_t sync_words[16];
  moe_cache c;
  std::memset(&c, 0, sizeof(c));
  c.num_slots = 2560;
  c.k_victims = 8;
  c.bp_mbps = 52700;
  c.bh_mbps = 77300;
  CHECK(moe_layer_kernel_count(&q, &c, 1) == 3);
  c.sync = sync_words;
  CHECK(moe_layer_kernel_count(&q, &c, 1) == 1);
  CHECK(moe_layer_kernel_count(&q, &c, 8) == 3);
  CHECK(moe_layer_kernel_count(&q, nullptr, 1) == 0);
  CHECK(moe_layer_kernel_count(&q, &c, 65) == 0);
  // argument refusals (nothing reaches the device)
  CHECK(moe_route(&q, nullptr, 1, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr) ==
        MOE_EINVAL);
  CHECK(moe_route(&bad, nullptr, 1, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr) ==
        MOE_EINVAL);
  CHECK(moe_route(&q, nullptr, 0, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr) == MOE_OK);
  int32_t ids_bad[2] = {0, 40 * 256};
  int32_t tabs[8];
  c.slot_of_id = tabs;
  c.id_of_slot = tabs;
  c.ts = reinterpret_cast<uint32_t*>(tabs);
  c.clock = reinterpret_cast<uint32_t*>(tabs);
  CHECK(moe_cache_place(&q, &c, ids_bad, 2, nullptr) == MOE_EINVAL);
  int32_t ids_rep[2] = {5, 5};
  CHECK(moe_cache_place(&q, &c, ids_rep, 2, nullptr) == MOE_EINVAL);
  moe_plan p;
  std::memset(&p, 0, sizeof(p));
  p.capacity = 4;
  CHECK(moe_cache_step(&q, &c, 0, ids_rep, 1, &p, 0, nullptr) != MOE_OK);  // capacity < T*k
  const moe_spec big = spec(1, 7168, 2048, 256, 8);
  moe_cache cb = c;
  cb.slot_pool = tabs;
  cb.bank = tabs;
  int32_t dummy[4];
  moe_plan pb;
  std::memset(&pb, 0, sizeof(pb));
  pb.capacity = 64 * 8;
  pb.uniq = pb.hit_ids = pb.hit_slots = pb.fill_ids = pb.fill_slots = pb.evicted_ids =
      pb.direct_ids = pb.victims = pb.counts = pb.err = dummy;
  CHECK(moe_expert_ffn_noalloc(&big, &cb, 0, &pb, dummy, 64, dummy, reinterpret_cast<float*>(dummy),
                               nullptr, reinterpret_cast<float*>(dummy), nullptr) ==
        MOE_ECAPACITY);
  // FP4 prefill passes the format check; the stack buffer fails the 256-byte
  // workspace alignment before anything is launched
  CHECK(moe_prefill_workspace_bytes(&nv, 4) > 0);
  CHECK(moe_expert_ffn_prefill(&nv, dummy, dummy, 4, dummy, reinterpret_cast<float*>(dummy),
                               nullptr, nullptr, dummy + 1, 1 << 20,
                               reinterpret_cast<float*>(dummy), nullptr) == MOE_EINVAL);
  // elastic resize: host-side rejections
  CHECK(moe_slots_for_budget(&nv, -1) == -1);
  CHECK(moe_slots_for_budget(&nv, 0) == 0);
  CHECK(moe_cache_resize_workspace_bytes(&cb, 0) == 0);
  CHECK(moe_cache_resize(&nv, &cb, 0, dummy, 1 << 20, nullptr) == MOE_EINVAL);
  CHECK(moe_cache_resize(&nv, &cb, 4, dummy, 4, nullptr) == MOE_ECAPACITY);
  // layer prefetch: a layer out of range and NULL pointers are refused before the copy
  CHECK(moe_layer_prefetch(&nv, dummy, nv.num_layers, dummy, nullptr) == MOE_EINVAL);
  CHECK(moe_layer_prefetch(&nv, dummy, -1, dummy, nullptr) == MOE_EINVAL);
  CHECK(moe_layer_prefetch(&nv, nullptr, 0, dummy, nullptr) == MOE_EINVAL);
  CHECK(moe_layer_prefetch(&nv, dummy, 0, nullptr, nullptr) == MOE_EINVAL);
  if (g_fail) return 1;
  std::printf("abi sanitizer run: ok\n");
  return 0;
}
