// C ABI entry points of libmoe (declared in include/moe.h): argument checks
// on the host, then kernel launches on the caller's stream.  Nothing here
// allocates device memory or synchronises the host.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <vector>

#include "moe_internal.cuh"

namespace moe {
// The double buffer's whole-layer copy (prefill.cu): a copy kernel of one
// 256-thread CTA per SM, or cudaMemcpyAsync when an address or the size is not
// a multiple of 16 bytes.
cudaError_t launch_layer_copy(const void* src, void* dst, size_t bytes, cudaStream_t st);
}  // namespace moe

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_err[0] = '\0';
  return MOE_OK;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(MOE_ECUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int check_spec(const moe_spec* s) {
  if (!s) return fail(MOE_EINVAL, "spec is NULL");
  if (s->num_layers < 1) return fail(MOE_EINVAL, "num_layers must be >= 1");
  if (s->hidden < 64 || s->hidden % 64) return fail(MOE_EINVAL, "hidden must be a multiple of 64");
  if (s->inter < 64 || s->inter % 64) return fail(MOE_EINVAL, "inter must be a multiple of 64");
  if (s->num_experts < 1 || s->num_experts > moe::kMaxExperts)
    return fail(MOE_EINVAL, "num_experts must be in 1..%d", moe::kMaxExperts);
  if (s->top_k < 1 || s->top_k > s->num_experts || s->top_k > 64)
    return fail(MOE_EINVAL, "top_k must be in 1..min(num_experts, 64)");
  if (s->format != MOE_FORMAT_INT4 && s->format != MOE_FORMAT_MXFP4 &&
      s->format != MOE_FORMAT_NVFP4)
    return fail(MOE_EINVAL, "unknown expert format %d", s->format);
  if (s->format == MOE_FORMAT_INT4 && s->group_size != moe::kGroup)
    return fail(MOE_EUNSUPPORTED, "group_size must be 64");
  if ((int64_t)s->num_layers * s->num_experts > (int64_t)1 << 30)
    return fail(MOE_EINVAL, "num_layers * num_experts too large");
  if (s->router == MOE_ROUTER_SIGMOID_GROUP) {
    if (s->n_groups < 1 || s->num_experts % s->n_groups)
      return fail(MOE_EINVAL, "num_experts must be a multiple of n_groups");
    if (s->n_groups > 32) return fail(MOE_EUNSUPPORTED, "n_groups > 32");
    if (s->num_experts / s->n_groups < 2) return fail(MOE_EINVAL, "groups need >= 2 experts");
    if (s->topk_groups < 1 || s->topk_groups > s->n_groups)
      return fail(MOE_EINVAL, "topk_groups must be in 1..n_groups");
    if (s->top_k > s->topk_groups * (s->num_experts / s->n_groups))
      return fail(MOE_EINVAL, "top_k exceeds the experts of the kept groups");
  } else if (s->router != MOE_ROUTER_SOFTMAX_TOPK) {
    return fail(MOE_EINVAL, "unknown router %d", s->router);
  }
  if (s->has_shared != 0 && s->has_shared != 1) return fail(MOE_EINVAL, "has_shared must be 0/1");
  if (s->has_shared && s->shared_inter != s->inter)
    return fail(MOE_EUNSUPPORTED, "shared_inter must equal inter");
  return MOE_OK;
}

int check_cache(const moe_spec* s, const moe_cache* c, bool need_data) {
  if (!c) return fail(MOE_EINVAL, "cache is NULL");
  if (c->num_slots < 1) return fail(MOE_EINVAL, "num_slots must be >= 1");
  if (c->k_victims < 1 || c->k_victims > moe::kMaxVictims)
    return fail(MOE_EINVAL, "k_victims must be in 1..%d", moe::kMaxVictims);
  if (c->bp_mbps <= 0 || c->bh_mbps <= 0) return fail(MOE_EINVAL, "bandwidths must be > 0");
  if (!c->slot_of_id || !c->id_of_slot || !c->ts || !c->clock)
    return fail(MOE_EINVAL, "cache table pointer is NULL");
  if (c->policy < MOE_POLICY_SHARED_LRU || c->policy > MOE_POLICY_STATIC)
    return fail(MOE_EINVAL, "unknown cache policy %d", c->policy);
  if (c->policy == MOE_POLICY_LAYER_LRU && c->num_slots < s->num_layers)
    return fail(MOE_EINVAL, "the per-layer LRU needs num_slots >= num_layers (%d < %d)",
                c->num_slots, s->num_layers);
  if (need_data) {
    if (!c->slot_pool || !c->bank) return fail(MOE_EINVAL, "slot_pool / bank is NULL");
    if (!aligned(c->slot_pool, 16) || !aligned(c->bank, 16))
      return fail(MOE_EINVAL, "slot_pool / bank must be 16-byte aligned");
  }
  return MOE_OK;
}

int check_plan(const moe_plan* p, int need) {
  if (!p) return fail(MOE_EINVAL, "plan is NULL");
  if (!p->uniq || !p->hit_ids || !p->hit_slots || !p->fill_ids || !p->fill_slots ||
      !p->evicted_ids || !p->direct_ids || !p->victims || !p->counts || !p->err)
    return fail(MOE_EINVAL, "plan buffer pointer is NULL");
  if (p->capacity < need)
    return fail(MOE_ECAPACITY, "plan capacity %d < T*k = %d", p->capacity, need);
  return MOE_OK;
}

int do_route(const moe_spec* spec, const void* x, int32_t T, const void* w_router,
             const float* bias, float* logits, int32_t* ids, float* weights, cudaStream_t st) {
  if (!x || !w_router || !logits || !ids || !weights)
    return fail(MOE_EINVAL, "moe_route: NULL argument");
  if (!aligned(x, 16) || !aligned(w_router, 16))
    return fail(MOE_EINVAL, "moe_route: x and w_router must be 16-byte aligned");
  cudaError_t e = moe::launch_router_logits(static_cast<const uint16_t*>(x),
                                            static_cast<const uint16_t*>(w_router), T,
                                            spec->num_experts, spec->hidden, logits, st);
  if (e != cudaSuccess) return cuda_fail(e, "router logits launch");
  e = moe::launch_router_select(*spec, logits, bias, T, ids, weights, st);
  if (e != cudaSuccess) return cuda_fail(e, "router select launch");
  return MOE_OK;
}

moe::CacheArgs cache_args(const moe_spec* spec, moe_cache* c, int32_t layer, const int32_t* ids,
                          int32_t T, moe_plan* plan) {
  moe::CacheArgs a;
  a.E = spec->num_experts;
  a.layer = layer;
  a.n_ids = T * spec->top_k;
  // per-layer LRU: layer's own range of floor(S / L) slots; else all S slots
  const bool per_layer = c->policy == MOE_POLICY_LAYER_LRU;
  a.S = per_layer ? c->num_slots / spec->num_layers : c->num_slots;
  a.S0 = per_layer ? layer * a.S : 0;
  a.no_fill = c->policy == MOE_POLICY_STATIC;
  a.K = c->k_victims;
  a.n_slots = c->num_slots;
  a.n_bank = spec->num_layers * spec->num_experts;
  a.bp = c->bp_mbps;
  a.bh = c->bh_mbps;
  a.ids = ids;
  a.slot_of_id = c->slot_of_id;
  a.id_of_slot = c->id_of_slot;
  a.ts = c->ts;
  a.clock = c->clock;
  a.plan = *plan;
  return a;
}

// The whole decode layer step as one cooperative kernel (ffn_coop.cu): the
// cache carries sync words and the shape is one it serves.
bool layer_one_kernel(const moe_spec* spec, const moe_cache* c, int32_t T) {
  return c->sync != nullptr &&
         moe::layer_fused_supported(spec->hidden, spec->inter, spec->num_experts, spec->top_k, T,
                                    spec->has_shared, c->k_victims, spec->router,
                                    spec->n_groups);
}

int do_cache_step(const moe_spec* spec, moe_cache* c, int32_t layer, const int32_t* ids,
                  int32_t T, moe_plan* plan, int32_t do_fill, cudaStream_t st,
                  uint32_t* zero_words = nullptr, int n_zero = 0) {
  moe::CacheArgs a = cache_args(spec, c, layer, ids, T, plan);
  a.zero_words = zero_words;
  a.n_zero = n_zero;
  cudaError_t e = moe::launch_cache_step(a, st);
  if (e != cudaSuccess) return cuda_fail(e, "cache step launch");
  if (do_fill) {
    e = moe::launch_fill_copy(*plan, c->k_victims, static_cast<const uint8_t*>(c->bank),
                              static_cast<uint8_t*>(c->slot_pool),
                              moe::expert_blob_bytes(spec->hidden, spec->inter, spec->format), st);
    if (e != cudaSuccess) return cuda_fail(e, "fill copy launch");
  }
  return MOE_OK;
}

// The fill copy of a decode layer step runs beside the FFN on a side stream
// owned by the library (one per host thread and device): the FFN reads the
// experts being filled from the bank, and the caller's stream waits for the
// copy before its next work.  Fork and join are event record / wait pairs,
// so they also hold inside a captured graph.  The stream and its events are
// created on the first call that is not being captured (creation is not
// allowed during capture); until then the copy stays on the caller's stream.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

SideStream* side_stream(cudaStream_t st) {
  thread_local SideStream tab[64];
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return nullptr;
  SideStream& r = tab[d];
  if (r.s) return &r;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
    return nullptr;
  if (cudaStreamCreateWithFlags(&r.s, cudaStreamNonBlocking) != cudaSuccess) {
    r.s = nullptr;
    return nullptr;
  }
  if (cudaEventCreateWithFlags(&r.fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&r.join, cudaEventDisableTiming) != cudaSuccess) {
    cudaStreamDestroy(r.s);
    r.s = nullptr;
    return nullptr;
  }
  return &r;
}

int check_step_args(const moe_spec* spec, int32_t layer, int32_t T) {
  if (layer < 0 || layer >= spec->num_layers) return fail(MOE_EINVAL, "layer out of range");
  if (T < 0) return fail(MOE_EINVAL, "T must be >= 0");
  if ((int64_t)T * spec->top_k > moe::kMaxRouted)
    return fail(MOE_ECAPACITY, "T*k = %lld exceeds %d", (long long)T * spec->top_k,
                moe::kMaxRouted);
  return MOE_OK;
}

// moe_debug_inject_ffn_stall: consumed by the next do_ffn
std::atomic<int> g_inject_stall{0};

// fuse_fill: the streaming FFN kernels also write F's blobs into their slots
// (the caller launches no fill copy); only when ffn_fill_fusable holds.
// ctr_zeroed: the control step launched just before cleared the FFN's counter
// words (moe_layer_forward); otherwise the FFN launch clears them itself.
moe::FfnArgs ffn_args(const moe_spec* spec, const moe_cache* c, int32_t layer,
                      const moe_plan* plan, const void* x, int32_t T, const int32_t* ids,
                      const float* weights, const void* shared, void* ws, float* y,
                      bool fuse_fill) {
  moe::FfnArgs a;
  a.H = spec->hidden;
  a.I = spec->inter;
  a.E = spec->num_experts;
  a.k = spec->top_k;
  a.layer = layer;
  a.T = T;
  a.has_shared = spec->has_shared;
  a.format = spec->format;
  a.blob_bytes = moe::expert_blob_bytes(a.H, a.I, a.format);
  a.bank = static_cast<const uint8_t*>(c->bank);
  a.pool = static_cast<const uint8_t*>(c->slot_pool);
  a.n_bank = spec->num_layers * spec->num_experts;
  a.n_pool = c->num_slots;
  a.slot_of_id = c->slot_of_id;
  a.uniq = plan->uniq;
  a.counts = plan->counts;
  a.fill_ids = plan->fill_ids;
  a.fill_slots = plan->fill_slots;
  a.fill_fused = fuse_fill ? 1 : 0;
  a.pool_w = static_cast<uint8_t*>(c->slot_pool);
  a.tab_slot_of_id = c->slot_of_id;
  a.tab_id_of_slot = c->id_of_slot;
  a.tab_ts = c->ts;
  a.inject_stall = g_inject_stall.exchange(0);
  a.err = plan->err;
  a.x = static_cast<const uint16_t*>(x);
  a.ids = ids;
  a.weights = weights;
  a.shared = static_cast<const uint8_t*>(shared);
  a.y = y;
  moe::ffn_carve_workspace(a, ws);
  return a;
}

int do_ffn(const moe_spec* spec, const moe_cache* c, int32_t layer, const moe_plan* plan,
           const void* x, int32_t T, const int32_t* ids, const float* weights, const void* shared,
           void* ws, size_t ws_bytes, float* y, cudaStream_t st, bool fuse_fill = false,
           bool ctr_zeroed = false) {
  if (T > moe::kMaxDecodeT) return fail(MOE_EUNSUPPORTED, "decode FFN supports T <= %d",
                                        moe::kMaxDecodeT);
  if (!x || !ids || !weights || !y || !ws) return fail(MOE_EINVAL, "moe_expert_ffn: NULL argument");
  if (spec->has_shared && !shared) return fail(MOE_EINVAL, "spec has a shared expert: pass its blob");
  if (!aligned(x, 16) || !aligned(ws, 256) || (shared && !aligned(shared, 16)))
    return fail(MOE_EINVAL, "x (16 B), shared (16 B) and workspace (256 B) alignment");
  const size_t need = moe::ffn_workspace_bytes(spec->hidden, spec->inter, spec->top_k, T,
                                               spec->has_shared);
  if (ws_bytes < need) return fail(MOE_ECAPACITY, "workspace %zu < %zu bytes", ws_bytes, need);
  if (spec->format != MOE_FORMAT_INT4 &&
      !moe::ffn_coop_supported(spec->hidden, spec->inter, spec->top_k, T, spec->has_shared))
    return fail(MOE_EUNSUPPORTED,
                "FP4 experts need hidden %% 1024 == 0, inter %% 512 == 0 and T <= 8");
  moe::FfnArgs a = ffn_args(spec, c, layer, plan, x, T, ids, weights, shared, ws, y, fuse_fill);
  cudaError_t e = moe::launch_ffn_decode(a, st, ctr_zeroed);
  if (e != cudaSuccess) return cuda_fail(e, "decode FFN launch");
  return MOE_OK;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace

extern "C" {

const char* moe_last_error(void) { return g_err; }

const char* moe_version(void) { return "moe-gb300 0.1 (sm_103a)"; }

size_t moe_expert_bytes(const moe_spec* spec) {
  if (check_spec(spec) != MOE_OK) return 0;
  return (size_t)moe::expert_blob_bytes(spec->hidden, spec->inter, spec->format);
}

int moe_route(const moe_spec* spec, const void* x, int32_t T, const void* w_router,
              const float* bias, float* logits, int32_t* ids, float* weights,
              moe_stream_t stream) {
  int rc = check_spec(spec);
  if (rc) return rc;
  if (T < 0) return fail(MOE_EINVAL, "T must be >= 0");
  if (T == 0) return ok();
  rc = do_route(spec, x, T, w_router, bias, logits, ids, weights, (cudaStream_t)stream);
  return rc ? rc : ok();
}

int moe_cache_reset(const moe_spec* spec, moe_cache* cache, moe_stream_t stream) {
  int rc = check_spec(spec);
  if (rc) return rc;
  rc = check_cache(spec, cache, false);
  if (rc) return rc;
  cudaError_t e = moe::launch_cache_reset(cache->slot_of_id,
                                          spec->num_layers * spec->num_experts,
                                          cache->id_of_slot, cache->ts, cache->num_slots,
                                          cache->clock, cache->sync, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cache reset launch");
  return ok();
}

int moe_cache_place(const moe_spec* spec, moe_cache* cache, const int32_t* ids, int32_t n,
                    moe_stream_t stream) {
  int rc = check_spec(spec);
  if (rc) return rc;
  rc = check_cache(spec, cache, false);
  if (rc) return rc;
  if (n < 0 || (n > 0 && !ids)) return fail(MOE_EINVAL, "moe_cache_place: bad id list");
  const int L = spec->num_layers, E = spec->num_experts, S = cache->num_slots;
  const int64_t n_ids = (int64_t)L * E;
  const bool per_layer = cache->policy == MOE_POLICY_LAYER_LRU;
  const int range = per_layer ? S / L : S;  // slots one layer (or all of them) may use
  std::vector<int32_t> slot_of_id((size_t)n_ids, -1), id_of_slot((size_t)S, -1);
  std::vector<int32_t> used(per_layer ? L : 1, 0);
  // the whole list is checked before anything on the device is written
  for (int32_t i = 0; i < n; ++i) {
    const int32_t u = ids[i];
    if (u < 0 || u >= n_ids)
      return fail(MOE_EINVAL, "moe_cache_place: id %d outside [0, L*E)", u);
    if (slot_of_id[(size_t)u] >= 0) return fail(MOE_EINVAL, "moe_cache_place: id %d repeated", u);
    const int l = per_layer ? u / E : 0;
    if (used[l] >= range)
      return fail(MOE_EINVAL, "moe_cache_place: more ids than the %d slots %s", range,
                  per_layer ? "of one layer" : "of the cache");
    const int32_t v = l * range + used[l]++;
    slot_of_id[(size_t)u] = v;
    id_of_slot[(size_t)v] = u;
  }
  const cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(cache->slot_of_id, slot_of_id.data(),
                                  (size_t)n_ids * sizeof(int32_t), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(cache->id_of_slot, id_of_slot.data(), (size_t)S * sizeof(int32_t),
                        cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(cache->ts, 0, (size_t)S * sizeof(uint32_t), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(cache->clock, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess && cache->sync)
    e = cudaMemsetAsync(cache->sync, 0, MOE_CACHE_SYNC_WORDS * sizeof(uint32_t), st);
  if (cache->slot_pool && cache->bank) {
    const int64_t blob = moe::expert_blob_bytes(spec->hidden, spec->inter, spec->format);
    for (int32_t i = 0; i < n && e == cudaSuccess; ++i) {
      const int32_t u = ids[i];
      e = cudaMemcpyAsync(static_cast<uint8_t*>(cache->slot_pool) + slot_of_id[(size_t)u] * blob,
                          static_cast<const uint8_t*>(cache->bank) + (int64_t)u * blob,
                          (size_t)blob, cudaMemcpyDeviceToDevice, st);
    }
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);  // the host tables die on return
  if (e != cudaSuccess) return cuda_fail(e, "moe_cache_place");
  return ok();
}

int64_t moe_slots_for_budget(const moe_spec* spec, int64_t free_bytes) {
  if (check_spec(spec) != MOE_OK) return -1;
  if (free_bytes < 0) {
    fail(MOE_EINVAL, "moe_slots_for_budget: free_bytes < 0");
    return -1;
  }
  ok();
  return free_bytes / moe::expert_blob_bytes(spec->hidden, spec->inter, spec->format);
}

size_t moe_cache_resize_workspace_bytes(const moe_cache* cache, int32_t new_slots) {
  if (!cache || cache->num_slots < 1 || new_slots < 1) return 0;
  return moe::resize_workspace_bytes(cache->num_slots, new_slots);
}

int moe_cache_resize(const moe_spec* spec, moe_cache* cache, int32_t new_slots, void* workspace,
                     size_t workspace_bytes, moe_stream_t stream) {
  int rc = check_spec(spec);
  if (rc) return rc;
  rc = check_cache(spec, cache, false);
  if (rc) return rc;
  if (cache->policy != MOE_POLICY_SHARED_LRU)
    return fail(MOE_EUNSUPPORTED, "moe_cache_resize: the shared LRU policy only");
  if (new_slots < 1) return fail(MOE_EINVAL, "moe_cache_resize: new_slots must be >= 1");
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 4)
    return fail(MOE_EINVAL, "moe_cache_resize: workspace NULL or not 4-byte aligned");
  const size_t need = moe::resize_workspace_bytes(cache->num_slots, new_slots);
  if (workspace_bytes < need)
    return fail(MOE_ECAPACITY, "moe_cache_resize: workspace %zu < %zu bytes", workspace_bytes,
                need);
  if (cache->slot_pool && reinterpret_cast<uintptr_t>(cache->slot_pool) % 16)
    return fail(MOE_EINVAL, "moe_cache_resize: slot_pool must be 16-byte aligned");
  const cudaError_t e = moe::launch_cache_resize(
      cache->slot_of_id, spec->num_layers * spec->num_experts, cache->id_of_slot, cache->ts,
      cache->num_slots, new_slots, static_cast<uint8_t*>(cache->slot_pool),
      moe::expert_blob_bytes(spec->hidden, spec->inter, spec->format),
      static_cast<int32_t*>(workspace), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cache resize launch");
  cache->num_slots = new_slots;
  return ok();
}

int moe_cache_step(const moe_spec* spec, moe_cache* cache, int32_t layer, const int32_t* ids,
                   int32_t T, moe_plan* plan, int32_t do_fill, moe_stream_t stream) {
  int rc = check_spec(spec);
  if (rc) return rc;
  rc = check_cache(spec, cache, do_fill != 0);
  if (rc) return rc;
  rc = check_step_args(spec, layer, T);
  if (rc) return rc;
  if (T == 0) return ok();
  if (!ids) return fail(MOE_EINVAL, "ids is NULL");
  rc = check_plan(plan, T * spec->top_k);
  if (rc) return rc;
  rc = do_cache_step(spec, cache, layer, ids, T, plan, do_fill, (cudaStream_t)stream);
  return rc ? rc : ok();
}

size_t moe_ffn_workspace_bytes(const moe_spec* spec, int32_t T) {
  if (check_spec(spec) != MOE_OK || T < 1) return 0;
  return moe::ffn_workspace_bytes(spec->hidden, spec->inter, spec->top_k, T, spec->has_shared);
}

int moe_expert_ffn(const moe_spec* spec, const moe_cache* cache, int32_t layer,
                   const moe_plan* plan, const void* x, int32_t T, const int32_t* ids,
                   const float* weights, const void* shared, void* workspace,
                   size_t workspace_bytes, float* y, moe_stream_t stream) {
  int rc = check_spec(spec);
  if (rc) return rc;
  rc = check_cache(spec, cache, true);
  if (rc) return rc;
  rc = check_step_args(spec, layer, T);
  if (rc) return rc;
  if (T == 0) return ok();
  rc = check_plan(plan, T * spec->top_k);
  if (rc) return rc;
  rc = do_ffn(spec, cache, layer, plan, x, T, ids, weights, shared, workspace, workspace_bytes, y,
              (cudaStream_t)stream);
  return rc ? rc : ok();
}

size_t moe_layer_workspace_bytes(const moe_spec* spec, int32_t T) {
  if (check_spec(spec) != MOE_OK || T < 1) return 0;
  return align256((size_t)T * spec->num_experts * 4) +
         moe::ffn_workspace_bytes(spec->hidden, spec->inter, spec->top_k, T, spec->has_shared);
}

int moe_debug_inject_ffn_stall(int32_t on) {
  g_inject_stall.store(on ? 1 : 0);
  return MOE_OK;
}

int32_t moe_layer_kernel_count(const moe_spec* spec, const moe_cache* cache, int32_t T) {
  if (check_spec(spec) != MOE_OK || !cache || T < 1 || T > moe::kMaxDecodeT) return 0;
  if (layer_one_kernel(spec, cache, T)) return 1;
  const bool fused_sel = T <= moe::kSelFusedMaxT && spec->num_experts <= moe::kSelFusedMaxE;
  const bool fused_fill =
      moe::ffn_fill_fusable(spec->hidden, spec->inter, spec->top_k, T, spec->has_shared);
  const bool coop =
      moe::ffn_coop_supported(spec->hidden, spec->inter, spec->top_k, T, spec->has_shared);
  // logits, [select], control step, [fill copy], FFN (one cooperative kernel, or
  // gate/up and down)
  return 1 + (fused_sel ? 0 : 1) + 1 + (fused_fill ? 0 : 1) + (coop ? 1 : 2);
}

int moe_layer_forward(const moe_spec* spec, moe_cache* cache, int32_t layer, const void* x,
                      int32_t T, const void* w_router, const float* bias, const void* shared,
                      moe_plan* plan, int32_t* ids, float* weights, void* workspace,
                      size_t workspace_bytes, float* y, moe_stream_t stream) {
  int rc = check_spec(spec);
  if (rc) return rc;
  rc = check_cache(spec, cache, true);
  if (rc) return rc;
  rc = check_step_args(spec, layer, T);
  if (rc) return rc;
  if (T == 0) return ok();
  if (T > moe::kMaxDecodeT)
    return fail(MOE_EUNSUPPORTED, "decode layer supports T <= %d", moe::kMaxDecodeT);
  rc = check_plan(plan, T * spec->top_k);
  if (rc) return rc;
  if (!workspace || !aligned(workspace, 256)) return fail(MOE_EINVAL, "workspace must be 256-B aligned");
  const size_t need = moe_layer_workspace_bytes(spec, T);
  if (workspace_bytes < need)
    return fail(MOE_ECAPACITY, "workspace %zu < %zu bytes", workspace_bytes, need);
  cudaStream_t st = (cudaStream_t)stream;
  float* logits = static_cast<float*>(workspace);
  const size_t lbytes = align256((size_t)T * spec->num_experts * 4);
  if (layer_one_kernel(spec, cache, T)) {
    if (!x || !w_router || !ids || !weights || !y)
      return fail(MOE_EINVAL, "moe_layer_forward: NULL argument");
    if (spec->has_shared && !shared) return fail(MOE_EINVAL, "spec has a shared expert: pass its blob");
    if (!aligned(x, 16) || !aligned(w_router, 16) || (shared && !aligned(shared, 16)))
      return fail(MOE_EINVAL, "moe_layer_forward: x, w_router and shared must be 16-byte aligned");
    moe::FfnArgs a = ffn_args(spec, cache, layer, plan, x, T, ids, weights, shared,
                              static_cast<uint8_t*>(workspace) + lbytes, y, true);
    a.ctr = cache->sync + moe::kSyncCtr;
    a.n_ctr = MOE_CACHE_SYNC_WORDS - moe::kSyncCtr;
    moe::LayerFuse lf;
    lf.w_router = static_cast<const uint16_t*>(w_router);
    lf.sel_bias = bias;
    lf.logits = logits;
    lf.router = spec->router;
    lf.n_groups = spec->n_groups;
    lf.topk_groups = spec->topk_groups;
    lf.scale = spec->routed_scale;
    lf.ids_out = ids;
    lf.wts_out = weights;
    lf.sync = cache->sync;
    lf.c = cache_args(spec, cache, layer, ids, T, plan);
    const cudaError_t e = moe::launch_layer_fused(a, lf, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode layer kernel launch");
    return ok();
  }
  // fill copy: written by the streaming FFN kernels as they read F from the
  // bank when both run for this shape (FreeToken "method steps": the miss
  // path copies the expert into its slot), else a copy kernel beside the FFN
  const bool fused_fill = moe::ffn_fill_fusable(spec->hidden, spec->inter, spec->top_k, T,
                                                spec->has_shared);
  SideStream* ss = fused_fill ? nullptr : side_stream(st);
  // the cooperative FFN's counter words, cleared by the control step
  const bool coop = moe::ffn_coop_supported(spec->hidden, spec->inter, spec->top_k, T,
                                            spec->has_shared);
  moe::FfnArgs carve;
  carve.H = spec->hidden;
  carve.I = spec->inter;
  carve.k = spec->top_k;
  carve.T = T;
  carve.has_shared = spec->has_shared;
  moe::ffn_carve_workspace(carve, static_cast<uint8_t*>(workspace) + lbytes);
  if (T <= moe::kSelFusedMaxT && spec->num_experts <= moe::kSelFusedMaxE) {
    // logits kernel, then the selection inside the control step's CTA
    if (!x || !w_router || !ids || !weights) return fail(MOE_EINVAL, "moe_layer_forward: NULL argument");
    if (!aligned(x, 16) || !aligned(w_router, 16))
      return fail(MOE_EINVAL, "moe_layer_forward: x and w_router must be 16-byte aligned");
    cudaError_t e = moe::launch_router_logits(static_cast<const uint16_t*>(x),
                                              static_cast<const uint16_t*>(w_router), T,
                                              spec->num_experts, spec->hidden, logits, st);
    if (e != cudaSuccess) return cuda_fail(e, "router logits launch");
    moe::CacheArgs a = cache_args(spec, cache, layer, ids, T, plan);
    if (coop) {
      a.zero_words = carve.ctr;
      a.n_zero = carve.n_ctr;
    }
    moe::SelArgs sa;
    sa.logits = logits;
    sa.bias = bias;
    sa.T = T;
    sa.k = spec->top_k;
    sa.router = spec->router;
    sa.n_groups = spec->n_groups;
    sa.topk_groups = spec->topk_groups;
    sa.scale = spec->routed_scale;
    sa.ids = ids;
    sa.wts = weights;
    e = moe::launch_cache_step_sel(a, sa, st);
    if (e != cudaSuccess) return cuda_fail(e, "control step launch");
    if (!ss && !fused_fill) {
      e = moe::launch_fill_copy(*plan, cache->k_victims, static_cast<const uint8_t*>(cache->bank),
                                static_cast<uint8_t*>(cache->slot_pool),
                                moe::expert_blob_bytes(spec->hidden, spec->inter, spec->format),
                                st);
      if (e != cudaSuccess) return cuda_fail(e, "fill copy launch");
    }
  } else {
    rc = do_route(spec, x, T, w_router, bias, logits, ids, weights, st);
    if (rc) return rc;
    rc = do_cache_step(spec, cache, layer, ids, T, plan, (ss || fused_fill) ? 0 : 1, st,
                       coop ? carve.ctr : nullptr, coop ? carve.n_ctr : 0);
    if (rc) return rc;
  }
  if (ss) {  // fill copy beside the FFN
    cudaError_t e = cudaEventRecord(ss->fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->s, ss->fork, 0);
    if (e != cudaSuccess) return cuda_fail(e, "fill fork");
    e = moe::launch_fill_copy(*plan, cache->k_victims, static_cast<const uint8_t*>(cache->bank),
                              static_cast<uint8_t*>(cache->slot_pool),
                              moe::expert_blob_bytes(spec->hidden, spec->inter, spec->format),
                              ss->s);
    if (e == cudaSuccess) e = cudaEventRecord(ss->join, ss->s);
    if (e != cudaSuccess) return cuda_fail(e, "fill copy launch");
  }
  rc = do_ffn(spec, cache, layer, plan, x, T, ids, weights, shared,
              static_cast<uint8_t*>(workspace) + lbytes, workspace_bytes - lbytes, y, st,
              fused_fill, coop);
  if (ss) {
    const cudaError_t e = cudaStreamWaitEvent(st, ss->join, 0);
    if (e != cudaSuccess && !rc) return cuda_fail(e, "fill join");
  }
  return rc ? rc : ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// On-device B_P / B_H measurement.
namespace {

constexpr int kProfCopies = 2;  // blobs per timed fill copy

struct ProfLayout {
  size_t copy, counts_c, ids_c, slots_c, counts_f, uniq, fill_ids, err, ids, wts, x, y, ffn, total;
};

ProfLayout prof_layout(const moe_spec* s) {
  ProfLayout L;
  const size_t se = moe::expert_blob_bytes(s->hidden, s->inter, s->format);
  const size_t k = (size_t)s->top_k;
  size_t o = 0;
  auto take = [&](size_t b) {
    const size_t at = o;
    o += align256(b);
    return at;
  };
  L.copy = take((size_t)kProfCopies * se);
  L.counts_c = take(8 * 4);
  L.ids_c = take(kProfCopies * 4);
  L.slots_c = take(kProfCopies * 4);
  L.counts_f = take(8 * 4);
  L.uniq = take(k * 4);
  L.fill_ids = take(k * 4);
  L.err = take(4);
  L.ids = take(k * 4);
  L.wts = take(k * 4);
  L.x = take((size_t)s->hidden * 2);
  L.y = take((size_t)s->hidden * 4);
  L.ffn = take(moe::ffn_workspace_bytes(s->hidden, s->inter, s->top_k, 1, 0));
  L.total = o;
  return L;
}

// Milliseconds of `reps` launches of fn on st (after two untimed ones).
template <typename F>
cudaError_t time_reps(F fn, int reps, cudaStream_t st, float* ms) {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaError_t e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  for (int i = 0; e == cudaSuccess && i < 2; ++i) e = fn();
  if (e == cudaSuccess) e = cudaEventRecord(e0, st);
  for (int i = 0; e == cudaSuccess && i < reps; ++i) e = fn();
  if (e == cudaSuccess) e = cudaEventRecord(e1, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaEventElapsedTime(ms, e0, e1);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  return e;
}

}  // namespace

extern "C" size_t moe_profile_workspace_bytes(const moe_spec* spec) {
  if (check_spec(spec) != MOE_OK) return 0;
  return prof_layout(spec).total;
}

extern "C" int moe_profile_bandwidths(const moe_spec* spec, const moe_cache* cache,
                                      int32_t layer, void* workspace, size_t workspace_bytes,
                                      int32_t reps, int32_t* bp_mbps, int32_t* bh_mbps,
                                      moe_stream_t stream) {
  int rc = check_spec(spec);
  if (rc) return rc;
  rc = check_cache(spec, cache, true);
  if (rc) return rc;
  if (layer < 0 || layer >= spec->num_layers) return fail(MOE_EINVAL, "layer out of range");
  if (reps < 1) return fail(MOE_EINVAL, "reps must be >= 1");
  if (!bp_mbps || !bh_mbps) return fail(MOE_EINVAL, "moe_profile_bandwidths: NULL output");
  if (spec->top_k > spec->num_experts) return fail(MOE_EINVAL, "top_k > num_experts");
  if (!workspace || !aligned(workspace, 256)) return fail(MOE_EINVAL, "workspace must be 256-B aligned");
  const ProfLayout L = prof_layout(spec);
  if (workspace_bytes < L.total)
    return fail(MOE_ECAPACITY, "workspace %zu < %zu bytes", workspace_bytes, L.total);
  cudaStream_t st = (cudaStream_t)stream;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
    return fail(MOE_EINVAL, "moe_profile_bandwidths cannot run during stream capture");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto i32 = [&](size_t off) { return reinterpret_cast<int32_t*>(ws + off); };
  const int E = spec->num_experts, k = spec->top_k;
  const int64_t se = moe::expert_blob_bytes(spec->hidden, spec->inter, spec->format);

  // fill plan: experts 0, 1 of the layer into scratch blobs 0, 1
  int32_t hc[8] = {0, 0, 0, 0, kProfCopies, 0, 0, 0};
  int32_t hid[kProfCopies], hsl[kProfCopies];
  for (int i = 0; i < kProfCopies; ++i) {
    hid[i] = layer * E + (i % E);
    hsl[i] = i;
  }
  // FFN plan: experts 0..k-1 of the layer for one token, all executed, none filling
  int32_t hf[8] = {k, 0, k, 0, 0, k, 0, 0};
  int32_t huniq[64], hids[64];
  float hw[64];
  for (int j = 0; j < k; ++j) {
    huniq[j] = layer * E + j;
    hids[j] = j;
    hw[j] = 1.0f / (float)k;
  }
  cudaError_t e = cudaMemcpyAsync(i32(L.counts_c), hc, sizeof(hc), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(i32(L.ids_c), hid, sizeof(hid), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(i32(L.slots_c), hsl, sizeof(hsl), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(i32(L.counts_f), hf, sizeof(hf), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(i32(L.uniq), huniq, k * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws + L.fill_ids, 0xff, (size_t)k * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws + L.err, 0, 4, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(i32(L.ids), hids, k * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ws + L.wts, hw, k * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws + L.x, 0, (size_t)spec->hidden * 2, st);
  // the host arrays above are read before this call returns
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "profile setup");

  moe_plan fp{};
  fp.counts = i32(L.counts_c);
  fp.fill_ids = i32(L.ids_c);
  fp.fill_slots = i32(L.slots_c);
  const uint8_t* bank = static_cast<const uint8_t*>(cache->bank);
  float ms_p = 0.0f, ms_h = 0.0f;
  e = time_reps([&] { return moe::launch_fill_copy(fp, kProfCopies, bank, ws + L.copy, se, st); },
                reps, st, &ms_p);
  if (e != cudaSuccess) return cuda_fail(e, "profile fill copy");

  moe::FfnArgs a;
  a.H = spec->hidden;
  a.I = spec->inter;
  a.E = E;
  a.k = k;
  a.layer = layer;
  a.T = 1;
  a.has_shared = 0;
  a.format = spec->format;
  a.blob_bytes = se;
  a.bank = bank;
  a.pool = static_cast<const uint8_t*>(cache->slot_pool);
  a.n_bank = spec->num_layers * E;
  a.n_pool = cache->num_slots;
  a.slot_of_id = cache->slot_of_id;
  a.uniq = i32(L.uniq);
  a.counts = i32(L.counts_f);
  a.fill_ids = i32(L.fill_ids);
  a.err = i32(L.err);
  a.x = reinterpret_cast<const uint16_t*>(ws + L.x);
  a.ids = i32(L.ids);
  a.weights = reinterpret_cast<const float*>(ws + L.wts);
  a.shared = nullptr;
  a.y = reinterpret_cast<float*>(ws + L.y);
  moe::ffn_carve_workspace(a, ws + L.ffn);
  e = time_reps([&] { return moe::launch_ffn_decode(a, st); }, reps, st, &ms_h);
  if (e != cudaSuccess) return cuda_fail(e, "profile FFN");
  int32_t derr = 0;
  e = cudaMemcpy(&derr, ws + L.err, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "profile FFN status");
  if (derr) return fail(MOE_ECUDA, "profile FFN flagged device error bits 0x%x", derr);
  const double bp = (double)kProfCopies * se * reps / (ms_p * 1e-3) / 1e6;
  const double bh = (double)k * se * reps / (ms_h * 1e-3) / 1e6;
  *bp_mbps = (int32_t)(bp < 2e9 ? (bp < 1.0 ? 1.0 : bp) : 2e9);
  *bh_mbps = (int32_t)(bh < 2e9 ? (bh < 1.0 ? 1.0 : bh) : 2e9);
  return ok();
}

// ---------------------------------------------------------------------------
// Prefill entry points.
namespace {

int check_prefill(const moe_spec* s, int32_t T) {
  if (T < 0) return fail(MOE_EINVAL, "T must be >= 0");
  if (s->hidden % 256 || s->inter % 128)
    return fail(MOE_EUNSUPPORTED, "prefill needs hidden %% 256 == 0 and inter %% 128 == 0");
  if (s->num_experts > 1023) return fail(MOE_EUNSUPPORTED, "prefill supports num_experts <= 1023");
  if ((int64_t)T * (s->top_k + 1) > ((int64_t)1 << 30)) return fail(MOE_EINVAL, "T too large");
  return MOE_OK;
}

size_t prefill_ws(const moe_spec* s, int32_t T) {
  return align256((size_t)T * s->num_experts * 4) +
         moe::prefill_workspace_bytes(s->hidden, s->inter, s->num_experts, s->top_k, T);
}

int do_prefill(const moe_spec* spec, const void* experts, const void* x, int32_t T,
               const int32_t* ids, const float* weights, const void* shared, int32_t* err,
               void* ws, size_t ws_bytes, float* y, cudaStream_t st) {
  if (!experts || !x || !ids || !weights || !y || !ws)
    return fail(MOE_EINVAL, "prefill: NULL argument");
  if (spec->has_shared && !shared) return fail(MOE_EINVAL, "spec has a shared expert: pass its blob");
  if (!aligned(experts, 16) || !aligned(x, 16) || !aligned(y, 16) || !aligned(ws, 256) ||
      (shared && !aligned(shared, 16)))
    return fail(MOE_EINVAL, "prefill: experts/x/y/shared need 16 B, workspace 256 B alignment");
  const size_t need = moe::prefill_workspace_bytes(spec->hidden, spec->inter, spec->num_experts,
                                                   spec->top_k, T);
  if (ws_bytes < need) return fail(MOE_ECAPACITY, "workspace %zu < %zu bytes", ws_bytes, need);
  moe::PrefillBufs b{};
  moe::prefill_carve(b, ws, spec->hidden, spec->inter, spec->num_experts, spec->top_k, T);
  moe::GemmArgs a = {};
  a.H = spec->hidden;
  a.I = spec->inter;
  a.E = spec->num_experts;
  a.k = spec->top_k;
  a.T = T;
  a.format = spec->format;
  a.blob_bytes = moe::expert_blob_bytes(a.H, a.I, a.format);
  a.experts = static_cast<const uint8_t*>(experts);
  a.shared = static_cast<const uint8_t*>(shared);
  a.weights = weights;
  a.err = err;
  cudaError_t e = moe::launch_prefill_ffn(a, b, static_cast<const uint16_t*>(x), ids,
                                          spec->has_shared, y, st);
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return MOE_OK;
}

}  // namespace

extern "C" size_t moe_prefill_workspace_bytes(const moe_spec* spec, int32_t T) {
  if (check_spec(spec) != MOE_OK || T < 1 || check_prefill(spec, T) != MOE_OK) return 0;
  return prefill_ws(spec, T);
}

extern "C" int moe_layer_prefetch(const moe_spec* spec, const void* bank, int32_t layer,
                                  void* dst, moe_stream_t stream) {
  int rc = check_spec(spec);
  if (rc) return rc;
  if (layer < 0 || layer >= spec->num_layers) return fail(MOE_EINVAL, "layer out of range");
  if (!bank || !dst) return fail(MOE_EINVAL, "moe_layer_prefetch: NULL argument");
  const size_t se = (size_t)moe::expert_blob_bytes(spec->hidden, spec->inter, spec->format);
  const size_t bytes = se * spec->num_experts;
  const uint8_t* src = static_cast<const uint8_t*>(bank) + (size_t)layer * bytes;
  cudaError_t e = moe::launch_layer_copy(src, dst, bytes, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "layer copy");
  return ok();
}

extern "C" int moe_expert_ffn_prefill(const moe_spec* spec, const void* layer_experts,
                                      const void* x, int32_t T, const int32_t* ids,
                                      const float* weights, const void* shared, int32_t* err,
                                      void* workspace, size_t workspace_bytes, float* y,
                                      moe_stream_t stream) {
  int rc = check_spec(spec);
  if (rc) return rc;
  rc = check_prefill(spec, T);
  if (rc) return rc;
  if (T == 0) return ok();
  rc = do_prefill(spec, layer_experts, x, T, ids, weights, shared, err, workspace,
                  workspace_bytes, y, (cudaStream_t)stream);
  return rc ? rc : ok();
}

extern "C" int moe_layer_forward_prefill(const moe_spec* spec, const void* layer_experts,
                                         const void* x, int32_t T, const void* w_router,
                                         const float* bias, const void* shared, int32_t* ids,
                                         float* weights, int32_t* err, void* workspace,
                                         size_t workspace_bytes, float* y, moe_stream_t stream) {
  int rc = check_spec(spec);
  if (rc) return rc;
  rc = check_prefill(spec, T);
  if (rc) return rc;
  if (T == 0) return ok();
  if (!workspace || !aligned(workspace, 256))
    return fail(MOE_EINVAL, "workspace must be 256-B aligned");
  if (workspace_bytes < prefill_ws(spec, T))
    return fail(MOE_ECAPACITY, "workspace %zu < %zu bytes", workspace_bytes, prefill_ws(spec, T));
  cudaStream_t st = (cudaStream_t)stream;
  float* logits = static_cast<float*>(workspace);
  const size_t lb = align256((size_t)T * spec->num_experts * 4);
  rc = do_route(spec, x, T, w_router, bias, logits, ids, weights, st);
  if (rc) return rc;
  rc = do_prefill(spec, layer_experts, x, T, ids, weights, shared, err,
                  static_cast<uint8_t*>(workspace) + lb, workspace_bytes - lb, y, st);
  return rc ? rc : ok();
}

// ---------------------------------------------------------------------------
// moe_expert_ffn_noalloc: the decode FFN with its scratch in a file-scope
// device array instead of a caller workspace, for callers that may not
// allocate device memory.  The array's device address is looked up once per
// device (host code cannot use the symbol itself as a device pointer).
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kNoAllocMaxDevices = 64;
// The array's device address per device, looked up on first use.  Atomic:
// host threads may make their first call concurrently (each stores the same
// address).  A device reset reloads the module and invalidates the address;
// moe.h asks callers not to use this entry point across a reset.
std::atomic<void*> g_noalloc_ptr[kNoAllocMaxDevices];

int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kNoAllocMaxDevices)
    return fail(MOE_EUNSUPPORTED, "device ordinal %d >= %d", dev, kNoAllocMaxDevices);
  void* p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    g_noalloc_ptr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return MOE_OK;
}

}  // namespace

extern "C" int moe_expert_ffn_noalloc(const moe_spec* spec, const moe_cache* cache,
                                      int32_t layer, const moe_plan* plan, const void* x,
                                      int32_t T, const int32_t* ids, const float* weights,
                                      const void* shared, float* y, moe_stream_t stream) {
  int rc = check_spec(spec);
  if (rc) return rc;
  rc = check_cache(spec, cache, true);
  if (rc) return rc;
  rc = check_step_args(spec, layer, T);
  if (rc) return rc;
  if (T == 0) return ok();
  rc = check_plan(plan, T * spec->top_k);
  if (rc) return rc;
  if (T > moe::kMaxDecodeT)
    return fail(MOE_EUNSUPPORTED, "decode FFN supports T <= %d", moe::kMaxDecodeT);
  const size_t need = moe::ffn_workspace_bytes(spec->hidden, spec->inter, spec->top_k, T,
                                               spec->has_shared);
  if (need > MOE_NOALLOC_SCRATCH_BYTES)
    return fail(MOE_ECAPACITY,
                "moe_expert_ffn_noalloc: this size needs %zu scratch bytes, the built-in "
                "array holds %zu; use moe_expert_ffn with a workspace",
                need, (size_t)MOE_NOALLOC_SCRATCH_BYTES);
  void* ws = nullptr;
  rc = noalloc_scratch(&ws);
  if (rc) return rc;
  rc = do_ffn(spec, cache, layer, plan, x, T, ids, weights, shared, ws,
              (size_t)MOE_NOALLOC_SCRATCH_BYTES, y, (cudaStream_t)stream);
  return rc ? rc : ok();
}

