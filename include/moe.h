/*
 * moe.h -- C ABI of libmoe.so, the GB300 (sm_103a) MoE expert step.
 *
 * One MoE layer step, entirely on one GPU:
 *   moe_route          router scoring: softmax-top-k or sigmoid-group
 *                      (Edge0 §2 "MoE routing")
 *   moe_cache_step     device control step: dedup of the routed ids lE+e, hit /
 *                      miss against the shared slot table, q* split of the
 *                      misses into a fill set F and a direct set C, single-pass
 *                      choice of K LRU victims, table update, and the fill
 *                      copies bank -> slot pool (FreeToken summary "core
 *                      method", "method steps", "novelty"; FreeToken reader
 *                      "Semantic-Aware Expert Caching", "Elastic Memory
 *                      Management")
 *   moe_cache_place    setup: preload a chosen expert set (static placement
 *                      or warm start); moe_cache.policy picks the shared LRU,
 *                      a per-layer LRU or static placement (the replacement
 *                      policies the pages compare)
 *   moe_cache_resize   elastic re-division of the slot pool at a safe point
 *                      between steps; moe_slots_for_budget gives the slot
 *                      count of a memory budget (FreeToken reader "Elastic
 *                      Memory Management")
 *   moe_expert_ffn     int4 affine group-64 SwiGLU experts down(silu(gate(x)) *
 *                      up(x)) over G = H u F (H from the slot pool; F, the
 *                      experts filled in this step, from their bank bytes,
 *                      identical to the slot copy) and over C read in place
 *                      from the bank, combined with the routing
 *                      weights (Edge0 §3.1 "math convention"; FreeToken summary
 *                      "core method": exact merge of the partial sums)
 *   moe_layer_forward  the three above in stream order
 * plus the prefill path (whole-layer copy and grouped GEMM; FreeToken summary
 * "method steps", reader "System Architecture" ping-pong buffers).
 *
 * Conventions shared by every entry point
 *   Memory   Every pointer named *device* must point to device memory that
 *            the caller owns (for instance a torch tensor's data_ptr()).  The
 *            library never allocates, frees or keeps a pointer after a call
 *            returns; scratch space is passed in as `workspace`.
 *   Streams  Every call is asynchronous on `stream` (a cudaStream_t; NULL is
 *            the legacy default stream).  No call synchronises the host, and
 *            all device-side sizes ("valid counts") live in device memory,
 *            so every call can be captured in a CUDA graph.  The exceptions
 *            are the setup-time calls moe_cache_place and
 *            moe_profile_bandwidths, which synchronise `stream`.
 *   Errors   Every int-returning call returns MOE_OK or a negative code.
 *            Arguments are validated on the host before anything is launched;
 *            on failure nothing is launched and moe_last_error() describes the
 *            problem (a thread-local string).  Nothing aborts or traps.
 *            Problems that only the device can see (a routed id outside
 *            [0, E)) set a bit in plan->err and the offending entry is skipped.
 *   Layout   Expert blob (one per (layer, expert); bank index l*E + e;
 *            size moe_expert_bytes, a multiple of 256 bytes):
 *              Wg codes [I][H/2] | Wu codes [I][H/2] | Wd codes [H][I/2]   (u8,
 *              two int4 codes per byte, the low nibble is the even column)
 *              Wg scale [I][H/64] | Wg bias [I][H/64] | Wu scale | Wu bias |
 *              Wd scale [H][I/64] | Wd bias [H][I/64]                      (bf16)
 *            Weight w = scale * q + bias with q in 0..15 (Edge0 §2
 *            "Quantisation": int4 affine, group 64, scale and bias).
 *            Hidden states x are bf16 [T][H] row-major; router weights bf16
 *            [E][H]; outputs fp32.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

enum {
  MOE_OK = 0,
  MOE_EINVAL = -1,       /* bad argument (null pointer, bad size, misalignment) */
  MOE_ECUDA = -2,        /* a CUDA runtime call failed (launch error, ...) */
  MOE_EUNSUPPORTED = -3, /* valid but not supported by this build */
  MOE_ECAPACITY = -4,    /* a buffer (plan, workspace) is too small */
  MOE_ETIMEOUT = -5      /* a bounded device wait gave up */
};

enum { MOE_ROUTER_SOFTMAX_TOPK = 0, MOE_ROUTER_SIGMOID_GROUP = 1 };

/* Expert weight formats (moe_spec.format).  The pages' deployed models keep
 * their experts in NVFP4 (Qwen3.6, GLM-5.2) or MXFP4 (DeepSeek-V4-Flash)
 * (FreeToken summary "Key results" table); Edge0 §2 "Quantisation" uses int4
 * affine.  FP4 elements are E2M1 (1 sign, 2 exponent, 1 mantissa bit, bias 1)
 * with one scale per block of a row: MXFP4 blocks of 32 with an E8M0 scale
 * 2^(e - 127); NVFP4 blocks of 16 with an FP8 E4M3 scale times one fp32 scale
 * per matrix.  FP4 blob layout (moe_expert_bytes):
 *   Wg codes [I][H/2] | Wu codes [I][H/2] | Wd codes [H][I/2]   (low nibble =
 *   even column) | Wg scales [I][H/B] | Wu scales [I][H/B] | Wd scales [H][I/B]
 *   (one byte per block) | NVFP4: fp32 matrix scales of Wg, Wu, Wd
 * rounded up to 256 bytes.  FP4 experts run in the decode FFN where its
 * one-kernel form serves the shape (hidden % 1024 == 0, inter % 512 == 0,
 * T <= 8); MXFP4 block scales must lie in 2^-32 .. 2^7 (E8M0 bytes 95..134:
 * smaller ones contribute 0, larger ones overflow).  Prefill takes all three
 * formats: FP4 weights are dequantised exactly to bf16 (E2M1 times the block
 * scale) for the tensor-core GEMMs, with no limit on the MXFP4 scales beyond
 * bf16's own range. */
enum { MOE_FORMAT_INT4 = 0, MOE_FORMAT_MXFP4 = 1, MOE_FORMAT_NVFP4 = 2 };

/* Device-side error bits written to plan->err[0] (OR-ed, never cleared by the
 * library; the caller may zero it).  MOE_DERR_RANGE: checked builds only
 * (libmoe_checked.so, compiled with -DMOE_CHECKED): a cache-table entry read
 * on the device lay outside its range and was treated as absent. */
enum { MOE_DERR_BAD_ID = 1, MOE_DERR_WAIT = 2, MOE_DERR_RANGE = 4 };

/* Model description (Edge0 §3 "MoESpec": expert count, routing family,
 * quantisation, layout). */
typedef struct moe_spec {
  int32_t num_layers;   /* L */
  int32_t hidden;       /* H, multiple of 64 (the router needs a multiple of 8) */
  int32_t inter;        /* I, expert intermediate size, multiple of 64 */
  int32_t num_experts;  /* E routed experts per layer, 1..1024 */
  int32_t top_k;        /* k experts per token, 1..min(E, 64) */
  int32_t router;       /* MOE_ROUTER_* */
  int32_t n_groups;     /* sigmoid-group: expert groups (E % n_groups == 0) */
  int32_t topk_groups;  /* sigmoid-group: groups kept per token */
  float routed_scale;   /* sigmoid-group: factor applied after renormalising */
  int32_t group_size;   /* int4 quantisation group, must be 64 (FP4 formats fix their own) */
  int32_t has_shared;   /* 1: an always-on shared expert, added with weight 1 */
  int32_t shared_inter; /* its intermediate size (must equal inter) */
  int32_t format;       /* MOE_FORMAT_*: expert weight format (0: int4 affine) */
} moe_spec;

/* Replacement policy of a slot cache (moe_cache.policy).  FreeToken's own
 * policy is the shared LRU (summary "core method"); the other two are the
 * placements its miss-rate comparison replays on the same routing traces
 * (summary "Key results"; reader Figure 4(b)) and Edge0's per-layer "hot"
 * resident set (Edge0 §3.1 "executor paths").
 *   MOE_POLICY_SHARED_LRU  one LRU over all S slots, all layers
 *   MOE_POLICY_LAYER_LRU   layer l owns slots [l*S_l, (l+1)*S_l) with
 *                          S_l = floor(S / L) and runs its own LRU there;
 *                          the S - L*S_l slots past the last range are unused
 *   MOE_POLICY_STATIC      the slots hold what moe_cache_place put there; a
 *                          step never fills (q = 0: every miss goes to C) */
enum { MOE_POLICY_SHARED_LRU = 0, MOE_POLICY_LAYER_LRU = 1, MOE_POLICY_STATIC = 2 };

/* The shared expert slot cache (FreeToken summary "core method": one pool
 * for all MoE layers, one slot per (layer, expert) pair).  The struct itself
 * lives on the host; the tables live on the device. */
typedef struct moe_cache {
  int32_t num_slots;   /* S >= 1 */
  int32_t k_victims;   /* K, victims chosen per step, 1..32 */
  int32_t bp_mbps;     /* B_P: fill bandwidth, MB/s (e.g. 52700) */
  int32_t bh_mbps;     /* B_H: direct-execute bandwidth, MB/s (e.g. 77300) */
  int32_t* slot_of_id; /* device [L*E]: slot holding id, or -1 */
  int32_t* id_of_slot; /* device [S]: id held by slot, or -1 */
  uint32_t* ts;        /* device [S]: last step the router selected it; 0 = empty */
  uint32_t* clock;     /* device [1]: step counter, advanced once per cache step */
  void* slot_pool;     /* device [S * S_e] bytes, 16-byte aligned */
  const void* bank;    /* device [L * E * S_e] bytes, 16-byte aligned */
  int32_t policy;      /* MOE_POLICY_*; MOE_POLICY_LAYER_LRU needs S >= L */
  uint32_t* sync;      /* device [MOE_CACHE_SYNC_WORDS] or NULL: words the one-kernel decode
                          layer step (moe_layer_forward) uses to coordinate its CTAs.  They
                          must be zero before the first step: moe_cache_reset and
                          moe_cache_place clear them, and every step leaves them zero.  With
                          NULL, moe_layer_forward runs its multi-kernel form. */
} moe_cache;

/* Words behind moe_cache.sync (16 KB; 4-byte aligned). */
#define MOE_CACHE_SYNC_WORDS 4096

/* Fixed-shape step buffers with device-side valid counts (FreeToken summary
 * "novelty": routing-dependent control kept as data).  All device pointers,
 * each list `capacity` entries long except victims (k_victims entries). */
typedef struct moe_plan {
  int32_t capacity;     /* >= T * top_k of the call */
  int32_t* uniq;        /* ascending unique ids l*E+e routed this step */
  int32_t* hit_ids;     /* H: resident ids (ascending) */
  int32_t* hit_slots;   /*    and their slots */
  int32_t* fill_ids;    /* F: misses copied into the cache (ascending) */
  int32_t* fill_slots;  /*    and the victim slots they went to */
  int32_t* evicted_ids; /*    id previously held by that slot, or -1 */
  int32_t* direct_ids;  /* C: misses executed in place from the bank */
  int32_t* victims;     /* the K victims in (ts, slot) order; -1 = none */
  int32_t* counts;      /* [8]: n_uniq n_hit n_miss q n_fill n_direct n_victims now */
  int32_t* err;         /* [1]: MOE_DERR_* bits */
} moe_plan;

/* Last error message of this thread ("" if none).  Never NULL. */
const char* moe_last_error(void);

/* Library version string. */
const char* moe_version(void);

/* Bytes of one expert blob for (hidden, inter): 3HI/2 + 3HI/64 * 4 rounded up
 * to 256 (Edge0 §3.1 "problem": 1.77 MB per expert at H=2048, I=512).
 * Returns 0 for an invalid spec. */
size_t moe_expert_bytes(const moe_spec* spec);

/* ------------------------------------------------------------------------
 * moe_route -- router scoring (Edge0 §2 "MoE routing").
 *   x          device bf16 [T][H]
 *   w_router   device bf16 [E][H]
 *   bias       device fp32 [E] or NULL (sigmoid-group only: added to the
 *              sigmoid scores for selection, never to the weights)
 *   logits     device fp32 [T][E] out: l = x . W_r^T, fp32, fixed summation
 *              order (8-element chunks, chunk c to lane c mod 32, lanes
 *              combined by an xor butterfly 16, 8, 4, 2, 1)
 *   ids        device int32 [T][k] out: expert index e in rank order
 *   weights    device fp32 [T][k] out
 * softmax-top-k : top k logits (ties: lower index), w = exp(l - lmax) / sum,
 *                 sum over the k in rank order.
 * sigmoid-group : s = sigmoid(l), sel = s + bias; groups ranked by the sum of
 *                 their two largest sel; top `topk_groups` groups kept; top k
 *                 sel inside them; w = s / sum(s) * routed_scale.
 * exp is the library's own (Cody-Waite reduction, degree-7 Taylor, exact
 * 2^n scaling) so routing is bit-reproducible against a CPU restatement.
 * T >= 0 (T == 0 launches nothing).
 * ------------------------------------------------------------------------ */
int moe_route(const moe_spec* spec, const void* x, int32_t T, const void* w_router,
              const float* bias, float* logits, int32_t* ids, float* weights,
              moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_cache_reset -- empty the cache: slot_of_id[*] = -1, id_of_slot[*] = -1,
 * ts[*] = 0, clock = 0.
 * ------------------------------------------------------------------------ */
int moe_cache_reset(const moe_spec* spec, moe_cache* cache, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_cache_place -- empty the cache, then preload a chosen set of experts:
 * the static placements of the pages' baselines (hot experts pinned at load
 * time; whole layers assigned to the GPU), or a warm start for an LRU.
 *   ids      HOST int32 [n]: bank ids l*E + e, distinct, in [0, L*E)
 *   n        0 <= n; n <= S (policy LAYER_LRU: ids of one layer <= S_l)
 * ids[i] goes to slot i (SHARED_LRU, STATIC) or, for LAYER_LRU, to slot
 * l*S_l + (number of ids of layer l before it in the list); every other slot
 * is emptied; ts = 0 everywhere (placed, not yet used); clock = 0.  When the
 * cache has a slot pool and bank, each placed blob is copied bank -> slot.
 * The list is checked on the host before anything is written (MOE_EINVAL
 * leaves the cache untouched).  Synchronises `stream` before it returns
 * (the tables are staged from host memory); not capturable.
 * ------------------------------------------------------------------------ */
int moe_cache_place(const moe_spec* spec, moe_cache* cache, const int32_t* ids, int32_t n,
                    moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_slots_for_budget -- slots of moe_expert_bytes(spec) that `free_bytes`
 * of device memory hold: floor(free_bytes / S_e) (FreeToken reader "Elastic
 * Memory Management": 10 slots of 0.5 GB in 5 GB, 8 in 4 GB, 12 in 6 GB).
 * Returns -1 for an invalid spec or free_bytes < 0.
 * ------------------------------------------------------------------------ */
int64_t moe_slots_for_budget(const moe_spec* spec, int64_t free_bytes);

/* Scratch bytes moe_cache_resize needs to go from cache->num_slots to
 * new_slots slots: 4 * (8 + 3 * max(S, new_slots)).  0 for a NULL cache or
 * new_slots < 1. */
size_t moe_cache_resize_workspace_bytes(const moe_cache* cache, int32_t new_slots);

/* ------------------------------------------------------------------------
 * moe_cache_resize -- re-divide the shared slot pool from S = cache->num_slots
 * to new_slots slots at a safe point between steps (FreeToken reader "Elastic
 * Memory Management": the excess slots are evicted when the budget shrinks,
 * new slots appear when it grows; the bank and the routing never change, so
 * every later output is what it would have been with the same resident set).
 *   Shrink: while more than new_slots slots are occupied, the occupied slot
 *     with the smallest key (ts, slot) is evicted (the order of the victim
 *     scan: the least recently routed expert goes first); then the kept
 *     experts in slots >= new_slots move, blob and ts, to the free slots below
 *     new_slots, both taken in ascending slot order.
 *   Growth: slots [S, new_slots) start empty (id -1, ts 0); nothing moves.
 *   Slots from min(S, new_slots) to max(S, new_slots) are left empty, and the
 *   clock does not move.
 * The caller guarantees that id_of_slot, ts and (if set) slot_pool hold
 * max(S, new_slots) entries.  Policy MOE_POLICY_SHARED_LRU only
 * (MOE_EUNSUPPORTED otherwise).  On success cache->num_slots = new_slots.
 *   workspace  device, 4-byte aligned, >= moe_cache_resize_workspace_bytes:
 *              int32 [0] evicted count, [1] moved count, [2] occupied slots
 *              after, [3] MOE_DERR_RANGE if the tables were not a bijection
 *              (then the tables are unchanged while cache->num_slots is
 *              new_slots: moe_cache_reset or moe_cache_place the cache before
 *              its next step); from word 8: the move sources, the move
 *              destinations and the evicted ids (ascending slot order),
 *              max(S, new_slots) words each.
 * No step of this cache may run concurrently (a safe point); asynchronous on
 * `stream`, two kernels (one for a growth or a cache without a pool).
 * ------------------------------------------------------------------------ */
int moe_cache_resize(const moe_spec* spec, moe_cache* cache, int32_t new_slots, void* workspace,
                     size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_cache_step -- one decode control step for layer `layer` (one CTA),
 * then (do_fill != 0) the fill copies bank[F_i] -> slot_pool[victim_i].
 *   ids      device int32 [T][k]: routed expert indices of this layer
 *   plan     capacity >= T*k; written with the step's sets and counts
 * Steps (FreeToken summary "method steps"; reader "Semantic-Aware Expert
 * Caching", "Elastic Memory Management"):
 *   now = ++clock; U = sorted unique {layer*E + id}; H = ids of U with a slot,
 *   their ts = now; M = U \ H ascending, m = |M|;
 *   q = m if B_H <= B_P else floor((2*m*B_P + B_H) / (2*B_H))  (round half up
 *   of m*B_P/B_H); victims = the K smallest (ts, slot) over slots with
 *   ts != now, in one pass; n_fill = min(q, K, #victims); F = M[:n_fill] into
 *   victims[:n_fill] (old ids evicted, ts = now); C = M[n_fill:] (not cached).
 * Policy: LAYER_LRU takes victims from layer's own slot range only; STATIC
 *   sets q = 0 (victims are still listed, nothing is filled).
 * Requires T*k <= 1024 and T*k <= plan->capacity (else MOE_ECAPACITY).
 * With do_fill == 0 only the tables change (trace replay).
 * ------------------------------------------------------------------------ */
int moe_cache_step(const moe_spec* spec, moe_cache* cache, int32_t layer, const int32_t* ids,
                   int32_t T, moe_plan* plan, int32_t do_fill, moe_stream_t stream);

/* Scratch bytes moe_expert_ffn needs for T tokens (0 for an invalid spec). */
size_t moe_ffn_workspace_bytes(const moe_spec* spec, int32_t T);

/* ------------------------------------------------------------------------
 * moe_expert_ffn -- decode expert FFN and combine (T <= 64).
 *   Executes every id in plan->uniq (H from its slot; F and C in place from
 *   the bank: an id cached before this step is read from the slot pool, an id
 *   in plan->fill_ids or without a slot from the bank, so the FFN does not
 *   depend on the fill copies) plus the shared expert:
 *     y[t] = sum_j weights[t][j] * expert(ids[t][j])(x[t]) + shared(x[t])
 *   expert(x) = Wd (silu(Wg x) * (Wu x)), dequantised int4, fp32 accumulate.
 *   The routed terms are added in rank order j, then the shared term.
 *   x        device bf16 [T][H];  ids, weights as written by moe_route
 *   shared   device blob of the shared expert, or NULL (needs has_shared)
 *   workspace device, >= moe_ffn_workspace_bytes(spec, T), 256-byte aligned
 *   y        device fp32 [T][H] out
 * ------------------------------------------------------------------------ */
int moe_expert_ffn(const moe_spec* spec, const moe_cache* cache, int32_t layer,
                   const moe_plan* plan, const void* x, int32_t T, const int32_t* ids,
                   const float* weights, const void* shared, void* workspace,
                   size_t workspace_bytes, float* y, moe_stream_t stream);

/* Scratch bytes moe_layer_forward needs for T tokens. */
size_t moe_layer_workspace_bytes(const moe_spec* spec, int32_t T);

/* ------------------------------------------------------------------------
 * moe_layer_forward -- moe_route, moe_cache_step (with fill) and
 * moe_expert_ffn for one decode layer, no host sync.
 *   ids, weights  device out [T][k] (the routing decision, kept for the caller)
 *   workspace     >= moe_layer_workspace_bytes(spec, T)
 * One kernel: when `cache->sync` is set and the shape allows it (the
 * cooperative FFN's shape: hidden % 1024 == 0, inter % 512 == 0, T <= 8; and
 * T*k <= 32, k_victims <= 8, num_experts <= 256), the whole step -- router
 * logits, selection, control step, FFN and fills -- is one cooperative kernel
 * (moe_layer_kernel_count == 1); it uses the cache's sync words and leaves
 * them zero.  Otherwise the step is a chain of kernels.
 * The fill copies (bank -> slot of every F expert): when a decode FFN kernel
 * carries them (the cooperative kernel; the streaming kernels for hidden %
 * 512 == 0, inter % 256 == 0, T <= 8, T*k + shared <= 128), it writes each F
 * expert's bytes into its slot as it reads them from the bank (FreeToken
 * summary "method steps": the miss path fills the slot), so no separate copy
 * runs.  Otherwise a copy kernel runs beside the FFN on a stream owned by the
 * library and `stream` waits for it before any later work.  Either way
 * everything the call enqueues is complete, in order, from the caller's
 * stream's view (also when the stream is being captured into a graph), and
 * the slot contents are the same.
 * ------------------------------------------------------------------------ */
int moe_layer_forward(const moe_spec* spec, moe_cache* cache, int32_t layer, const void* x,
                      int32_t T, const void* w_router, const float* bias, const void* shared,
                      moe_plan* plan, int32_t* ids, float* weights, void* workspace,
                      size_t workspace_bytes, float* y, moe_stream_t stream);

/* Test hook for failure detection without a GPU fault.  With on != 0 the
 * next decode FFN call of this process (moe_expert_ffn or moe_layer_forward,
 * on a shape the cooperative or streaming kernels serve) issues no weight
 * copies: the kernel's warps find their stages never filled, give up after
 * their bounded wait (2^31 SM clock cycles after 1024 polling rounds, about a
 * second at full clock), set MOE_DERR_WAIT in plan->err and return; y of that
 * call is undefined.  When the call carried the step's fills (moe_layer_forward)
 * the experts it filled are unmapped again (slot_of_id = -1, the slot empty,
 * ts 0), so the cache never maps a partly written slot.  The flag is cleared
 * by that call (or by on == 0); the device context stays usable and the next
 * call runs normally.  Any bounded wait that runs out for another reason has
 * the same effect.  Returns MOE_OK. */
int moe_debug_inject_ffn_stall(int32_t on);

/* Kernels one moe_layer_forward call on `cache` launches for T tokens (for
 * graph sizing and launch accounting); 0 for an invalid spec, a NULL cache or
 * T outside 1..64. */
int32_t moe_layer_kernel_count(const moe_spec* spec, const moe_cache* cache, int32_t T);

/* ------------------------------------------------------------------------
 * Prefill (FreeToken summary "method steps": the GPU computes layer l from
 * one whole-layer buffer while the next layer is copied into the other; the
 * reader's "System Architecture" ping-pong buffers).  In prefill the routing
 * union covers nearly every expert, so the experts run as grouped GEMMs on
 * the tensor cores instead of through the slot cache.
 * Requires hidden % 256 == 0, inter % 128 == 0, num_experts <= 1023.
 * ------------------------------------------------------------------------ */

/* Scratch bytes moe_expert_ffn_prefill / moe_layer_forward_prefill need. */
size_t moe_prefill_workspace_bytes(const moe_spec* spec, int32_t T);

/* Copy the E expert blobs of `layer` (E * S_e bytes, contiguous in the bank)
 * into `dst` (device) on `stream`: the whole-layer fill of the double buffer.
 * Issue it on a second stream to overlap another layer's compute.  With bank
 * and dst 16-byte aligned the copy is one kernel of one 256-thread CTA per SM
 * (streaming loads and stores, no shared memory), small enough to share each
 * SM with the routing kernels of moe_route / moe_layer_forward_prefill, which
 * is where it overlaps best; otherwise it is a cudaMemcpyAsync.
 * MOE_EINVAL for a NULL pointer or a layer out of range. */
int moe_layer_prefetch(const moe_spec* spec, const void* bank, int32_t layer, void* dst,
                       moe_stream_t stream);

/* Prefill expert FFN + combine for T tokens (T >= 1).
 *   layer_experts  device, the E blobs of this layer (bank slice or a buffer
 *                  filled by moe_layer_prefetch)
 *   x              device bf16 [T][H];  ids int32 [T][k], weights fp32 [T][k]
 *   shared         shared expert blob or NULL (needs has_shared)
 *   err            device int32 [1] or NULL: MOE_DERR_* bits are OR-ed in
 *   y              device fp32 [T][H] out:  sum_j w[t][j] expert_{ids[t][j]}(x[t])
 *                  + shared(x[t]); each routed term is rounded to bf16 before
 *                  the fixed-order fp32 sum; h is bf16.
 * Steps: stable counting sort of the T*k assignments by expert, grouped GEMM
 * gate/up with SwiGLU, grouped GEMM down with the routing weight, combine. */
int moe_expert_ffn_prefill(const moe_spec* spec, const void* layer_experts, const void* x,
                           int32_t T, const int32_t* ids, const float* weights,
                           const void* shared, int32_t* err, void* workspace,
                           size_t workspace_bytes, float* y, moe_stream_t stream);

/* moe_route + moe_expert_ffn_prefill for one layer (ids / weights are outputs). */
int moe_layer_forward_prefill(const moe_spec* spec, const void* layer_experts, const void* x,
                              int32_t T, const void* w_router, const float* bias,
                              const void* shared, int32_t* ids, float* weights, int32_t* err,
                              void* workspace, size_t workspace_bytes, float* y,
                              moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_expert_ffn_noalloc -- moe_expert_ffn for callers that cannot allocate
 * device memory.  No counterpart on the pages: this is a library addition.
 *
 * Some callers of the decode FFN cannot call cudaMalloc or any allocating
 * routine: code that runs inside a host application's fixed device-memory
 * budget (an inference server or game engine whose pools own all device
 * memory), real-time loops that forbid allocation on the token path, and
 * plugins that are handed only input and output buffers.  For them this entry
 * point takes the same inputs and output as moe_expert_ffn but no workspace:
 * its scratch is one file-scope device array of MOE_NOALLOC_SCRATCH_BYTES
 * inside libmoe.so, which every GPU that loads the library holds until the
 * process exits.
 *   - Sizes whose scratch need (moe_ffn_workspace_bytes(spec, T)) exceeds
 *     MOE_NOALLOC_SCRATCH_BYTES are rejected with MOE_ECAPACITY.
 *   - The first call on a device looks up the array's device address for the
 *     current device (cudaGetSymbolAddress) and keeps it; make that first call
 *     before any stream capture.  A device reset (cudaDeviceReset) reloads the
 *     library's device code and invalidates the kept address: do not use this
 *     entry point on a device after resetting it.
 *   - All calls share the one array, which keeps the last call's contents
 *     (the arrival counters are cleared by every call).  Calls whose
 *     execution overlaps on the GPU (different streams, or different host
 *     threads) race on it and must not be issued; order them on one stream.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 * Results equal moe_expert_ffn's for the same inputs.
 * ------------------------------------------------------------------------ */
#define MOE_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
int moe_expert_ffn_noalloc(const moe_spec* spec, const moe_cache* cache, int32_t layer,
                           const moe_plan* plan, const void* x, int32_t T, const int32_t* ids,
                           const float* weights, const void* shared, float* y,
                           moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_profile_bandwidths -- measure B_P and B_H on this device
 * (FreeToken summary "method steps": B_P and B_H are measured on the deployed
 * machine before q* is used; "weaknesses": they drift, so they should be
 * re-measured rather than read once from a specification sheet).
 *   B_P: expert blobs copied from the bank by the library's fill copy (the
 *        same kernel as the step's fills), into scratch inside `workspace`,
 *        never into the slot pool.  Rate = blob bytes moved per second.
 *   B_H: the decode expert FFN (T = 1, the spec's top_k experts 0..k-1 of
 *        `layer`, no shared expert) executed where the cache tables place
 *        those experts (slot if resident, else in place from the bank).
 *        Rate = expert weight bytes executed per second.
 * Both are returned in MB/s (1 MB = 10^6 bytes), the units of
 * moe_cache.bp_mbps / bh_mbps, so the result can be stored there directly.
 *   cache          tables and bank are read, nothing is written (tables,
 *                  recency stamps, clock and slot pool are left unchanged)
 *   layer          0 <= layer < num_layers
 *   workspace      device, >= moe_profile_workspace_bytes(spec), 256-B aligned;
 *                  its contents are overwritten
 *   reps           >= 1 timed repetitions of each measurement (after 2 warm-up)
 *   bp_mbps, bh_mbps  host out-pointers
 * Unlike the step entry points this call synchronises the stream (it reads
 * CUDA event timings) and creates and destroys two CUDA events; it must not
 * be called during stream capture.
 * ------------------------------------------------------------------------ */
size_t moe_profile_workspace_bytes(const moe_spec* spec);
int moe_profile_bandwidths(const moe_spec* spec, const moe_cache* cache, int32_t layer,
                           void* workspace, size_t workspace_bytes, int32_t reps,
                           int32_t* bp_mbps, int32_t* bh_mbps, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
