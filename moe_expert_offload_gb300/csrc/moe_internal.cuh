// Internal declarations of libmoe (not part of the C ABI).
#pragma once

#include <cuda.h>  // CUtensorMap and its enums (types only)
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kGroup = 64;
constexpr int kMaxRouted = 1024;  // T*k limit of the single-CTA control step
constexpr int kMaxVictims = 32;
constexpr int kMaxDecodeT = 64;
constexpr int kMaxExperts = 1024;

// Byte offsets of the nine sections of an expert blob.
struct BlobOffsets {
  int64_t gq, uq, dq, gs, gb, us, ub, ds, db, total;
};

__host__ __device__ inline BlobOffsets blob_offsets(int64_t H, int64_t I) {
  BlobOffsets o;
  const int64_t cgu = I * H / 2, cd = H * I / 2;
  const int64_t sgu = I * (H / kGroup) * 2, sd = H * (I / kGroup) * 2;
  o.gq = 0;
  o.uq = cgu;
  o.dq = 2 * cgu;
  o.gs = o.dq + cd;
  o.gb = o.gs + sgu;
  o.us = o.gb + sgu;
  o.ub = o.us + sgu;
  o.ds = o.ub + sgu;
  o.db = o.ds + sd;
  o.total = ((o.db + sd) + 255) / 256 * 256;
  return o;
}

// FP4 expert blob (MOE_FORMAT_MXFP4 / NVFP4): E2M1 codes laid out as the
// int4 codes, then one scale byte per block of each matrix, then (NVFP4) the
// three fp32 matrix scales; the total rounded up to 256 bytes.
struct Fp4Offsets {
  int64_t gq, uq, dq, gs, us, ds, mat, total;
  int block;  // elements per scale: 32 (MXFP4) or 16 (NVFP4)
};

__host__ __device__ inline Fp4Offsets fp4_offsets(int64_t H, int64_t I, int format) {
  Fp4Offsets o;
  o.block = format == MOE_FORMAT_NVFP4 ? 16 : 32;
  const int64_t hi = H * I;
  o.gq = 0;
  o.uq = hi / 2;
  o.dq = hi;
  o.gs = hi / 2 * 3;
  o.us = o.gs + hi / o.block;
  o.ds = o.us + hi / o.block;
  o.mat = o.ds + hi / o.block;
  o.total = (o.mat + (format == MOE_FORMAT_NVFP4 ? 12 : 0) + 255) / 256 * 256;
  return o;
}

// Bytes of one expert blob of the given format.
inline int64_t expert_blob_bytes(int64_t H, int64_t I, int format) {
  return format == MOE_FORMAT_INT4 ? blob_offsets(H, I).total : fp4_offsets(H, I, format).total;
}

// Checked builds (-DMOE_CHECKED): cache-table entries read on the device are
// range-checked before they index anything; an entry outside its range ORs
// MOE_DERR_RANGE into the error word and is treated as absent.  In normal
// builds the check compiles away.
__device__ __forceinline__ bool checked_ok(bool in_range, int32_t* err) {
#ifdef MOE_CHECKED
  if (!in_range) {
    if (err) atomicOr(err, MOE_DERR_RANGE);
    return false;
  }
#else
  (void)in_range;
  (void)err;
#endif
  return true;
}

// Programmatic dependent launch (the decode layer path).  A kernel launched
// with launch_pdl may be scheduled while the previous kernel in the stream is
// still running: it calls griddep_wait() before its first access to memory
// that a predecessor writes or reads, and griddep_launch() so that its own
// dependent can be scheduled early.  After a predecessor that never signals
// (any other kernel) it simply starts when that kernel has finished.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Tiled TMA descriptor over u32 elements, rank <= 5, 128-byte swizzle (or
// none): dims[0] innermost, strides[i] = bytes between consecutive indices of
// dimension i + 1.  Returns cudaErrorNotSupported without a driver encoder.
cudaError_t encode_tiled_u32(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                             const uint64_t* strides, const uint32_t* box,
                             bool swizzle128 = true);

// ---------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error.
cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* w, int T, int E, int H,
                                 float* logits, cudaStream_t st);
cudaError_t launch_router_select(const moe_spec& sp, const float* logits, const float* bias,
                                 int T, int32_t* ids, float* weights, cudaStream_t st);

// The victim scan covers slots [S0, S0 + S): all S slots of the pool for the
// shared LRU and static placement, layer's own range for the per-layer LRU.
// no_fill (static placement) makes q = 0.
struct CacheArgs {
  int E = 0, layer = 0, n_ids = 0, S0 = 0, S = 0, K = 0, bp = 0, bh = 0, no_fill = 0;
  int n_slots = 0, n_bank = 0;  // all slots of the pool; L * E (range checks)
  // words the step clears for the decode FFN that follows it (its counters)
  uint32_t* zero_words = nullptr;
  int n_zero = 0;
  const int32_t* ids = nullptr;
  int32_t *slot_of_id = nullptr, *id_of_slot = nullptr;
  uint32_t *ts = nullptr, *clock = nullptr;
  moe_plan plan{};
};
cudaError_t launch_cache_step(const CacheArgs& a, cudaStream_t st);
// Router selection done inside the control step's CTA (decode layer step with
// T <= 16 tokens and E <= 256 experts): one warp per token reads its logits
// and writes ids / weights before the control step reads them.
struct SelArgs {
  const float* logits = nullptr;
  const float* bias = nullptr;
  int T = 0, k = 0, router = 0, n_groups = 0, topk_groups = 0;
  float scale = 0.0f;
  int32_t* ids = nullptr;
  float* wts = nullptr;
};
constexpr int kSelFusedMaxT = 16, kSelFusedMaxE = 256;

// One-kernel decode layer step (ffn_coop.cu): the router logits, the
// selection and the control step run inside the cooperative decode FFN
// kernel.  Layout of the cache's sync words (moe_cache.sync, zero between
// steps): the logits count, the fill publication flag, then the FFN's counter
// block (FfnArgs::ctr).
constexpr int kSyncLogits = 0, kSyncFill = 1, kSyncCtr = 4;
struct LayerFuse {
  const uint16_t* w_router = nullptr;  // [E][H] bf16
  const float* sel_bias = nullptr;     // [E] or null (sigmoid-group selection)
  float* logits = nullptr;             // [T][E] scratch
  int router = 0, n_groups = 0, topk_groups = 0;
  float scale = 0.0f;
  int32_t* ids_out = nullptr;          // [T][k] routed ids (written, then read by every CTA)
  float* wts_out = nullptr;            // [T][k] routing weights
  uint32_t* sync = nullptr;            // the cache's sync words
  CacheArgs c;                         // the control step (c.ids == ids_out)
};
cudaError_t launch_cache_step_sel(const CacheArgs& a, const SelArgs& s, cudaStream_t st);
cudaError_t launch_cache_reset(int32_t* slot_of_id, int n_ids, int32_t* id_of_slot, uint32_t* ts,
                               int S, uint32_t* clock, uint32_t* sync, cudaStream_t st);
cudaError_t launch_fill_copy(const moe_plan& plan, int K, const uint8_t* bank, uint8_t* pool,
                             int64_t blob_bytes, cudaStream_t st);
// Elastic re-division of the shared slot pool from S to S_new slots (resize.cu).
size_t resize_workspace_bytes(int S, int S_new);
cudaError_t launch_cache_resize(int32_t* slot_of_id, int n_ids, int32_t* id_of_slot, uint32_t* ts,
                                int S, int S_new, uint8_t* pool, int64_t blob_bytes, int32_t* ws,
                                cudaStream_t st);

struct FfnArgs {
  // every member has a zero default, so a caller that fills in only some
  // fields never hands a kernel an indeterminate flag or pointer
  int H = 0, I = 0, E = 0, k = 0, layer = 0, T = 0, has_shared = 0;
  int format = 0;  // MOE_FORMAT_*
  int64_t blob_bytes = 0;
  const uint8_t* bank = nullptr;
  const uint8_t* pool = nullptr;
  const int32_t* slot_of_id = nullptr;
  const int32_t* uniq = nullptr;
  const int32_t* counts = nullptr;
  const int32_t* fill_ids = nullptr;    // F of this step (counts[4] entries)
  const int32_t* fill_slots = nullptr;  // and their slots
  // 1: the streaming kernels also write each F expert's blob into its slot as
  // they read it from the bank (the step's fill copy, fused); set only when
  // both streaming kernels run (ffn_fill_fusable)
  int fill_fused = 0;
  uint8_t* pool_w = nullptr;  // the slot pool, written when fill_fused
  int inject_stall = 0;       // test hook: the gate/up producer issues no copies
  int32_t* err = nullptr;
  const uint16_t* x = nullptr;
  const int32_t* ids = nullptr;
  const float* weights = nullptr;
  const uint8_t* shared = nullptr;
  float* h = nullptr;         // [max_entries][T][I]
  float* partial = nullptr;   // [T][k + has_shared][H]
  uint32_t* tick = nullptr;   // [ceil(H / 16)] arrival counters, one per 16-row tile of y
  float* y = nullptr;         // [T][H]
  int max_entries = 0;
  int n_bank = 0;             // blobs in the bank (num_layers * E)
  int n_pool = 0;             // slots in the pool
  // cooperative decode kernel (ffn_coop.cu): counter words [n_ctr] that must
  // be zero when the kernel starts (cleared by the control step or by a
  // memset ahead of the launch), and the cache tables it restores when a
  // bounded wait gave up while the call carried the step's fills
  uint32_t* ctr = nullptr;
  int n_ctr = 0;
  int32_t* tab_slot_of_id = nullptr;
  int32_t* tab_id_of_slot = nullptr;
  uint32_t* tab_ts = nullptr;
};
// Where the FFN reads a routed id's weights: its slot when it was cached
// before this step (H), else in place from the bank (C, and F: an expert being
// filled in this step is read from the bank, byte-identical to its new slot,
// so the FFN need not wait for the fill copy).  Returns the slot or -1; with
// fs, also the slot an F expert goes to (-1 for H and C; only when the call
// carries the fill, the one case fill_slots is set).
// The slot, the fill count and the first fill ids (and slots) are loaded
// together, no load waiting for another's result beyond the fill count, since
// this sits on the FFN's start-up path.
__device__ __forceinline__ int32_t ffn_slot(const FfnArgs& a, int32_t id,
                                            int32_t* fs = nullptr) {
  int32_t slot = a.slot_of_id[id];
  if (!checked_ok(slot >= -1 && slot < a.n_pool, a.err)) slot = -1;
  const int nf = a.counts[4];
  const bool want = fs != nullptr && a.fill_fused;
  bool filled = false;
  int32_t fv = -1;
  for (int i0 = 0; i0 < nf; i0 += 8) {
    int32_t f[8], v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      f[q] = i0 + q < nf ? a.fill_ids[i0 + q] : -1;
      v[q] = want && i0 + q < nf ? a.fill_slots[i0 + q] : -1;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (f[q] == id) {
        filled = true;
        fv = v[q];
      }
  }
  if (fs) *fs = want ? fv : -1;
  return (slot < 0 || filled) ? -1 : slot;
}

size_t ffn_workspace_bytes(int H, int I, int k, int T, int has_shared);
void ffn_carve_workspace(FfnArgs& a, void* ws);
// Counter words at the end of the decode FFN workspace (ffn_carve_workspace
// points FfnArgs::ctr / n_ctr at them): the arrival counters of the 16-row
// output tiles, plus the cooperative kernel's per-entry readiness counters
// and its completion and failure words and per (entry, token) maxima of h.
inline int ffn_ctr_words(int H, int max_entries) {
  return (H + 15) / 16 + 9 * max_entries + 4;
}
// ctr_zeroed: the counter words are known to be zero (cleared by the control
// step just before); otherwise a memset clears them ahead of a kernel that
// needs them.
cudaError_t launch_ffn_decode(const FfnArgs& a, cudaStream_t st, bool ctr_zeroed = false);
// The cooperative decode kernel serves this shape: H % 1024 == 0,
// I % 512 == 0, 1 <= T <= 8, T * k <= 512, T * k + shared <= 128, and its
// shared-memory plan fits.  Its counters (FfnArgs::ctr) must be zero at
// launch.
bool ffn_coop_supported(int H, int I, int k, int T, int has_shared);
cudaError_t launch_ffn_coop(const FfnArgs& a, cudaStream_t st);
// The one-kernel step serves this shape: the cooperative FFN's, T k <= 32
// routed ids, K <= 8 victims, E <= 256 experts, k <= 64.
bool layer_fused_supported(int H, int I, int E, int k, int T, int has_shared, int K, int router,
                           int n_groups);
cudaError_t launch_layer_fused(const FfnArgs& a, const LayerFuse& lf, cudaStream_t st);
// Both streaming decode kernels run for this shape, so they can carry the
// step's fill copy (FfnArgs::fill_fused).
bool ffn_fill_fusable(int H, int I, int k, int T, int has_shared);
// streaming gate/up phase (T <= 8, H % 256 == 0): persistent CTAs fed by
// cp.async.bulk stages
cudaError_t launch_ffn_gate_up_stream(const FfnArgs& a, int n_tick, cudaStream_t st);
size_t ffn_stream_smem(int H, int T);
// streaming down phase (T <= 8, I % 256 == 0): launched as a programmatic
// dependent of the gate/up kernel
cudaError_t launch_ffn_down_stream(const FfnArgs& a, cudaStream_t st);
size_t ffn_down_stream_smem(int H, int I, int T);

// ------------------------------------------------------------------ prefill
constexpr int kPrefillTileRows = 256;  // rows of one grouped-GEMM m-tile

struct GemmArgs {
  int H, I, E, k, T;
  int64_t blob_bytes;
  const uint8_t* experts;   // E blobs of this layer, contiguous
  const uint8_t* shared;    // shared expert blob (group E) or null
  const uint16_t* a_src;    // mode 1: x_perm [T][H]; mode 2: h_perm [R][I]
  const int32_t* perm;      // permuted row -> assignment (t*k + j, or T*k + t)
  const int32_t* tile_g;    // m-tile -> group (expert, or E for the shared one)
  const int32_t* tile_row0; // m-tile -> first permuted row
  const int32_t* tile_rows; // m-tile -> rows (<= kPrefillTileRows)
  const int32_t* n_tiles;   // device count of m-tiles
  const float* weights;     // [T][k]
  uint16_t* h_out;          // mode 1 output: h_perm [R][I], K-permuted
  uint16_t* y_out;          // mode 2 output: y_assign [T][k+1][H]
  int32_t* err;             // device error bits (MOE_DERR_*), may be null
  int format;               // MOE_FORMAT_* of the expert blobs
};

struct PrefillBufs {
  uint16_t* x_perm;
  int32_t* counts;          // [E + 1]
  int32_t* offsets;         // [E + 2]
  int32_t* perm;            // [T*k + T]
  int32_t* tile_g;
  int32_t* tile_row0;
  int32_t* tile_rows;
  int32_t* n_tiles;
  uint16_t* h_perm;         // [T*k + T][I]
  uint16_t* y_assign;       // [T][k + 1][H]
  int32_t* chunk_cnt;       // [nch][E]: assignments of each expert per chunk of ids
  int32_t* chunk_base;      // [nch][E]: where each chunk's ids of an expert start in perm
  int nch;
  int max_tiles;
};

size_t prefill_workspace_bytes(int H, int I, int E, int k, int T);
void prefill_carve(PrefillBufs& b, void* ws, int H, int I, int E, int k, int T);
cudaError_t launch_prefill_ffn(const GemmArgs& base, const PrefillBufs& b, const uint16_t* x,
                               const int32_t* ids, int has_shared, float* y, cudaStream_t st);
cudaError_t launch_grouped_gemm(int mode, const GemmArgs& a, int max_tiles, cudaStream_t st);

}  // namespace moe
