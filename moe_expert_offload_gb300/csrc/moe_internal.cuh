// Internal declarations of libmoe (not part of the C ABI).
#pragma once

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

// ---------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error.
cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* w, int T, int E, int H,
                                 float* logits, cudaStream_t st);
cudaError_t launch_router_select(const moe_spec& sp, const float* logits, const float* bias,
                                 int T, int32_t* ids, float* weights, cudaStream_t st);

struct CacheArgs {
  int E, layer, n_ids, S, K, bp, bh;
  const int32_t* ids;
  int32_t *slot_of_id, *id_of_slot;
  uint32_t *ts, *clock;
  moe_plan plan;
};
cudaError_t launch_cache_step(const CacheArgs& a, cudaStream_t st);
cudaError_t launch_cache_reset(int32_t* slot_of_id, int n_ids, int32_t* id_of_slot, uint32_t* ts,
                               int S, uint32_t* clock, cudaStream_t st);
cudaError_t launch_fill_copy(const moe_plan& plan, int K, const uint8_t* bank, uint8_t* pool,
                             int64_t blob_bytes, cudaStream_t st);

struct FfnArgs {
  int H, I, E, k, layer, T, has_shared;
  int64_t blob_bytes;
  const uint8_t* bank;
  const uint8_t* pool;
  const int32_t* slot_of_id;
  const int32_t* uniq;
  const int32_t* counts;
  int32_t* err;
  const uint16_t* x;
  const int32_t* ids;
  const float* weights;
  const uint8_t* shared;
  float* h;         // [max_entries][T][I]
  float* partial;   // [T][k + has_shared][H]
  uint32_t* tick;   // [H / rows per down block] arrival counters
  float* y;         // [T][H]
  int max_entries;
};
size_t ffn_workspace_bytes(int H, int I, int k, int T, int has_shared);
void ffn_carve_workspace(FfnArgs& a, void* ws);
cudaError_t launch_ffn_decode(const FfnArgs& a, cudaStream_t st);

}  // namespace moe
