// Arguments shared by the tree-verification attention kernels (internal).
#pragma once

#include <stdint.h>

#include "kernels.h"

namespace tsv {

struct RopeTable {
  double inv_freq[64];  // theta^(-2m/D), m < D/2
};

struct AttnArgs {
  // cache
  void* k_cache;
  void* v_cache;
  const int32_t* block_table;
  int64_t capacity;
  int layout, max_blocks, num_blocks;
  // per request
  const int32_t* prefix_len;
  const int32_t* num_nodes;
  const int32_t* position_ids;
  const uint32_t* mask;
  int mask_words;
  int32_t* err;
  void* out;  // [B, max_nodes, Hq, D]
  // workspace
  void* q_rot;
  float* o_part;
  float* ml;
  int32_t* valid;
  // sizes
  int max_nodes, hq, hkv, group, head_dim, rows_pad, max_prefix;
  int tile_keys, tiles_per_split, nsplit;
};

// Query rows per tensor-core CTA (one 128-row M tile).
constexpr int TC_M_GROUP = 128;

// Most key splits of one row block on the tensor-core path.
#define TSV_ATTN_MAX_SPLITS 32

bool tc_supported(const AttnPlan& p);
int launch_attn_tc(const AttnPlan& p, const AttnArgs& a, float scale_log2, void* out,
                   cudaStream_t stream);
// tcgen05 path with cp.async-fed K/V rings (attn_umma.cu): bf16, head_dim 128, sm_100+;
// keys in tiles of 128.
bool umma_supported(const AttnPlan& p);
int launch_attn_umma(const AttnPlan& p, const AttnArgs& a, float scale_log2, void* out,
                     cudaStream_t stream);
// Warp-level tensor-core path (mma.sync, attn_mma.cu): bf16, head_dim 128, sm_80+; keys
// in tiles of MMA_TILE_KEYS.
constexpr int MMA_TILE_KEYS = 64;
constexpr int MMA_M_GROUP = 128;
int launch_attn_mma(const AttnPlan& p, const AttnArgs& a, float scale_log2, void* out,
                    cudaStream_t stream);
// Log-sum-exp merge of the key splits into the bf16 output (rows of requests that took
// one split are left as the attention kernel wrote them).
int launch_split_merge(const AttnPlan& p, const AttnArgs& a, void* out, cudaStream_t stream);

}  // namespace tsv
