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

}  // namespace tsv
