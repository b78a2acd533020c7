// Internal launchers (one per kernel family); argument checks happen in api.cu.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/tsv.h"

namespace tsv {

int launch_build_meta(const int32_t* parents, const int32_t* num_nodes, const int32_t* prefix_len,
                      int batch, int max_nodes, int max_depth, uint32_t* mask,
                      int32_t* position_ids, int32_t* retrieve, int32_t* num_leaves,
                      int32_t* next_token, int32_t* next_sibling, int32_t* err,
                      cudaStream_t stream);

int launch_grow_mask(uint32_t* mask, int32_t* position_ids, const int32_t* new_parents,
                     const int32_t* prefix_len, int batch, int first_new, int count,
                     int max_nodes, int32_t* err, cudaStream_t stream);

int launch_accept_compact(const int32_t* tokens, const int32_t* next_token,
                          const int32_t* next_sibling, const int32_t* target,
                          const int32_t* num_nodes, const int32_t* prefix_len,
                          const int32_t* tree_valid, int batch,
                          int max_nodes, int max_depth, const tsv_kv_cache* cache,
                          int32_t* accept_path, int32_t* accept_len, int32_t* bonus,
                          int32_t* slot_map, int32_t* new_prefix_len, int32_t* err,
                          cudaStream_t stream);

// KV compaction of a path chosen by another kernel: accept_path / accept_len as written,
// code[b] = that request's status (only TSV_REQ_OK requests move rows).
int launch_compact_given(const int32_t* num_nodes, const int32_t* prefix_len, int batch,
                         int max_nodes, int max_depth, const tsv_kv_cache* cache,
                         const int32_t* code, int32_t* accept_path, int32_t* accept_len,
                         cudaStream_t stream);

// Non-greedy acceptance.
struct SampleArgs {
  const float* logits;       // [batch, max_nodes, vocab]
  const float* draft_probs;  // [batch, max_nodes, vocab] or null (target-only)
  int vocab;
  const float* temperature;  // [batch] each
  const int32_t* top_k;
  const float* top_p;
  const float* min_p;
  const float* u_node;       // [batch, max_nodes]
  const float* u_final;      // [batch]
  const int32_t* tokens;
  const int32_t* next_token;
  const int32_t* next_sibling;
  const int32_t* num_nodes;
  const int32_t* prefix_len;
  const int32_t* tree_valid;
  int batch, max_nodes, max_depth;
};
size_t sample_ws_bytes(int batch, int max_nodes);
int launch_target_probs(const SampleArgs& a, float* probs, void* ws, cudaStream_t stream);
int launch_sample_accept(const SampleArgs& a, const tsv_kv_cache* cache, int32_t* accept_path,
                         int32_t* accept_len, int32_t* bonus, int32_t* slot_map,
                         int32_t* new_prefix_len, int32_t* err, void* ws, cudaStream_t stream);

// Draft expansion.
struct TopkPlan {
  int chunks;         // CTAs per row in the streaming stage (workspace slots per row)
  int chunk_len;      // vocab entries per chunk (multiple of 4)
  bool persistent;    // large batch: one CTA per SM over equal shares of all entries
  bool cluster;       // small batch: one CTA per row, a thread-block cluster per request
  size_t ws_bytes;
};
TopkPlan plan_topk(int batch, int rows, int vocab, int top_k);
int launch_topk_expand(const float* logits, int batch, int rows, int64_t row_stride, int vocab,
                       int top_k, int level, const float* front_score_in,
                       const int32_t* front_store_in, int store_cap, int32_t* store_token,
                       float* store_score, int32_t* store_parent, int32_t* front_token_out,
                       float* front_score_out, int32_t* front_store_out, void* ws,
                       const TopkPlan& plan, bool product, cudaStream_t stream);
// Outputs of the tree metadata build (the arrays of tsv_tree_build_meta).
struct MetaOut {
  uint32_t* mask;
  int32_t* position_ids;
  int32_t* retrieve;
  int32_t* num_leaves;
  int32_t* next_token;
  int32_t* next_sibling;
  int32_t* err;
};
// meta (may be null): also build the selected trees' metadata in the same launch, with
// prefix_len and max_depth as tsv_tree_build_meta takes them.
int launch_select_final(const int32_t* store_token, const float* store_score,
                        const int32_t* store_parent, int batch, int num_candidates,
                        int store_cap, int total_tokens, const int32_t* root_token,
                        int max_nodes, int32_t* tokens, int32_t* parents, int32_t* num_nodes,
                        const int32_t* prefix_len, int max_depth, const MetaOut* meta,
                        cudaStream_t stream);

// Expansion variants.
int launch_draft_to_target(int32_t* tokens, const int32_t* num_nodes, int batch, int max_nodes,
                           const int32_t* d2t, int draft_vocab, int32_t* err,
                           cudaStream_t stream);
int launch_fixed_level(const float* logits, int batch, int frontier, int64_t row_stride,
                       int vocab, int width, int first_node, int first_parent, int max_nodes,
                       int32_t* tokens, int32_t* parents, cudaStream_t stream);

// Tree-verification attention.
struct AttnPlan {
  int batch, max_nodes, hq, hkv, group, head_dim, dtype;
  int rows;           // max_nodes * group (query rows per kv head)
  int rows_pad;       // rows rounded up to the M tile
  int tile_keys;      // keys per split unit
  int nsplit;         // splits along the keys
  int tiles_per_split;
  int max_prefix;
  bool tensor_core;   // a bf16 tensor-core path (q_rot in bf16, M tiles of 128 rows)
  bool umma;          // that path is the tcgen05 kernel (else the mma.sync one)
  size_t off_qrot, off_opart, off_ml, off_valid, ws_bytes;
};
AttnPlan plan_attn(const tsv_attn_shape* shape, const tsv_kv_cache* cache);
// Host checks of every tree-verification attention entry point (shape, cache, pointers,
// alignment, scalars): TSV_OK or TSV_ERR_INVALID_ARG; *empty is set for a batch of 0
// (nothing to launch). The workspace is each entry point's own check.
int attn_call_check(const tsv_attn_shape* shape, const tsv_kv_cache* cache, const void* q,
                    const void* k_new, const void* v_new, const int32_t* prefix_len,
                    const int32_t* num_nodes, const int32_t* position_ids, const uint32_t* mask,
                    float rope_theta, float softmax_scale, const void* out, bool* empty);
int launch_attn(const AttnPlan& plan, const void* q, const void* k_new, const void* v_new,
                const tsv_kv_cache* cache, const int32_t* prefix_len, const int32_t* num_nodes,
                const int32_t* position_ids, const uint32_t* mask, float rope_theta,
                float softmax_scale, void* out, void* ws, int32_t* err, cudaStream_t stream);

// Target lm-head argmax (the greedy token at every node).
struct LmPlan {
  int m_tiles;        // 128-row tiles of the node rows
  int chunks;         // 32-entry pieces of the vocabulary
  int splits;         // vocabulary ranges (CTAs per row tile), whole chunks each
  size_t ws_bytes;    // one 64-bit key per (split, row)
};
LmPlan plan_lm_head(int rows, int vocab);
bool lm_head_supported();
int launch_lm_head_argmax(const LmPlan& plan, const void* hidden, const void* weight, int rows,
                          int hidden_size, int vocab, int32_t* argmax, float* max_logit,
                          void* ws, cudaStream_t stream);

}  // namespace tsv
