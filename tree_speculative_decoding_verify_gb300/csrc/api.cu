// C ABI entry points: host-side argument checks, workspace sizing and dispatch.
// Nothing here touches the GPU before the checks pass.
#include <stdio.h>

#include <mutex>

#include "attn_common.cuh"
#include "common.cuh"
#include "kernels.h"

namespace tsv {

static thread_local int g_last_cuda_error = 0;

void record_cuda_error(cudaError_t e) { g_last_cuda_error = (int)e; }

int launch_status() {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return TSV_ERR_CUDA;
  }
  return TSV_OK;
}

namespace {
constexpr int MAX_DEVICES = 64;
int g_sms[MAX_DEVICES];
int g_cc[MAX_DEVICES];
std::mutex g_mu;

void load_device(int* sms, int* cc) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
    cudaGetLastError();
    *sms = 148;
    *cc = 0;
    return;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_sms[dev] == 0) {
    int s = 0, ma = 0, mi = 0;
    cudaDeviceGetAttribute(&s, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&ma, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev);
    cudaGetLastError();
    g_sms[dev] = s > 0 ? s : 148;
    g_cc[dev] = 10 * ma + mi;
  }
  *sms = g_sms[dev];
  *cc = g_cc[dev];
}
}  // namespace

int device_sm_count() {
  int s, c;
  load_device(&s, &c);
  return s;
}

int device_cc() {
  int s, c;
  load_device(&s, &c);
  return c;
}

static bool cache_ok(const tsv_kv_cache* c, bool need_layers) {
  if (!c || !c->k || !c->v) return false;
  if (c->dtype != TSV_DTYPE_F32 && c->dtype != TSV_DTYPE_BF16) return false;
  if (c->num_kv_heads < 1 || (c->head_dim != 64 && c->head_dim != 128)) return false;
  if (c->layout == TSV_KV_CONTIGUOUS) {
    if (c->capacity < TSV_KV_BLOCK || c->capacity % TSV_KV_BLOCK) return false;
  } else if (c->layout == TSV_KV_PAGED) {
    if (!c->block_table || c->max_blocks < 1 || c->num_blocks < 1) return false;
  } else {
    return false;
  }
  if (need_layers && (c->num_layers < 1 || (c->num_layers > 1 && c->layer_stride <= 0)))
    return false;
  const int esize = c->dtype == TSV_DTYPE_BF16 ? 2 : 4;
  if ((reinterpret_cast<uintptr_t>(c->k) | reinterpret_cast<uintptr_t>(c->v)) % 16) return false;
  if (need_layers && c->num_layers > 1 && (c->layer_stride * esize) % 16) return false;
  return true;
}

}  // namespace tsv

using namespace tsv;

namespace {
inline bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }
}  // namespace

static bool attn_shape_ok(const tsv_attn_shape* s, const tsv_kv_cache* c) {
  if (!s || !cache_ok(c, false)) return false;
  if (s->batch < 0 || s->max_nodes < 1 || s->max_nodes > TSV_MAX_NODES || s->max_prefix < 0)
    return false;
  if (s->num_q_heads < 1 || s->num_q_heads % c->num_kv_heads) return false;
  if ((int64_t)s->batch * c->num_kv_heads > 65535) return false;  // grid.y/z limit
  if ((int64_t)s->max_nodes * (s->num_q_heads / c->num_kv_heads) > 1024) return false;
  return true;
}

namespace tsv {
int attn_call_check(const tsv_attn_shape* shape, const tsv_kv_cache* cache, const void* q,
                    const void* k_new, const void* v_new, const int32_t* prefix_len,
                    const int32_t* num_nodes, const int32_t* position_ids, const uint32_t* mask,
                    float rope_theta, float softmax_scale, const void* out, bool* empty) {
  *empty = false;
  if (!attn_shape_ok(shape, cache)) return TSV_ERR_INVALID_ARG;
  if (!(rope_theta > 0.f) || !(softmax_scale > 0.f)) return TSV_ERR_INVALID_ARG;
  if (shape->batch == 0) {
    *empty = true;
    return TSV_OK;
  }
  if (!q || !k_new || !v_new || !prefix_len || !num_nodes || !position_ids || !mask || !out)
    return TSV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out))
    return TSV_ERR_INVALID_ARG;
  return TSV_OK;
}
}  // namespace tsv


extern "C" {

const char* tsv_version(void) { return "tsv 0.1.0 (sm_103a)"; }

const char* tsv_status_string(int status) {
  switch (status) {
    case TSV_OK: return "ok";
    case TSV_ERR_INVALID_ARG: return "invalid argument";
    case TSV_ERR_UNSUPPORTED: return "unsupported";
    case TSV_ERR_WORKSPACE: return "workspace missing or too small";
    case TSV_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int tsv_last_cuda_error(void) { return g_last_cuda_error; }

int tsv_tree_build_meta(const int32_t* parents, const int32_t* num_nodes,
                        const int32_t* prefix_len, int batch, int max_nodes, int max_depth,
                        uint32_t* mask, int32_t* position_ids, int32_t* retrieve_indices,
                        int32_t* num_leaves, int32_t* next_token, int32_t* next_sibling,
                        int32_t* err, tsv_stream_t stream) {
  if (batch < 0 || max_nodes < 1 || max_nodes > TSV_MAX_NODES || max_depth < 0 ||
      max_depth > TSV_MAX_DEPTH)
    return TSV_ERR_INVALID_ARG;
  if (batch == 0) return TSV_OK;
  if (!parents || !num_nodes || !prefix_len || !mask || !position_ids || !retrieve_indices ||
      !num_leaves || !next_token || !next_sibling)
    return TSV_ERR_INVALID_ARG;
  return launch_build_meta(parents, num_nodes, prefix_len, batch, max_nodes, max_depth, mask,
                           position_ids, retrieve_indices, num_leaves, next_token, next_sibling,
                           err, (cudaStream_t)stream);
}

int tsv_draft_grow_mask(uint32_t* mask, int32_t* position_ids, const int32_t* new_parents,
                        const int32_t* prefix_len, int batch, int first_new, int count,
                        int max_nodes, int32_t* err, tsv_stream_t stream) {
  if (batch < 0 || max_nodes < 2 || max_nodes > TSV_MAX_NODES || first_new < 1 || count < 1 ||
      (int64_t)first_new + count > max_nodes)
    return TSV_ERR_INVALID_ARG;
  if (batch == 0) return TSV_OK;
  if (!mask || !position_ids || !new_parents || !prefix_len) return TSV_ERR_INVALID_ARG;
  return launch_grow_mask(mask, position_ids, new_parents, prefix_len, batch, first_new, count,
                          max_nodes, err, (cudaStream_t)stream);
}

size_t tsv_draft_topk_expand_workspace_size(int batch, int rows, int vocab, int top_k) {
  if (batch < 1 || rows < 1 || vocab < 1 || top_k < 1 || top_k > TSV_MAX_TOPK) return 0;
  return plan_topk(batch, rows, vocab, top_k).ws_bytes;
}

int tsv_draft_topk_expand_launches(int batch, int rows, int vocab, int top_k) {
  if (batch < 1 || rows < 1 || vocab < 1 || top_k < 1 || top_k > TSV_MAX_TOPK) return 0;
  return plan_topk(batch, rows, vocab, top_k).persistent ? 2 : 1;
}

static int topk_expand(const float* logits, int batch, int rows, int64_t row_stride, int vocab,
                       int top_k, int level, const float* front_score_in,
                       const int32_t* front_store_in, int store_cap, int32_t* store_token,
                       float* store_score, int32_t* store_parent, int32_t* front_token_out,
                       float* front_score_out, int32_t* front_store_out, void* workspace,
                       size_t workspace_bytes, bool product, cudaStream_t stream) {
  if (batch < 0 || top_k < 1 || top_k > TSV_MAX_TOPK || vocab < top_k || row_stride < vocab ||
      level < 1 || rows < 1 || rows > TSV_MAX_TOPK)
    return TSV_ERR_INVALID_ARG;
  if ((level == 1) != (rows == 1) || (level > 1 && rows != top_k)) return TSV_ERR_INVALID_ARG;
  if ((int64_t)batch * rows > 65535) return TSV_ERR_INVALID_ARG;  // grid.y limit
  const int64_t off = level == 1 ? 0 : top_k + (int64_t)(level - 2) * top_k * top_k;
  if (off + (int64_t)rows * top_k > store_cap) return TSV_ERR_INVALID_ARG;
  if (batch == 0) return TSV_OK;
  if (!logits || !store_token || !store_score || !store_parent || !front_token_out ||
      !front_score_out || !front_store_out)
    return TSV_ERR_INVALID_ARG;
  if (level > 1 && (!front_score_in || !front_store_in)) return TSV_ERR_INVALID_ARG;
  const TopkPlan plan = plan_topk(batch, rows, vocab, top_k);
  if (!workspace || workspace_bytes < plan.ws_bytes) return TSV_ERR_WORKSPACE;
  return launch_topk_expand(logits, batch, rows, row_stride, vocab, top_k, level, front_score_in,
                            front_store_in, store_cap, store_token, store_score, store_parent,
                            front_token_out, front_score_out, front_store_out, workspace, plan,
                            product, stream);
}

int tsv_draft_topk_expand(const float* logits, int batch, int rows, int64_t row_stride,
                          int vocab, int top_k, int level, const float* front_score_in,
                          const int32_t* front_store_in, int store_cap, int32_t* store_token,
                          float* store_score, int32_t* store_parent, int32_t* front_token_out,
                          float* front_score_out, int32_t* front_store_out, void* workspace,
                          size_t workspace_bytes, tsv_stream_t stream) {
  return topk_expand(logits, batch, rows, row_stride, vocab, top_k, level, front_score_in,
                     front_store_in, store_cap, store_token, store_score, store_parent,
                     front_token_out, front_score_out, front_store_out, workspace,
                     workspace_bytes, false, (cudaStream_t)stream);
}

int tsv_draft_topk_expand_product(const float* logits, int batch, int rows, int64_t row_stride,
                                  int vocab, int top_k, int level, const float* front_score_in,
                                  const int32_t* front_store_in, int store_cap,
                                  int32_t* store_token, float* store_score,
                                  int32_t* store_parent, int32_t* front_token_out,
                                  float* front_score_out, int32_t* front_store_out,
                                  void* workspace, size_t workspace_bytes, tsv_stream_t stream) {
  return topk_expand(logits, batch, rows, row_stride, vocab, top_k, level, front_score_in,
                     front_store_in, store_cap, store_token, store_score, store_parent,
                     front_token_out, front_score_out, front_store_out, workspace,
                     workspace_bytes, true, (cudaStream_t)stream);
}

int tsv_draft_to_target(int32_t* tokens, const int32_t* num_nodes, int batch, int max_nodes,
                        const int32_t* d2t, int draft_vocab, int32_t* err, tsv_stream_t stream) {
  if (batch < 0 || max_nodes < 1 || max_nodes > TSV_MAX_NODES || draft_vocab < 1)
    return TSV_ERR_INVALID_ARG;
  if (batch == 0) return TSV_OK;
  if (!tokens || !num_nodes || !d2t) return TSV_ERR_INVALID_ARG;
  return launch_draft_to_target(tokens, num_nodes, batch, max_nodes, d2t, draft_vocab, err,
                                (cudaStream_t)stream);
}

int tsv_draft_fixed_level(const float* logits, int batch, int frontier, int64_t row_stride,
                          int vocab, int width, int first_node, int first_parent, int max_nodes,
                          int32_t* tokens, int32_t* parents, tsv_stream_t stream) {
  if (batch < 0 || frontier < 1 || width < 1 || width > TSV_MAX_TOPK || vocab < width ||
      row_stride < vocab || max_nodes < 1 || max_nodes > TSV_MAX_NODES || first_parent < 0 ||
      first_parent + frontier > first_node ||
      (int64_t)first_node + (int64_t)frontier * width > max_nodes ||
      (int64_t)batch * frontier > 65535)
    return TSV_ERR_INVALID_ARG;
  if (batch == 0) return TSV_OK;
  if (!logits || !tokens || !parents) return TSV_ERR_INVALID_ARG;
  return launch_fixed_level(logits, batch, frontier, row_stride, vocab, width, first_node,
                            first_parent, max_nodes, tokens, parents, (cudaStream_t)stream);
}

int tsv_draft_select_final(const int32_t* store_token, const float* store_score,
                           const int32_t* store_parent, int batch, int num_candidates,
                           int store_cap, int total_tokens, const int32_t* root_token,
                           int max_nodes, int32_t* tokens, int32_t* parents, int32_t* num_nodes,
                           tsv_stream_t stream) {
  if (batch < 0 || total_tokens < 1 || num_candidates < total_tokens || num_candidates > 4096 ||
      store_cap < num_candidates || max_nodes < total_tokens + 1 || max_nodes > TSV_MAX_NODES)
    return TSV_ERR_INVALID_ARG;
  if (batch == 0) return TSV_OK;
  if (!store_token || !store_score || !store_parent || !root_token || !tokens || !parents)
    return TSV_ERR_INVALID_ARG;
  return launch_select_final(store_token, store_score, store_parent, batch, num_candidates,
                             store_cap, total_tokens, root_token, max_nodes, tokens, parents,
                             num_nodes, nullptr, 0, nullptr, (cudaStream_t)stream);
}

int tsv_draft_select_tree(const int32_t* store_token, const float* store_score,
                          const int32_t* store_parent, int batch, int num_candidates,
                          int store_cap, int total_tokens, const int32_t* root_token,
                          int max_nodes, int32_t* tokens, int32_t* parents, int32_t* num_nodes,
                          const int32_t* prefix_len, int max_depth, uint32_t* mask,
                          int32_t* position_ids, int32_t* retrieve_indices, int32_t* num_leaves,
                          int32_t* next_token, int32_t* next_sibling, int32_t* err,
                          tsv_stream_t stream) {
  if (batch < 0 || total_tokens < 1 || num_candidates < total_tokens || num_candidates > 4096 ||
      store_cap < num_candidates || max_nodes < total_tokens + 1 || max_nodes > TSV_MAX_NODES ||
      max_depth < 0 || max_depth > TSV_MAX_DEPTH)
    return TSV_ERR_INVALID_ARG;
  if (batch == 0) return TSV_OK;
  if (!store_token || !store_score || !store_parent || !root_token || !tokens || !parents ||
      !prefix_len || !mask || !position_ids || !retrieve_indices || !num_leaves || !next_token ||
      !next_sibling)
    return TSV_ERR_INVALID_ARG;
  const MetaOut meta{mask, position_ids, retrieve_indices, num_leaves, next_token, next_sibling,
                     err};
  return launch_select_final(store_token, store_score, store_parent, batch, num_candidates,
                             store_cap, total_tokens, root_token, max_nodes, tokens, parents,
                             num_nodes, prefix_len, max_depth, &meta, (cudaStream_t)stream);
}

size_t tsv_tree_verify_attn_workspace_size(const tsv_attn_shape* shape,
                                           const tsv_kv_cache* cache) {
  if (!attn_shape_ok(shape, cache)) return 0;
  return plan_attn(shape, cache).ws_bytes;
}

int tsv_tree_verify_attn_launches(const tsv_attn_shape* shape, const tsv_kv_cache* cache) {
  if (!attn_shape_ok(shape, cache)) return 0;
  const AttnPlan p = plan_attn(shape, cache);
  return p.tensor_core ? (p.nsplit > 1 ? 3 : 2) : 3;
}

int tsv_tree_verify_attn(const tsv_attn_shape* shape, const void* q, const void* k_new,
                         const void* v_new, const tsv_kv_cache* cache,
                         const int32_t* prefix_len, const int32_t* num_nodes,
                         const int32_t* position_ids, const uint32_t* mask, float rope_theta,
                         float softmax_scale, void* out, void* workspace,
                         size_t workspace_bytes, int32_t* err, tsv_stream_t stream) {
  bool empty = false;
  const int st = attn_call_check(shape, cache, q, k_new, v_new, prefix_len, num_nodes,
                                 position_ids, mask, rope_theta, softmax_scale, out, &empty);
  if (st != TSV_OK || empty) return st;
  const AttnPlan plan = plan_attn(shape, cache);
  if (!workspace || workspace_bytes < plan.ws_bytes ||
      reinterpret_cast<uintptr_t>(workspace) % 256)
    return TSV_ERR_WORKSPACE;
  return launch_attn(plan, q, k_new, v_new, cache, prefix_len, num_nodes, position_ids, mask,
                     rope_theta, softmax_scale, out, workspace, err, (cudaStream_t)stream);
}

size_t tsv_lm_head_argmax_workspace_size(int rows, int vocab) {
  if (rows < 0 || rows > (1 << 24) || vocab < 1) return 0;
  return plan_lm_head(rows, vocab).ws_bytes;
}

int tsv_lm_head_argmax(const void* hidden, const void* weight, int rows, int hidden_size,
                       int vocab, int32_t* argmax, float* max_logit, void* workspace,
                       size_t workspace_bytes, tsv_stream_t stream) {
  if (rows < 0 || rows > (1 << 24) || vocab < 1 || hidden_size < 64 || hidden_size % 64)
    return TSV_ERR_INVALID_ARG;
  if (rows == 0) return TSV_OK;
  if (!hidden || !weight || !argmax) return TSV_ERR_INVALID_ARG;
  if (((uintptr_t)hidden | (uintptr_t)weight) & 15u) return TSV_ERR_INVALID_ARG;
  if (!lm_head_supported()) return TSV_ERR_UNSUPPORTED;
  const LmPlan plan = plan_lm_head(rows, vocab);
  if (!workspace || workspace_bytes < plan.ws_bytes || ((uintptr_t)workspace & 255u))
    return TSV_ERR_WORKSPACE;
  return launch_lm_head_argmax(plan, hidden, weight, rows, hidden_size, vocab, argmax, max_logit,
                               workspace, (cudaStream_t)stream);
}

size_t tsv_tree_sample_accept_workspace_size(int batch, int max_nodes) {
  if (batch < 0 || max_nodes < 1 || max_nodes > TSV_MAX_NODES) return 0;
  return sample_ws_bytes(batch, max_nodes);
}

static bool sample_sizes_ok(int batch, int max_nodes, int vocab) {
  return batch >= 0 && batch <= 65535 && max_nodes >= 1 && max_nodes <= TSV_MAX_NODES &&
         vocab >= 1 && vocab <= TSV_MAX_SAMPLE_VOCAB;
}

int tsv_tree_sample_accept(const float* target_logits, const float* draft_probs, int vocab,
                           const float* temperature, const int32_t* top_k, const float* top_p,
                           const float* min_p, const float* u_node, const float* u_final,
                           const int32_t* tokens, const int32_t* next_token,
                           const int32_t* next_sibling, const int32_t* num_nodes,
                           const int32_t* prefix_len, const int32_t* tree_valid, int batch,
                           int max_nodes, int max_depth, const tsv_kv_cache* cache,
                           int32_t* accept_path, int32_t* accept_len, int32_t* bonus_token,
                           int32_t* slot_map, int32_t* new_prefix_len, int32_t* err,
                           void* workspace, size_t workspace_bytes, tsv_stream_t stream) {
  if (!sample_sizes_ok(batch, max_nodes, vocab) || max_depth < 0 || max_depth > TSV_MAX_DEPTH)
    return TSV_ERR_INVALID_ARG;
  if (cache && !cache_ok(cache, true)) return TSV_ERR_INVALID_ARG;
  if (batch == 0) return TSV_OK;
  if (!target_logits || !temperature || !top_k || !top_p || !min_p || !u_node || !u_final ||
      !tokens || !next_token || !next_sibling || !num_nodes || !prefix_len || !accept_path ||
      !accept_len || !bonus_token || !slot_map || !new_prefix_len)
    return TSV_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < sample_ws_bytes(batch, max_nodes) ||
      ((uintptr_t)workspace & 255u))
    return TSV_ERR_WORKSPACE;
  const SampleArgs a{target_logits, draft_probs, vocab, temperature, top_k, top_p, min_p,
                     u_node, u_final, tokens, next_token, next_sibling, num_nodes, prefix_len,
                     tree_valid, batch, max_nodes, max_depth};
  return launch_sample_accept(a, cache, accept_path, accept_len, bonus_token, slot_map,
                              new_prefix_len, err, workspace, (cudaStream_t)stream);
}

int tsv_target_probs(const float* target_logits, int vocab, const float* temperature,
                     const int32_t* top_k, const float* top_p, const float* min_p,
                     const int32_t* num_nodes, int batch, int max_nodes, float* probs,
                     void* workspace, size_t workspace_bytes, tsv_stream_t stream) {
  if (!sample_sizes_ok(batch, max_nodes, vocab)) return TSV_ERR_INVALID_ARG;
  if (batch == 0) return TSV_OK;
  if (!target_logits || !temperature || !top_k || !top_p || !min_p || !num_nodes || !probs)
    return TSV_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < sample_ws_bytes(batch, max_nodes) ||
      ((uintptr_t)workspace & 255u))
    return TSV_ERR_WORKSPACE;
  const SampleArgs a{target_logits, nullptr, vocab, temperature, top_k, top_p, min_p,
                     nullptr, nullptr, nullptr, nullptr, nullptr, num_nodes, nullptr,
                     nullptr, batch, max_nodes, 0};
  return launch_target_probs(a, probs, workspace, (cudaStream_t)stream);
}

int tsv_accept_and_compact(const int32_t* tokens, const int32_t* next_token,
                           const int32_t* next_sibling, const int32_t* target_argmax,
                           const int32_t* num_nodes, const int32_t* prefix_len,
                           const int32_t* tree_valid, int batch,
                           int max_nodes, int max_depth, const tsv_kv_cache* cache,
                           int32_t* accept_path, int32_t* accept_len, int32_t* bonus_token,
                           int32_t* slot_map, int32_t* new_prefix_len, int32_t* err,
                           tsv_stream_t stream) {
  if (batch < 0 || max_nodes < 1 || max_nodes > TSV_MAX_NODES || max_depth < 0 ||
      max_depth > TSV_MAX_DEPTH)
    return TSV_ERR_INVALID_ARG;
  if (cache && !cache_ok(cache, true)) return TSV_ERR_INVALID_ARG;
  if (batch == 0) return TSV_OK;
  if (!tokens || !next_token || !next_sibling || !target_argmax || !num_nodes || !prefix_len ||
      !accept_path || !accept_len || !bonus_token || !slot_map || !new_prefix_len)
    return TSV_ERR_INVALID_ARG;
  return launch_accept_compact(tokens, next_token, next_sibling, target_argmax, num_nodes,
                               prefix_len, tree_valid, batch, max_nodes, max_depth, cache,
                               accept_path,
                               accept_len, bonus_token, slot_map, new_prefix_len, err,
                               (cudaStream_t)stream);
}

}  // extern "C"
