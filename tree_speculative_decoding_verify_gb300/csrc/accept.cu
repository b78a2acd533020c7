// Greedy acceptance walk and KV compaction.
//
// Pages: "推理系统手册 · 投机解码进阶：树形草稿与 EAGLE", section 实现
// (tree_speculative_generate: from the root, step to the lowest-numbered child whose
// token equals the target's argmax at the current node; stop when there is none; the
// bonus token is the argmax at the last accepted node; the accepted nodes' KV is reused,
// not recomputed); "TensorRT-LLM 源码完全拆解(二十二): EAGLE-3 一体式草稿", section
// 验证:在树上走一条路径 (the walk follows the next_token / next_sibling lists) and
// section 接受之后:KV 从树形搬回线性 (the accepted KV moves to consecutive slots).
//
// One CTA per (request, copy unit); a copy unit is one (layer, kv head,
// keys-or-values) plane. Every CTA of a request repeats the (tiny) walk from shared
// memory, so no CTA waits for another. With `given` the walk has been made already (the
// non-greedy acceptance writes the path, its length and a per-request code first) and
// the kernel only moves the rows.
#include "common.cuh"
#include "kernels.h"
#include "kv_view.cuh"

namespace tsv {
namespace {

constexpr int THREADS = 128;
constexpr int UNITS_PER_CTA = 1;  // copy units per CTA: each CTA pays one load round trip
constexpr int MAX_ROW_BYTES = 128 * 4;  // head_dim 128 in f32

__global__ void __launch_bounds__(THREADS)
accept_compact_kernel(const int32_t* __restrict__ tokens, const int32_t* __restrict__ next_token,
                      const int32_t* __restrict__ next_sibling, const int32_t* __restrict__ target,
                      const int32_t* __restrict__ num_nodes, const int32_t* __restrict__ prefix_len,
                      const int32_t* __restrict__ tree_valid, int max_nodes, int max_depth,
                      CacheView cache, bool has_cache, const int32_t* __restrict__ given,
                      int32_t* __restrict__ accept_path, int32_t* __restrict__ accept_len,
                      int32_t* __restrict__ bonus, int32_t* __restrict__ slot_map,
                      int32_t* __restrict__ new_prefix_len, int32_t* __restrict__ err) {
  __shared__ int32_t s_tok[TSV_MAX_NODES], s_next[TSV_MAX_NODES], s_sib[TSV_MAX_NODES],
      s_tgt[TSV_MAX_NODES];
  __shared__ int32_t s_path[TSV_MAX_DEPTH + 1];
  __shared__ int s_len, s_code;
  __shared__ __align__(16) unsigned char s_rows[TSV_MAX_DEPTH * MAX_ROW_BYTES];

  griddep_wait();
  griddep_launch();
  const int b = blockIdx.x;
  const int64_t row0 = (int64_t)b * max_nodes;
  const int T = num_nodes[b];
  const int P = prefix_len[b];
  const bool size_ok = T >= 1 && T <= max_nodes && P >= 0;
  if (given) {
    // the path, its length and the request's code come from the walk already made
    if (threadIdx.x == 0) {
      const int cols = max_depth + 1;
      const int len = min(max(accept_len[b], 1), cols);
      for (int i = 0; i < len; ++i) s_path[i] = accept_path[(int64_t)b * cols + i];
      s_len = len;
      s_code = given[b];
    }
    __syncthreads();
  } else {
  for (int i = threadIdx.x; i < max_nodes; i += THREADS) {
    const bool in = size_ok && i < T;
    s_tok[i] = in ? tokens[row0 + i] : -1;
    s_next[i] = in ? next_token[row0 + i] : -1;
    s_sib[i] = in ? next_sibling[row0 + i] : -1;
    s_tgt[i] = target[row0 + i];
  }
  __syncthreads();

  if (threadIdx.x == 0) {
    int code = size_ok ? TSV_REQ_OK : TSV_REQ_BAD_SIZE;
    int len = 1, node = 0;
    s_path[0] = 0;
    // a request without a valid tree takes the single-token path: the root alone
    const bool has_tree = !tree_valid || tree_valid[b] != 0;
    if (code == TSV_REQ_OK && has_tree) {
      // Every step goes one level down; a valid tree has at most max_depth levels.
      for (int step = 0; step <= max_depth; ++step) {
        const int pred = s_tgt[node];
        // Children are listed in ascending node order, so the chain strictly increases
        // and ends within T hops.
        int c = s_next[node];
        int prev = node;
        while (c >= 0) {
          if (c <= prev || c >= T) { code = TSV_REQ_BAD_LINKS; break; }
          if (s_tok[c] == pred) break;
          prev = c;
          c = s_sib[c];
        }
        if (code != TSV_REQ_OK || c < 0) break;
        if (len == max_depth + 1) { code = TSV_REQ_BAD_LINKS; break; }
        s_path[len++] = c;
        node = c;
      }
    }
    if (code == TSV_REQ_OK && has_cache) {
      if ((int64_t)P + T > cache_slots(cache)) code = TSV_REQ_CAPACITY;
      for (int i = 0; code == TSV_REQ_OK && i < len; ++i) {
        bool ok = true;
        slot_offset(cache, b, 0, P + s_path[i], &ok);
        slot_offset(cache, b, 0, P + i, &ok);
        if (!ok) code = TSV_REQ_BAD_BLOCK;
      }
    }
    if (code != TSV_REQ_OK) len = 1;
    s_len = len;
    s_code = code;
  }
  __syncthreads();
  }
  const int len = s_len;
  const int code = s_code;

  if (blockIdx.y == 0 && !given) {
    const int cols = max_depth + 1;
    for (int i = threadIdx.x; i < cols; i += THREADS) {
      const bool in = i < len;
      accept_path[(int64_t)b * cols + i] = in ? s_path[i] : -1;
      slot_map[((int64_t)b * cols + i) * 2 + 0] = in ? P + s_path[i] : -1;
      slot_map[((int64_t)b * cols + i) * 2 + 1] = in ? P + i : -1;
    }
    if (threadIdx.x == 0) {
      accept_len[b] = len;
      bonus[b] = s_tgt[s_path[len - 1]];
      new_prefix_len[b] = (size_ok ? P : 0) + len;
      if (err) err[b] = code;
    }
  }
  if (!has_cache || code != TSV_REQ_OK || len == 1) return;

  // Compaction: slot P + i <- slot P + path[i] for i in [1, len). Rows are staged in
  // shared memory first, so overlapping sources and destinations are safe.
  const int chunks = cache.row_bytes / 16;
  const int units = cache.num_layers * cache.hkv * 2;
  for (int u = blockIdx.y * UNITS_PER_CTA; u < min(units, (blockIdx.y + 1) * UNITS_PER_CTA); ++u) {
    const int layer = u / (cache.hkv * 2);
    const int h = (u >> 1) % cache.hkv;
    char* base = ((u & 1) ? cache.v : cache.k) + (int64_t)layer * cache.layer_stride_bytes;
    const int total = (len - 1) * chunks;
    for (int t = threadIdx.x; t < total; t += THREADS) {
      const int i = 1 + t / chunks, ch = t % chunks;
      bool ok = true;
      const int64_t src = slot_offset(cache, b, h, P + s_path[i], &ok);
      reinterpret_cast<int4*>(s_rows)[(i - 1) * chunks + ch] =
          reinterpret_cast<const int4*>(base + src)[ch];
    }
    __syncthreads();
    for (int t = threadIdx.x; t < total; t += THREADS) {
      const int i = 1 + t / chunks, ch = t % chunks;
      if (s_path[i] == i) continue;
      bool ok = true;
      const int64_t dst = slot_offset(cache, b, h, P + i, &ok);
      reinterpret_cast<int4*>(base + dst)[ch] =
          reinterpret_cast<const int4*>(s_rows)[(i - 1) * chunks + ch];
    }
    __syncthreads();
  }
}

}  // namespace

int launch_accept_compact(const int32_t* tokens, const int32_t* next_token,
                          const int32_t* next_sibling, const int32_t* target,
                          const int32_t* num_nodes, const int32_t* prefix_len,
                          const int32_t* tree_valid, int batch,
                          int max_nodes, int max_depth, const tsv_kv_cache* cache,
                          int32_t* accept_path, int32_t* accept_len, int32_t* bonus,
                          int32_t* slot_map, int32_t* new_prefix_len, int32_t* err,
                          cudaStream_t stream) {
  const CacheView cv = make_cache_view(cache);
  int ctas_y = 1;
  if (cache)
    ctas_y = (int)ceil_div((int64_t)cache->num_layers * cache->num_kv_heads * 2, UNITS_PER_CTA);
  dim3 grid(batch, ctas_y);
  return launch_pdl(accept_compact_kernel, grid, dim3(THREADS), 0, stream, tokens, next_token,
                    next_sibling, target, num_nodes, prefix_len, tree_valid, max_nodes,
                    max_depth, cv,
                    cache != nullptr, static_cast<const int32_t*>(nullptr), accept_path, accept_len, bonus, slot_map, new_prefix_len,
                    err);
}

}  // namespace tsv

namespace tsv {

int launch_compact_given(const int32_t* num_nodes, const int32_t* prefix_len, int batch,
                         int max_nodes, int max_depth, const tsv_kv_cache* cache,
                         const int32_t* code, int32_t* accept_path, int32_t* accept_len,
                         cudaStream_t stream) {
  const CacheView cv = make_cache_view(cache);
  const int ctas_y =
      (int)ceil_div((int64_t)cache->num_layers * cache->num_kv_heads * 2, UNITS_PER_CTA);
  return launch_pdl(accept_compact_kernel, dim3(batch, ctas_y), dim3(THREADS), 0, stream,
                    static_cast<const int32_t*>(nullptr), static_cast<const int32_t*>(nullptr),
                    static_cast<const int32_t*>(nullptr), static_cast<const int32_t*>(nullptr),
                    num_nodes, prefix_len, static_cast<const int32_t*>(nullptr), max_nodes,
                    max_depth, cv, true, code, accept_path, accept_len,
                    static_cast<int32_t*>(nullptr), static_cast<int32_t*>(nullptr),
                    static_cast<int32_t*>(nullptr), static_cast<int32_t*>(nullptr));
}

}  // namespace tsv
