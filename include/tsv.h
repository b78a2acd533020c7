/*
 * tsv.h — C ABI of the GB300 (sm_103a) tree speculative-decoding verification library.
 *
 * Hot path of EAGLE-2/3 dynamic-tree speculative decoding, one GPU:
 *   tsv_draft_topk_expand   one level of the draft tree expansion (per-row log-softmax +
 *                           top-k, cumulative scores, joint top-k pruning)
 *   tsv_draft_select_final  the total_tokens best candidates laid out as a tree
 *   tsv_draft_select_tree   tsv_draft_select_final and tsv_tree_build_meta in one launch
 *   tsv_draft_topk_expand_product, tsv_draft_to_target, tsv_draft_fixed_level
 *                           expansion variants: probability-product scores, the d2t id
 *                           map, fixed-branching trees
 *   tsv_tree_build_meta     ancestor bitmask, positions, retrieve_indices, child/sibling links
 *   tsv_draft_grow_mask     the drafter's mask and positions grown by one level
 *   tsv_tree_verify_attn    RoPE + KV append + tree-masked split-KV attention of every node
 *   tsv_lm_head_argmax      the target's greedy token at every node (lm_head GEMM with an
 *                           argmax epilogue; the logits are never written)
 *   tsv_accept_and_compact  greedy acceptance walk + move of the accepted KV to
 *                           consecutive slots
 *   tsv_tree_sample_accept  non-greedy acceptance: filtered target probabilities per node,
 *                           tree rejection walk, correction sample, KV move
 *   tsv_target_probs        the filtered target probabilities themselves
 *
 * Pages cited (by title):
 *   [TRT]    "TensorRT-LLM 源码完全拆解(二十二): EAGLE-3 一体式草稿——三层隐状态、草稿循环
 *            与动态树验证"
 *   [HB]     "推理系统手册 · 投机解码进阶：树形草稿与 EAGLE"
 *   [EAGLE2] the EAGLE v2 dynamic-tree walkthrough (initialize_tree / topK_generate /
 *            tree_decoding / evaluate_posterior), sections 3-5
 *   [MO]     "EAGLE头结构深潜: Model Optimizer 投机解码草稿模型的内部设计"
 *
 * Conventions for every call:
 *   - Every array pointer is a DEVICE pointer owned by the caller, unless stated. The
 *     library allocates no memory and keeps no state between calls beyond a per-device
 *     cache of device attributes.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     and never synchronise the host. They can be captured into a CUDA graph. Kernels
 *     are launched with programmatic stream serialization: a kernel may be scheduled
 *     while the previous work of the stream finishes, but it waits for that work to
 *     complete before its first memory access, so stream order holds as usual.
 *   - The return value is a tsv_status. Host-side checks (null pointers, sizes,
 *     workspace) happen before anything is launched; on failure nothing is launched.
 *   - Data-dependent faults (a malformed tree, a request that does not fit its cache)
 *     are found on the device: a per-request code is written to the caller's `err`
 *     array (where the call has one) and that request's outputs are left in the
 *     documented safe state. Nothing traps; every device loop is bounded.
 *   - Node 0 of every tree is the root (the last token the target model committed);
 *     parents precede children; parents[0] == -1.
 *   - Integer arrays are int32 unless stated; "[a, b]" is a row-major shape.
 */
#ifndef TSV_H
#define TSV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* tsv_stream_t; /* a cudaStream_t */

/* ---- status codes (return values) ---- */
enum tsv_status {
  TSV_OK = 0,
  TSV_ERR_INVALID_ARG = 1, /* null pointer, size out of range, inconsistent sizes */
  TSV_ERR_UNSUPPORTED = 2, /* dtype / head_dim / device not supported */
  TSV_ERR_WORKSPACE = 3,   /* workspace pointer null or too small */
  TSV_ERR_CUDA = 4         /* a CUDA call failed; see tsv_last_cuda_error() */
};

/* ---- per-request device error codes (written to err[b]) ---- */
enum tsv_request_error {
  TSV_REQ_OK = 0,
  TSV_REQ_BAD_ROOT = 1,     /* parents[b][0] != -1 */
  TSV_REQ_BAD_PARENT = 2,   /* some parents[b][i] outside [0, i) */
  TSV_REQ_TOO_DEEP = 3,     /* a root-to-node path longer than max_depth + 1 nodes */
  TSV_REQ_BAD_SIZE = 4,     /* num_nodes[b] outside [1, max_nodes] or prefix_len[b] < 0 */
  TSV_REQ_CAPACITY = 5,     /* prefix_len[b] + num_nodes[b] does not fit the KV cache */
  TSV_REQ_BAD_BLOCK = 6,    /* a block-table entry outside [0, num_blocks) */
  TSV_REQ_BAD_LINKS = 7,    /* child/sibling links leave the tree */
  TSV_REQ_TIMEOUT = 8,      /* a bounded device-side wait gave up (the request's outputs
                               are not valid; the GPU context stays usable) */
  TSV_REQ_BAD_TOKEN = 9     /* a draft token outside the d2t table (tsv_draft_to_target) */
};

/* ---- limits ---- */
#define TSV_MAX_NODES 256 /* nodes per tree, root included */
#define TSV_MAX_TOPK 16   /* top_k of the expansion */
#define TSV_MAX_DEPTH 64  /* max_depth (edges from the root to the deepest node) */
#define TSV_KV_BLOCK 64   /* tokens per paged KV block */
#define TSV_MAX_SAMPLE_VOCAB (1 << 20) /* vocabulary of tsv_tree_sample_accept */

/* ---- element types ---- */
enum tsv_dtype { TSV_DTYPE_F32 = 0, TSV_DTYPE_BF16 = 1 };

/* ---- KV cache description ---- */
enum tsv_kv_layout {
  TSV_KV_CONTIGUOUS = 0, /* k, v: [batch, num_kv_heads, capacity, head_dim] */
  TSV_KV_PAGED = 1       /* k, v: [num_blocks, num_kv_heads, TSV_KV_BLOCK, head_dim];
                            slot s of request b lives in block block_table[b][s / 64],
                            row s % 64 */
};

typedef struct {
  void* k;                     /* keys of layer 0 (keys are stored already rotated) */
  void* v;                     /* values of layer 0 */
  int dtype;                   /* tsv_dtype of k and v */
  int num_kv_heads;            /* Hkv */
  int head_dim;                /* D: 64 or 128 */
  int layout;                  /* tsv_kv_layout */
  int64_t capacity;            /* CONTIGUOUS: slots per (request, kv head), a multiple of 64 */
  const int32_t* block_table;  /* PAGED: [batch, max_blocks] (device) */
  int max_blocks;              /* PAGED: columns of block_table */
  int num_blocks;              /* PAGED: blocks in the pool */
  int num_layers;              /* layers reachable from k/v (>= 1) */
  int64_t layer_stride;        /* elements from one layer's k (or v) to the next layer's */
} tsv_kv_cache;

/* Library version string and a readable name for a tsv_status. */
const char* tsv_version(void);
const char* tsv_status_string(int status);
/* cudaError_t of the last failed CUDA call made by this library on this thread. */
int tsv_last_cuda_error(void);

/* --------------------------------------------------------------------------------
 * tsv_draft_topk_expand — one level of the dynamic draft tree.
 *
 * [EAGLE2] section 3 (树的生长, topK_generate): every frontier row takes its top_k
 * tokens with their log-probabilities; a candidate's cumulative score is its parent's
 * score plus its log-probability (cu_scores = topk_p + scores[:, None]); a joint
 * top_k over the rows * top_k candidates gives the next frontier. [TRT] section
 * 树的三套账: candidates are laid out parent-major (flat = s * top_k + c), so the
 * parent row of a flat index is flat / top_k.
 *
 * logits           fp32, row (b, s) at logits + (b * rows + s) * row_stride; the row's
 *                  first `vocab` entries are the draft logits of frontier node s of
 *                  request b. Level 1 has rows == 1 (the root), later levels
 *                  rows == top_k (the previous level's frontier, best first).
 * level            1-based expansion level: 1 for the base layer, 2 .. depth + 1 after.
 * front_score_in   fp32 [batch, rows]: cumulative score of each frontier node
 * front_store_in   int32 [batch, rows]: store index of each frontier node
 *                  (both NULL at level 1: the root has score 0 and store index -1)
 * store_*          [batch, store_cap]: the candidate store. This level writes entries
 *                  off .. off + rows * top_k - 1, off = 0 at level 1 and
 *                  top_k + (level - 2) * top_k^2 after: the token id, the fp32
 *                  cumulative score and the store index of the parent (-1: root).
 * front_*_out      [batch, top_k]: the next frontier, best first (token id, fp32
 *                  cumulative score, store index). Must not alias the *_in arrays.
 * workspace        device scratch of tsv_draft_topk_expand_workspace_size() bytes,
 *                  zero-filled by the caller before its first use; every call leaves
 *                  it fit for the next (its first bytes hold per-request counters that
 *                  each call returns to zero). One workspace sized for rows = top_k
 *                  serves every level of a request batch.
 *
 * Order and ties: higher values first; equal values go to the lower token id (per
 * row) and to the lower flat index (joint). Log-probabilities are x - logsumexp(row),
 * the log-sum-exp accumulated in fp32 with exact (two-sum) group additions, rounded
 * to fp32; cumulative scores are fp32 sums. Returns TSV_ERR_INVALID_ARG for top_k
 * outside [1, TSV_MAX_TOPK], vocab < top_k, row_stride < vocab, a store too small for
 * this level, or rows inconsistent with level.
 * ------------------------------------------------------------------------------ */
size_t tsv_draft_topk_expand_workspace_size(int batch, int rows, int vocab, int top_k);
/* Kernels one tsv_draft_topk_expand (or _product) call of this shape launches on its stream
 * when the logits rows are 16-byte aligned: 1, or 2 for a large batch (the streaming
 * kernel over equal shares of all rows, then one merge per request). 0 for a shape the
 * call rejects. Host only, no device work. */
int tsv_draft_topk_expand_launches(int batch, int rows, int vocab, int top_k);
int tsv_draft_topk_expand(const float* logits, int batch, int rows, int64_t row_stride,
                          int vocab, int top_k, int level, const float* front_score_in,
                          const int32_t* front_store_in, int store_cap, int32_t* store_token,
                          float* store_score, int32_t* store_parent, int32_t* front_token_out,
                          float* front_score_out, int32_t* front_store_out, void* workspace,
                          size_t workspace_bytes, tsv_stream_t stream);

/* --------------------------------------------------------------------------------
 * tsv_draft_select_final — keep the total_tokens best candidates as a tree.
 *
 * [EAGLE2] section 3: after the last level, the total_tokens highest cumulative
 * scores among the num_candidates = top_k + depth * top_k^2 stored candidates are
 * kept (ties to the lower store index). The kept candidates become nodes 1 ..
 * total_tokens in ascending store index, node 0 is the root; a node's parent is the
 * node of its parent's store index, or 0 for first-level candidates. Because a
 * log-probability is never positive, a kept candidate's parent is always kept.
 *
 * tokens, parents  [batch, max_nodes] out: entries 0 .. total_tokens hold the tree,
 *                  the rest are set to -1.
 * num_nodes        [batch] out (may be NULL): total_tokens + 1.
 * root_token       [batch]: token of node 0.
 * Returns TSV_ERR_INVALID_ARG unless 1 <= total_tokens <= num_candidates <= store_cap
 * and total_tokens + 1 <= max_nodes <= TSV_MAX_NODES, num_candidates <= 4096.
 * ------------------------------------------------------------------------------ */
int tsv_draft_select_final(const int32_t* store_token, const float* store_score,
                           const int32_t* store_parent, int batch, int num_candidates,
                           int store_cap, int total_tokens, const int32_t* root_token,
                           int max_nodes, int32_t* tokens, int32_t* parents, int32_t* num_nodes,
                           tsv_stream_t stream);

/* --------------------------------------------------------------------------------
 * tsv_draft_topk_expand_product — tsv_draft_topk_expand with the probability-product
 * scores of [TRT] section 树的三套账 (_select_topk_draft_tokens: a candidate's score is
 * its parent's score times its own probability, new_scores * previous_scores, ranked
 * as they are; base layer: the probabilities). The child's probability is expf of its
 * fp32 log-probability; the product is an fp32 product. Same arguments, layout, ranking
 * rule (larger score, then the lower flat index) and workspace; front_score_in / out
 * and store_score hold the products. tsv_draft_select_final ranks them unchanged.
 * ------------------------------------------------------------------------------ */
int tsv_draft_topk_expand_product(const float* logits, int batch, int rows, int64_t row_stride,
                                  int vocab, int top_k, int level, const float* front_score_in,
                                  const int32_t* front_store_in, int store_cap,
                                  int32_t* store_token, float* store_score,
                                  int32_t* store_parent, int32_t* front_token_out,
                                  float* front_score_out, int32_t* front_store_out,
                                  void* workspace, size_t workspace_bytes, tsv_stream_t stream);

/* --------------------------------------------------------------------------------
 * tsv_draft_to_target — draft-vocabulary ids to target ids, in place.
 *
 * [MO] section 独立小lm_head草稿词表压缩: a drafter with a smaller vocabulary; the d2t
 * buffer maps each draft id back (draft_token = d2t[draft_token]).
 * tokens      [batch, max_nodes] in/out: nodes 1 .. num_nodes[b]-1 become d2t[token];
 *             node 0 (the root, already a target token) is not touched. An id outside
 *             [0, draft_vocab) becomes -1 (it matches no target token).
 * num_nodes   [batch] in; d2t [draft_vocab] int32 in (device).
 * err         [batch] out (may be NULL): TSV_REQ_BAD_TOKEN where an id was outside the
 *             table, else TSV_REQ_OK.
 * ------------------------------------------------------------------------------ */
int tsv_draft_to_target(int32_t* tokens, const int32_t* num_nodes, int batch, int max_nodes,
                        const int32_t* d2t, int draft_vocab, int32_t* err, tsv_stream_t stream);

/* --------------------------------------------------------------------------------
 * tsv_draft_fixed_level — one level of a fixed-branching draft tree.
 *
 * [HB] section 实现 (build_draft_tree): level l gives every frontier node its
 * top-branching[l] tokens, appended frontier node by frontier node.
 * logits      [batch, frontier, vocab] fp32, rows row_stride floats apart: row f is the
 *             draft's logits at the level's f-th frontier node (NaN never wins).
 * width       tokens per frontier node, 1 .. TSV_MAX_TOPK, <= vocab.
 * first_node  node index of the level's first new node; first_parent that of the first
 *             frontier node (the frontier is first_parent .. first_parent+frontier-1).
 * tokens, parents [batch, max_nodes] out: for f < frontier, r < width, node
 *             first_node + f*width + r gets the f-th row's r-th best token (larger logit,
 *             then the lower id) and parent first_parent + f. Other entries untouched;
 *             the caller writes the root (node 0, parent -1) and num_nodes.
 * Returns TSV_ERR_INVALID_ARG for sizes out of range or nodes past max_nodes.
 * ------------------------------------------------------------------------------ */
int tsv_draft_fixed_level(const float* logits, int batch, int frontier, int64_t row_stride,
                          int vocab, int width, int first_node, int first_parent, int max_nodes,
                          int32_t* tokens, int32_t* parents, tsv_stream_t stream);

/* --------------------------------------------------------------------------------
 * tsv_tree_build_meta — tree metadata, one warp per tree.
 *
 * [HB] section 实现 (tree_mask, depths; positions = prefix length + depth) and section
 * 为什么要用树 (every node sees the prefix, its ancestors and itself; siblings share a
 * position); [TRT] section 树构建内核做了什么 (bit-packed mask, 32 positions per
 * word; retrieve_next_token / retrieve_next_sibling, -1 where absent); [EAGLE2]
 * section 3 (retrieve_indices: one root-to-leaf path per leaf).
 *
 * parents          [batch, max_nodes] in: parent node of each node (entries at and
 *                  beyond num_nodes[b] are ignored).
 * num_nodes        [batch] in: nodes of request b, root included, in [1, max_nodes].
 * prefix_len       [batch] in: committed KV length P_b (>= 0).
 * max_depth        deepest allowed node (edges from the root), <= TSV_MAX_DEPTH.
 * mask             [batch, max_nodes, W] uint32 out, W = ceil(max_nodes / 32): bit j % 32
 *                  of word j / 32 in row i is set iff node j is node i or an ancestor.
 * position_ids     [batch, max_nodes] out: P_b + depth(i).
 * retrieve_indices [batch, max_nodes, max_depth + 1] out: row r is the r-th leaf (in
 *                  ascending node order), columns are the node indices from the root
 *                  to that leaf, -1 padded; rows >= num_leaves[b] are all -1.
 * num_leaves       [batch] out.
 * next_token       [batch, max_nodes] out: lowest-numbered child, or -1.
 * next_sibling     [batch, max_nodes] out: next higher-numbered child of the same
 *                  parent, or -1.
 * err              [batch] out: tsv_request_error. On an error the request's outputs
 *                  hold the root-only tree (every row sees only itself, positions
 *                  P_b, one retrieve row [0, -1, ...], no links, num_leaves 1), so a
 *                  later verification accepts only the root.
 * Rows and columns at and beyond num_nodes[b] are zero (mask) or -1 (the rest);
 * position_ids there are P_b.
 * ------------------------------------------------------------------------------ */
int tsv_tree_build_meta(const int32_t* parents, const int32_t* num_nodes,
                        const int32_t* prefix_len, int batch, int max_nodes, int max_depth,
                        uint32_t* mask, int32_t* position_ids, int32_t* retrieve_indices,
                        int32_t* num_leaves, int32_t* next_token, int32_t* next_sibling,
                        int32_t* err, tsv_stream_t stream);

/* --------------------------------------------------------------------------------
 * tsv_draft_select_tree — tsv_draft_select_final followed by tsv_tree_build_meta of
 * the selected trees, in one launch.
 *
 * [EAGLE2] section 3 (the total_tokens best candidates as a tree, then the tree's
 * retrieve_indices) with the metadata of [HB] section 实现 and [TRT] section
 * 树构建内核做了什么. The arguments up to num_nodes are those of tsv_draft_select_final
 * (num_nodes may be NULL); prefix_len .. err are those of tsv_tree_build_meta, whose
 * parents and num_nodes are the selected trees here (total_tokens + 1 nodes). Every
 * output and every error state is the one of the two calls made in order; err may be
 * NULL. Returns TSV_ERR_INVALID_ARG where either call would.
 * ------------------------------------------------------------------------------ */
int tsv_draft_select_tree(const int32_t* store_token, const float* store_score,
                          const int32_t* store_parent, int batch, int num_candidates,
                          int store_cap, int total_tokens, const int32_t* root_token,
                          int max_nodes, int32_t* tokens, int32_t* parents, int32_t* num_nodes,
                          const int32_t* prefix_len, int max_depth, uint32_t* mask,
                          int32_t* position_ids, int32_t* retrieve_indices, int32_t* num_leaves,
                          int32_t* next_token, int32_t* next_sibling, int32_t* err,
                          tsv_stream_t stream);

/* --------------------------------------------------------------------------------
 * tsv_draft_grow_mask — the drafter's ancestor mask, grown by one level.
 *
 * [TRT] section 首步变长、后续定长 (_build_mask_and_position): per draft level the mask is
 * the block matrix [[old mask, 0], [the new nodes' parents' rows, tree_mask_init]] (old
 * nodes see no new node; a new node sees its parent's ancestors, its parent and itself),
 * and a new node's position is its parent's plus one. The attention of the drafter's
 * nodes is then tsv_tree_verify_attn with this mask and these positions.
 * mask          [batch, max_nodes, ceil(max_nodes/32)] uint32 in/out, the layout of
 *               tsv_tree_build_meta. Rows first_new .. first_new+count-1 are written;
 *               rows below first_new are read (their parents' rows) and not changed.
 *               With first_new == 1 the root's row (bit 0) is written first.
 * position_ids  [batch, max_nodes] in/out: new nodes get their parent's position + 1
 *               (with first_new == 1 the root gets prefix_len[b]).
 * new_parents   [batch, count] in: node index of each new node's parent, in
 *               [0, first_new).
 * prefix_len    [batch] in (read when first_new == 1).
 * err           [batch] out (may be NULL): TSV_REQ_BAD_PARENT where a parent was out of
 *               range (that node's row holds only its own bit, its position is -1).
 * ------------------------------------------------------------------------------ */
int tsv_draft_grow_mask(uint32_t* mask, int32_t* position_ids, const int32_t* new_parents,
                        const int32_t* prefix_len, int batch, int first_new, int count,
                        int max_nodes, int32_t* err, tsv_stream_t stream);

/* --------------------------------------------------------------------------------
 * tsv_tree_verify_attn — tree verification attention of one layer.
 *
 * [HB] section 实现 (forward_with_mask) and section 为什么要用树; [EAGLE2] section 4
 * (tree_decoding); [TRT] section CUDA Graph 里的掩码重排 (the target attention reads
 * the padded [N, ceil(N/32)] bit mask directly).
 * For every request b, node i < T_b = num_nodes[b] and query head h:
 *   q' = RoPE(q[b, i, h], position_ids[b, i]),  k' = RoPE(k_new[b, i, h / G], same)
 *   k' and v_new[b, i, .] are written to cache slot P_b + i (P_b = prefix_len[b]);
 *   out[b, i, h] = softmax_j(scale * q' . K_j) V_j over cache slots j < P_b + T_b,
 *   where slot j < P_b is always visible and slot P_b + t is visible iff bit t of
 *   mask row i is set. G = num_q_heads / num_kv_heads (grouped-query attention).
 * RoPE is the rotate-half form with inverse frequencies rope_theta^(-2m/D).
 *
 * shape            batch, max_nodes (node stride of q/k_new/v_new/out), num_q_heads,
 *                  max_prefix (an upper bound on every prefix_len[b], used to size
 *                  the split-KV grid).
 * q, out           [batch, max_nodes, num_q_heads, head_dim], cache->dtype.
 * k_new, v_new     [batch, max_nodes, num_kv_heads, head_dim], cache->dtype.
 *                  q, k_new, v_new and out start on 16-byte boundaries (the kernels
 *                  move 16 bytes per access); TSV_ERR_INVALID_ARG otherwise.
 * cache            one layer's KV cache (num_layers/layer_stride are ignored). The
 *                  prefix keys must already be rotated. On return slots P_b ..
 *                  P_b + T_b - 1 hold the tree's rotated keys and its values, and the
 *                  slots from P_b + T_b up to the next slot index that is a multiple of
 *                  16 are zero (the tensor-core path reads keys in steps of 16).
 * position_ids, mask  as produced by tsv_tree_build_meta for the same max_nodes.
 * workspace        tsv_tree_verify_attn_workspace_size(shape, cache) bytes of device
 *                  scratch, 256-byte aligned.
 * err              [batch] out (may be NULL): TSV_REQ_BAD_SIZE, TSV_REQ_CAPACITY or
 *                  TSV_REQ_BAD_BLOCK; such a request's outputs are zero and its cache
 *                  is left untouched. TSV_REQ_TIMEOUT if a bounded wait of the
 *                  tensor-core kernel gave up (its outputs are then not valid).
 * Supported: bf16 with head_dim 128 (tcgen05/TMEM tensor-core path), bf16 or f32 with
 * head_dim 64 or 128 (CUDA-core path). num_q_heads % num_kv_heads == 0,
 * max_nodes * G <= 1024.
 * ------------------------------------------------------------------------------ */
typedef struct {
  int batch;
  int max_nodes;
  int num_q_heads;
  int max_prefix;
} tsv_attn_shape;

size_t tsv_tree_verify_attn_workspace_size(const tsv_attn_shape* shape,
                                           const tsv_kv_cache* cache);
/* Kernels one tsv_tree_verify_attn call with this shape and cache launches on its stream:
 * the prep, the attention kernel and, when the plan splits the keys of a row block, the
 * split merge. 0 when the shape is not supported. Host only, no device work. */
int tsv_tree_verify_attn_launches(const tsv_attn_shape* shape, const tsv_kv_cache* cache);
int tsv_tree_verify_attn(const tsv_attn_shape* shape, const void* q, const void* k_new,
                         const void* v_new, const tsv_kv_cache* cache,
                         const int32_t* prefix_len, const int32_t* num_nodes,
                         const int32_t* position_ids, const uint32_t* mask, float rope_theta,
                         float softmax_scale, void* out, void* workspace,
                         size_t workspace_bytes, int32_t* err, tsv_stream_t stream);

/* --------------------------------------------------------------------------------
 * tsv_tree_verify_attn_noalloc — tsv_tree_verify_attn for callers that cannot allocate.
 *
 * The pages have no counterpart of this call; it exists for this library's users. Some
 * callers cannot call cudaMalloc: their device memory is entirely owned by their own
 * pool or arena, or they run in a latency-critical loop where an allocation (which can
 * synchronize the device) is not acceptable, and they cannot size and keep a workspace
 * themselves. This call computes exactly what tsv_tree_verify_attn computes, with the
 * same arguments minus the workspace, and allocates nothing: its scratch is a fixed
 * device array of TSV_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that
 * loads the library holds until the process exits.
 *
 * - Returns TSV_ERR_WORKSPACE when the call would need more scratch than that
 *   (tsv_tree_verify_attn_workspace_size tells how much a shape needs).
 * - The first call on a device looks up the array's device address on that device
 *   (cudaGetSymbolAddress); make that first call before any stream capture. The address
 *   is kept per device together with the CUDA context it was found in: after a device
 *   reset (cudaDeviceReset), or from another context on that device, the next call looks
 *   it up again, so that call too should come before any capture.
 * - Its host checks are those of tsv_tree_verify_attn (the same function runs them), so
 *   both calls return the same status for the same invalid arguments.
 * - Every call on a device shares the one array, and a call leaves its contents behind.
 *   Nothing in it has to start at zero. Calls whose GPU work overlaps (on different
 *   streams, without ordering between them) race on the array and give wrong results.
 * ------------------------------------------------------------------------------ */
#define TSV_NOALLOC_SCRATCH_BYTES (32u << 20) /* 32 MiB per device */

int tsv_tree_verify_attn_noalloc(const tsv_attn_shape* shape, const void* q, const void* k_new,
                                 const void* v_new, const tsv_kv_cache* cache,
                                 const int32_t* prefix_len, const int32_t* num_nodes,
                                 const int32_t* position_ids, const uint32_t* mask,
                                 float rope_theta, float softmax_scale, void* out, int32_t* err,
                                 tsv_stream_t stream);

/* --------------------------------------------------------------------------------
 * tsv_lm_head_argmax — the target model's greedy token at every tree node.
 *
 * [HB] section 实现 (the verifier's forward returns lm_head(norm(x)) for every node; the
 * walk takes pred = logits[node].argmax()); [EAGLE2] section 5 (evaluate_posterior
 * compares each candidate with the target's argmax at its parent); [TRT] section
 * 验证:在树上走一条路径 (target_predict, the argmax at every node, feeds the walk).
 *
 * For every row m: argmax[m] = argmax_v sum_k hidden[m, k] * weight[v, k], the LOWEST v
 * among equal maxima; max_logit[m] = that maximum. bf16 inputs, products accumulated in
 * fp32 on the tensor cores; the maximum is taken over the fp32 logits, so two logits
 * closer than the fp32 accumulation error may order differently from an exact sum.
 *
 * hidden           [rows, hidden_size] bf16 in: final-normed hidden state of every node
 *                  (a batch of trees flattened to rows, e.g. batch * max_nodes).
 * weight           [vocab, hidden_size] bf16 in: the lm_head matrix, row-major.
 * rows             0 .. 2^24 (0 launches nothing).
 * hidden_size      a positive multiple of 64.
 * vocab            >= 1, < 2^31.
 * argmax           [rows] out: the greedy token per row (-1 if a bounded device-side
 *                  wait gave up; never on a healthy GPU).
 * max_logit        [rows] fp32 out (may be NULL): the logit of argmax[m] (NaN with -1).
 * workspace        device scratch of tsv_lm_head_argmax_workspace_size(rows, vocab)
 *                  bytes (depends on the device's SM count), 256-byte aligned.
 * hidden and weight must be 16-byte aligned (they are read with the tensor-memory
 * accelerator). Returns TSV_ERR_UNSUPPORTED on a device without tcgen05 (sm_100 and
 * later), TSV_ERR_INVALID_ARG for a null pointer, a misaligned input or a size out of
 * range, TSV_ERR_WORKSPACE for a missing or small workspace.
 * ------------------------------------------------------------------------------ */
size_t tsv_lm_head_argmax_workspace_size(int rows, int vocab);
int tsv_lm_head_argmax(const void* hidden, const void* weight, int rows, int hidden_size,
                       int vocab, int32_t* argmax, float* max_logit, void* workspace,
                       size_t workspace_bytes, tsv_stream_t stream);

/* --------------------------------------------------------------------------------
 * tsv_tree_sample_accept — non-greedy acceptance on the tree (rejection sampling).
 *
 * [TRT] section 非贪心:只靠目标分布的拒绝采样: the target's logits at every node are
 * filtered into probabilities with the request's sampling parameters (temperature,
 * top-k, top-p, min-p); the walk follows next_token / next_sibling, makes a probability
 * test for each candidate and, where it stops, samples a correction token from the
 * target's distribution ("target-only": no draft probabilities needed).
 * [HB] section 练习, exercise 2 (采样时的树): accept candidate x with probability
 * min(1, p(x)/q(x)); on a rejection p <- norm(max(0, p - q)) and try the next candidate;
 * all rejected: sample one token from the last residual.
 *
 * Per node, the filtered distribution (in this order):
 *   temperature  <= 0 or NaN: greedy (all mass on the first maximum);
 *   top_k        keep the top_k largest logits, ties to the lower token id (<= 0 or
 *                >= vocab: off; 1: greedy);
 *   top_p        on the renormalised result, in that order, keep every token whose
 *                preceding mass is below top_p of the total (the crossing token is kept;
 *                >= 1 or NaN: off; <= 0: only the first token);
 *   min_p        keep tokens whose mass is at least min(min_p, 1) times the largest
 *                (<= 0 or NaN: off);
 * then p(v) = exp((l_v - max l) / temperature) over the kept tokens, normalised. Masses
 * are fp32 (2^((l - m) log2(e) / T)); the sums that decide are compensated fp32 sums
 * in a fixed order, so a call gives the same result on every run.
 * The walk: at the current node take its children in ascending node order; child c
 * with token x is accepted when u_node[c] < min(1, p(x) / q(x)), q(x) = 1 for
 * target-only (draft_probs NULL). Draft-aware: draft_probs[b][node] is the distribution
 * q the node's children were drawn from, one after another without replacement (they
 * are distinct tokens), so the j-th child is tested against q_j = q with the tokens of
 * the children rejected before it set to 0, renormalised (q_0 = q as given). A
 * rejection replaces p by the residual (target-only: p without x; draft-aware:
 * max(0, p - q_j)), renormalised; a residual of zero mass leaves p as it was; if q_j has
 * no mass left the later children are tested against 0 (accepted where p > 0). The
 * output then follows the target distribution exactly when the children were drawn
 * that way. An accepted child becomes the current node. Where no child is accepted
 * (or there are none) the walk stops and bonus_token is sampled from the current
 * residual by inverse CDF in token-id order: the smallest t whose running sum exceeds
 * u_final[b] times the total.
 *
 * target_logits    [batch, max_nodes, vocab] fp32 in (NaN reads as -inf).
 * draft_probs      [batch, max_nodes, vocab] fp32 in, or NULL (target-only).
 * temperature, top_p, min_p  [batch] fp32 in; top_k [batch] int32 in.
 * u_node           [batch, max_nodes] fp32 in: uniforms in [0, 1), one per node (the
 *                  test of node c as a candidate of its parent).
 * u_final          [batch] fp32 in: uniform in [0, 1) of the final sample.
 * tokens, next_token, next_sibling, num_nodes, prefix_len, tree_valid, max_depth,
 * cache, accept_path, accept_len, slot_map, new_prefix_len, err: as for
 *                  tsv_accept_and_compact (a request without a tree, or with an error,
 *                  accepts the root alone and its token is sampled at the root; with
 *                  TSV_REQ_BAD_SIZE bonus_token is -1).
 * bonus_token      [batch] out: the sampled token where the walk stopped.
 * workspace        tsv_tree_sample_accept_workspace_size(batch, max_nodes) bytes,
 *                  256-byte aligned; nothing in it has to start at zero.
 * Returns TSV_ERR_INVALID_ARG for a null pointer, vocab outside [1,
 * TSV_MAX_SAMPLE_VOCAB], or sizes out of range.
 * ------------------------------------------------------------------------------ */
size_t tsv_tree_sample_accept_workspace_size(int batch, int max_nodes);
int tsv_tree_sample_accept(const float* target_logits, const float* draft_probs, int vocab,
                           const float* temperature, const int32_t* top_k, const float* top_p,
                           const float* min_p, const float* u_node, const float* u_final,
                           const int32_t* tokens, const int32_t* next_token,
                           const int32_t* next_sibling, const int32_t* num_nodes,
                           const int32_t* prefix_len, const int32_t* tree_valid, int batch,
                           int max_nodes, int max_depth, const tsv_kv_cache* cache,
                           int32_t* accept_path, int32_t* accept_len, int32_t* bonus_token,
                           int32_t* slot_map, int32_t* new_prefix_len, int32_t* err,
                           void* workspace, size_t workspace_bytes, tsv_stream_t stream);

/* tsv_target_probs — the filtered target probabilities of tsv_tree_sample_accept,
 * written out: probs [batch, max_nodes, vocab] fp32 (rows of nodes at or past
 * num_nodes[b] are not written). Same arguments and workspace. */
int tsv_target_probs(const float* target_logits, int vocab, const float* temperature,
                     const int32_t* top_k, const float* top_p, const float* min_p,
                     const int32_t* num_nodes, int batch, int max_nodes, float* probs,
                     void* workspace, size_t workspace_bytes, tsv_stream_t stream);

/* --------------------------------------------------------------------------------
 * tsv_accept_and_compact — greedy acceptance walk and KV compaction.
 *
 * [HB] section 实现 (tree_speculative_generate: from the root, step to the child whose
 * token equals the target's argmax at the current node, the lowest-numbered one;
 * stop when none matches; the bonus token is the argmax at the last accepted node;
 * only the accepted nodes' KV is kept, nothing is recomputed); [TRT] section
 * 验证:在树上走一条路径 (the walk follows next_token / next_sibling) and section
 * 接受之后:KV 从树形搬回线性 (the accepted nodes' KV moves to consecutive slots).
 *
 * tokens           [batch, max_nodes] in: node tokens (node 0 = root).
 * next_token, next_sibling  [batch, max_nodes] in: links from tsv_tree_build_meta.
 * tree_valid       [batch] in (may be NULL: every request has a tree): 0 = the request
 *                  has no valid tree this step ([TRT] section 每请求一份树,按 slot 存放:
 *                  its slot was released); it takes the single-token path: only the
 *                  root is accepted, its bonus token is target_argmax at the root and
 *                  the cache is not touched.
 * target_argmax    [batch, max_nodes] in: the target model's argmax at every node.
 * cache            may be NULL (walk only). Otherwise, for every layer l <
 *                  num_layers, kv head and i < accept_len[b]:
 *                  slot P_b + i <- slot P_b + accept_path[b][i] (keys and values).
 * accept_path      [batch, max_depth + 1] out: accepted node indices, root first,
 *                  -1 padded.
 * accept_len       [batch] out: accepted nodes including the root (>= 1).
 * bonus_token      [batch] out: target_argmax at the last accepted node.
 * slot_map         [batch, max_depth + 1, 2] out: (source slot, destination slot) per
 *                  accepted node, -1 padded.
 * new_prefix_len   [batch] out: P_b + accept_len[b].
 * err              [batch] out (may be NULL): TSV_REQ_BAD_SIZE, TSV_REQ_BAD_LINKS,
 *                  TSV_REQ_CAPACITY or TSV_REQ_BAD_BLOCK; on an error only the root is
 *                  accepted and the cache is not touched.
 * ------------------------------------------------------------------------------ */
int tsv_accept_and_compact(const int32_t* tokens, const int32_t* next_token,
                           const int32_t* next_sibling, const int32_t* target_argmax,
                           const int32_t* num_nodes, const int32_t* prefix_len,
                           const int32_t* tree_valid, int batch,
                           int max_nodes, int max_depth, const tsv_kv_cache* cache,
                           int32_t* accept_path, int32_t* accept_len, int32_t* bonus_token,
                           int32_t* slot_map, int32_t* new_prefix_len, int32_t* err,
                           tsv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TSV_H */
