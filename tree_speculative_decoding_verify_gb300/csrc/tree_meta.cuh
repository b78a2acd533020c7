// Tree metadata of one request by one warp (internal): ancestor bitmask, positions,
// retrieve_indices and child/sibling links. Used by tsv_tree_build_meta's kernel and by
// the final selection when it builds the tree it has just laid out.
//
// Pages: "推理系统手册 · 投机解码进阶：树形草稿与 EAGLE", section 实现 (tree_mask: a node
// sees itself and its ancestors; depths; position = prefix length + depth);
// "TensorRT-LLM 源码完全拆解(二十二): EAGLE-3 一体式草稿", section 树构建内核做了什么
// (bit-packed mask of 32 positions per word, retrieve_next_token / next_sibling lists,
// -1 where absent); the EAGLE v2 dynamic-tree walkthrough, section 3 (retrieve_indices,
// one root-to-leaf path per leaf).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace tsv {

// Request b's metadata, called by one whole warp: parents_b [max_nodes] holds the
// request's parents (global or shared memory), T its node count and P its prefix length as
// given; par, dep, first, last are the warp's TSV_MAX_NODES-entry shared-memory scratch.
__device__ __forceinline__ void build_meta_warp(int b, const int32_t* parents_b,
                                                int T, int P, int max_nodes, int max_depth,
                                                const MetaOut& o, int32_t* par, int32_t* dep,
                                                int32_t* first, int32_t* last) {
  const int lane = threadIdx.x & 31;
  uint32_t* mask = o.mask;
  int32_t* position_ids = o.position_ids;
  int32_t* retrieve = o.retrieve;
  int32_t* num_leaves = o.num_leaves;
  int32_t* next_token = o.next_token;
  int32_t* next_sibling = o.next_sibling;
  int32_t* err = o.err;
  const int words = (max_nodes + 31) >> 5;
  const int cols = max_depth + 1;
  const int64_t row0 = (int64_t)b * max_nodes;

  int code = TSV_REQ_OK;
  if (T < 1 || T > max_nodes || P < 0) code = TSV_REQ_BAD_SIZE;
  const int Tn = code == TSV_REQ_OK ? T : 0;

  // Stage parents; check parent-first order.
  bool bad_parent = false;
  for (int i = lane; i < max_nodes; i += 32) {
    int p = i < Tn ? parents_b[i] : -1;
    par[i] = p;
    first[i] = -1;
    last[i] = -1;
    if (i > 0 && i < Tn && (p < 0 || p >= i)) bad_parent = true;
  }
  __syncwarp();
  if (code == TSV_REQ_OK && par[0] != -1) code = TSV_REQ_BAD_ROOT;
  if (code == TSV_REQ_OK && __any_sync(FULL, bad_parent)) code = TSV_REQ_BAD_PARENT;

  // Depth of every node: walk up (parents precede children, so the walk ends at the
  // root within i steps); deeper than max_depth is an error.
  bool too_deep = false;
  if (code == TSV_REQ_OK) {
    for (int i = lane; i < Tn; i += 32) {
      int d = 0, j = i;
      while (j > 0 && d <= max_depth) { j = par[j]; ++d; }
      if (j > 0 || d > max_depth) too_deep = true;
      dep[i] = d;
    }
    if (__any_sync(FULL, too_deep)) code = TSV_REQ_TOO_DEEP;
  }
  __syncwarp();

  if (code != TSV_REQ_OK) {
    // Root-only state: every row sees itself, no links, one retrieve row [0, -1, ...].
    const int pos = P < 0 ? 0 : P;
    for (int i = lane; i < max_nodes; i += 32) {
      for (int w = 0; w < words; ++w)
        mask[(row0 + i) * words + w] = (w == (i >> 5)) ? (1u << (i & 31)) : 0u;
      position_ids[row0 + i] = pos;
      next_token[row0 + i] = -1;
      next_sibling[row0 + i] = -1;
      for (int c = 0; c < cols; ++c)
        retrieve[(row0 + i) * cols + c] = (i == 0 && c == 0) ? 0 : -1;
    }
    if (lane == 0) {
      num_leaves[b] = 1;
      if (err) err[b] = code;
    }
    return;
  }

  // Mask rows: for every word, walk from the node up to the root and keep the bits
  // that fall in that word. Rows at and beyond T are zero.
  for (int i = lane; i < max_nodes; i += 32) {
    for (int w = 0; w < words; ++w) {
      uint32_t bits = 0;
      if (i < T) {
        int j = i;
        while (true) {
          if ((j >> 5) == w) bits |= 1u << (j & 31);
          if (j == 0) break;
          j = par[j];
        }
      }
      mask[(row0 + i) * words + w] = bits;
    }
    position_ids[row0 + i] = P + (i < T ? dep[i] : 0);
  }

  // Child/sibling links, 32 nodes at a time in ascending order: lanes with the same
  // parent form a group; inside a chunk the next sibling is the next lane of the group,
  // across chunks it is linked through last[parent].
  for (int i = lane; i < max_nodes; i += 32) {
    next_token[row0 + i] = -1;
    next_sibling[row0 + i] = -1;
  }
  __syncwarp();
  for (int base = 1; base < T; base += 32) {
    const int i = base + lane;
    const bool live = i < T;
    const int p = live ? par[i] : -1 - lane;  // dead lanes get distinct keys
    const unsigned grp = __match_any_sync(FULL, p);
    const unsigned above = grp & ~((2u << lane) - 1u);      // group lanes after me
    const bool leader = live && (grp & ((1u << lane) - 1u)) == 0;  // lowest lane of group
    const bool tail = live && above == 0;
    if (live && !tail) next_sibling[row0 + i] = base + __ffs(above) - 1;
    const int prev = leader ? last[p] : -1;
    __syncwarp();
    if (leader) {
      if (prev < 0) {
        first[p] = i;
        next_token[row0 + p] = i;
      } else {
        next_sibling[row0 + prev] = i;
      }
    }
    if (tail) last[p] = i;
    __syncwarp();
  }

  // Leaves in ascending order; each leaf's root-to-leaf path is one retrieve row.
  int leaves_before = 0;
  for (int base = 0; base < max_nodes; base += 32) {
    const int i = base + lane;
    const bool leaf = i < T && first[i] < 0;
    const unsigned bal = __ballot_sync(FULL, leaf);
    const int rank = leaves_before + __popc(bal & ((1u << lane) - 1u));
    if (leaf) {
      const int d = dep[i];
      int64_t r = (row0 + rank) * cols;
      for (int c = d + 1; c < cols; ++c) retrieve[r + c] = -1;
      int j = i;
      for (int c = d; c >= 0; --c) {
        retrieve[r + c] = j;
        j = c > 0 ? par[j] : j;
      }
    }
    leaves_before += __popc(bal);
  }
  for (int r = leaves_before + lane; r < max_nodes; r += 32)
    for (int c = 0; c < cols; ++c) retrieve[(row0 + r) * cols + c] = -1;
  if (lane == 0) {
    num_leaves[b] = leaves_before;
    if (err) err[b] = TSV_REQ_OK;
  }
}

}  // namespace tsv
