// Tree metadata, one warp per tree: ancestor bitmask, positions, retrieve_indices and
// child/sibling links.
//
// Pages: "推理系统手册 · 投机解码进阶：树形草稿与 EAGLE", section 实现 (tree_mask: a node
// sees itself and its ancestors; depths; position = prefix length + depth);
// "TensorRT-LLM 源码完全拆解(二十二): EAGLE-3 一体式草稿", section 树构建内核做了什么
// (bit-packed mask of 32 positions per word, retrieve_next_token / next_sibling lists,
// -1 where absent); the EAGLE v2 dynamic-tree walkthrough, section 3 (retrieve_indices,
// one root-to-leaf path per leaf).
#include "common.cuh"
#include "kernels.h"

namespace tsv {
namespace {

constexpr int WARPS = 4;

__global__ void __launch_bounds__(WARPS * 32)
build_meta_kernel(const int32_t* __restrict__ parents, const int32_t* __restrict__ num_nodes,
                  const int32_t* __restrict__ prefix_len, int batch, int max_nodes,
                  int max_depth, uint32_t* __restrict__ mask, int32_t* __restrict__ position_ids,
                  int32_t* __restrict__ retrieve, int32_t* __restrict__ num_leaves,
                  int32_t* __restrict__ next_token, int32_t* __restrict__ next_sibling,
                  int32_t* __restrict__ err) {
  __shared__ int32_t s_par[WARPS][TSV_MAX_NODES];
  __shared__ int32_t s_depth[WARPS][TSV_MAX_NODES];
  __shared__ int32_t s_first[WARPS][TSV_MAX_NODES];  // first child of a node, -1
  __shared__ int32_t s_last[WARPS][TSV_MAX_NODES];   // last child seen so far, -1
  griddep_wait();
  griddep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * WARPS + warp;
  if (b >= batch) return;
  int32_t* par = s_par[warp];
  int32_t* dep = s_depth[warp];
  int32_t* first = s_first[warp];
  int32_t* last = s_last[warp];

  const int words = (max_nodes + 31) >> 5;
  const int cols = max_depth + 1;
  const int64_t row0 = (int64_t)b * max_nodes;
  const int T = num_nodes[b];
  const int P = prefix_len[b];

  int code = TSV_REQ_OK;
  if (T < 1 || T > max_nodes || P < 0) code = TSV_REQ_BAD_SIZE;
  const int Tn = code == TSV_REQ_OK ? T : 0;

  // Stage parents; check parent-first order.
  bool bad_parent = false;
  for (int i = lane; i < max_nodes; i += 32) {
    int p = i < Tn ? parents[row0 + i] : -1;
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

constexpr int GT = 128;

__global__ void __launch_bounds__(GT)
grow_mask_kernel(uint32_t* __restrict__ mask, int32_t* __restrict__ position_ids,
                 const int32_t* __restrict__ new_parents, const int32_t* __restrict__ prefix_len,
                 int first_new, int count, int max_nodes, int32_t* __restrict__ err) {
  __shared__ int s_bad;
  griddep_wait();
  griddep_launch();
  const int b = blockIdx.x;
  const int W = (max_nodes + 31) / 32;
  uint32_t* m = mask + (int64_t)b * max_nodes * W;
  int32_t* pos = position_ids + (int64_t)b * max_nodes;
  if (threadIdx.x == 0) {
    s_bad = 0;
    if (first_new == 1) {  // the first level also writes the root's row
      for (int w = 0; w < W; ++w) m[w] = w == 0 ? 1u : 0u;
      pos[0] = prefix_len[b];
    }
  }
  __syncthreads();
  // new node n = first_new + j: words of its parent's row (bits of old nodes only) and
  // its own bit
  for (int e = threadIdx.x; e < count * W; e += GT) {
    const int j = e / W, w = e % W, n = first_new + j;
    const int p = new_parents[(int64_t)b * count + j];
    const bool ok = p >= 0 && p < first_new;
    uint32_t word = ok && w * 32 < first_new ? m[(int64_t)p * W + w] : 0u;
    if (w == (n >> 5)) word |= 1u << (n & 31);
    m[(int64_t)n * W + w] = word;
    if (w == 0) {
      pos[n] = ok ? pos[p] + 1 : -1;
      if (!ok) s_bad = 1;
    }
  }
  __syncthreads();
  if (err && threadIdx.x == 0) err[b] = s_bad ? TSV_REQ_BAD_PARENT : TSV_REQ_OK;
}

}  // namespace

int launch_build_meta(const int32_t* parents, const int32_t* num_nodes, const int32_t* prefix_len,
                      int batch, int max_nodes, int max_depth, uint32_t* mask,
                      int32_t* position_ids, int32_t* retrieve, int32_t* num_leaves,
                      int32_t* next_token, int32_t* next_sibling, int32_t* err,
                      cudaStream_t stream) {
  dim3 grid((unsigned)ceil_div(batch, WARPS));
  return launch_pdl(build_meta_kernel, grid, dim3(WARPS * 32), 0, stream, parents, num_nodes,
                    prefix_len, batch, max_nodes, max_depth, mask, position_ids, retrieve,
                    num_leaves, next_token, next_sibling, err);
}

int launch_grow_mask(uint32_t* mask, int32_t* position_ids, const int32_t* new_parents,
                     const int32_t* prefix_len, int batch, int first_new, int count,
                     int max_nodes, int32_t* err, cudaStream_t stream) {
  return launch_pdl(grow_mask_kernel, dim3(batch), dim3(GT), 0, stream, mask, position_ids,
                    new_parents, prefix_len, first_new, count, max_nodes, err);
}

}  // namespace tsv
