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
#include "tree_meta.cuh"

namespace tsv {
namespace {

constexpr int WARPS = 4;

__global__ void __launch_bounds__(WARPS * 32)
build_meta_kernel(const int32_t* __restrict__ parents, const int32_t* __restrict__ num_nodes,
                  const int32_t* __restrict__ prefix_len, int batch, int max_nodes,
                  int max_depth, MetaOut o) {
  __shared__ int32_t s_par[WARPS][TSV_MAX_NODES];
  __shared__ int32_t s_depth[WARPS][TSV_MAX_NODES];
  __shared__ int32_t s_first[WARPS][TSV_MAX_NODES];  // first child of a node, -1
  __shared__ int32_t s_last[WARPS][TSV_MAX_NODES];   // last child seen so far, -1
  griddep_wait();
  griddep_launch();
  const int warp = threadIdx.x >> 5;
  const int b = blockIdx.x * WARPS + warp;
  if (b >= batch) return;
  build_meta_warp(b, parents + (int64_t)b * max_nodes, num_nodes[b], prefix_len[b], max_nodes,
                  max_depth, o, s_par[warp], s_depth[warp], s_first[warp], s_last[warp]);
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
  MetaOut o{mask, position_ids, retrieve, num_leaves, next_token, next_sibling, err};
  return launch_pdl(build_meta_kernel, grid, dim3(WARPS * 32), 0, stream, parents, num_nodes,
                    prefix_len, batch, max_nodes, max_depth, o);
}

int launch_grow_mask(uint32_t* mask, int32_t* position_ids, const int32_t* new_parents,
                     const int32_t* prefix_len, int batch, int first_new, int count,
                     int max_nodes, int32_t* err, cudaStream_t stream) {
  return launch_pdl(grow_mask_kernel, dim3(batch), dim3(GT), 0, stream, mask, position_ids,
                    new_parents, prefix_len, first_new, count, max_nodes, err);
}

}  // namespace tsv
