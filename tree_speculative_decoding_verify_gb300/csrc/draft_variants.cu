// Variants of the draft expansion: the draft-to-target id map and fixed-branching levels.
//
// Pages: "EAGLE头结构深潜: Model Optimizer 投机解码草稿模型的内部设计", section
// 独立小lm_head草稿词表压缩 (the drafter predicts over a smaller vocabulary; a d2t buffer maps
// every draft id back to the target's: draft_token = d2t[draft_token]);
// "推理系统手册 · 投机解码进阶：树形草稿与 EAGLE", section 实现 (build_draft_tree: level l
// gives every frontier node its top-branching[l] tokens, appended frontier node by
// frontier node, so the tree's shape is fixed and only its tokens depend on the draft).
//
//   draft_to_target_kernel  one CTA per request: nodes 1 .. num_nodes-1 through the table
//       (the root is a token the target committed already); an id outside the table maps
//       to -1, which no target token equals, and marks the request TSV_REQ_BAD_TOKEN.
//   fixed_level_kernel      one CTA per (frontier node, request): the row's `width` best
//       tokens (larger logit, then the lower id) by `width` passes of a block-wide maximum
//       over the keys below the previous pick; each pass after the first reads the row
//       from L2. Writes the new nodes' tokens and (fixed) parents.
#include "common.cuh"
#include "kernels.h"

namespace tsv {
namespace {

constexpr int MT = 128;  // threads of the map kernel
constexpr int XT = 256;  // threads of the fixed-level kernel

__global__ void __launch_bounds__(MT)
draft_to_target_kernel(int32_t* __restrict__ tokens, const int32_t* __restrict__ num_nodes,
                       int max_nodes, const int32_t* __restrict__ d2t, int draft_vocab,
                       int32_t* __restrict__ err) {
  __shared__ int s_bad;
  griddep_wait();
  griddep_launch();
  const int b = blockIdx.x;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  const int n = min(num_nodes[b], max_nodes);
  int bad = 0;
  for (int i = 1 + threadIdx.x; i < n; i += MT) {
    int32_t* t = tokens + (int64_t)b * max_nodes + i;
    const int x = *t;
    const bool in = x >= 0 && x < draft_vocab;
    *t = in ? d2t[x] : -1;
    bad |= !in;
  }
  if (bad) s_bad = 1;
  __syncthreads();
  if (err && threadIdx.x == 0) err[b] = s_bad ? TSV_REQ_BAD_TOKEN : TSV_REQ_OK;
}

__device__ __forceinline__ unsigned long long row_key(float l, int v) {
  unsigned u = __float_as_uint(l != l ? -INFINITY : l);  // NaN never wins
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned)(~(unsigned)v);
}

__global__ void __launch_bounds__(XT)
fixed_level_kernel(const float* __restrict__ logits, int frontier, int64_t row_stride, int vocab,
                   int width, int first_node, int first_parent, int max_nodes,
                   int32_t* __restrict__ tokens, int32_t* __restrict__ parents) {
  __shared__ unsigned long long s_w[XT / 32];
  griddep_wait();
  griddep_launch();
  const int f = blockIdx.x, b = blockIdx.y;
  const float* row = logits + ((int64_t)b * frontier + f) * row_stride;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long prev = ~0ull;
  for (int r = 0; r < width; ++r) {
    unsigned long long best = 0ull;
    for (int v = threadIdx.x; v < vocab; v += XT) {
      const unsigned long long k = row_key(__ldg(row + v), v);
      if (k < prev) best = max(best, k);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) best = max(best, __shfl_xor_sync(FULL, best, o));
    if (lane == 0) s_w[warp] = best;
    __syncthreads();
    best = lane < XT / 32 ? s_w[lane] : 0ull;
#pragma unroll
    for (int o = 16; o; o >>= 1) best = max(best, __shfl_xor_sync(FULL, best, o));
    __syncthreads();  // s_w is rewritten by the next pick
    prev = best;
    if (threadIdx.x == 0) {
      const int64_t at = (int64_t)b * max_nodes + first_node + f * width + r;
      tokens[at] = (int32_t)(~(unsigned)(best & 0xffffffffu));
      parents[at] = first_parent + f;
    }
  }
}

}  // namespace

int launch_draft_to_target(int32_t* tokens, const int32_t* num_nodes, int batch, int max_nodes,
                           const int32_t* d2t, int draft_vocab, int32_t* err,
                           cudaStream_t stream) {
  return launch_pdl(draft_to_target_kernel, dim3(batch), dim3(MT), 0, stream, tokens, num_nodes,
                    max_nodes, d2t, draft_vocab, err);
}

int launch_fixed_level(const float* logits, int batch, int frontier, int64_t row_stride,
                       int vocab, int width, int first_node, int first_parent, int max_nodes,
                       int32_t* tokens, int32_t* parents, cudaStream_t stream) {
  return launch_pdl(fixed_level_kernel, dim3(frontier, batch), dim3(XT), 0, stream, logits,
                    frontier, row_stride, vocab, width, first_node, first_parent, max_nodes,
                    tokens, parents);
}

}  // namespace tsv
