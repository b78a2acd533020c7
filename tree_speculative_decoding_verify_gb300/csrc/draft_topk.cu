// Draft tree expansion: per-row log-softmax + top-k, cumulative scores, joint top-k,
// and the final total_tokens selection.
//
// Page: the EAGLE v2 dynamic-tree walkthrough, section 3 (树的生长, topK_generate):
// each frontier row takes its top_k tokens and log-probabilities, a candidate's score is
// its parent's score plus its log-probability (cu_scores = topk_p + scores[:, None]), a
// joint top_k over the top_k * top_k candidates forms the next frontier, and after the
// last level the total_tokens best of all stored candidates are kept. Candidate layout
// follows "TensorRT-LLM 源码完全拆解(二十二)", section 树的三套账 (flat = parent * K +
// child, parent = flat / K).
//
// One kernel per level. Each CTA streams one (row, vocab chunk) once with 128-bit loads:
//   - top-k: a warp-cooperative select. Every warp keeps its best 16 candidates spread
//     over lanes 0-15 and a warp-uniform threshold (its 16th best). A thread only
//     buffers elements that beat the threshold (a handful per row after the first few
//     hundred); when any buffer is nearly full, the whole warp merges buffers and list
//     by a 16-round tournament, so no lane ever runs a divergent insertion.
//   - log-sum-exp: exp(x - ref) against the thread's running maximum ref, summed in fp32
//     groups of 16 terms flushed into an fp64 accumulator. Keeping ref at the maximum
//     makes x - ref exact for every term that matters; when a new maximum arrives the
//     old (ref, sum) pair is parked and combined once at the end (one fp64 exp), so the
//     log-sum-exp is good to about 1e-9 and the fp32 log-probabilities round like fp64.
// The warps' lists merge into the chunk's top-k; the last CTA of a request to finish
// (an atomic ticket) merges the chunks of every row, writes the level's candidates to
// the store and runs the joint top-K of the cumulative scores.
#include <float.h>
#include <limits.h>
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace tsv {
namespace {

constexpr int KMAX = TSV_MAX_TOPK;  // 16: warp list length
constexpr int A_THREADS = 256;
constexpr int A_WARPS = A_THREADS / 32;
constexpr int MAX_CHUNKS = 32;
constexpr int BUF = 8;              // per-thread candidate buffer

struct ChunkStat {
  double sum;  // sum of exp(x - ref) over the chunk
  float ref;
  float pad;
};

struct TopkWs {
  ChunkStat* stat;     // [rows_total, chunks]
  float* val;          // [rows_total, chunks, K]
  int32_t* idx;        // [rows_total, chunks, K]
  unsigned* tickets;   // [batch] finished chunk CTAs of each request (zeroed per call)
};

__host__ __device__ inline TopkWs carve(void* ws, int rows_total, int chunks, int k) {
  char* p = static_cast<char*>(ws);
  TopkWs w;
  const size_t n = (size_t)rows_total * chunks;
  w.stat = reinterpret_cast<ChunkStat*>(p);
  p += (n * sizeof(ChunkStat) + 255) & ~size_t(255);
  w.val = reinterpret_cast<float*>(p);
  p += (n * k * sizeof(float) + 255) & ~size_t(255);
  w.idx = reinterpret_cast<int32_t*>(p);
  p += (n * k * sizeof(int32_t) + 255) & ~size_t(255);
  w.tickets = reinterpret_cast<unsigned*>(p);
  return w;
}

// Order-preserving unsigned image of a float (larger float -> larger unsigned).
__device__ __forceinline__ unsigned ord(float v) {
  const unsigned u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Warp-wide best (value, index) pair — larger value, then lower index — with two
// hardware warp reductions; every lane gets the pair and the lane that holds it.
__device__ __forceinline__ void warp_argmax(float& v, int& i, int& lane_of) {
  const unsigned u = ord(v);
  const unsigned umax = __reduce_max_sync(FULL, u);
  const unsigned imin = __reduce_min_sync(FULL, u == umax ? (unsigned)i : 0xffffffffu);
  const unsigned own = __ballot_sync(FULL, u == umax && (unsigned)i == imin);
  lane_of = __ffs(own) - 1;
  v = __shfl_sync(FULL, v, lane_of);
  i = (int)imin;
}

// Sum of (ref_i, s_i) pairs over a warp against the warp's largest reference: one fp64
// exp per lane whose reference differs (none when they all agree), then fp64 adds.
__device__ __forceinline__ void warp_combine(float& r, double& s) {
  float R = r;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) R = fmaxf(R, __shfl_xor_sync(FULL, R, o));
  if (r != R) s = (s == 0.0) ? 0.0 : s * exp((double)r - (double)R);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(FULL, s, o);
  r = R;
}

__device__ __forceinline__ float4 ld_stream(const float4* p) {
  float4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}

// Per-thread streaming state.
struct Stream {
  // exp-sum
  float ref;    // running maximum
  float g;      // fp32 sum of the current group
  double d;     // fp64 sum against ref
  float ref0;   // parked older reference (-inf: none)
  double d0;    // parked sum against ref0
  // top-k: warp list slot (lanes 0-15), warp threshold, own buffer
  float lv;
  int li;
  float thr_v;
  int thr_i;
  float bv[BUF];
  int bi[BUF];
  int bc;
};

__device__ __forceinline__ void flush(Stream& st) {
  st.d += (double)st.g;
  st.g = 0.f;
}

// d0 * e^(ref0 - ref) + d: the rare merge of two parked sums, kept out of line.
__device__ __noinline__ double merge_pair(double d0, float ref0, double d, float ref) {
  return d0 * exp((double)ref0 - (double)ref) + d;
}

__device__ __forceinline__ void consider(Stream& st, float x, int idx) {
  if (x > st.ref) {  // new maximum: park the old pair
    flush(st);
    st.d0 = st.ref0 == -INFINITY ? st.d : merge_pair(st.d0, st.ref0, st.d, st.ref);
    st.ref0 = st.ref;
    st.d = 0.0;
    st.ref = x;
  }
  st.g += expf(x - st.ref);
  if (better(x, idx, st.thr_v, st.thr_i)) {
#pragma unroll
    for (int s = 0; s < BUF; ++s) {
      if (s == st.bc) { st.bv[s] = x; st.bi[s] = idx; }
    }
    ++st.bc;
  }
}

// Warp merge: new list = best k of (list, all buffers), held by lanes 0 .. k-1;
// threshold = its k-th entry.
__device__ __forceinline__ void warp_merge(Stream& st, int lane, int k) {
  // (inlined at three sites: the streaming loop, its tail and the final merge)
  unsigned taken = 0;       // bit s: buffer slot s used; bit BUF: list slot used
  float nv = -INFINITY;
  int ni = INT_MAX;
  for (int r = 0; r < k; ++r) {
    float v = -INFINITY;
    int i = INT_MAX, which = -1;
    if (lane < k && !(taken >> BUF & 1u) && better(st.lv, st.li, v, i)) {
      v = st.lv; i = st.li; which = BUF;
    }
#pragma unroll
    for (int s = 0; s < BUF; ++s) {
      if (s < st.bc && !(taken >> s & 1u) && better(st.bv[s], st.bi[s], v, i)) {
        v = st.bv[s]; i = st.bi[s]; which = s;
      }
    }
    int who = lane;
    float wv = v;
    int wi = i;
    warp_argmax(wv, wi, who);
    if (lane == who && which >= 0) taken |= 1u << which;
    if (lane == r) { nv = wv; ni = wi; }
  }
  st.lv = nv;
  st.li = ni;
  st.thr_v = __shfl_sync(FULL, nv, k - 1);
  st.thr_i = __shfl_sync(FULL, ni, k - 1);
  st.bc = 0;
}

__global__ void __launch_bounds__(A_THREADS)
topk_level_kernel(const float* __restrict__ logits, int64_t row_stride, int vocab, int rows, int k,
                  int chunks, int chunk_len, int level, bool vec, TopkWs ws,
                  const float* __restrict__ front_score_in, const int32_t* __restrict__ front_store_in,
                  int store_cap, int32_t* __restrict__ store_token, float* __restrict__ store_score,
                  int32_t* __restrict__ store_parent, int32_t* __restrict__ front_token_out,
                  float* __restrict__ front_score_out, int32_t* __restrict__ front_store_out) {
  __shared__ float s_wv[A_WARPS][KMAX];
  __shared__ int s_wi[A_WARPS][KMAX];
  __shared__ float s_red[A_WARPS];
  __shared__ double s_sum[A_WARPS];
  __shared__ float s_cv[A_WARPS][MAX_CHUNKS * KMAX];
  __shared__ int s_ci[A_WARPS][MAX_CHUNKS * KMAX];
  __shared__ float s_cu[KMAX * KMAX];
  __shared__ int s_tok[KMAX * KMAX];
  __shared__ bool s_last;

  const int row = blockIdx.y, chunk = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* x = logits + (int64_t)row * row_stride;
  const int start = chunk * chunk_len;
  const int end = min(vocab, start + chunk_len);

  Stream st;
  st.g = 0.f;
  st.d = 0.0;
  st.ref0 = -INFINITY;
  st.d0 = 0.0;
  st.lv = -INFINITY;
  st.li = INT_MAX;
  st.thr_v = -INFINITY;
  st.thr_i = INT_MAX;
  st.bc = 0;
#pragma unroll
  for (int s = 0; s < BUF; ++s) { st.bv[s] = -INFINITY; st.bi[s] = INT_MAX; }

  // Common starting reference: the largest of the first elements every thread sees.
  float first = -INFINITY;
  for (int e = start + tid * 4; e < min(end, start + tid * 4 + 4); ++e) first = fmaxf(first, x[e]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) first = fmaxf(first, __shfl_xor_sync(FULL, first, o));
  if (lane == 0) s_red[warp] = first;
  __syncthreads();
  first = s_red[0];
#pragma unroll
  for (int w = 1; w < A_WARPS; ++w) first = fmaxf(first, s_red[w]);
  st.ref = fmaxf(first, -FLT_MAX);  // finite, so x = -inf gives a zero term

  // Every thread takes 4 consecutive entries per step (one 128-bit load when the row is
  // 16-byte aligned), two steps prefetched ahead; after each step the warp merges if some
  // buffer could overflow on the next one. All lanes run the same number of steps.
  const int steps = (end - start + 4 * A_THREADS - 1) / (4 * A_THREADS);
  auto load4 = [&](int it) -> float4 {
    const int e = start + 4 * (it * A_THREADS + tid);
    if (vec && e + 3 < end) return ld_stream(reinterpret_cast<const float4*>(x + e));
    float4 r;
    r.x = e < end ? x[e] : -INFINITY;
    r.y = e + 1 < end ? x[e + 1] : -INFINITY;
    r.z = e + 2 < end ? x[e + 2] : -INFINITY;
    r.w = e + 3 < end ? x[e + 3] : -INFINITY;
    return r;
  };
  const float4 none = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  float4 a = steps > 0 ? load4(0) : none;
  float4 bnext = steps > 1 ? load4(1) : none;
  for (int it = 0; it < steps; ++it) {
    const float4 c = it + 2 < steps ? load4(it + 2) : none;
    const int e = start + 4 * (it * A_THREADS + tid);
    if (e < end) consider(st, a.x, e);
    if (e + 1 < end) consider(st, a.y, e + 1);
    if (e + 2 < end) consider(st, a.z, e + 2);
    if (e + 3 < end) consider(st, a.w, e + 3);
    if (__any_sync(FULL, st.bc > BUF - 4)) warp_merge(st, lane, k);
    if ((it & 3) == 3) flush(st);
    a = bnext;
    bnext = c;
  }
  flush(st);
  warp_merge(st, lane, k);  // the warp's final best k

  // exp-sum: fold the parked pair, then combine over the block.
  if (st.ref0 != -INFINITY) st.d += st.d0 * exp((double)st.ref0 - (double)st.ref);
  float R = st.ref;
  double part = st.d;
  warp_combine(R, part);
  __syncthreads();  // s_red was read for the starting reference
  if (lane == 0) { s_red[warp] = R; s_sum[warp] = part; }
  if (lane < k) { s_wv[warp][lane] = st.lv; s_wi[warp][lane] = st.li; }
  __syncthreads();
  if (warp == 0) {
    // block top-k: 8 sorted warp lists, lanes 0-7 hold the list heads
    int ptr = 0;
    const size_t base = ((size_t)row * chunks + chunk) * k;
    for (int r = 0; r < k; ++r) {
      float v = lane < A_WARPS ? s_wv[lane][ptr] : -INFINITY;
      int i = lane < A_WARPS ? s_wi[lane][ptr] : INT_MAX;
      int who = lane;
      warp_argmax(v, i, who);
      if (lane == who) ++ptr;
      if (lane == 0) { ws.val[base + r] = v; ws.idx[base + r] = i; }
    }
    float rr = lane < A_WARPS ? s_red[lane] : -INFINITY;
    double ss = lane < A_WARPS ? s_sum[lane] : 0.0;
    warp_combine(rr, ss);
    if (lane == 0) {
      ChunkStat cs;
      cs.sum = ss;
      cs.ref = rr;
      cs.pad = 0.f;
      ws.stat[(size_t)row * chunks + chunk] = cs;
    }
  }

  // The last CTA of this request to finish merges its rows and runs the joint top-K.
  const int b = row / rows;
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned t = atomicAdd(&ws.tickets[b], 1u);
    s_last = (t == (unsigned)(rows * chunks - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const int off = level == 1 ? 0 : k + (level - 2) * k * k;
  const int64_t srow = (int64_t)b * store_cap;
  for (int s = warp; s < rows; s += A_WARPS) {
    const int r0 = b * rows + s;
    float Rr = -INFINITY;
    double sum = 0.0;
    if (lane < chunks) {  // written by other CTAs: read through L2
      const ChunkStat* cs = &ws.stat[(size_t)r0 * chunks + lane];
      Rr = __ldcg(&cs->ref);
      sum = __ldcg(&cs->sum);
    }
    warp_combine(Rr, sum);
    const double lse = (double)Rr + log(sum);
    float* cv = s_cv[warp];
    int* ci = s_ci[warp];
    for (int t = lane; t < chunks * k; t += 32) {
      const int c = t / k, j = t % k;
      const size_t g = ((size_t)r0 * chunks + c) * k + j;
      cv[c * KMAX + j] = __ldcg(ws.val + g);
      ci[c * KMAX + j] = __ldcg(ws.idx + g);
    }
    __syncwarp();
    const float pscore = level == 1 ? 0.0f : front_score_in[r0];
    const int pstore = level == 1 ? -1 : front_store_in[r0];
    int ptr = 0;
    for (int r = 0; r < k; ++r) {
      float v = (lane < chunks) ? cv[lane * KMAX + ptr] : -INFINITY;
      int i = (lane < chunks) ? ci[lane * KMAX + ptr] : INT_MAX;
      int who = lane;
      warp_argmax(v, i, who);
      if (lane == who) ++ptr;
      if (lane == 0) {
        const float logp = (float)((double)v - lse);
        const float cu = pscore + logp;
        const int flat = s * k + r;
        store_token[srow + off + flat] = i;
        store_score[srow + off + flat] = cu;
        store_parent[srow + off + flat] = pstore;
        s_cu[flat] = cu;
        s_tok[flat] = i;
      }
    }
    __syncwarp();
  }
  __syncthreads();

  // Joint top-K over the rows * K cumulative scores (ties to the lower flat index).
  if (warp == 0) {
    const int n = rows * k;
    unsigned taken = 0;  // bit j: flat lane + 32 j taken
    for (int r = 0; r < k; ++r) {
      float v = -INFINITY;
      int i = INT_MAX;
      for (int j = 0; lane + 32 * j < n; ++j) {
        const int f = lane + 32 * j;
        if (!(taken >> j & 1u) && better(s_cu[f], f, v, i)) { v = s_cu[f]; i = f; }
      }
      int who = lane;
      warp_argmax(v, i, who);
      if (lane == who) taken |= 1u << ((i - lane) / 32);
      if (lane == 0) {
        front_token_out[b * k + r] = s_tok[i];
        front_score_out[b * k + r] = v;
        front_store_out[b * k + r] = off + i;
      }
    }
    if (lane == 0) ws.tickets[b] = 0u;
  }
}

// ---- final selection --------------------------------------------------------------
// Bitonic sort of 64-bit keys (descending score, then ascending store index) in shared
// memory; the first total_tokens keys are the kept candidates, numbered in ascending
// store index by a block prefix sum.
constexpr int F_THREADS = 512;

__device__ __forceinline__ uint64_t sel_key(float score, int idx) {
  uint32_t u = __float_as_uint(score);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // ascending float order as unsigned
  return ((uint64_t)(~u) << 32) | (uint32_t)idx;     // ascending key = descending score
}

__global__ void __launch_bounds__(F_THREADS)
select_final_kernel(const int32_t* __restrict__ store_token, const float* __restrict__ store_score,
                    const int32_t* __restrict__ store_parent, int C, int npow2, int store_cap,
                    int total, const int32_t* __restrict__ root_token, int max_nodes,
                    int32_t* __restrict__ tokens, int32_t* __restrict__ parents,
                    int32_t* __restrict__ num_nodes) {
  extern __shared__ unsigned char smem[];
  uint64_t* s_key = reinterpret_cast<uint64_t*>(smem);          // [npow2]
  int* s_node = reinterpret_cast<int*>(s_key + npow2);          // [C]
  __shared__ int s_warp[F_THREADS / 32];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t srow = (int64_t)b * store_cap;
  for (int c = tid; c < npow2; c += F_THREADS)
    s_key[c] = c < C ? sel_key(store_score[srow + c], c) : ~0ull;
  for (int c = tid; c < C; c += F_THREADS) s_node[c] = 0;
  __syncthreads();
  for (int size = 2; size <= npow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = tid; t < npow2 / 2; t += F_THREADS) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const uint64_t a = s_key[lo], c = s_key[hi];
        if ((a > c) == up) { s_key[lo] = c; s_key[hi] = a; }
      }
      __syncthreads();
    }
  }
  for (int r = tid; r < total; r += F_THREADS) s_node[(int)(s_key[r] & 0xffffffffu)] = 1;
  __syncthreads();
  // Node numbers in ascending store index: each thread owns a contiguous segment.
  const int seg = (C + F_THREADS - 1) / F_THREADS;
  const int c0 = min(C, tid * seg), c1 = min(C, c0 + seg);
  int mine = 0;
  for (int c = c0; c < c1; ++c) mine += s_node[c];
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int before = incl - mine;
  for (int w = 0; w < warp; ++w) before += s_warp[w];
  for (int c = c0; c < c1; ++c) {
    if (s_node[c]) s_node[c] = 1 + before++;
  }
  __syncthreads();
  const int64_t trow = (int64_t)b * max_nodes;
  for (int n = tid; n < max_nodes; n += F_THREADS) {
    if (n > total) { tokens[trow + n] = -1; parents[trow + n] = -1; }
  }
  if (tid == 0) {
    tokens[trow] = root_token[b];
    parents[trow] = -1;
    if (num_nodes) num_nodes[b] = total + 1;
  }
  for (int c = tid; c < C; c += F_THREADS) {
    const int node = s_node[c];
    if (!node) continue;
    tokens[trow + node] = store_token[srow + c];
    const int p = store_parent[srow + c];
    parents[trow + node] = (p >= 0 && p < C) ? s_node[p] : 0;
  }
}

}  // namespace

TopkPlan plan_topk(int batch, int rows, int vocab, int top_k) {
  TopkPlan p{};
  const int64_t rows_total = (int64_t)batch * rows;
  const int64_t target = 4LL * device_sm_count();
  int chunks = (int)std::min<int64_t>(MAX_CHUNKS, std::max<int64_t>(1, ceil_div(target, rows_total)));
  // at least 8192 entries per chunk (short chunks are all fixed cost), lengths a
  // multiple of 4
  chunks = (int)std::max<int64_t>(1, std::min<int64_t>(chunks, ceil_div(vocab, 8192)));
  int chunk_len = (int)round_up(ceil_div(vocab, chunks), 4);
  chunks = (int)ceil_div(vocab, chunk_len);
  p.chunks = chunks;
  p.chunk_len = chunk_len;
  const size_t n = (size_t)rows_total * chunks;
  p.ws_bytes = align256(n * sizeof(ChunkStat)) + align256(n * top_k * sizeof(float)) +
               align256(n * top_k * sizeof(int32_t)) + align256((size_t)batch * sizeof(unsigned));
  return p;
}

int launch_topk_expand(const float* logits, int batch, int rows, int64_t row_stride, int vocab,
                       int top_k, int level, const float* front_score_in,
                       const int32_t* front_store_in, int store_cap, int32_t* store_token,
                       float* store_score, int32_t* store_parent, int32_t* front_token_out,
                       float* front_score_out, int32_t* front_store_out, void* ws,
                       const TopkPlan& plan, cudaStream_t stream) {
  const int rows_total = batch * rows;
  TopkWs w = carve(ws, rows_total, plan.chunks, top_k);
  if (cudaMemsetAsync(w.tickets, 0, (size_t)batch * sizeof(unsigned), stream) != cudaSuccess)
    return launch_status();
  dim3 grid(plan.chunks, rows_total);
  const bool vec = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) && (row_stride % 4 == 0);
  topk_level_kernel<<<grid, A_THREADS, 0, stream>>>(
      logits, row_stride, vocab, rows, top_k, plan.chunks, plan.chunk_len, level, vec, w,
      front_score_in, front_store_in, store_cap, store_token, store_score, store_parent,
      front_token_out, front_score_out, front_store_out);
  return launch_status();
}

int launch_select_final(const int32_t* store_token, const float* store_score,
                        const int32_t* store_parent, int batch, int num_candidates,
                        int store_cap, int total_tokens, const int32_t* root_token,
                        int max_nodes, int32_t* tokens, int32_t* parents, int32_t* num_nodes,
                        cudaStream_t stream) {
  int npow2 = 2;
  while (npow2 < num_candidates) npow2 <<= 1;
  const size_t smem = (size_t)npow2 * sizeof(uint64_t) + (size_t)num_candidates * sizeof(int);
  if (smem > 48 * 1024) {
    static bool attr = false;
    if (!attr) {
      if (cudaFuncSetAttribute(select_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               64 * 1024) != cudaSuccess)
        return launch_status();
      attr = true;
    }
  }
  select_final_kernel<<<batch, F_THREADS, smem, stream>>>(store_token, store_score, store_parent,
                                                          num_candidates, npow2, store_cap,
                                                          total_tokens, root_token, max_nodes,
                                                          tokens, parents, num_nodes);
  return launch_status();
}

}  // namespace tsv
