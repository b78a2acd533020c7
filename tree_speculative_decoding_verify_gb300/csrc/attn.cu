// Tree-verification attention: RoPE + KV append (prep), split-KV partial attention
// (CUDA-core path here; the bf16 tensor-core paths live in attn_umma.cu and
// attn_mma.cu) and the
// log-sum-exp merges of the split partials.
//
// Pages: "推理系统手册 · 投机解码进阶：树形草稿与 EAGLE", section 实现 (forward_with_mask:
// every node attends to the whole committed prefix and, among the tree nodes, to its
// ancestors and itself; grouped-query heads share a KV head) and section 为什么要用树
// (RoPE position = prefix length + depth); the EAGLE v2 walkthrough, section 4
// (tree_decoding: one target pass over all nodes under tree_mask).
//
// Workspace layout (all offsets 256-byte aligned):
//   q_rot  [B, Hkv, rows_pad, D]  rotated queries, row r = node * G + g (bf16 for the
//                                 tensor-core path, f32 otherwise); padding rows are 0
//   o_part [B, Hkv, nsplit, rows_pad, D] f32  unnormalised partial outputs
//   ml     [B, Hkv, nsplit, rows_pad, 2]  f32  (running max m in log2 units, sum l)
//   valid  [B] int32                      request passed the device checks
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "attn_common.cuh"
#include "common.cuh"
#include "kernels.h"

namespace tsv {
namespace {

constexpr int PREP_THREADS = 128;
constexpr int SIMT_WARPS = 8;
constexpr int MERGE_WARPS = 8;
constexpr float LOG2E = 1.4426950408889634f;

// ---- device checks shared by the prep kernel ------------------------------------
__device__ int request_code(const AttnArgs& a, int b) {
  const int T = a.num_nodes[b], P = a.prefix_len[b];
  if (T < 1 || T > a.max_nodes || P < 0 || P > a.max_prefix) return TSV_REQ_BAD_SIZE;
  // slots the kernels touch: the tree, then zeros up to the next multiple of 16
  const int64_t need = ((int64_t)P + T + 15) & ~15LL;
  if (a.layout == TSV_KV_CONTIGUOUS) return need > a.capacity ? TSV_REQ_CAPACITY : TSV_REQ_OK;
  if (need > (int64_t)a.max_blocks * TSV_KV_BLOCK) return TSV_REQ_CAPACITY;
  return TSV_REQ_OK;
}

template <typename T>
__device__ __forceinline__ T* slot_ptr(const AttnArgs& a, T* base, int b, int h, int slot) {
  if (a.layout == TSV_KV_CONTIGUOUS)
    return base + (((int64_t)b * a.hkv + h) * a.capacity + slot) * a.head_dim;
  const int blk = a.block_table[(int64_t)b * a.max_blocks + slot / TSV_KV_BLOCK];
  return base + (((int64_t)blk * a.hkv + h) * TSV_KV_BLOCK + slot % TSV_KV_BLOCK) * a.head_dim;
}

// Eight consecutive elements of T as one (bf16) or two (f32) 16-byte accesses.
template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { u = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void store(__nv_bfloat16* p) const { *reinterpret_cast<uint4*>(p) = u; }
  __device__ __forceinline__ void zero() { u = make_uint4(0, 0, 0, 0); }
  __device__ __forceinline__ void get(float (&f)[8]) const {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ __forceinline__ void set(const float (&f)[8]) {
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  }
};
template <> struct Vec8<float> {
  float4 x, y;
  __device__ __forceinline__ void load(const float* p) {
    x = reinterpret_cast<const float4*>(p)[0];
    y = reinterpret_cast<const float4*>(p)[1];
  }
  __device__ __forceinline__ void store(float* p) const {
    reinterpret_cast<float4*>(p)[0] = x;
    reinterpret_cast<float4*>(p)[1] = y;
  }
  __device__ __forceinline__ void zero() { x = y = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void get(float (&f)[8]) const {
    f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w; f[4] = y.x; f[5] = y.y; f[6] = y.z; f[7] = y.w;
  }
  __device__ __forceinline__ void set(const float (&f)[8]) {
    x = make_float4(f[0], f[1], f[2], f[3]);
    y = make_float4(f[4], f[5], f[6], f[7]);
  }
};

// Rotate-half RoPE of elements m0 .. m0 + 7 of both halves of one head vector.
template <typename T, typename U>
__device__ __forceinline__ void rope8(const T* src, U* dst, int m0, int half, const float* cs,
                                      const float* sn) {
  Vec8<T> a, b;
  a.load(src + m0);
  b.load(src + m0 + half);
  float x1[8], x2[8], y1[8], y2[8];
  a.get(x1);
  b.get(x2);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float c = cs[m0 + e], s = sn[m0 + e];
    y1[e] = x1[e] * c - x2[e] * s;
    y2[e] = x2[e] * c + x1[e] * s;
  }
  Vec8<U> o1, o2;
  o1.set(y1);
  o2.set(y2);
  o1.store(dst + m0);
  o2.store(dst + m0 + half);
}

// One CTA per (node, request): rotate q and k at position_ids, append k/v to the cache and
// zero the cache slots after the tree up to the next multiple of 16; for a node past the
// tree (or a request that failed its checks) zero its output row. Every access moves 16
// bytes. Query rows of the workspace that belong to no node are left as they are: rows
// are independent in every kernel, and such rows are never stored.
template <typename T, typename QT>
__global__ void __launch_bounds__(PREP_THREADS)
prep_kernel(AttnArgs a, const T* __restrict__ q, const T* __restrict__ k_new,
            const T* __restrict__ v_new, RopeTable rope) {
  __shared__ float s_cos[64], s_sin[64];
  griddep_wait();
  griddep_launch();
  const int i = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int D = a.head_dim, H = D / 2, G = a.group;
  int code = request_code(a, b);
  if (code == TSV_REQ_OK && a.layout == TSV_KV_PAGED) {
    const int P = a.prefix_len[b], Tn = a.num_nodes[b];
    const int nblk = (int)((((P + Tn + 15) & ~15) + TSV_KV_BLOCK - 1) / TSV_KV_BLOCK);
    bool bad = false;
    for (int j = tid; j < nblk; j += PREP_THREADS) {
      const int blk = a.block_table[(int64_t)b * a.max_blocks + j];
      bad |= blk < 0 || blk >= a.num_blocks;
    }
    if (__syncthreads_or(bad)) code = TSV_REQ_BAD_BLOCK;
  }
  const bool ok = code == TSV_REQ_OK;
  if (i == 0) {
    if (tid == 0) {
      a.valid[b] = ok ? 1 : 0;
      if (a.err) a.err[b] = code;
    }
  }
  const int Tn = ok ? a.num_nodes[b] : 0;
  const int P = ok ? a.prefix_len[b] : 0;
  const int V8 = D / 8, H8 = H / 8;

  if (i < Tn) {
    const int pos = a.position_ids[(int64_t)b * a.max_nodes + i];
    if (tid < H) {
      // angle in fp64, reduced to [-pi, pi] before the fp32 sin/cos
      const double ang = (double)pos * rope.inv_freq[tid];
      const double two_pi = 6.283185307179586;
      const double red = ang - two_pi * rint(ang * (1.0 / two_pi));
      float sn, cs;
      sincosf((float)red, &sn, &cs);
      s_cos[tid] = cs;
      s_sin[tid] = sn;
    }
    __syncthreads();
    QT* qr = reinterpret_cast<QT*>(a.q_rot);
    const int64_t qbase = (int64_t)b * a.hkv * a.rows_pad;
    const T* qi = q + ((int64_t)b * a.max_nodes + i) * a.hq * D;
    for (int e = tid; e < a.hq * H8; e += PREP_THREADS) {
      const int h = e / H8, m0 = (e % H8) * 8;
      rope8(qi + h * D, qr + ((qbase + (int64_t)(h / G) * a.rows_pad) + (int64_t)i * G + h % G) * D,
            m0, H, s_cos, s_sin);
    }
    const T* ki = k_new + ((int64_t)b * a.max_nodes + i) * a.hkv * D;
    for (int e = tid; e < a.hkv * H8; e += PREP_THREADS) {
      const int h = e / H8, m0 = (e % H8) * 8;
      rope8(ki + h * D, slot_ptr(a, reinterpret_cast<T*>(a.k_cache), b, h, P + i), m0, H, s_cos,
            s_sin);
    }
    const T* vi = v_new + ((int64_t)b * a.max_nodes + i) * a.hkv * D;
    for (int e = tid; e < a.hkv * V8; e += PREP_THREADS) {
      const int h = e / V8, d0 = (e % V8) * 8;
      Vec8<T> x;
      x.load(vi + h * D + d0);
      x.store(slot_ptr(a, reinterpret_cast<T*>(a.v_cache), b, h, P + i) + d0);
    }
    if (i == Tn - 1) {  // zero the slots after the tree up to the next multiple of 16
      const int pad = ((P + Tn + 15) & ~15) - (P + Tn);
      Vec8<T> z;
      z.zero();
      for (int e = tid; e < pad * a.hkv * V8; e += PREP_THREADS) {
        const int j = e / (a.hkv * V8), h = (e / V8) % a.hkv, d0 = (e % V8) * 8;
        z.store(slot_ptr(a, reinterpret_cast<T*>(a.k_cache), b, h, P + Tn + j) + d0);
        z.store(slot_ptr(a, reinterpret_cast<T*>(a.v_cache), b, h, P + Tn + j) + d0);
      }
    }
  } else {
    // no node here (or the request failed its checks): its output row is zero
    T* o = reinterpret_cast<T*>(a.out) + ((int64_t)b * a.max_nodes + i) * a.hq * D;
    Vec8<T> z;
    z.zero();
    for (int e = tid; e < a.hq * V8; e += PREP_THREADS) z.store(o + e * 8);
  }
}

// ---- CUDA-core split-KV attention: one warp per (query row, split) ---------------
template <typename T, int D>
__global__ void __launch_bounds__(SIMT_WARPS * 32)
simt_attn_kernel(AttnArgs a, float scale_log2) {
  constexpr int PER = D / 32;
  griddep_wait();
  griddep_launch();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = blockIdx.x * SIMT_WARPS + warp;
  const int split = blockIdx.y;
  const int b = blockIdx.z / a.hkv, kv = blockIdx.z % a.hkv;
  if (!a.valid[b]) return;
  const int Tn = a.num_nodes[b], P = a.prefix_len[b];
  if (r >= Tn * a.group) return;
  const int node = r / a.group;
  const int keys = P + Tn;
  const int n_tiles = (keys + a.tile_keys - 1) / a.tile_keys;
  const int t0 = split * a.tiles_per_split;
  const int t1 = min(n_tiles, t0 + a.tiles_per_split);
  if (t0 >= t1) return;
  const int j0 = t0 * a.tile_keys, j1 = min(keys, t1 * a.tile_keys);

  const float* qr = reinterpret_cast<const float*>(a.q_rot) +
                    (((int64_t)b * a.hkv + kv) * a.rows_pad + r) * D;
  float qv[PER], o[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) { qv[e] = qr[lane + 32 * e]; o[e] = 0.f; }
  const uint32_t* mrow = a.mask + ((int64_t)b * a.max_nodes + node) * a.mask_words;
  float m = -INFINITY, l = 0.f;
  const T* kc = reinterpret_cast<const T*>(a.k_cache);
  const T* vc = reinterpret_cast<const T*>(a.v_cache);
  for (int j = j0; j < j1; ++j) {
    if (j >= P) {
      const int t = j - P;
      if (!((mrow[t >> 5] >> (t & 31)) & 1u)) continue;
    }
    const T* kr = slot_ptr(a, kc, b, kv, j);
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) dot += qv[e] * to_f32(kr[lane + 32 * e]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(FULL, dot, off);
    const float s = dot * scale_log2;
    const float mn = fmaxf(m, s);
    const float alpha = exp2f(m - mn);
    const float p = exp2f(s - mn);
    l = l * alpha + p;
    const T* vr = slot_ptr(a, vc, b, kv, j);
#pragma unroll
    for (int e = 0; e < PER; ++e) o[e] = o[e] * alpha + p * to_f32(vr[lane + 32 * e]);
    m = mn;
  }
  const int64_t prow = (((int64_t)b * a.hkv + kv) * a.nsplit + split) * a.rows_pad + r;
#pragma unroll
  for (int e = 0; e < PER; ++e) a.o_part[prow * D + lane + 32 * e] = o[e];
  if (lane == 0) {
    a.ml[prow * 2 + 0] = m;
    a.ml[prow * 2 + 1] = l;
  }
}

// ---- merge: one warp per (request, kv head, query row); warp-shuffle LSE ---------
template <typename T>
__global__ void __launch_bounds__(MERGE_WARPS * 32)
merge_kernel(AttnArgs a, T* __restrict__ out) {
  griddep_wait();
  griddep_launch();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = blockIdx.x * MERGE_WARPS + warp;
  const int b = blockIdx.y / a.hkv, kv = blockIdx.y % a.hkv;
  if (r >= a.max_nodes * a.group) return;
  const int D = a.head_dim;
  const int node = r / a.group, g = r % a.group;
  T* dst = out + (((int64_t)b * a.max_nodes + node) * a.hq + kv * a.group + g) * D;
  const bool live = a.valid[b] && node < a.num_nodes[b];
  if (!live) {
    for (int d = lane; d < D; d += 32) dst[d] = from_f32<T>(0.f);
    return;
  }
  const int keys = a.prefix_len[b] + a.num_nodes[b];
  const int n_tiles = (keys + a.tile_keys - 1) / a.tile_keys;
  const int nsp = (n_tiles + a.tiles_per_split - 1) / a.tiles_per_split;
  const int64_t pbase = ((int64_t)b * a.hkv + kv) * a.nsplit;
  // running (M, L) over this lane's splits, then a warp-shuffle combine
  float M = -INFINITY, L = 0.f;
  for (int s = lane; s < nsp; s += 32) {
    const float ms = a.ml[((pbase + s) * a.rows_pad + r) * 2 + 0];
    const float ls = a.ml[((pbase + s) * a.rows_pad + r) * 2 + 1];
    if (ms == -INFINITY) continue;
    const float mn = fmaxf(M, ms);
    L = L * exp2f(M - mn) + ls * exp2f(ms - mn);
    M = mn;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(FULL, M, off);
    const float l2 = __shfl_xor_sync(FULL, L, off);
    const float mn = fmaxf(M, m2);
    if (mn != -INFINITY) {
      L = (M == -INFINITY ? 0.f : L * exp2f(M - mn)) + (m2 == -INFINITY ? 0.f : l2 * exp2f(m2 - mn));
      M = mn;
    }
  }
  const float inv = 1.f / L;
  for (int d = lane; d < D; d += 32) {
    float acc = 0.f;
    for (int s = 0; s < nsp; ++s) {
      const float ms = a.ml[((pbase + s) * a.rows_pad + r) * 2 + 0];
      if (ms == -INFINITY) continue;
      acc += exp2f(ms - M) * a.o_part[((pbase + s) * a.rows_pad + r) * D + d];
    }
    dst[d] = from_f32<T>(acc * inv);
  }
}

// ---- split merge of the bf16 tensor-core paths: one warp per query row -------------
// Combines the key splits of the rows whose request took more than one split: lane s
// holds split s's (m, l) (m in log2 units), the warp forms the log-sum-exp weights
// w_s = 2^(m_s - M) / L, and lane c accumulates output columns 4c .. 4c + 3 over the splits
// (eight partial loads in flight), written as bf16. Rows of a single-split request were
// written by the attention kernel itself; rows past the tree were zeroed by the prep.
constexpr int SMERGE_ROWS = 8;  // warps (query rows) per CTA

__global__ void __launch_bounds__(SMERGE_ROWS * 32)
split_merge_kernel(const AttnArgs a, __nv_bfloat16* __restrict__ out) {
  griddep_wait();
  griddep_launch();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = blockIdx.x * SMERGE_ROWS + warp;
  const int b = blockIdx.y / a.hkv, h = blockIdx.y % a.hkv;
  if (!a.valid[b]) return;
  const int T = a.num_nodes[b], P = a.prefix_len[b];
  if (r >= T * a.group) return;
  const int n_tiles = (P + T + a.tile_keys - 1) / a.tile_keys;
  const int nsp = (n_tiles + a.tiles_per_split - 1) / a.tiles_per_split;
  if (nsp <= 1) return;
  const int64_t pbase = ((int64_t)b * a.hkv + h) * a.nsplit;
  float2 ml = make_float2(-INFINITY, 0.f);
  if (lane < nsp) ml = reinterpret_cast<const float2*>(a.ml)[(pbase + lane) * a.rows_pad + r];
  float M = ml.x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, o));
  const float e = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
  float L = ml.y * e;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(FULL, L, o);
  const float w = L > 0.f ? e / L : 0.f;  // this lane's split weight
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* src = reinterpret_cast<const float4*>(a.o_part) + (pbase * a.rows_pad + r) * 32 + lane;
  const int64_t stride = (int64_t)a.rows_pad * 32;  // float4s between splits
  for (int s0 = 0; s0 < nsp; s0 += 8) {
    float4 x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      x[u] = s0 + u < nsp ? __ldcg(src + (s0 + u) * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float ws = __shfl_sync(FULL, w, (s0 + u) & 31);
      if (s0 + u < nsp && ws != 0.f) {  // a split with no visible key holds no partial
        acc.x += ws * x[u].x;
        acc.y += ws * x[u].y;
        acc.z += ws * x[u].z;
        acc.w += ws * x[u].w;
      }
    }
  }
  const int node = r / a.group;
  __nv_bfloat16* dst = out + (((int64_t)b * a.max_nodes + node) * a.hq + h * a.group + r % a.group) * 128;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  reinterpret_cast<uint2*>(dst)[lane] =
      make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
}

}  // namespace

int launch_split_merge(const AttnPlan& p, const AttnArgs& a, void* out, cudaStream_t stream) {
  dim3 gm((unsigned)ceil_div(p.rows, SMERGE_ROWS), p.batch * p.hkv);
  return launch_pdl(split_merge_kernel, gm, dim3(SMERGE_ROWS * 32), 0, stream, a,
                    static_cast<__nv_bfloat16*>(out));
}

AttnPlan plan_attn(const tsv_attn_shape* shape, const tsv_kv_cache* cache) {
  AttnPlan p{};
  p.batch = shape->batch;
  p.max_nodes = shape->max_nodes;
  p.hq = shape->num_q_heads;
  p.hkv = cache->num_kv_heads;
  p.group = p.hq / p.hkv;
  p.head_dim = cache->head_dim;
  p.dtype = cache->dtype;
  p.max_prefix = shape->max_prefix;
  p.rows = p.max_nodes * p.group;
  // bf16 with head_dim 128: the tcgen05 kernel (attn_umma.cu) on sm_100+, else the
  // warp-level tensor-core kernel (attn_mma.cu)
  p.tensor_core = p.dtype == TSV_DTYPE_BF16 && p.head_dim == 128 && device_cc() >= 80;
  p.umma = p.tensor_core && umma_supported(p);
  p.rows_pad = (int)round_up(p.rows, p.tensor_core ? MMA_M_GROUP : 8);
  p.tile_keys = p.umma ? 128 : (p.tensor_core ? MMA_TILE_KEYS : 128);
  const int64_t keys_max = (int64_t)p.max_prefix + p.max_nodes;
  const int64_t n_tiles = ceil_div(keys_max, p.tile_keys);
  const int sms = device_sm_count();
  if (p.tensor_core) {
    // One CTA per SM. Splits: the count with the shortest estimated makespan for
    // full-length requests (waves x (tiles per split + 2 tiles of fixed cost: the ring's
    // fill and the epilogue)), at least one full wave; partials stay under about half of
    // the KV bytes.
    const int64_t units = (int64_t)p.batch * p.hkv * ceil_div(p.rows, MMA_M_GROUP);
    const int64_t rows_g = std::min<int64_t>(p.rows, MMA_M_GROUP);
    const int64_t cap = std::max<int64_t>(
        1, std::min<int64_t>({n_tiles, keys_max / (2 * rows_g), (int64_t)TSV_ATTN_MAX_SPLITS}));
    int64_t best = 1, best_cost = INT64_MAX;
    for (int64_t ns = 1; ns <= cap; ++ns) {
      const int64_t tps = ceil_div(n_tiles, ns);
      const int64_t eff = ceil_div(n_tiles, tps);
      const int64_t cost = ceil_div(units * eff, sms) * (tps + 2);
      if (cost < best_cost) { best_cost = cost; best = ns; }
    }
    best = std::min(cap, std::max(best, ceil_div((int64_t)sms, units)));
    p.tiles_per_split = (int)ceil_div(n_tiles, best);
  } else {
    const int64_t ctas = (int64_t)p.batch * p.hkv;
    int64_t nsplit = std::max<int64_t>(1, ceil_div(2LL * sms, ctas));
    nsplit = std::min<int64_t>(nsplit, n_tiles);
    p.tiles_per_split = (int)ceil_div(n_tiles, nsplit);
  }
  p.nsplit = (int)ceil_div(n_tiles, p.tiles_per_split);
  const size_t qsize = p.tensor_core ? 2 : 4;
  const size_t planes = (size_t)p.batch * p.hkv;
  size_t off = 0;
  p.off_qrot = off;
  off += align256(planes * p.rows_pad * p.head_dim * qsize);
  p.off_opart = off;
  off += align256(planes * p.nsplit * p.rows_pad * p.head_dim * sizeof(float));
  p.off_ml = off;
  off += align256(planes * p.nsplit * p.rows_pad * 2 * sizeof(float));
  p.off_valid = off;
  off += align256((size_t)p.batch * sizeof(int32_t));
  p.ws_bytes = off;
  return p;
}

int launch_attn(const AttnPlan& p, const void* q, const void* k_new, const void* v_new,
                const tsv_kv_cache* cache, const int32_t* prefix_len, const int32_t* num_nodes,
                const int32_t* position_ids, const uint32_t* mask, float rope_theta,
                float softmax_scale, void* out, void* ws, int32_t* err, cudaStream_t stream) {
  char* w = static_cast<char*>(ws);
  AttnArgs a{};
  a.k_cache = cache->k;
  a.v_cache = cache->v;
  a.block_table = cache->block_table;
  a.capacity = cache->capacity;
  a.layout = cache->layout;
  a.max_blocks = cache->max_blocks;
  a.num_blocks = cache->num_blocks;
  a.prefix_len = prefix_len;
  a.num_nodes = num_nodes;
  a.position_ids = position_ids;
  a.mask = mask;
  a.mask_words = (p.max_nodes + 31) / 32;
  a.err = err;
  a.out = out;
  a.q_rot = w + p.off_qrot;
  a.o_part = reinterpret_cast<float*>(w + p.off_opart);
  a.ml = reinterpret_cast<float*>(w + p.off_ml);
  a.valid = reinterpret_cast<int32_t*>(w + p.off_valid);
  a.max_nodes = p.max_nodes;
  a.hq = p.hq;
  a.hkv = p.hkv;
  a.group = p.group;
  a.head_dim = p.head_dim;
  a.rows_pad = p.rows_pad;
  a.max_prefix = p.max_prefix;
  a.tile_keys = p.tile_keys;
  a.tiles_per_split = p.tiles_per_split;
  a.nsplit = p.nsplit;

  RopeTable rope{};
  for (int m = 0; m < p.head_dim / 2; ++m)
    rope.inv_freq[m] = pow((double)rope_theta, -2.0 * m / p.head_dim);
  const float scale_log2 = softmax_scale * LOG2E;

  dim3 gprep(p.max_nodes, p.batch);
  const dim3 bprep(PREP_THREADS);
  const bool bf16 = p.dtype == TSV_DTYPE_BF16;
  int st;
  if (bf16) {
    using T = __nv_bfloat16;
    if (p.tensor_core)
      st = launch_pdl(prep_kernel<T, T>, gprep, bprep, 0, stream, a, (const T*)q,
                      (const T*)k_new, (const T*)v_new, rope);
    else
      st = launch_pdl(prep_kernel<T, float>, gprep, bprep, 0, stream, a, (const T*)q,
                      (const T*)k_new, (const T*)v_new, rope);
  } else {
    st = launch_pdl(prep_kernel<float, float>, gprep, bprep, 0, stream, a, (const float*)q,
                    (const float*)k_new, (const float*)v_new, rope);
  }
  if (st != TSV_OK) return st;

  if (p.tensor_core) {
    // tensor-core attention plus, when the plan splits the keys, the separate
    // warp-per-row split merge kernel
    return p.umma ? launch_attn_umma(p, a, scale_log2, out, stream)
                  : launch_attn_mma(p, a, scale_log2, out, stream);
  } else {
    dim3 gs((unsigned)ceil_div(p.rows, SIMT_WARPS), p.nsplit, p.batch * p.hkv);
    const dim3 bs(SIMT_WARPS * 32);
    if (bf16) {
      if (p.head_dim == 128) st = launch_pdl(simt_attn_kernel<__nv_bfloat16, 128>, gs, bs, 0, stream, a, scale_log2);
      else st = launch_pdl(simt_attn_kernel<__nv_bfloat16, 64>, gs, bs, 0, stream, a, scale_log2);
    } else {
      if (p.head_dim == 128) st = launch_pdl(simt_attn_kernel<float, 128>, gs, bs, 0, stream, a, scale_log2);
      else st = launch_pdl(simt_attn_kernel<float, 64>, gs, bs, 0, stream, a, scale_log2);
    }
    if (st != TSV_OK) return st;
  }

  dim3 gm((unsigned)ceil_div(p.rows, MERGE_WARPS), p.batch * p.hkv);
  const dim3 bm(MERGE_WARPS * 32);
  if (bf16) return launch_pdl(merge_kernel<__nv_bfloat16>, gm, bm, 0, stream, a, (__nv_bfloat16*)out);
  return launch_pdl(merge_kernel<float>, gm, bm, 0, stream, a, (float*)out);
}

}  // namespace tsv
