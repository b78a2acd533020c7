// Non-greedy acceptance on the tree: the target's filtered distribution at every node and
// the rejection walk.
//
// Pages: "TensorRT-LLM 源码完全拆解(二十二): EAGLE-3 一体式草稿", section
// 非贪心:只靠目标分布的拒绝采样 (the target's logits at every node are filtered into
// probabilities with the request's temperature / top-k / top-p / min-p; the walk follows
// next_token / next_sibling, tests each candidate against the target's probability and,
// where it stops, samples a correction token from the target's distribution);
// "推理系统手册 · 投机解码进阶：树形草稿与 EAGLE", section 练习, exercise 2 (采样时的树) and
// its answer (accept a candidate x with probability min(1, p(x)/q(x)); on a rejection
// p <- norm(max(0, p - q)) and try the next candidate; all rejected: sample from the
// residual).
//
// Target-only is the rule with q = the point mass on the candidate (accept x with
// probability p(x); a rejection removes x from p); draft-aware takes one draft
// distribution q per node from the caller, from which the node's children (distinct
// tokens) were drawn without replacement: the j-th candidate is tested against q with
// the j - 1 tokens drawn before it removed and renormalised, q_j = q / D_j off those
// tokens (D_0 = 1, D_j = sum(q) - the q of the rejected tokens), and the residual after
// its rejection is norm(max(0, p_j - q_j)).
//
// Kernels:
//   filter_stats_kernel   one 1024-thread CTA per (node, request), 68 KB of shared memory.
//       A node's filtered distribution is described by the largest
//       logit m, c = log2(e)/temperature, a 64-bit key threshold, a min-p bound and the
//       normaliser Z: token v is kept when its key (logit order, then the lower token id)
//       is at least the threshold and its mass e_v = 2^(l_v c - m c) (one FFMA and the
//       hardware base-2 exponential) at least the min-p bound; p(v) = e_v / Z. Every pass
//       keeps four 16-byte loads in flight per thread. The first pass finds m (a float
//       maximum and its first token); the second sums Z (fp32 groups of 16 terms, each
//       added exactly into a (hi, lo) pair) and builds the histogram.
//       Thresholds: a histogram of d = (m - l_v) c over 4096 linear bins of [0, 32) (the
//       last bin also takes everything beyond) with exact 32-bit counts and fp32 masses
//       locates the bins where the top-k count or the top-p mass is reached; those bins'
//       tokens are then gathered, with the compensated mass of everything before them,
//       sorted by key in shared memory and scanned. The fp32 sums that decide use a fixed
//       order, so the result is the same on every run; the atomic fp32 bin masses only
//       choose which bins to gather (with a margin, and a check that widens it). A bin
//       range of more than 2048 tokens goes to a 64-bit radix select instead.
//   sample_walk_kernel    one 512-thread CTA per request: the walk (the logits of a
//       node's candidates are gathered in one round of loads), the residual passes of the
//       draft-aware rule, and the final inverse-CDF sample: per-warp sums of 2048-token
//       tiles, the crossing tile, then a block scan inside it.
//   accept_compact_kernel (accept.cu), given-path mode: the accepted KV rows move.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "kv_view.cuh"

namespace tsv {
namespace {

typedef unsigned long long u64;

constexpr int FT = 1024;    // threads of the filter kernel
constexpr int NB = 4096;    // histogram bins (4 per filter thread)
constexpr float DR = 32.f;  // bins cover d in [0, 32)
constexpr int CAP = 2048;   // tokens gathered and sorted in shared memory
constexpr int WT = 512;     // threads of the walk kernel
constexpr int TILE = 4 * WT;  // tokens per tile of the final sample
constexpr int MAX_TILES = TSV_MAX_SAMPLE_VOCAB / TILE;
static_assert(NB == 4 * FT, "bin scans take four bins per thread");
static_assert(CAP == 2 * FT, "list scans take two entries per thread");

struct RowStats {
  u64 thr;     // kept: key >= thr
  float z;     // sum of the kept masses
  float m;     // largest logit
  float c;     // log2(e) / temperature; 0 = greedy (only the first maximum is kept)
  float mc;    // m * c rounded once: a token's mass is 2^(l c - mc)
  float minp;  // kept: mass >= minp
};

__device__ __forceinline__ float clean(float l) { return l != l ? -INFINITY : l; }
// Order-preserving key: larger logit first, then the lower token id.
__device__ __forceinline__ u64 vkey(float l, int v) {
  unsigned u = __float_as_uint(l);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((u64)u << 32) | (unsigned)(~(unsigned)v);
}
__device__ __forceinline__ float key_value(u64 k) {
  const unsigned u = (unsigned)(k >> 32);
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}
// A token's mass relative to the largest logit is 2^t with t = l c - m c, the exponent
// from one FFMA against mc = m c rounded once per row (t <= 0 up to that rounding; -inf
// for l = -inf), and 2^t from the hardware's base-2 exponential (relative error a few
// units in the last place; masses below 2^-126 flush to zero). Greedy rows (c = 0) keep
// mass 1. Every pass and the walk use these two functions, so the masses agree exactly.
__device__ __forceinline__ float ex2a(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float expo(float l, float c, float mc) { return fmaf(l, c, -mc); }
__device__ __forceinline__ float emass(float l, float c, float mc) {
  return c == 0.f ? 1.f : ex2a(expo(l, c, mc));
}
// Histogram bin of exponent t: d = -t in [0, DR) over NB linear bins; -t >= DR (and
// l = -inf) -> the last bin. Non-decreasing as l decreases.
__device__ __forceinline__ int bin_t(float t) {
  return t > -DR ? min(NB - 1, (int)(-t * (NB / DR))) : NB - 1;
}
__device__ __forceinline__ int bin_of(float l, float c, float mc) { return bin_t(expo(l, c, mc)); }
// key(l, v) >= k0 with the float order first: the 64-bit key only decides a tie in value
// (float order and key order agree on unequal values; -0 and +0 compare equal as floats
// and are then told apart by their keys). kv = key_floor(k0); k0 = 0 keeps every token
// (every key is positive).
__device__ __forceinline__ float key_floor(u64 k0) { return k0 ? key_value(k0) : -INFINITY; }
__device__ __forceinline__ bool key_at_least(float l, int v, float kv, u64 k0) {
  return l > kv || (l == kv && vkey(l, v) >= k0);
}
__device__ __forceinline__ float kept_mass(const RowStats& st, float l, int v) {
  if (!key_at_least(l, v, key_floor(st.thr), st.thr)) return 0.f;
  const float e = emass(l, st.c, st.mc);
  return e >= st.minp ? e : 0.f;
}

// Compensated fp32 sum (the additions of one thread in a fixed order).
struct Kahan {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float y = x - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
  }
  __device__ __forceinline__ float value() const { return s - c; }
};

// Visit every token of a row: f(v, logit), NaN read as -inf; four loads in flight.
template <class F>
__device__ __forceinline__ void for_row(const float* __restrict__ row, int V, bool vec, F&& f) {
  const int bd = blockDim.x;
  if (vec) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int n4 = V >> 2;
    int j = threadIdx.x;
    for (; j + 3 * bd < n4; j += 4 * bd) {
      float4 x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) x[u] = __ldg(r4 + j + u * bd);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = 4 * (j + u * bd);
        f(v, clean(x[u].x));
        f(v + 1, clean(x[u].y));
        f(v + 2, clean(x[u].z));
        f(v + 3, clean(x[u].w));
      }
    }
    for (; j < n4; j += bd) {
      const float4 x = __ldg(r4 + j);
      f(4 * j, clean(x.x));
      f(4 * j + 1, clean(x.y));
      f(4 * j + 2, clean(x.z));
      f(4 * j + 3, clean(x.w));
    }
  } else {
    int v = threadIdx.x;
    for (; v + 3 * bd < V; v += 4 * bd) {
      float x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) x[u] = __ldg(row + v + u * bd);
#pragma unroll
      for (int u = 0; u < 4; ++u) f(v + u * bd, clean(x[u]));
    }
    for (; v < V; v += bd) f(v, clean(__ldg(row + v)));
  }
}

// for_row with g() called after every batch of (up to) 16 tokens a thread visits, and
// after its last tokens: g closes a group of fp32 terms (see Pair).
template <class F, class G>
__device__ __forceinline__ void for_row_batched(const float* __restrict__ row, int V, bool vec,
                                                F&& f, G&& g) {
  const int bd = blockDim.x;
  if (vec) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int n4 = V >> 2;
    int j = threadIdx.x;
    for (; j + 3 * bd < n4; j += 4 * bd) {
      float4 x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) x[u] = __ldg(r4 + j + u * bd);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = 4 * (j + u * bd);
        f(v, clean(x[u].x));
        f(v + 1, clean(x[u].y));
        f(v + 2, clean(x[u].z));
        f(v + 3, clean(x[u].w));
      }
      g();
    }
    for (; j < n4; j += bd) {
      const float4 x = __ldg(r4 + j);
      f(4 * j, clean(x.x));
      f(4 * j + 1, clean(x.y));
      f(4 * j + 2, clean(x.z));
      f(4 * j + 3, clean(x.w));
    }
  } else {
    int v = threadIdx.x;
    for (; v + 3 * bd < V; v += 4 * bd) {
      float x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) x[u] = __ldg(row + v + u * bd);
#pragma unroll
      for (int u = 0; u < 4; ++u) f(v + u * bd, clean(x[u]));
      g();
    }
    for (; v < V; v += bd) f(v, clean(__ldg(row + v)));
  }
  g();
}

// Exact sum of two floats as an unevaluated pair (Knuth's TwoSum): s + e == a + b.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bp = s - a;
  e = (a - (s - bp)) + (b - bp);
}
// A thread's sum of many masses: fp32 groups of at most 16 terms (each term at most a
// few units), every group added exactly into an unevaluated (hi, lo) pair.
struct Pair {
  float hi = 0.f, lo = 0.f, g = 0.f;
  __device__ __forceinline__ void close() {
    float s, e;
    two_sum(hi, g, s, e);
    e += lo;
    hi = s + e;
    lo = e - (hi - s);
    g = 0.f;
  }
  __device__ __forceinline__ float value() const { return hi + lo; }
};

// ---- block-wide helpers (any multiple of 32 threads up to 1024); fixed order ---------
template <typename Tv>
__device__ Tv warp_sum(Tv x) {
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(FULL, x, o);
  return x;
}
template <typename Tv>
__device__ Tv block_sum(Tv x, Tv* sb) {
  x = warp_sum(x);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (l == 0) sb[w] = x;
  __syncthreads();
  x = l < nw ? sb[l] : (Tv)0;
  return warp_sum(x);
}
__device__ u64 block_max_u64(u64 x, u64* sb) {
  for (int o = 16; o; o >>= 1) x = max(x, __shfl_xor_sync(FULL, x, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (l == 0) sb[w] = x;
  __syncthreads();
  x = l < nw ? sb[l] : 0ull;
  for (int o = 16; o; o >>= 1) x = max(x, __shfl_xor_sync(FULL, x, o));
  return x;
}
// Inclusive scan across the block; *total = the block's sum.
template <typename Tv>
__device__ Tv block_scan(Tv x, Tv* sb, Tv* total) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int o = 1; o < 32; o <<= 1) {
    const Tv y = __shfl_up_sync(FULL, x, o);
    if (l >= o) x += y;
  }
  __syncthreads();
  if (l == 31) sb[w] = x;
  __syncthreads();
  Tv base = 0, tot = 0;
  for (int i = 0; i < nw; ++i) {
    const Tv s = sb[i];
    if (i < w) base += s;
    tot += s;
  }
  *total = tot;
  return x + base;
}

// ---- filter kernel ------------------------------------------------------------------
struct FilterSmem {
  unsigned cnt[NB];
  float mass[NB];
  // bin masses during the histogram pass as 32-bit fixed point: bin b's masses lie in
  // (2^-(o+1), 2^-o] with o = b / 128 (its octave of d), so a mass times 2^o is in (1/2, 1]
  // and is added as round(mass * 2^(o + qs)), qs = 32 - bits(V): no bin can overflow.
  // Integer shared-memory atomics cost a fraction of fp32 ones.
  unsigned qm[NB];
  u64 lkey[CAP];
  float lmass[CAP];
  u64 tkey[CAP / 2];  // unsorted copy for the ranking sort
  float tmass[CAP / 2];
  u64 sb[32];
  float sf[32];
  unsigned su[32];
  u64 s_prefix;
  float s_f;
  int s_lo, s_hi, s_n, s_j;
};

__device__ void sort_desc(u64* key, float* val, int n) {  // n a power of two
  for (int k = 2; k <= n; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int p = i ^ j;
        if (p > i) {
          const bool desc = (i & k) == 0;
          const u64 a = key[i], b = key[p];
          if ((a < b) == desc) {
            key[i] = b;
            key[p] = a;
            const float t = val[i];
            val[i] = val[p];
            val[p] = t;
          }
        }
      }
      __syncthreads();
    }
}

// Tokens with bin in [lo, hi] and key >= kmin gathered into S.lkey / S.lmass (sorted by
// key, descending); returns the compensated mass of the tokens with bin < lo (and key >=
// kmin), and in *n the number gathered (more than CAP: not gathered).
__device__ float gather_bins(FilterSmem& S, const float* row, int V, bool vec, float c, float mc,
                             int lo, int hi, u64 kmin, int* n) {
  if (threadIdx.x == 0) S.s_n = 0;
  __syncthreads();
  const float kv = key_floor(kmin);
  Pair pre;
  for_row_batched(row, V, vec, [&](int v, float l) {
    const float t = expo(l, c, mc);
    const int bn = bin_t(t);
    if (bn > hi) return;
    if (kmin != 0ull && !key_at_least(l, v, kv, kmin)) return;
    const float e = ex2a(t);  // non-greedy rows only (c > 0)
    if (bn < lo) {
      pre.g += e;
      return;
    }
    const int pos = atomicAdd(&S.s_n, 1);
    if (pos < CAP) {
      S.lkey[pos] = vkey(l, v);
      S.lmass[pos] = e;
    }
  }, [&] { pre.close(); });
  const float before = block_sum<float>(pre.value(), S.sf);  // synchronises
  *n = S.s_n;
  if (*n <= CAP / 2) {
    // rank by counting (keys are distinct): two barriers instead of a sorting network
    const int nn = *n;
    for (int j = threadIdx.x; j < nn; j += blockDim.x) {
      S.tkey[j] = S.lkey[j];
      S.tmass[j] = S.lmass[j];
    }
    __syncthreads();
    for (int j = threadIdx.x; j < nn; j += blockDim.x) {
      const u64 kj = S.tkey[j];
      int r = 0;
      for (int q = 0; q < nn; ++q) r += S.tkey[q] > kj;
      S.lkey[r] = kj;
      S.lmass[r] = S.tmass[j];
    }
  } else if (*n <= CAP) {
    int np = 2;
    while (np < *n) np <<= 1;
    for (int j = *n + threadIdx.x; j < np; j += blockDim.x) {
      S.lkey[j] = 0ull;
      S.lmass[j] = 0.f;
    }
    __syncthreads();
    sort_desc(S.lkey, S.lmass, np);
  }
  __syncthreads();
  return before;
}

// First entry j of the sorted list whose running mass (after `before`) reaches target;
// n - 1 when none does. *incl = before + the list's mass up to and including j.
__device__ int list_cross(FilterSmem& S, int n, float before, float target, float* incl) {
  if (n <= 0) {
    *incl = before;
    return -1;
  }
  const int j0 = threadIdx.x * 2;
  const float a = j0 < n ? S.lmass[j0] : 0.f;
  const float b = j0 + 1 < n ? S.lmass[j0 + 1] : 0.f;
  float tot;
  const float inc = block_scan<float>(a + b, S.sf, &tot);
  if (threadIdx.x == 0) S.s_j = n - 1;
  __syncthreads();
  const float ex = before + (inc - a - b);
  // the first crossing: the lowest j with before + prefix >= target
  if (j0 < n && ex + a >= target) atomicMin(&S.s_j, j0);
  else if (j0 + 1 < n && ex + a + b >= target) atomicMin(&S.s_j, j0 + 1);
  __syncthreads();
  const int j = S.s_j;
  if (threadIdx.x == (j >> 1)) S.s_f = ex + a + ((j & 1) ? b : 0.f);
  __syncthreads();
  *incl = S.s_f;
  return j;
}

// Fixed-order sum of the sorted list's masses 0 .. upto.
__device__ float list_prefix(FilterSmem& S, int upto) {
  const int j0 = threadIdx.x * 2;
  float x = 0.f;
  if (j0 <= upto) x += S.lmass[j0];
  if (j0 + 1 <= upto) x += S.lmass[j0 + 1];
  return block_sum<float>(x, S.sf);
}

// Bins [lo, hi] (contiguous) whose approximate running mass interval, widened by eps,
// contains target: the bins the exact crossing can be in. Bins past `last` are empty.
__device__ void candidate_bins(FilterSmem& S, float target, float eps, int last) {
  const int j0 = threadIdx.x * 4;
  float loc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) loc += j0 + i <= last ? S.mass[j0 + i] : 0.f;
  float tot;
  const float inc = block_scan<float>(loc, S.sf, &tot);
  if (threadIdx.x == 0) {
    S.s_lo = NB;
    S.s_hi = -1;
  }
  __syncthreads();
  float ex = inc - loc;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int bn = j0 + i;
    if (bn > last) break;
    const float in = ex + S.mass[bn];
    if (ex - eps <= target && target <= in + eps) {
      atomicMin(&S.s_lo, bn);
      atomicMax(&S.s_hi, bn);
    }
    ex = in;
  }
  __syncthreads();
  if (threadIdx.x == 0 && S.s_hi < 0) {  // rounding left no bin: take them all
    S.s_lo = 0;
    S.s_hi = last;
  }
  __syncthreads();
}

// Exact selection among the tokens with bin in [lo, hi] and key >= kmin, in descending key
// order: mode 0 -> the token of rank `want` (0-based); mode 1 -> the first token at which
// `before` + the running mass reaches `target` (the last token when none does). A radix
// select over the 64-bit keys, eight digits of 8 bits, most significant first. Used only
// when the candidate tokens do not fit the sorted list (mode 1 sums its digit masses with
// fp32 atomics, so on that path the result may depend on their order).
__device__ u64 radix_select(FilterSmem& S, const float* row, int V, bool vec, float c, float mc,
                            int lo, int hi, u64 kmin, int mode, unsigned want, float target) {
  unsigned* hc = reinterpret_cast<unsigned*>(S.lkey);  // 256-entry histograms
  float* hm = S.lmass;
  // every thread has read the shared results of the step before (the gathered count in
  // S.s_n, the crossing mass in S.s_f) before thread 0 overwrites them: without this
  // barrier a late reader could see the new values and take another branch of the
  // block-uniform control flow
  __syncthreads();
  if (threadIdx.x == 0) {
    S.s_prefix = 0ull;
    S.s_n = (int)want;
    S.s_f = target;
  }
  for (int d = 7; d >= 0; --d) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) {
      hc[i] = 0u;
      hm[i] = 0.f;
    }
    __syncthreads();
    const u64 prefix = S.s_prefix;
    const int sh = 8 * d;
    for_row(row, V, vec, [&](int v, float l) {
      const int bn = bin_of(l, c, mc);
      if (bn < lo || bn > hi) return;
      const u64 k = vkey(l, v);
      if (k < kmin) return;
      if (d < 7 && (k >> (sh + 8)) != prefix) return;
      const int bk = (int)((k >> sh) & 255ull);
      atomicAdd(&hc[bk], 1u);
      if (mode == 1) atomicAdd(&hm[bk], emass(l, c, mc));
    });
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned w = (unsigned)S.s_n;
      float t = S.s_f;
      unsigned acc = 0;
      float macc = 0.f;
      int pick = -1, last = 0;
      for (int bk = 255; bk >= 0; --bk) {
        if (hc[bk] == 0u) continue;
        last = bk;
        if (mode == 0 ? (acc + hc[bk] > w) : (macc + hm[bk] >= t)) {
          pick = bk;
          break;
        }
        acc += hc[bk];
        macc += hm[bk];
      }
      if (pick >= 0) {
        S.s_n = (int)(w - acc);
        S.s_f = t - macc;
      } else {  // not reached: the last token (every later digit takes its last)
        S.s_n = 0x7fffffff;
        S.s_f = INFINITY;
      }
      S.s_prefix = (prefix << 8) | (u64)(pick >= 0 ? pick : last);
    }
    __syncthreads();
  }
  return S.s_prefix;
}

// Compensated mass of the tokens with key >= kmin (and mass >= minp).
__device__ float kept_total(FilterSmem& S, const float* row, int V, bool vec, float c, float mc,
                            u64 kmin, float minp) {
  const float kv = key_floor(kmin);
  Pair acc;
  for_row_batched(row, V, vec, [&](int v, float l) {
    if (!key_at_least(l, v, kv, kmin)) return;
    const float e = emass(l, c, mc);
    if (e >= minp) acc.g += e;
  }, [&] { acc.close(); });
  return block_sum<float>(acc.value(), S.sf);
}

__global__ void __launch_bounds__(FT, 1)
filter_stats_kernel(const SampleArgs a, RowStats* __restrict__ stats, float* __restrict__ probs) {
  extern __shared__ __align__(16) unsigned char smraw[];
  FilterSmem& S = *reinterpret_cast<FilterSmem*>(smraw);
  griddep_wait();
  griddep_launch();
  const int i = blockIdx.x, b = blockIdx.y;
  const int T = a.max_nodes, V = a.vocab;
  const int n = a.num_nodes[b];
  if (i >= min(n, T)) return;  // absent node (or a request whose size is invalid)
  const float* row = a.logits + ((int64_t)b * T + i) * V;
  const bool vec = (V & 3) == 0 && ((uintptr_t)row & 15u) == 0;

  // the largest logit and its first token (a thread visits its tokens in ascending id)
  float mx = -INFINITY;
  int mi = -1;
  for_row(row, V, vec, [&](int v, float l) {
    if (l > mx || mi < 0) {
      mx = l;
      mi = v;
    }
  });
  const u64 maxkey = block_max_u64(mi >= 0 ? vkey(mx, mi) : 0ull, S.sb);
  const float m = key_value(maxkey);
  const float tau = a.temperature[b];
  const int k = a.top_k[b];
  const float pp = a.top_p[b];
  const float mp = a.min_p[b];
  RowStats st;
  st.m = m;
  const bool greedy = !(tau > 0.f) || k == 1 || pp <= 0.f || isinf(m);
  if (greedy) {
    st.thr = maxkey;
    st.z = 1.f;
    st.c = 0.f;
    st.mc = 0.f;
    st.minp = 0.f;
  } else {
    const float c = 1.4426950408889634f / tau;
    const float mc = m * c;
    st.mc = mc;
    const bool topk_on = k > 1 && k < V;
    const bool topp_on = pp < 1.f;
    st.c = c;
    st.minp = mp > 0.f ? fminf(mp, 1.f) : 0.f;
    u64 thr = 0ull;
    float z = -1.f;  // the kept mass when a scan below has it already
    if (topk_on || topp_on) {
      for (int j = threadIdx.x; j < NB; j += FT) {
        S.cnt[j] = 0u;
        S.qm[j] = 0u;
      }
      const int qs = __clz(V);  // 32 - bits(V)
      __syncthreads();
      // The open last bin takes no atomics (with a peaked row most tokens land there, all
      // on one address); its count and mass follow from the totals below.
      Pair all;
      for_row_batched(row, V, vec, [&](int v, float l) {
        const float t = expo(l, c, mc);
        const float e = ex2a(t);
        all.g += e;
        const int bn = bin_t(t);
        if (bn == NB - 1) return;
        if (topk_on) atomicAdd(&S.cnt[bn], 1u);
        if (topp_on)  // e * 2^(octave + qs), rounded
          atomicAdd(&S.qm[bn], __float2uint_rn(e * __int_as_float((127 + qs + (bn >> 7)) << 23)));
      }, [&] { all.close(); });
      float z1 = block_sum<float>(all.value(), S.sf);  // synchronises
      {
        unsigned cl = 0;
        float ml = 0.f;
        for (int j = threadIdx.x; j < NB - 1; j += FT) {
          cl += S.cnt[j];
          const float mj =
              topp_on ? (float)S.qm[j] * __int_as_float((127 - qs - (j >> 7)) << 23) : 0.f;
          S.mass[j] = mj;
          ml += mj;
        }
        const unsigned ca = block_sum<unsigned>(cl, S.su);
        const float ma = block_sum<float>(ml, S.sf);
        if (threadIdx.x == 0) {
          S.cnt[NB - 1] = (unsigned)V - ca;
          S.mass[NB - 1] = fmaxf(0.f, z1 - ma);
        }
        __syncthreads();
      }
      int bk = NB - 1;  // last bin of the top-k set
      u64 thr_k = 0ull;
      if (topk_on) {
        // the bin holding the k-th token: exact counts
        const int j0 = threadIdx.x * 4;
        unsigned loc = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) loc += S.cnt[j0 + q];
        unsigned tot;
        const unsigned inc = block_scan<unsigned>(loc, S.su, &tot);
        unsigned ex = inc - loc;
        if (ex < (unsigned)k && (unsigned)k <= inc) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (ex + S.cnt[j0 + q] >= (unsigned)k) {
              S.s_lo = j0 + q;
              S.s_j = (int)((unsigned)k - 1u - ex);  // rank inside the bin
              break;
            }
            ex += S.cnt[j0 + q];
          }
        }
        __syncthreads();
        bk = S.s_lo;
        const int r = S.s_j;
        int ng;
        const float before = gather_bins(S, row, V, vec, c, mc, bk, bk, 0ull, &ng);
        if (ng <= CAP) {
          thr_k = S.lkey[r];
          // the top-k mass: everything before bin bk, then the list up to rank r
          z1 = before + list_prefix(S, r);
        } else {
          thr_k = radix_select(S, row, V, vec, c, mc, bk, bk, 0ull, 0, (unsigned)r, 0.f);
          z1 = kept_total(S, row, V, vec, c, mc, thr_k, 0.f);
        }
        z = z1;
      }
      thr = thr_k;
      if (topp_on) {
        const float target = pp * z1;
        // the bins the crossing can be in (the top-k set ends inside bin bk; its part of
        // bin bk replaces the bin's mass)
        if (topk_on) {
          // mass of bin bk inside the set = z1 - the bins before it (approximate)
          float loc = 0.f;
          for (int j = threadIdx.x; j < bk; j += FT) loc += S.mass[j];
          const float pre = block_sum<float>(loc, S.sf);
          if (threadIdx.x == 0) S.mass[bk] = fmaxf(0.f, z1 - pre);
          __syncthreads();
        }
        candidate_bins(S, target, 1e-4f * z1 + 1e-30f, bk);
        int lo = S.s_lo, hi = S.s_hi;
        u64 thr_p = maxkey;
        float zp = -1.f;
        for (int tries = 0; tries < 3; ++tries) {
          if (tries == 2) {  // the last try: the exact select over every bin the crossing
                             // can be in (no gather pass first: its list would be unused)
            thr_p = radix_select(S, row, V, vec, c, mc, 0, bk, thr_k, 1, 0u, target);
            zp = -1.f;
            break;
          }
          int ng;
          const float before = gather_bins(S, row, V, vec, c, mc, lo, hi, thr_k, &ng);
          if (ng > CAP) {  // too many for the sorted list: the exact select over these bins
            thr_p = radix_select(S, row, V, vec, c, mc, lo, hi, thr_k, 1, 0u, target - before);
            zp = -1.f;
            break;
          }
          if (before >= target && lo > 0) {  // the crossing is earlier: widen down
            hi = lo - 1;
            lo = 0;
            continue;
          }
          float incl;
          const int j = list_cross(S, ng, before, target, &incl);
          if (incl < target && hi < bk) {  // the crossing is later: widen up
            lo = hi + 1;
            hi = bk;
            continue;
          }
          if (ng > 0) {
            thr_p = S.lkey[j];
            zp = incl;
          }
          break;
        }
        thr = max(thr_k, thr_p);
        z = thr_p >= thr_k ? zp : z;
      }
    }
    st.thr = thr;
    if (z < 0.f || st.minp > 0.f) z = kept_total(S, row, V, vec, c, mc, thr, st.minp);
    st.z = z;
  }
  if (threadIdx.x == 0) stats[(int64_t)b * T + i] = st;
  if (probs) {
    float* out = probs + ((int64_t)b * T + i) * V;
    const float inv = 1.f / st.z;
    for_row(row, V, false, [&](int v, float l) { out[v] = kept_mass(st, l, v) * inv; });
  }
}

// ---- walk kernel --------------------------------------------------------------------
struct WalkSmem {
  int tok[TSV_MAX_NODES], nxt[TSV_MAX_NODES], sib[TSV_MAX_NODES];
  int kids[TSV_MAX_NODES];
  float kl[TSV_MAX_NODES], kq[TSV_MAX_NODES];
  int removed[TSV_MAX_NODES];
  float rmass[TSV_MAX_NODES];
  // draft-aware, per rejection j at this node: the residual's normaliser (0: p kept as
  // it was) and 1 / D_j, the normaliser of the q that candidate was tested against
  float zr[TSV_MAX_NODES];
  float qi[TSV_MAX_NODES + 1];
  float qrem;  // D of the next candidate: sum(q) less the q of the rejected tokens
  int path[TSV_MAX_DEPTH + 1];
  float tile[MAX_TILES];
  float sf[32];
  RowStats st;
  float zcur;  // target-only: the current node's normaliser after its removals
  float target;
  int node, len, code, nk, acc, nrem, nz, pick, ptile;
};

// Draft-aware residual probability of token v (draft probability q) after `nz`
// rejections at this node. A rejected token already has residual 0 after its own
// rejection (it was rejected only if p_j < q_j there), so removing it from the later
// q_j changes nothing here.
__device__ __forceinline__ float resid_p(const WalkSmem& W, float l, int v, float q) {
  float r = kept_mass(W.st, l, v) / W.st.z;
  for (int j = 0; j < W.nz; ++j)
    if (W.zr[j] > 0.f) r = fmaxf(0.f, r - q * W.qi[j]) / W.zr[j];
  return r;
}
// Weight of token v (logit l, draft probability q) in the final sample, before the
// target-only removals.
__device__ __forceinline__ float final_w(const WalkSmem& W, bool draft, float l, int v, float q) {
  return draft ? resid_p(W, l, v, q) : kept_mass(W.st, l, v);
}
__device__ __forceinline__ bool removed_tok(const WalkSmem& W, int v) {
  for (int r = 0; r < W.nrem; ++r)
    if (W.removed[r] == v) return true;
  return false;
}

__global__ void __launch_bounds__(WT)
sample_walk_kernel(const SampleArgs a, const RowStats* __restrict__ stats, CacheView cache,
                   bool has_cache, int32_t* __restrict__ accept_path,
                   int32_t* __restrict__ accept_len, int32_t* __restrict__ bonus,
                   int32_t* __restrict__ slot_map, int32_t* __restrict__ new_prefix_len,
                   int32_t* __restrict__ err, int32_t* __restrict__ code_out) {
  __shared__ WalkSmem W;
  griddep_wait();
  griddep_launch();
  const int b = blockIdx.x;
  const int T = a.max_nodes, V = a.vocab;
  const int64_t row0 = (int64_t)b * T;
  const int n = a.num_nodes[b];
  const int P = a.prefix_len[b];
  const bool size_ok = n >= 1 && n <= T && P >= 0;
  const bool draft = a.draft_probs != nullptr;
  for (int i = threadIdx.x; i < T; i += WT) {
    const bool in = size_ok && i < n;
    W.tok[i] = in ? a.tokens[row0 + i] : -1;
    W.nxt[i] = in ? a.next_token[row0 + i] : -1;
    W.sib[i] = in ? a.next_sibling[row0 + i] : -1;
  }
  if (threadIdx.x == 0) {
    W.node = 0;
    W.len = 1;
    W.path[0] = 0;
    W.code = size_ok ? TSV_REQ_OK : TSV_REQ_BAD_SIZE;
    W.nrem = 0;
    W.nz = 0;
    if (size_ok) {
      W.st = stats[row0];
      W.zcur = W.st.z;
    }
  }
  __syncthreads();
  const bool has_tree = !a.tree_valid || a.tree_valid[b] != 0;

  if (W.code == TSV_REQ_OK && has_tree) {
    for (int step = 0; step <= a.max_depth; ++step) {
      const int node = W.node;
      const float* lrow = a.logits + (row0 + node) * V;
      const float* qrow = draft ? a.draft_probs + (row0 + node) * V : nullptr;
      if (threadIdx.x == 0) {
        W.st = stats[row0 + node];
        W.zcur = W.st.z;
        W.nrem = 0;
        W.nz = 0;
        W.qi[0] = 1.f;
        W.acc = -1;
        // children in ascending node order: the chain strictly increases within [0, n)
        int nk = 0, c = W.nxt[node], prev = node;
        while (c >= 0) {
          if (c <= prev || c >= n) {
            W.code = TSV_REQ_BAD_LINKS;
            nk = 0;
            break;
          }
          W.kids[nk++] = c;
          prev = c;
          c = W.sib[c];
        }
        W.nk = nk;
      }
      __syncthreads();
      const int nk = W.nk;
      for (int j = threadIdx.x; j < nk; j += WT) {
        const int x = W.tok[W.kids[j]];
        const bool in = x >= 0 && x < V;
        W.kl[j] = in ? clean(lrow[x]) : -INFINITY;
        W.kq[j] = !draft ? 1.f : (in ? qrow[x] : 0.f);
      }
      __syncthreads();
      for (int j = 0; j < nk; ++j) {
        if (threadIdx.x == 0) {
          const int c = W.kids[j];
          const int x = W.tok[c];
          const bool in = x >= 0 && x < V;
          const float km = in ? kept_mass(W.st, W.kl[j], x) : 0.f;
          float p, q = W.kq[j];
          if (!draft) {
            bool gone = false;
            for (int r = 0; r < W.nrem; ++r) gone |= W.removed[r] == x;
            p = gone ? 0.f : km / W.zcur;
            q = 1.f;
          } else {
            p = in ? resid_p(W, W.kl[j], x, q) : 0.f;
            q *= W.qi[W.nz];
          }
          const float ratio = q > 0.f ? p / q : (p > 0.f ? INFINITY : 0.f);
          const float u = a.u_node[row0 + c];
          if (u < fminf(1.f, ratio)) {
            W.acc = j;
          } else if (!draft && p > 0.f && W.zcur - km > 0.f) {
            // the residual without x (a residual of zero mass keeps p as it was)
            W.zcur -= km;
            W.removed[W.nrem] = x;
            W.rmass[W.nrem] = km;
            W.nrem++;
          }
        }
        __syncthreads();
        if (W.acc >= 0) break;
        if (draft) {
          // residual normaliser: sum over v of max(0, p_j(v) - q_j(v)); the first pass
          // at a node also sums q
          const int nz = W.nz;
          const float qs = W.qi[nz];
          Kahan part, qtot;
          for (int v = threadIdx.x; v < V; v += WT) {
            const float q = qrow[v];
            part.add(fmaxf(0.f, resid_p(W, clean(lrow[v]), v, q) - q * qs));
            if (nz == 0) qtot.add(q);
          }
          const float zn = block_sum<float>(part.value(), W.sf);
          const float qsum = nz == 0 ? block_sum<float>(qtot.value(), W.sf) : 0.f;
          if (threadIdx.x == 0) {
            // the next sibling was drawn from q without the tokens drawn before it
            W.qrem = (nz == 0 ? qsum : W.qrem) - W.kq[j];
            W.qi[nz + 1] = W.qrem > 0.f ? 1.f / W.qrem : 0.f;
            W.zr[nz] = zn > 0.f ? zn : 0.f;
            W.nz = nz + 1;
          }
          __syncthreads();
        }
      }
      if (W.acc < 0) break;
      if (threadIdx.x == 0) {
        if (W.len == a.max_depth + 1) {
          W.code = TSV_REQ_BAD_LINKS;
        } else {
          W.path[W.len++] = W.kids[W.acc];
          W.node = W.kids[W.acc];
        }
      }
      __syncthreads();
      if (W.code != TSV_REQ_OK) break;
    }
  }
  if (threadIdx.x == 0 && W.code == TSV_REQ_OK && has_cache) {
    if ((int64_t)P + n > cache_slots(cache)) W.code = TSV_REQ_CAPACITY;
    for (int i = 0; W.code == TSV_REQ_OK && i < W.len; ++i) {
      bool ok = true;
      slot_offset(cache, b, 0, P + W.path[i], &ok);
      slot_offset(cache, b, 0, P + i, &ok);
      if (!ok) W.code = TSV_REQ_BAD_BLOCK;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && W.code != TSV_REQ_OK && size_ok) {
    // on an error only the root is accepted; its token comes from the root's own
    // distribution
    W.node = 0;
    W.len = 1;
    W.nrem = 0;
    W.nz = 0;
    W.st = stats[row0];
    W.zcur = W.st.z;
  }
  __syncthreads();

  // ---- the sample where the walk stopped: the smallest t whose running weight exceeds
  // u * total. Tiles of TILE tokens: warp w sums tiles w, w + 16, ...; the crossing tile
  // is found from the tile sums in order; a block scan inside it finds the token.
  int token = -1;
  if (size_ok) {
    const int node = W.node;
    const float* lrow = a.logits + (row0 + node) * V;
    const float* qrow = draft ? a.draft_probs + (row0 + node) * V : nullptr;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = (V + TILE - 1) / TILE;
    for (int t = warp; t < ntiles; t += WT / 32) {
      // lane l takes tokens t*TILE + 4*(l + 32 q) .. +3, q = 0..15, eight loads in flight
      const int base = t * TILE + 4 * lane;
      float s = 0.f;
      for (int h = 0; h < 2; ++h) {
        float lv[32], qv[32];
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int v = base + 128 * (8 * h + q) + e;
            lv[4 * q + e] = v < V ? __ldg(lrow + v) : -INFINITY;
            qv[4 * q + e] = draft && v < V ? __ldg(qrow + v) : 0.f;
          }
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int v = base + 128 * (8 * h + q) + e;
            if (v < V) s += final_w(W, draft, clean(lv[4 * q + e]), v, qv[4 * q + e]);
          }
      }
      const float ts = warp_sum(s);
      if (lane == 0) W.tile[t] = ts;
    }
    __syncthreads();
    if (threadIdx.x == 0 && !draft)  // the target-only removals
      for (int r = 0; r < W.nrem; ++r) W.tile[W.removed[r] / TILE] -= W.rmass[r];
    __syncthreads();
    if (threadIdx.x == 0) {
      Kahan tot;
      int lastpos = -1;
      for (int t = 0; t < ntiles; ++t) {
        tot.add(W.tile[t]);
        if (W.tile[t] > 0.f) lastpos = t;
      }
      const float target = a.u_final[b] * tot.value();
      Kahan run;
      int pt = -1;
      for (int t = 0; t < ntiles; ++t) {
        if (W.tile[t] > 0.f && run.value() + W.tile[t] > target) {
          pt = t;
          break;
        }
        run.add(W.tile[t]);
      }
      // rounding put the target past the last positive tile: its last token
      W.target = pt >= 0 ? target - run.value() : INFINITY;
      W.ptile = pt >= 0 ? pt : max(lastpos, 0);
      W.pick = 0x7fffffff;
    }
    __syncthreads();
    const int t = W.ptile;
    const int v0 = t * TILE + threadIdx.x * 4;
    float w4[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int v = v0 + q;
      w4[q] = v < V && !(!draft && removed_tok(W, v))
                  ? final_w(W, draft, clean(lrow[v]), v, draft ? qrow[v] : 0.f)
                  : 0.f;
    }
    const float mine = w4[0] + w4[1] + w4[2] + w4[3];
    float tot;
    const float incl = block_scan<float>(mine, W.sf, &tot);
    float acc = incl - mine;
    const float target = W.target;
    int found = -1, lastpos = -1;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (w4[q] > 0.f) {
        lastpos = v0 + q;
        if (found < 0 && acc + w4[q] > target) found = v0 + q;
      }
      acc += w4[q];
    }
    if (found >= 0) atomicMin(&W.pick, found);
    __syncthreads();
    if (W.pick == 0x7fffffff) {
      // rounding put the target past the tile's last positive weight: take that token
      __syncthreads();
      if (threadIdx.x == 0) W.pick = -1;
      __syncthreads();
      if (lastpos >= 0) atomicMax(&W.pick, lastpos);
      __syncthreads();
    }
    token = W.pick;
  }

  const int cols = a.max_depth + 1;
  const int len = W.len;
  for (int i = threadIdx.x; i < cols; i += WT) {
    const bool in = i < len;
    accept_path[(int64_t)b * cols + i] = in ? W.path[i] : -1;
    slot_map[((int64_t)b * cols + i) * 2 + 0] = in ? P + W.path[i] : -1;
    slot_map[((int64_t)b * cols + i) * 2 + 1] = in ? P + i : -1;
  }
  if (threadIdx.x == 0) {
    accept_len[b] = len;
    bonus[b] = token;
    new_prefix_len[b] = (size_ok ? P : 0) + len;
    if (err) err[b] = W.code;
    code_out[b] = W.code;
  }
}

struct SampleWs {
  RowStats* stats;
  int32_t* code;
};
SampleWs carve(void* ws, int batch, int max_nodes) {
  char* p = static_cast<char*>(ws);
  SampleWs w;
  w.stats = reinterpret_cast<RowStats*>(p);
  w.code = reinterpret_cast<int32_t*>(p + align256((size_t)batch * max_nodes * sizeof(RowStats)));
  return w;
}

int launch_filter(const SampleArgs& a, RowStats* stats, float* probs, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return TSV_ERR_UNSUPPORTED;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(filter_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(FilterSmem)) != cudaSuccess)
      return launch_status();
    attr_set[dev] = true;
  }
  return launch_pdl(filter_stats_kernel, dim3(a.max_nodes, a.batch), dim3(FT), sizeof(FilterSmem),
                    stream, a, stats, probs);
}

}  // namespace

size_t sample_ws_bytes(int batch, int max_nodes) {
  return align256((size_t)batch * max_nodes * sizeof(RowStats)) +
         align256((size_t)batch * sizeof(int32_t));
}

int launch_target_probs(const SampleArgs& a, float* probs, void* ws, cudaStream_t stream) {
  const SampleWs w = carve(ws, a.batch, a.max_nodes);
  return launch_filter(a, w.stats, probs, stream);
}

int launch_sample_accept(const SampleArgs& a, const tsv_kv_cache* cache, int32_t* accept_path,
                         int32_t* accept_len, int32_t* bonus, int32_t* slot_map,
                         int32_t* new_prefix_len, int32_t* err, void* ws, cudaStream_t stream) {
  const SampleWs w = carve(ws, a.batch, a.max_nodes);
  int st = launch_filter(a, w.stats, nullptr, stream);
  if (st != TSV_OK) return st;
  st = launch_pdl(sample_walk_kernel, dim3(a.batch), dim3(WT), 0, stream, a,
                  static_cast<const RowStats*>(w.stats), make_cache_view(cache), cache != nullptr,
                  accept_path, accept_len, bonus, slot_map, new_prefix_len, err, w.code);
  if (st != TSV_OK || !cache) return st;
  return launch_compact_given(a.num_nodes, a.prefix_len, a.batch, a.max_nodes, a.max_depth,
                              cache, w.code, accept_path, accept_len, stream);
}

}  // namespace tsv
