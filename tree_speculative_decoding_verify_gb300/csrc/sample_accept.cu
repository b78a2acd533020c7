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
// distribution q per node from the caller.
//
// Kernels:
//   filter_stats_kernel   one 1024-thread CTA per (node, request). A node's filtered
//       distribution is described by the largest logit m, c = log2(e)/temperature, a
//       64-bit key threshold, a min-p bound and the normaliser Z: token v is kept when
//       its key (logit order, then the lower token id) is at least the threshold and its
//       mass e_v = 2^((l_v - m) c) at least the min-p bound, and p(v) = e_v / Z. Masses
//       are summed as 40-bit fixed point, so every sum is exact and independent of the
//       order of the additions. The top-k and top-p thresholds come from a histogram of
//       d = (m - l_v) c over 4096 linear bins of [0, 32) (the last bin also takes
//       everything beyond), then an exact ordering of the one bin where the criterion is
//       met: its tokens sorted in shared memory, or, when the bin holds more than 4096
//       tokens or is the open last bin, a 64-bit radix select over its keys.
//   sample_walk_kernel    one 512-thread CTA per request: the walk (the logits of a
//       node's candidates are gathered in one round of loads), the residual passes of the
//       draft-aware rule, and the final inverse-CDF sample over the vocabulary (one
//       contiguous slice per thread, an exact integer scan for target-only).
//   accept_compact_kernel (accept.cu), given-path mode: the accepted KV rows move.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "kv_view.cuh"

namespace tsv {
namespace {

typedef unsigned long long u64;

constexpr int FT = 1024;                 // threads of the filter kernel
constexpr int NB = 4096;                 // histogram bins (4 per filter thread)
constexpr float DR = 32.f;               // bins cover d in [0, 32): masses down to 2^-32
constexpr int CAP = 4096;                // tokens of one bin sorted in shared memory
constexpr float FIXS = 1099511627776.0f;  // 2^40: masses as fixed point
constexpr int WT = 512;                  // threads of the walk kernel
static_assert(NB == 4 * FT, "cross_index takes four entries per thread");

struct RowStats {
  u64 thr;     // kept: key >= thr
  u64 z;       // sum of the kept masses (fixed point)
  float m;     // largest logit
  float c;     // log2(e) / temperature; 0 = greedy (only the first maximum is kept)
  float minp;  // kept: mass >= minp
  int valid;   // 1 once written
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
// Mass relative to the largest logit (1 there; 0 for -inf).
__device__ __forceinline__ float emass(float l, float m, float c) {
  return c == 0.f ? 1.f : exp2f((l - m) * c);
}
__device__ __forceinline__ u64 fixp(float e) { return (u64)(e * FIXS); }
__device__ __forceinline__ int bin_of(float l, float m, float c) {
  const float d = (m - l) * c;  // >= 0, non-decreasing as l decreases; NaN/inf -> last bin
  return d < DR ? min(NB - 1, (int)(d * (NB / DR))) : NB - 1;
}
__device__ __forceinline__ u64 kept_mass(const RowStats& st, float l, int v) {
  if (vkey(l, v) < st.thr) return 0ull;
  const float e = emass(l, st.m, st.c);
  return e >= st.minp ? fixp(e) : 0ull;
}

// Visit every token of a row: f(v, logit) with NaN read as -inf.
template <class F>
__device__ __forceinline__ void for_row(const float* __restrict__ row, int V, bool vec, F&& f) {
  if (vec) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    for (int j = threadIdx.x; j < (V >> 2); j += blockDim.x) {
      const float4 x = __ldg(r4 + j);
      f(4 * j, clean(x.x));
      f(4 * j + 1, clean(x.y));
      f(4 * j + 2, clean(x.z));
      f(4 * j + 3, clean(x.w));
    }
  } else {
    for (int v = threadIdx.x; v < V; v += blockDim.x) f(v, clean(__ldg(row + v)));
  }
}

// ---- block-wide helpers (any multiple of 32 threads up to 1024) -----------------------
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
__device__ u64 block_sum_u64(u64 x, u64* sb) {
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(FULL, x, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (l == 0) sb[w] = x;
  __syncthreads();
  x = l < nw ? sb[l] : 0ull;
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(FULL, x, o);
  return x;
}
// fixed order of additions: the result is the same on every run
__device__ double block_sum_f64(double x, double* sd) {
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(FULL, x, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (l == 0) sd[w] = x;
  __syncthreads();
  x = l < nw ? sd[l] : 0.0;
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(FULL, x, o);
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
  u64 cnt[NB];
  u64 mass[NB];
  u64 ckey[CAP];
  u64 cmass[CAP];
  u64 sb[32];
  u64 s_before, s_prefix, s_want;
  int s_res, s_n;
};

// Smallest j < n with vals[0] + ... + vals[j] >= target (target >= 1), or -1; *before =
// the sum of the entries before j. n <= 4 * blockDim.x.
__device__ int cross_index(const u64* vals, int n, u64 target, FilterSmem& S, u64* before) {
  const int j0 = threadIdx.x * 4;
  u64 loc = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (j0 + i < n) loc += vals[j0 + i];
  u64 tot;
  const u64 incl = block_scan<u64>(loc, S.sb, &tot);
  if (threadIdx.x == 0) S.s_res = -1;
  __syncthreads();
  u64 acc = incl - loc;
  if (acc < target && target <= incl) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const u64 x = j0 + i < n ? vals[j0 + i] : 0ull;
      if (acc + x >= target) {
        S.s_res = j0 + i;
        S.s_before = acc;
        break;
      }
      acc += x;
    }
  }
  __syncthreads();
  *before = S.s_before;
  return S.s_res;
}

__device__ void sort_desc(u64* key, u64* val, int n) {  // n a power of two
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
            const u64 t = val[i];
            val[i] = val[p];
            val[p] = t;
          }
        }
      }
      __syncthreads();
    }
}

// The tokens of bin `bsel` with key >= lo, sorted by key (descending) into S.ckey /
// S.cmass; returns how many (the caller has checked that they fit).
__device__ int collect_sorted(FilterSmem& S, const float* row, int V, bool vec, float m, float c,
                              int bsel, u64 lo) {
  if (threadIdx.x == 0) S.s_n = 0;
  __syncthreads();
  for_row(row, V, vec, [&](int v, float l) {
    if (bin_of(l, m, c) != bsel) return;
    const u64 k = vkey(l, v);
    if (k < lo) return;
    const int pos = atomicAdd(&S.s_n, 1);
    if (pos < CAP) {
      S.ckey[pos] = k;
      S.cmass[pos] = fixp(emass(l, m, c));
    }
  });
  __syncthreads();
  const int n = min(S.s_n, CAP);
  int np = 2;
  while (np < n) np <<= 1;
  for (int j = n + threadIdx.x; j < np; j += blockDim.x) {
    S.ckey[j] = 0ull;
    S.cmass[j] = 0ull;
  }
  __syncthreads();
  sort_desc(S.ckey, S.cmass, np);
  return n;
}

// Exact selection among the tokens of bin `bsel` with key >= lo, in descending key order:
// mode 0 -> the token of rank `want` (0-based); mode 1 -> the token at which the running
// mass first reaches `want` (>= 1; the last token when the bin's mass is smaller). A
// radix select over the 64-bit keys, eight digits of 8 bits, most significant first.
__device__ u64 radix_select(FilterSmem& S, const float* row, int V, bool vec, float m, float c,
                            int bsel, u64 lo, int mode, u64 want) {
  u64* hc = S.ckey;   // 256-entry histograms (the sorted list is not in use here)
  u64* hm = S.cmass;
  if (threadIdx.x == 0) {
    S.s_prefix = 0ull;
    S.s_want = want;
  }
  for (int d = 7; d >= 0; --d) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) {
      hc[i] = 0ull;
      hm[i] = 0ull;
    }
    __syncthreads();
    const u64 prefix = S.s_prefix;
    const int sh = 8 * d;
    for_row(row, V, vec, [&](int v, float l) {
      const u64 k = vkey(l, v);
      if (k < lo || bin_of(l, m, c) != bsel) return;
      if (d < 7 && (k >> (sh + 8)) != prefix) return;
      const int bk = (int)((k >> sh) & 255ull);
      atomicAdd(&hc[bk], 1ull);
      if (mode == 1) atomicAdd(&hm[bk], fixp(emass(l, m, c)));
    });
    __syncthreads();
    if (threadIdx.x == 0) {
      const u64 w = S.s_want;
      u64 acc = 0;
      int pick = -1, last = 0;
      for (int bk = 255; bk >= 0; --bk) {
        if (hc[bk] == 0ull) continue;
        last = bk;
        const u64 x = mode == 0 ? hc[bk] : hm[bk];
        if (mode == 0 ? (acc + x > w) : (acc + x >= w)) {
          pick = bk;
          break;
        }
        acc += x;
      }
      // not reached inside this bin: the last token (every later digit takes its last)
      S.s_want = pick >= 0 ? w - acc : ~0ull;
      S.s_prefix = (prefix << 8) | (u64)(pick >= 0 ? pick : last);
    }
    __syncthreads();
  }
  return S.s_prefix;
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

  u64 best = 0ull;
  for_row(row, V, vec, [&](int v, float l) { best = max(best, vkey(l, v)); });
  const u64 maxkey = block_max_u64(best, S.sb);
  const float m = key_value(maxkey);
  const float tau = a.temperature[b];
  const int k = a.top_k[b];
  const float pp = a.top_p[b];
  const float mp = a.min_p[b];
  RowStats st;
  st.m = m;
  st.valid = 1;
  const bool greedy = !(tau > 0.f) || k == 1 || pp <= 0.f || isinf(m);
  if (greedy) {
    st.thr = maxkey;
    st.z = fixp(1.f);
    st.c = 0.f;
    st.minp = 0.f;
  } else {
    const float c = 1.4426950408889634f / tau;
    const bool topk_on = k > 1 && k < V;
    const bool topp_on = pp < 1.f;
    st.c = c;
    st.minp = mp > 0.f ? fminf(mp, 1.f) : 0.f;
    u64 thr = 0ull;
    if (topk_on || topp_on) {
      for (int j = threadIdx.x; j < NB; j += FT) {
        S.cnt[j] = 0ull;
        S.mass[j] = 0ull;
      }
      __syncthreads();
      for_row(row, V, vec, [&](int v, float l) {
        const int bn = bin_of(l, m, c);
        atomicAdd(&S.cnt[bn], 1ull);
        const u64 w = fixp(emass(l, m, c));
        if (w) atomicAdd(&S.mass[bn], w);
      });
      __syncthreads();
      int bk = NB;          // bins from bk on are outside the top-k set
      bool listed = false;  // S.ckey / S.cmass hold the top-k part of bin bk, sorted
      int nlist = 0;
      u64 thr_k = 0ull;
      if (topk_on) {
        u64 before;
        bk = cross_index(S.cnt, NB, (u64)k, S, &before);  // k < V: always found
        const int r = k - 1 - (int)before;                // rank inside bin bk
        u64 part = 0ull;
        if (bk < NB - 1 && S.cnt[bk] <= (u64)CAP) {
          collect_sorted(S, row, V, vec, m, c, bk, 0ull);
          thr_k = S.ckey[r];
          listed = true;
          nlist = r + 1;
          for (int j = threadIdx.x; j <= r; j += FT) part += S.cmass[j];
        } else {
          thr_k = radix_select(S, row, V, vec, m, c, bk, 0ull, 0, (u64)r);
          for_row(row, V, vec, [&](int v, float l) {
            if (bin_of(l, m, c) == bk && vkey(l, v) >= thr_k) part += fixp(emass(l, m, c));
          });
        }
        const u64 mass_in = block_sum_u64(part, S.sb);
        // the histogram now describes the top-k set only
        for (int j = threadIdx.x; j < NB; j += FT) {
          if (j > bk) {
            S.cnt[j] = 0ull;
            S.mass[j] = 0ull;
          } else if (j == bk) {
            S.cnt[j] = (u64)(r + 1);
            S.mass[j] = mass_in;
          }
        }
        __syncthreads();
      }
      thr = thr_k;
      if (topp_on) {
        u64 loc = 0ull;
        for (int j = threadIdx.x; j < NB; j += FT) loc += S.mass[j];
        const u64 z1 = block_sum_u64(loc, S.sb);
        const u64 target = (u64)((double)pp * (double)z1);
        u64 thr_p;
        if (target == 0ull) {
          thr_p = maxkey;  // only the first token is kept
        } else {
          u64 before;
          const int bp = cross_index(S.mass, NB, target, S, &before);
          const u64 want = target - before;
          if (listed && bp == bk) {
            u64 b2;
            const int j = cross_index(S.cmass, nlist, want, S, &b2);
            thr_p = S.ckey[j < 0 ? nlist - 1 : j];
          } else if (bp < NB - 1 && S.cnt[bp] <= (u64)CAP) {
            const int nc = collect_sorted(S, row, V, vec, m, c, bp, thr_k);
            u64 b2;
            const int j = cross_index(S.cmass, nc, want, S, &b2);
            thr_p = S.ckey[j < 0 ? nc - 1 : j];
          } else {
            thr_p = radix_select(S, row, V, vec, m, c, bp, thr_k, 1, want);
          }
        }
        thr = max(thr_k, thr_p);
      }
    }
    st.thr = thr;
    u64 z = 0ull;
    for_row(row, V, vec, [&](int v, float l) { z += kept_mass(st, l, v); });
    st.z = block_sum_u64(z, S.sb);
  }
  if (threadIdx.x == 0) stats[(int64_t)b * T + i] = st;
  if (probs) {
    float* out = probs + ((int64_t)b * T + i) * V;
    const double inv = 1.0 / (double)st.z;
    for_row(row, V, false, [&](int v, float l) {
      out[v] = (float)((double)kept_mass(st, l, v) * inv);
    });
  }
}

// ---- walk kernel --------------------------------------------------------------------
struct WalkSmem {
  int tok[TSV_MAX_NODES], nxt[TSV_MAX_NODES], sib[TSV_MAX_NODES];
  int kids[TSV_MAX_NODES];
  float kl[TSV_MAX_NODES], kq[TSV_MAX_NODES];
  int removed[TSV_MAX_NODES];
  u64 rmass[TSV_MAX_NODES];
  float zr[TSV_MAX_NODES];  // draft-aware: normalisers of the residuals at this node
  int path[TSV_MAX_DEPTH + 1];
  u64 seg[WT];
  double segd[WT];
  u64 sb[32];
  double sd[32];
  RowStats st;
  u64 zcur;  // target-only: the current node's normaliser after its removals
  int node, len, code, nk, acc, nrem, nz, pick;
};

// Draft-aware residual probability of token v after `nz` rejections at this node.
__device__ __forceinline__ float resid_p(const WalkSmem& W, float l, int v, float q) {
  float r = (float)((double)kept_mass(W.st, l, v) / (double)W.st.z);
  for (int j = 0; j < W.nz; ++j) r = fmaxf(0.f, r - q) / W.zr[j];
  return r;
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
          const u64 km = in ? kept_mass(W.st, W.kl[j], x) : 0ull;
          float p, q = W.kq[j];
          if (!draft) {
            bool gone = false;
            for (int r = 0; r < W.nrem; ++r) gone |= W.removed[r] == x;
            p = gone ? 0.f : (float)((double)km / (double)W.zcur);
            q = 1.f;
          } else {
            p = in ? resid_p(W, W.kl[j], x, q) : 0.f;
          }
          const float ratio = q > 0.f ? p / q : (p > 0.f ? INFINITY : 0.f);
          const float u = a.u_node[row0 + c];
          if (u < fminf(1.f, ratio)) {
            W.acc = j;
          } else if (!draft && p > 0.f && W.zcur > km) {
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
          // residual normaliser: sum over v of max(0, p_j(v) - q(v))
          double part = 0.0;
          for (int v = threadIdx.x; v < V; v += WT) {
            const float q = qrow[v];
            part += (double)fmaxf(0.f, resid_p(W, clean(lrow[v]), v, q) - q);
          }
          const double zn = block_sum_f64(part, W.sd);
          if (threadIdx.x == 0 && zn > 0.0) W.zr[W.nz++] = (float)zn;
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

  // ---- the sample where the walk stopped: smallest t with prefix(t) > u * total -----
  int token = -1;
  if (size_ok) {
    const int node = W.node;
    const float* lrow = a.logits + (row0 + node) * V;
    const float* qrow = draft ? a.draft_probs + (row0 + node) * V : nullptr;
    const int L = (V + WT - 1) / WT;
    const int v0 = min(V, threadIdx.x * L), v1 = min(V, v0 + L);
    const float u = a.u_final[b];
    if (!draft) {
      u64 s = 0ull;
      for (int v = v0; v < v1; ++v) s += kept_mass(W.st, clean(lrow[v]), v);
      W.seg[threadIdx.x] = s;
      __syncthreads();
      if (threadIdx.x == 0)
        for (int r = 0; r < W.nrem; ++r) W.seg[min(WT - 1, W.removed[r] / L)] -= W.rmass[r];
      __syncthreads();
      const u64 mine = W.seg[threadIdx.x];
      u64 total;
      const u64 incl = block_scan<u64>(mine, W.sb, &total);
      const u64 target = (u64)((double)u * (double)total);
      if (threadIdx.x == 0) W.pick = -1;
      __syncthreads();
      u64 acc = incl - mine;
      if (acc <= target && target < incl) {
        for (int v = v0; v < v1; ++v) {
          bool gone = false;
          for (int r = 0; r < W.nrem; ++r) gone |= W.removed[r] == v;
          const u64 w = gone ? 0ull : kept_mass(W.st, clean(lrow[v]), v);
          if (acc + w > target) {
            W.pick = v;
            break;
          }
          acc += w;
        }
      }
      __syncthreads();
      token = W.pick;
    } else {
      double s = 0.0;
      for (int v = v0; v < v1; ++v) s += (double)resid_p(W, clean(lrow[v]), v, qrow[v]);
      double total;
      const double incl = block_scan<double>(s, W.segd, &total);
      const double target = (double)u * total;
      if (threadIdx.x == 0) W.pick = -1;
      __syncthreads();
      double acc = incl - s;
      if (acc <= target && target < incl) {
        for (int v = v0; v < v1; ++v) {
          const double w = (double)resid_p(W, clean(lrow[v]), v, qrow[v]);
          if (acc + w > target) {
            W.pick = v;
            break;
          }
          acc += w;
        }
      }
      __syncthreads();
      token = W.pick;
      if (token < 0) {
        // rounding put the target past the last positive entry: the last kept token
        if (threadIdx.x == 0) {
          for (int v = V - 1; v >= 0; --v)
            if (resid_p(W, clean(lrow[v]), v, qrow[v]) > 0.f) {
              W.pick = v;
              break;
            }
        }
        __syncthreads();
        token = W.pick;
      }
    }
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
