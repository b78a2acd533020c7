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
// One level runs one of three designs, chosen by plan_topk:
//   - small batches (rows of at most 32768 entries, every request's rows in one thread-
//     block cluster, the clusters in at most two waves): topk_row_kernel, one CTA per row
//     holding the row in registers; the rank-0 CTA of a request's cluster runs the joint
//     top-K over distributed shared memory (see its section below);
//   - large batches (every share of the level at least a row long): topk_stream_kernel,
//     a persistent kernel over equal shares of all rows' entries, then topk_merge_kernel;
//   - otherwise topk_level_kernel, one CTA per (row, vocab chunk); the chunk count per row
//     keeps the units in as few waves of resident CTAs as the makespan allows.
// In the last two, each unit is read once with 128-bit loads:
//   - log-sum-exp: fp32 terms 2^(x log2 e - ref log2 e) against a running reference,
//     summed in groups of 16 and added exactly (two-sum) into an unevaluated (hi, lo)
//     pair; the reference is raised, and the pair rescaled, only when an entry exceeds it
//     by more than 16 (natural log units). No fp64: it runs at a small fraction of the
//     fp32 rate on this part.
//   - top-k: a unit of one or two steps keeps its entries in registers. A longer unit
//     buffers the float4 groups whose largest entry beats a filter (the warp's k-th
//     value, or a CTA-wide bound: the best warp threshold, seeded with the k-th best of
//     the first step's 64 eight-lane group maxima) in the warp's shared-memory slice and
//     folds them into a register list 32 groups at a time. At the end a bound with k
//     entries of the unit at or above it leaves a handful of survivors, ranked by
//     counting in shared memory.
// The request merge (in topk_level_kernel the last CTA of a request to finish, found by
// an atomic ticket; after the persistent kernel, topk_merge_kernel) stages the request's
// chunk lists in shared memory, merges each row (k rounds of a warp tournament over list
// heads), writes the level's candidates to the store and ranks the rows' cumulative
// scores for the joint top-K.
#include <float.h>
#include <limits.h>
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tree_meta.cuh"

namespace tsv {
namespace {

constexpr int KMAX = TSV_MAX_TOPK;  // 16: longest warp list
constexpr int A_THREADS = 512;  // 16 warps: the request's merge gives every row a warp
constexpr int A_WARPS = A_THREADS / 32;
constexpr int MAX_CHUNKS = 32;
constexpr int MIN_CHUNK = 1024;     // vocab entries per chunk at least (4 per thread)
constexpr int GROUPS = 32;         // buffered groups of four entries per warp
constexpr int CTAS_PER_SM = 2;      // resident CTAs of the level kernel (launch bounds)
// the request merge stages rows x chunks x k (value, index) pairs in shared memory
// (and the rows' k cumulative scores and tokens)
constexpr int MERGE_SMEM_MAX = TSV_MAX_TOPK * (MAX_CHUNKS + 1) * TSV_MAX_TOPK * 8;
// survivors of a unit's finish (value, index): at most 8 register entries per thread
constexpr int SURV_MAX = 8 * A_THREADS;
constexpr float L2E = 1.4426950408889634f;
// Ring of a long unit: thread 0 copies the row chunk into shared memory in stages of four
// steps (8192 entries, 32 KB) with bulk copies, RING_STAGES ahead; the CTA consumes from
// shared memory. Units of at least RING_MIN entries on 16-byte aligned rows take it.
constexpr int RING_STAGES = 3;
constexpr int STAGE_F4 = 4 * A_THREADS;  // float4 groups per stage
constexpr int STAGE_ENTRIES = 4 * STAGE_F4;
constexpr int RING_BYTES = RING_STAGES * STAGE_ENTRIES * 4;
constexpr int RING_MIN = 2 * STAGE_ENTRIES;
// Ring of the persistent kernel (large batches): two CTAs per SM, so one CTA's piece
// finish overlaps the other's streaming.
constexpr int P_STAGES = 3;
constexpr int P_CTAS_PER_SM = 2;
constexpr int MAX_STAGES = P_STAGES > RING_STAGES ? P_STAGES : RING_STAGES;

struct ChunkStat {
  float ref;     // reference (a running maximum)
  float hi, lo;  // sum of exp(x - ref) over the chunk as an unevaluated fp32 pair
  float pad;
};

struct TopkWs {
  unsigned* tickets;   // [batch] finished chunk CTAs of each request: zero between calls
  ChunkStat* stat;     // [rows_total, chunks]
  float* val;          // [rows_total, chunks, K]
  int32_t* idx;        // [rows_total, chunks, K]
};

// The tickets come first, at the same place for every level of a request batch: the
// caller zeroes the workspace once and every call leaves them at zero.
__host__ __device__ inline TopkWs carve(void* ws, int batch, int rows_total, int chunks, int k) {
  char* p = static_cast<char*>(ws);
  TopkWs w;
  const size_t n = (size_t)rows_total * chunks;
  w.tickets = reinterpret_cast<unsigned*>(p);
  p += ((size_t)batch * sizeof(unsigned) + 255) & ~size_t(255);
  w.stat = reinterpret_cast<ChunkStat*>(p);
  p += (n * sizeof(ChunkStat) + 255) & ~size_t(255);
  w.val = reinterpret_cast<float*>(p);
  p += (n * k * sizeof(float) + 255) & ~size_t(255);
  w.idx = reinterpret_cast<int32_t*>(p);
  return w;
}

// Order-preserving unsigned image of a float (larger float -> larger unsigned).
__device__ __forceinline__ unsigned ord(float v) {
  const unsigned u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Warp-wide best (value, index) pair — larger value, then lower index — with one
// hardware warp reduction when the largest value is held by one lane (a second one
// breaks ties); every lane gets the pair and the lane that holds it.
__device__ __forceinline__ void warp_argmax(float& v, int& i, int& lane_of) {
  const unsigned u = ord(v);
  const unsigned umax = __reduce_max_sync(FULL, u);
  unsigned own = __ballot_sync(FULL, u == umax);
  if (own & (own - 1)) {  // several lanes hold the largest value: lowest index wins
    const unsigned imin = __reduce_min_sync(FULL, u == umax ? (unsigned)i : 0xffffffffu);
    own = __ballot_sync(FULL, u == umax && (unsigned)i == imin);
  }
  lane_of = __ffs(own) - 1;
  v = __shfl_sync(FULL, v, lane_of);
  i = __shfl_sync(FULL, i, lane_of);
}

// Compare-exchange of two (value, index) entries so that entry a is the better one.
__device__ __forceinline__ void cx(float& va, int& ia, float& vb, int& ib) {
  const bool sw = better(vb, ib, va, ia);
  const float tv = sw ? vb : va;
  const int ti = sw ? ib : ia;
  vb = sw ? va : vb;
  ib = sw ? ia : ib;
  va = tv;
  ia = ti;
}
// Sorts n register entries best first (odd-even transposition network, n rounds).
template <int N>
__device__ __forceinline__ void sort_entries(float (&v)[N], int (&ix)[N]) {
#pragma unroll
  for (int r = 0; r < N; ++r) {
#pragma unroll
    for (int t = r & 1; t + 1 < N; t += 2) cx(v[t], ix[t], v[t + 1], ix[t + 1]);
  }
}
// k rounds of a warp tournament over per-lane sorted entries: each round the best lane
// head wins and that lane shifts its entries up. Lane r receives the r-th best entry.
template <int N>
__device__ __forceinline__ void warp_select(float (&v)[N], int (&ix)[N], int rounds, int lane,
                                            float& out_v, int& out_i) {
  out_v = -INFINITY;
  out_i = INT_MAX;
  for (int r = 0; r < rounds; ++r) {
    float hv = v[0];
    int hi = ix[0], who = lane;
    warp_argmax(hv, hi, who);
    if (lane == r) { out_v = hv; out_i = hi; }
    if (lane == who) {
#pragma unroll
      for (int t = 0; t + 1 < N; ++t) { v[t] = v[t + 1]; ix[t] = ix[t + 1]; }
      v[N - 1] = -INFINITY;
      ix[N - 1] = INT_MAX;
    }
  }
}

// Exact sum of two floats as an unevaluated pair (Knuth's TwoSum): s + e == a + b.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bp = s - a;
  e = (a - (s - bp)) + (b - bp);
}
// (hi, lo) += (h2, l2), renormalised.
__device__ __forceinline__ void pair_add(float& hi, float& lo, float h2, float l2) {
  float s, e;
  two_sum(hi, h2, s, e);
  e += lo + l2;
  hi = s + e;
  lo = e - (hi - s);
}

// Sum of (ref_i, hi_i + lo_i) over a warp against the warp's largest reference: one
// fp32 exp per lane whose reference differs (none when they all agree), then pair adds.
__device__ __forceinline__ void warp_combine(float& r, float& hi, float& lo) {
  float R = r;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) R = fmaxf(R, __shfl_xor_sync(FULL, R, o));
  if (r != R) {
    const float f = hi == 0.f ? 0.f : expf(r - R);
    hi *= f;
    lo *= f;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float h2 = __shfl_xor_sync(FULL, hi, o), l2 = __shfl_xor_sync(FULL, lo, o);
    pair_add(hi, lo, h2, l2);
  }
  r = R;
}

__device__ __forceinline__ float4 ld_stream(const float4* p) {
  float4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct TopkSmem {
  float4 gv[A_WARPS][GROUPS];                  // per-warp buffered groups (warp-owned)
  int gi[A_WARPS][GROUPS];                     // index of a group's first entry
  float lv[A_WARPS][KMAX];                     // warp lists at the end of a unit
  int li[A_WARPS][KMAX];
  float red[A_WARPS];
  float shi[A_WARPS], slo[A_WARPS];
  unsigned long long gkey[A_THREADS / 8];      // best entry of each eight-lane group
  unsigned long long gthr;                     // key() of the best warp threshold
  unsigned long long tau;                      // bound of the unit's top k
  unsigned long long full[MAX_STAGES];         // ring: stage landed (bulk copy bytes)
  unsigned long long empty[MAX_STAGES];        // ring: every warp has read the stage
  int ns;                                      // survivors collected
  int fail;                                    // a ring wait gave up (never expected)
  bool last;
};

// Order-preserving 64-bit image of an entry: larger value first, then lower index. Real
// entries (index < INT_MAX) beat placeholders (-inf, INT_MAX) of the same value.
__device__ __forceinline__ unsigned long long key(float v, int i) {
  return ((unsigned long long)ord(v) << 32) | (unsigned)(~(unsigned)i);
}

// Per-thread log-sum-exp state: fp32 terms exp(x - ref) summed in groups of 16, each
// group added exactly into an unevaluated (hi, lo) pair. The reference is raised (and
// the pair rescaled) only when an entry exceeds it by more than RAISE, so terms stay
// below e^RAISE and the rare rescale is the only inexact step besides the terms.
constexpr float RAISE = 16.f;
struct Lse {
  float ref, rl, g, hi, lo;  // rl = ref * log2(e): a term is 2^(x log2(e) - rl), one FFMA
  __device__ __forceinline__ void flush() {
    pair_add(hi, lo, g, 0.f);
    g = 0.f;
  }
  // rare; inlined so the state stays in registers (an out-of-line member call would
  // keep it in local memory on the streaming path)
  __device__ __forceinline__ void raise(float m) {
    flush();
    const float f = expf(ref - m);
    hi *= f;
    lo *= f;
    ref = m;
    rl = m * L2E;
  }
  __device__ __forceinline__ float term(float x) const { return ex2(fmaf(x, L2E, -rl)); }
};

// Inverse of ord().
__device__ __forceinline__ float unord(unsigned o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// Streaming state of one thread for one (row, chunk) unit. The warp's top-k list lives
// in registers, entry r in lane r for r < k; entries not yet filled are placeholders
// (-inf, INT_MAX) that every real entry beats. A group of four entries whose largest
// beats the filter is buffered whole in the warp's shared-memory slice (one slot per
// lane, positions from a ballot: no atomics); the list absorbs the buffer when it is
// full and at the end of the unit.
struct UnitState {
  Lse lse;
  float lv;     // this lane's list entry
  int li;
  float thr;    // group filter: the larger of the warp's k-th value and the CTA-wide bound
  int cnt;      // warp-uniform number of buffered groups
};

// The list absorbs the buffered groups: lane t takes group t (four entries) beside its
// own list entry, sorts the five, and k rounds of a warp tournament pick the new list.
// Entries at or past `end` are placeholders. The warp's k-th value then bounds the
// unit's top k from below (k entries are at least that large), so every warp may filter
// with the largest such value (an atomicMax of its ord() image).
__device__ __forceinline__ void fold(TopkSmem& sm, UnitState& u, int warp, int lane, int k,
                                     int end) {
  __syncwarp();
  float v[5];
  int ix[5];
  v[0] = u.lv;
  ix[0] = u.li;
  const bool have = lane < u.cnt;
  const float4 g = have ? sm.gv[warp][lane] : make_float4(0.f, 0.f, 0.f, 0.f);
  const int e = have ? sm.gi[warp][lane] : end;
  const float gq[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    v[1 + q] = e + q < end ? gq[q] : -INFINITY;
    ix[1 + q] = e + q < end ? e + q : INT_MAX;
  }
  sort_entries(v, ix);
  warp_select(v, ix, k, lane, u.lv, u.li);
  u.cnt = 0;
  const float thr_v = __shfl_sync(FULL, u.lv, k - 1);
  const int thr_i = __shfl_sync(FULL, u.li, k - 1);
  if (lane == 0) atomicMax(&sm.gthr, key(thr_v, thr_i));
  u.thr = fmaxf(thr_v, unord((unsigned)(*reinterpret_cast<volatile unsigned long long*>(&sm.gthr) >> 32)));
  __syncwarp();  // the buffer slots are free again
}

// Log-sum-exp terms of four entries (-inf entries give zero terms).
// The log-sum-exp terms of four entries whose largest is m4 (-inf entries give zero
// terms); the caller flushes the group sum every four calls.
__device__ __forceinline__ void lse4(UnitState& u, float4 a, float m4) {
  if (m4 > u.lse.ref + RAISE) u.lse.raise(m4);
  u.lse.g += (u.lse.term(a.x) + u.lse.term(a.y)) + (u.lse.term(a.z) + u.lse.term(a.w));
}
__device__ __forceinline__ float max4(float4 a) { return fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)); }

// One streaming step: the log-sum-exp terms of entries e .. e + 3 and, when their largest
// beats the filter, the group into the warp's buffer (the list absorbs the buffer first
// when the new groups would not fit). Warp-uniform call.
__device__ __forceinline__ void step4(TopkSmem& sm, UnitState& u, int warp, int lane, int k,
                                      float4 a, int e, int end) {
  const float m4 = max4(a);
  lse4(u, a, m4);
  const bool q = m4 >= u.thr;
  const unsigned bal = __ballot_sync(FULL, q);
  if (bal) {  // warp-uniform and rare once the list holds k entries
    const int n = __popc(bal);
    if (u.cnt + n > GROUPS) fold(sm, u, warp, lane, k, end);
    if (q) {
      const int pos = u.cnt + __popc(bal & ((1u << lane) - 1u));
      sm.gv[warp][pos] = a;
      sm.gi[warp][pos] = e;
    }
    u.cnt += n;
  }
}

// The filter half of step4 for a group whose largest entry m4 is known (its exp-sum
// terms are added by the caller). Warp-uniform call.
__device__ __forceinline__ void filter4(TopkSmem& sm, UnitState& u, int warp, int lane, int k,
                                        float4 a, float m4, int e, int end) {
  const bool q = m4 >= u.thr;
  const unsigned bal = __ballot_sync(FULL, q);
  if (bal) {
    const int n = __popc(bal);
    if (u.cnt + n > GROUPS) fold(sm, u, warp, lane, k, end);
    if (q) {
      const int pos = u.cnt + __popc(bal & ((1u << lane) - 1u));
      sm.gv[warp][pos] = a;
      sm.gi[warp][pos] = e;
    }
    u.cnt += n;
  }
}

// Four consecutive steps of a thread (entries e, e + 4 A_THREADS, ...; every entry in
// range): one raise check and one filter vote for all sixteen entries, the exp-sum terms
// in the order of four step4 calls, then the group flush. The per-group filter runs only
// when some lane's sixteen entries reach the filter (rare once the list is full).
__device__ __forceinline__ void step16(TopkSmem& sm, UnitState& u, int warp, int lane, int k,
                                       const float4 (&a)[4], int e, int end) {
  float m[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) m[q] = max4(a[q]);
  const float m16 = fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
  if (m16 > u.lse.ref + RAISE) u.lse.raise(m16);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    u.lse.g += (u.lse.term(a[q].x) + u.lse.term(a[q].y)) + (u.lse.term(a[q].z) + u.lse.term(a[q].w));
  u.lse.flush();
  if (__any_sync(FULL, m16 >= u.thr)) {
#pragma unroll
    for (int q = 0; q < 4; ++q) filter4(sm, u, warp, lane, k, a[q], m[q], e + 4 * q * A_THREADS, end);
  }
}

// The k-th best of 64 keys (ties by position), written to *out by the thread that finds
// it; the whole CTA takes part: eight threads per key, each comparing it with eight of the
// 64, their counts added by shuffles. Block-uniform call; *out is read after the next
// barrier.
__device__ __forceinline__ void kth_of_64(const unsigned long long* keys, int k,
                                          unsigned long long* out) {
  static_assert(A_THREADS == 64 * 8, "eight threads per key");
  const int t = threadIdx.x >> 3, part = threadIdx.x & 7;
  const unsigned long long a = keys[t];
  int r = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int o = part * 8 + u;
    const unsigned long long b = keys[o];
    r += (b > a || (b == a && o < t)) ? 1 : 0;
  }
  r += __shfl_xor_sync(FULL, r, 1);
  r += __shfl_xor_sync(FULL, r, 2);
  r += __shfl_xor_sync(FULL, r, 4);
  if (part == 0 && r == k - 1) *out = a;
}

// Starts a unit's per-thread state (sm.gthr was set before the CTA's last barrier).
__device__ __forceinline__ void unit_begin(UnitState& u, float ref, unsigned long long gthr) {
  u.lse.ref = fmaxf(ref, -1e30f);  // finite (and so is ref * log2(e)): x = -inf gives a zero term
  u.lse.rl = u.lse.ref * L2E;
  u.lse.g = 0.f;
  u.lse.hi = 0.f;
  u.lse.lo = 0.f;
  u.lv = -INFINITY;
  u.li = INT_MAX;
  u.thr = unord((unsigned)(gthr >> 32));
  u.cnt = 0;
}

struct LevelArgs {
  const float* logits;
  int64_t row_stride;
  int vocab, rows, k, chunks, chunk_len, level;
  bool product;  // scores: parent score x child probability, else parent + log-probability
  bool ring;     // the launch has RING_BYTES of dynamic shared memory for long units
  int rows_total;  // batch * rows
  TopkWs ws;
  const float* front_score_in;
  const int32_t* front_store_in;
  int store_cap;
  int32_t* store_token;
  float* store_score;
  int32_t* store_parent;
  int32_t* front_token_out;
  float* front_score_out;
  int32_t* front_store_out;
};

// The request's merge, run by the CTA that finished its last unit: every row's chunk
// lists and exp-sums combine into the row's top-k log-probabilities and cumulative
// scores (written to the store), then the joint top-K over the rows. The request's chunk
// lists are staged in (dynamic) shared memory with one cooperative load; each merge is k
// rounds of a warp tournament over list heads, the winning lane stepping its pointer, so
// no list is held in registers. Out of line: it is rare, and inlined its registers would
// crowd the streaming loop.
__device__ __noinline__ void request_merge(const LevelArgs& p, int b, float4* stage) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = p.k, rows = p.rows, chunks = p.chunks;
  const int off = p.level == 1 ? 0 : k + (p.level - 2) * k * k;
  const int64_t srow = (int64_t)b * p.store_cap;
  // lists of the request: entry j of (row s, chunk c) at (s * chunks + c) * k + j
  const int n = rows * chunks * k;
  float* mv = reinterpret_cast<float*>(stage);
  int* mi = reinterpret_cast<int*>(mv + n);
  // the rows' cumulative scores and tokens (flat = row * k + j); through the declared
  // shared array the compiler emits shared-memory accesses (a generic pointer to the
  // static struct measured several times slower per tournament round)
  float* cu_s = reinterpret_cast<float*>(mi + n);
  int* tok_s = reinterpret_cast<int*>(cu_s + rows * k);
  const size_t g0 = (size_t)b * n;
  // eight loads per thread in flight before any store: one L2 round trip per 4096 entries
  for (int t0 = tid; t0 < n; t0 += 8 * A_THREADS) {
    float v8[8];
    int i8[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = t0 + u * A_THREADS;
      v8[u] = t < n ? __ldcg(p.ws.val + g0 + t) : 0.f;
      i8[u] = t < n ? __ldcg(p.ws.idx + g0 + t) : 0;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = t0 + u * A_THREADS;
      if (t < n) {
        mv[t] = v8[u];
        mi[t] = i8[u];
      }
    }
  }
  static_assert(A_WARPS >= TSV_MAX_TOPK, "one warp per frontier row");
  const int s = warp, r0 = b * rows + s;
  float4 cs = make_float4(-INFINITY, 0.f, 0.f, 0.f);
  if (warp < rows && lane < chunks)
    cs = __ldcg(reinterpret_cast<const float4*>(&p.ws.stat[(size_t)r0 * chunks + lane]));
  __syncthreads();
  if (warp < rows) {
    // warp s merges row s: lane c walks chunk c's sorted list
    const float pscore = p.level == 1 ? (p.product ? 1.0f : 0.0f) : p.front_score_in[r0];
    const int pstore = p.level == 1 ? -1 : p.front_store_in[r0];
    float Rr = cs.x, sh = cs.y, sl = cs.z;
    warp_combine(Rr, sh, sl);
    // log(hi + lo) = log(hi) + log1p(lo / hi); |lo / hi| is below an ulp, so the second
    // term is lo / hi
    const float lse_hi = Rr, lse_mid = logf(sh), lse_lo = sl / sh;
    const bool have = lane < chunks;
    const int lb = (s * chunks + lane) * k;
    int ptr = 0;
    float hv = have ? mv[lb] : -INFINITY;
    int hi = have ? mi[lb] : INT_MAX;
    float v = -INFINITY;
    int i = INT_MAX;
    for (int r = 0; r < k; ++r) {
      float wv = hv;
      int wi = hi, who = lane;
      warp_argmax(wv, wi, who);
      if (lane == r) { v = wv; i = wi; }
      if (lane == who) {
        ++ptr;
        hv = ptr < k ? mv[lb + ptr] : -INFINITY;
        hi = ptr < k ? mi[lb + ptr] : INT_MAX;
      }
    }
    if (lane < k) {
      const float logp = ((v - lse_hi) - lse_mid) - lse_lo;
      const float cu = p.product ? pscore * expf(logp) : pscore + logp;
      const int flat = s * k + lane;
      p.store_token[srow + off + flat] = i;
      p.store_score[srow + off + flat] = cu;
      p.store_parent[srow + off + flat] = pstore;
      cu_s[flat] = cu;
      tok_s[flat] = i;
    }
  }
  __syncthreads();

  // Joint top-K over the rows * K cumulative scores (ties to the lower flat index): entry
  // f's rank is the number of entries better than it; the K of rank below K are the
  // frontier, written to their rank.
  const int nf = rows * k;
  if (tid < nf) {
    const float cv = cu_s[tid];
    int rank = 0;
#pragma unroll 4
    for (int u = 0; u < nf; ++u) {
      const float o = cu_s[u];
      rank += (o > cv || (o == cv && u < tid)) ? 1 : 0;
    }
    if (rank < k) {
      p.front_token_out[b * k + rank] = tok_s[tid];
      p.front_score_out[b * k + rank] = cv;
      p.front_store_out[b * k + rank] = off + tid;
    }
  }
  if (tid == 0) p.ws.tickets[b] = 0u;
  __syncthreads();
}

// End of a unit. Every entry that can still reach the unit's top k is collected in
// shared memory by the whole CTA and ranked there. The bound tau is an entry key with k of
// the unit's entries at or above it: the k-th best of 64 candidates -- the eight-lane
// group maxima of a short unit, or the first four entries of every warp list when
// streaming (there also at least the best warp threshold) -- or 0, which every entry
// passes, when fewer than k candidates are entries. The survivors -- the warps' exact lists after a last
// fold (streaming) or the lanes' register entries (short unit) at or above tau -- hold the
// unit's top k; a survivor's rank is the number of survivors better than it. The last unit
// of the request to finish (an atomic ticket) then merges the request's rows. Called by
// the whole CTA; ng is the number of register groups per lane of a short unit (0 when
// streaming).
// surv: room for surv_cap survivors; merge_stage: the request merge's staging area.
// With also_empty the unit also stands for chunk + 1 of its row, which holds no entry
// (its list is placeholders and its exp-sum zero) and counts on the request's ticket.
// Without merge_here the request merge is left to topk_merge_kernel (no ticket).
__device__ void finish_unit(TopkSmem& sm, UnitState& u, const LevelArgs& p, int row, int chunk,
                            int end, int ng, float4 g0, float4 g1, int e0, int e1, float4* surv,
                            int surv_cap, float4* merge_stage, bool also_empty = false,
                            bool merge_here = true) {
  float* sv = reinterpret_cast<float*>(surv);
  int* si = reinterpret_cast<int*>(sv + surv_cap);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = p.k, rows = p.rows, chunks = p.chunks;
  u.lse.flush();
  float R = u.lse.ref, phi = u.lse.hi, plo = u.lse.lo;
  warp_combine(R, phi, plo);
  if (lane == 0) { sm.red[warp] = R; sm.shi[warp] = phi; sm.slo[warp] = plo; }
  const float gv[2][4] = {{g0.x, g0.y, g0.z, g0.w}, {g1.x, g1.y, g1.z, g1.w}};
  const int ge[2] = {e0, e1};
  if (ng == 0) {
    // the warp's exact top k (its last fold also raises the CTA-wide bound)
    if (u.cnt > 0) fold(sm, u, warp, lane, k, end);
    if (lane < k) { sm.lv[warp][lane] = u.lv; sm.li[warp][lane] = u.li; }
    static_assert(A_THREADS / 8 == 4 * A_WARPS, "four list heads per warp");
    if (lane < 4) sm.gkey[warp * 4 + lane] = lane < k ? key(u.lv, u.li) : 0ull;
  } else {
    unsigned long long best = 0ull;
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (t < ng && ge[t] + q < end) best = max(best, key(gv[t][q], ge[t] + q));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) best = max(best, __shfl_xor_sync(FULL, best, o));
    if ((lane & 7) == 0) sm.gkey[tid >> 3] = best;
  }
  if (tid == 0) sm.ns = 0;
  __syncthreads();
  kth_of_64(sm.gkey, k, &sm.tau);  // the 64 candidates' k-th best is tau
  __syncthreads();
  const unsigned long long tau = ng > 0 ? sm.tau : max(sm.tau, sm.gthr);

  // survivors, appended with one shared-memory atomic per warp and entry slot
  auto push = [&](bool keep, float v, int i) {  // warp-uniform call
    const unsigned bal = __ballot_sync(FULL, keep);
    if (bal) {
      const int leader = __ffs(bal) - 1;
      int at = 0;
      if (lane == leader) at = atomicAdd(&sm.ns, __popc(bal));
      at = __shfl_sync(FULL, at, leader);
      if (keep) {
        const int pos = at + __popc(bal & ((1u << lane) - 1u));
        sv[pos] = v;
        si[pos] = i;
      }
    }
  };
  if (ng == 0) {
    // list entries: thread t holds entry t % KMAX of warp t / KMAX
    const int w = tid / KMAX, j = tid % KMAX;
    const bool in = tid < A_WARPS * KMAX && j < k;
    const float v = in ? sm.lv[w][j] : -INFINITY;
    const int i = in ? sm.li[w][j] : INT_MAX;
    push(in && i != INT_MAX && key(v, i) >= tau, v, i);
  } else {
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (t < ng) push(ge[t] + q < end && key(gv[t][q], ge[t] + q) >= tau, gv[t][q], ge[t] + q);
  }
  __syncthreads();
  const int S = sm.ns;
  const size_t base = ((size_t)row * chunks + chunk) * k;
  for (int t = tid; t < S; t += A_THREADS) {
    const float v = sv[t];
    const int i = si[t];
    int rank = 0;
#pragma unroll 4
    for (int s2 = 0; s2 < S; ++s2) {
      const float o = sv[s2];
      rank += (o > v || (o == v && si[s2] < i)) ? 1 : 0;
    }
    if (rank < k) { p.ws.val[base + rank] = v; p.ws.idx[base + rank] = i; }
  }
  for (int t = S + tid; t < k; t += A_THREADS) {  // fewer than k entries in the unit
    p.ws.val[base + t] = -INFINITY;
    p.ws.idx[base + t] = INT_MAX;
  }
  if (also_empty) {
    for (int t = tid; t < k; t += A_THREADS) {
      p.ws.val[base + k + t] = -INFINITY;
      p.ws.idx[base + k + t] = INT_MAX;
    }
    if (tid == 0) {
      ChunkStat cs;
      cs.ref = -INFINITY;
      cs.hi = 0.f;
      cs.lo = 0.f;
      cs.pad = 0.f;
      p.ws.stat[(size_t)row * chunks + chunk + 1] = cs;
    }
  }
  if (warp == A_WARPS - 1) {  // the block's exp-sum
    float rr = lane < A_WARPS ? sm.red[lane] : -INFINITY;
    float hh = lane < A_WARPS ? sm.shi[lane] : 0.f, ll = lane < A_WARPS ? sm.slo[lane] : 0.f;
    warp_combine(rr, hh, ll);
    if (lane == 0) {
      ChunkStat cs;
      cs.ref = rr;
      cs.hi = hh;
      cs.lo = ll;
      cs.pad = 0.f;
      p.ws.stat[(size_t)row * chunks + chunk] = cs;
    }
  }

  // The last unit of this request to finish merges its rows and runs the joint top-K.
  const int b = row / rows;
  __syncthreads();
  if (!merge_here) return;  // every thread: the list and stat buffers are free again
  if (tid == 0) {
    __threadfence();
    const unsigned inc = also_empty ? 2u : 1u;
    const unsigned t = atomicAdd(&p.ws.tickets[b], inc);
    sm.last = (t + inc == (unsigned)(rows * chunks));
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  griddep_launch();  // the next kernel may be scheduled (it waits for this grid to finish)
  request_merge(p, b, merge_stage);
}

// ---- ring of bulk copies ---------------------------------------------------------------
__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ bool bar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for a ring barrier phase: after about a second (never expected: a bulk
// copy of this GPU's own memory always lands) the CTA is marked failed and its waits
// return at once, so the call finishes instead of hanging (the unit's result is then
// incomplete).
__device__ bool ring_wait(TopkSmem& sm, uint32_t bar, uint32_t parity) {
  if (bar_test(bar, parity)) return true;
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (uint32_t i = 0;; ++i) {
    if (bar_test(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&sm.fail)) return false;
    if ((i & 255u) == 255u) {
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > 1000000000ull) {
        sm.fail = 1;
        return false;
      }
    }
  }
}
// Stage i of the unit's chunk [start, end4) into ring slot i % RING_STAGES (thread 0).
__device__ __forceinline__ void ring_issue(TopkSmem& sm, uint32_t ring0, const float* x,
                                           int start, int end4, int i) {
  const int s = i % RING_STAGES;
  const int e0 = start + i * STAGE_ENTRIES;
  const uint32_t bytes = (uint32_t)min(STAGE_ENTRIES, end4 - e0) * 4u;  // a multiple of 16
  const uint32_t full = sa(&sm.full[s]);
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(full), "r"(bytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          ring0 + (uint32_t)s * (STAGE_ENTRIES * 4)),
      "l"(x + e0), "r"(bytes), "r"(full)
      : "memory");
}

// A long unit through the ring: the same per-thread entries, exp-sum grouping and filter
// as the streaming loop, sixteen entries (four steps) per stage read from shared memory,
// so the loads hold no registers and never stall the arithmetic.
__device__ __forceinline__ void stream_ring(TopkSmem& sm, const LevelArgs& p, int row, int chunk,
                                            int start, int end, const float* x) {
  extern __shared__ float4 dyn_smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int end4 = start + ((end - start) & ~3);  // entries the bulk copies bring
  const int nst = (end4 - start + STAGE_ENTRIES - 1) / STAGE_ENTRIES;
  const uint32_t ring0 = sa(dyn_smem);
  const float4 none = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  if (tid == 0) {
    for (int st = 0; st < RING_STAGES; ++st) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa(&sm.full[st])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&sm.empty[st])),
                   "r"(A_WARPS)
                   : "memory");
    }
    sm.fail = 0;
    sm.gthr = 0ull;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int i = 0; i < min(RING_STAGES, nst); ++i) ring_issue(sm, ring0, x, start, end4, i);
  }
  __syncthreads();
  // The first stage: the common starting reference (its largest entry) and the seed of the
  // CTA-wide bound, the k-th best of the maxima of 64 disjoint groups of 128 entries
  // (eight threads' sixteen entries each; a group maximum is an entry of the unit, so k
  // entries are at or above the seed).
  ring_wait(sm, sa(&sm.full[0]), 0);
  float first = -INFINITY;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (start + 4 * (tid + q * A_THREADS) < end4) first = fmaxf(first, max4(dyn_smem[tid + q * A_THREADS]));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) first = fmaxf(first, __shfl_xor_sync(FULL, first, o));
  if ((lane & 7) == 0) sm.gkey[tid >> 3] = key(first, INT_MAX);
#pragma unroll
  for (int o = 8; o < 32; o <<= 1) first = fmaxf(first, __shfl_xor_sync(FULL, first, o));
  if (lane == 0) sm.red[warp] = first;
  __syncthreads();
  kth_of_64(sm.gkey, p.k, &sm.gthr);
  first = sm.red[0];
#pragma unroll
  for (int w = 1; w < A_WARPS; ++w) first = fmaxf(first, sm.red[w]);
  __syncthreads();  // sm.red is reused by finish_unit; sm.gthr is seeded
  UnitState u;
  unit_begin(u, first, sm.gthr);
  const unsigned long long* gthr = &sm.gthr;
  int st = 0;  // ring slot and phase parity of stage i, advanced stage by stage
  uint32_t par = 0u;
  for (int i = 0; i < nst; ++i) {
    const bool ok = i == 0 || ring_wait(sm, sa(&sm.full[st]), par);
    const float4* stage = dyn_smem + st * STAGE_F4;
    const int eb = start + i * STAGE_ENTRIES + 4 * tid;  // entry of this thread's first group
    float4 cur[4];
    if (i + 1 < nst) {  // a full stage: every entry is in the unit
#pragma unroll
      for (int q = 0; q < 4; ++q) cur[q] = ok ? stage[tid + q * A_THREADS] : none;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) cur[q] = ok && eb + 4 * q * A_THREADS < end4 ? stage[tid + q * A_THREADS] : none;
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(&sm.empty[st])) : "memory");
    step16(sm, u, warp, lane, p.k, cur, eb, end);
    u.thr = fmaxf(u.thr, unord((unsigned)(*reinterpret_cast<const volatile unsigned long long*>(gthr) >> 32)));
    if (tid == 0 && i + RING_STAGES < nst) {
      // every warp has read this stage: it takes stage i + RING_STAGES
      if (ring_wait(sm, sa(&sm.empty[st]), par)) ring_issue(sm, ring0, x, start, end4, i + RING_STAGES);
    }
    if (++st == RING_STAGES) {
      st = 0;
      par ^= 1u;
    }
  }
  // entries past the last group of four (at most three), by warp 0
  if (warp == 0) {
    float4 t = none;
    int e = end;
    if (lane == 0 && end4 < end) {
      e = end4;
      t.x = x[end4];
      if (end4 + 1 < end) t.y = x[end4 + 1];
      if (end4 + 2 < end) t.z = x[end4 + 2];
    }
    step4(sm, u, warp, lane, p.k, t, e, end);
  }
  finish_unit(sm, u, p, row, chunk, end, 0, none, none, end, end, dyn_smem, SURV_MAX, dyn_smem);
}


// ---- large batches: persistent CTAs (two per SM), each over an equal share of all entries
// The rows' entries, laid end to end (row r at r * V), are cut into one contiguous share
// per CTA (multiples of four entries; each share at least a row long, so a row lies in at
// most two shares: its first piece is chunk 0 of the workspace, a second piece chunk 1).
// A CTA streams its pieces in order through one ring of P_STAGES bulk-copy stages
// (thread 0 issues them), so the copies of the next piece keep flowing while a piece is
// finished; every piece is a unit like those of topk_level_kernel (same entry order per
// thread, exp-sum grouping, filter, finish and request merge). A row that lies wholly in
// one share also accounts for its empty chunk 1.
constexpr int P_SURV = A_WARPS * KMAX;  // survivors of a streamed unit: the warp lists
constexpr int P_RING_BYTES = P_STAGES * STAGE_ENTRIES * 4;

// Share [lo, hi) of CTA c among g (flat entry indices, multiples of four).
__host__ __device__ inline void share_of(int64_t total, int g, int c, int64_t* lo, int64_t* hi) {
  *lo = ((int64_t)c * total / g) & ~(int64_t)3;
  *hi = c + 1 == g ? total : (((int64_t)(c + 1) * total / g) & ~(int64_t)3);
}

__global__ void __launch_bounds__(A_THREADS, 2) topk_stream_kernel(const LevelArgs p) {
  extern __shared__ float4 dyn_smem[];
  __shared__ TopkSmem sm;
  griddep_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.vocab;
  int64_t lo, hi;
  share_of((int64_t)p.rows_total * V, gridDim.x, blockIdx.x, &lo, &hi);
  float4* ring = dyn_smem;
  float4* surv = dyn_smem + P_RING_BYTES / 16;
  float4* mstage = surv + P_SURV * 8 / 16;
  const uint32_t ring0 = sa(ring);
  const float4 none = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  const int r_first = (int)(lo / V), r_last = hi > lo ? (int)((hi - 1) / V) : r_first - 1;
  // piece of row r inside the share: entries [e0, e1) of the row
  auto piece = [&](int r, int* e0, int* e1) {
    const int64_t a = lo - (int64_t)r * V, z = hi - (int64_t)r * V;
    *e0 = a > 0 ? (int)a : 0;
    *e1 = z < V ? (int)z : V;
  };
  // producer cursor (thread 0): the next stage to copy starts at entry pe of row pr
  int pr = r_first, pe = 0, pe1 = 0;
  if (pr <= r_last) piece(pr, &pe, &pe1);
  int islot = 0;  // ring slot of the next stage to copy (stages go round the ring in order)
  auto issue_next = [&]() {  // thread 0: copy the stage at the cursor, advance it
    if (pr > r_last) return;
    const int st = islot;
    const uint32_t bytes = (uint32_t)min(STAGE_ENTRIES, pe1 - pe) * 4u;  // a multiple of 16
    const uint32_t fb = sa(&sm.full[st]);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            ring0 + (uint32_t)st * (STAGE_ENTRIES * 4)),
        "l"(p.logits + (int64_t)pr * p.row_stride + pe), "r"(bytes), "r"(fb)
        : "memory");
    if (++islot == P_STAGES) islot = 0;
    pe += STAGE_ENTRIES;
    if (pe >= pe1 && ++pr <= r_last) piece(pr, &pe, &pe1);
  };
  if (tid == 0) {
    for (int st = 0; st < P_STAGES; ++st) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sa(&sm.full[st])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&sm.empty[st])),
                   "r"(A_WARPS)
                   : "memory");
    }
    sm.fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int i = 0; i < P_STAGES; ++i) issue_next();
  }
  __syncthreads();
  // ring slot and phase parity of the next stage to consume, advanced stage by stage
  // (no division in the loop)
  int cst = 0;
  uint32_t cpar = 0u;
  for (int r = r_first; r <= r_last; ++r) {
    int e0, e1;
    piece(r, &e0, &e1);
    const int nst = (e1 - e0 + STAGE_ENTRIES - 1) / STAGE_ENTRIES;
    // the piece's first stage: starting reference and seed of the CTA-wide bound
    {
      ring_wait(sm, sa(&sm.full[cst]), cpar);
      const float4* stage = ring + cst * STAGE_F4;
      float m = -INFINITY;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (e0 + 4 * (tid + q * A_THREADS) < e1) m = fmaxf(m, max4(stage[tid + q * A_THREADS]));
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
      if ((lane & 7) == 0) sm.gkey[tid >> 3] = key(m, INT_MAX);
#pragma unroll
      for (int o = 8; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
      if (lane == 0) sm.red[warp] = m;
      if (tid == 0) sm.gthr = 0ull;
      __syncthreads();
      kth_of_64(sm.gkey, p.k, &sm.gthr);
    }
    float first = sm.red[0];
#pragma unroll
    for (int w = 1; w < A_WARPS; ++w) first = fmaxf(first, sm.red[w]);
    __syncthreads();  // sm.red is reused by the finish; sm.gthr is seeded
    UnitState u;
    unit_begin(u, first, sm.gthr);
    const unsigned long long* gthr = &sm.gthr;
    for (int i = 0; i < nst; ++i) {
      const int st = cst;
      const uint32_t par = cpar;
      if (++cst == P_STAGES) {
        cst = 0;
        cpar ^= 1u;
      }
      const bool ok = i == 0 || ring_wait(sm, sa(&sm.full[st]), par);
      const float4* stage = ring + st * STAGE_F4;
      const int eb = e0 + i * STAGE_ENTRIES + 4 * tid;
      float4 cur[4];
      if (i + 1 < nst) {  // a full stage: every entry is in the piece
#pragma unroll
        for (int q = 0; q < 4; ++q) cur[q] = ok ? stage[tid + q * A_THREADS] : none;
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) cur[q] = ok && eb + 4 * q * A_THREADS < e1 ? stage[tid + q * A_THREADS] : none;
      }
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(&sm.empty[st])) : "memory");
      step16(sm, u, warp, lane, p.k, cur, eb, e1);
      u.thr = fmaxf(u.thr, unord((unsigned)(*reinterpret_cast<const volatile unsigned long long*>(gthr) >> 32)));
      if (tid == 0 && pr <= r_last) {
        // every warp has read stage g: its slot takes the next stage at the cursor
        if (ring_wait(sm, sa(&sm.empty[st]), par)) issue_next();
      }
    }
    finish_unit(sm, u, p, r, e0 == 0 ? 0 : 1, e1, 0, none, none, e1, e1, surv, P_SURV, mstage,
                e0 == 0 && e1 == V, false);
  }
  griddep_launch();  // the merge kernel may be scheduled (it waits for this grid)
}

// The request merges of the persistent kernel's level, one CTA per request, after it.
__global__ void __launch_bounds__(A_THREADS) topk_merge_kernel(const LevelArgs p) {
  extern __shared__ float4 dyn_smem[];
  griddep_wait();
  request_merge(p, blockIdx.x, dyn_smem);
}

// ---- streaming: one (row, chunk) unit per CTA -----------------------------------------
__global__ void __launch_bounds__(A_THREADS, CTAS_PER_SM)
topk_level_kernel(const LevelArgs p, bool vec) {
  extern __shared__ float4 dyn_smem[];
  __shared__ TopkSmem sm;
  griddep_wait();
  const int row = blockIdx.y, chunk = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* x = p.logits + (int64_t)row * p.row_stride;
  const int start = chunk * p.chunk_len;
  const int end = min(p.vocab, start + p.chunk_len);
  if (p.ring && vec && end - start >= RING_MIN) {
    stream_ring(sm, p, row, chunk, start, end, x);
    return;
  }

  // Every thread takes 4 consecutive entries per step (one 128-bit load when the row is
  // 16-byte aligned), up to three steps prefetched ahead.
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

  // Common starting reference: the largest of the first entries every thread sees. The
  // maxima of the eight-lane groups (32 entries each) of that first step also seed the
  // CTA-wide bound of a streaming unit.
  float first = fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) first = fmaxf(first, __shfl_xor_sync(FULL, first, o));
  if ((lane & 7) == 0) sm.gkey[tid >> 3] = key(first, INT_MAX);
#pragma unroll
  for (int o = 8; o < 32; o <<= 1) first = fmaxf(first, __shfl_xor_sync(FULL, first, o));
  if (lane == 0) sm.red[warp] = first;
  if (tid == 0) sm.gthr = 0ull;
  __syncthreads();
  if (steps > 2) kth_of_64(sm.gkey, p.k, &sm.gthr);
  first = sm.red[0];
#pragma unroll
  for (int w = 1; w < A_WARPS; ++w) first = fmaxf(first, sm.red[w]);
  __syncthreads();  // sm.red is reused by finish_unit; sm.gthr is seeded
  UnitState u;
  unit_begin(u, first, sm.gthr);

  const int e0 = start + 4 * tid;
  if (steps <= 2) {
    // short unit (one or two steps): every entry stays in registers for the finish
    lse4(u, a, max4(a));
    if (steps == 2) lse4(u, bnext, max4(bnext));
    finish_unit(sm, u, p, row, chunk, end, steps, a, bnext, e0, e0 + 4 * A_THREADS, dyn_smem,
                SURV_MAX, dyn_smem);
    return;
  }
  const unsigned long long* gthr = &sm.gthr;
  int it = 0;
  // Two steps in flight. Every fourth step the exp-sum group (16 terms) is flushed and
  // the filter takes up the CTA-wide bound.
  for (; it < steps; ++it) {
    const float4 c = it + 2 < steps ? load4(it + 2) : none;
    step4(sm, u, warp, lane, p.k, a, e0 + 4 * it * A_THREADS, end);
    a = bnext;
    bnext = c;
    if ((it & 3) == 3) {
      u.lse.flush();
      u.thr = fmaxf(u.thr, unord((unsigned)(*reinterpret_cast<const volatile unsigned long long*>(gthr) >> 32)));
    }
  }
  finish_unit(sm, u, p, row, chunk, end, 0, none, none, end, end, dyn_smem, SURV_MAX, dyn_smem);
}

// ---- small batches: one CTA per frontier row, a thread-block cluster per request -------
// A level of a few requests has too few rows to fill the GPU with (row, chunk) units unless
// they are short, and then the grid-wide ticket and the one-CTA request merge set its
// latency. Here a row is one CTA that holds the whole row in registers (R_NF groups of four
// entries per thread, all loads in flight at once), and the rows of a request form one
// cluster: every CTA stores its row's k cumulative scores and tokens into the rank-0 CTA's
// shared memory, which runs the joint top-K once the cluster barrier completes.
//   - log-sum-exp: the thread's terms against its own largest entry (none above 1),
//     summed in groups of 16 and added exactly into an unevaluated (hi, lo) pair, then
//     combined over the CTA as in the per-unit path.
//   - top-k: t1 = the k-th largest of the warps' largest values is at most the row's k-th
//     largest value, so the entries of value t1 or more hold the row's top k; a thread
//     scans only its groups whose largest entry reaches t1, and the survivors (a handful
//     on untied rows) are ranked by counting. When ties or ordered rows leave more
//     survivors than the buffer holds, an exact bound on (value, index) keys -- the k-th
//     best thread maximum, found among the thread maxima at or above the k-th best warp
//     maximum -- leaves at most k threads' entries.
constexpr int R_THREADS = 512;
constexpr int R_WARPS = R_THREADS / 32;
constexpr int R_NF = 16;                           // groups of four entries per thread
constexpr int R_MAX_VOCAB = 4 * R_NF * R_THREADS;  // 32768 entries per row
constexpr int R_SURV = KMAX * 4 * R_NF;            // k threads' entries (the exact bound)
constexpr int R_MAX_ROWS = 16;                     // cluster size (non-portable above 8)
static_assert(R_WARPS >= KMAX, "the bounds need k warp maxima");

struct RowSmem {
  unsigned long long wkey[R_WARPS];   // exact bound: each warp's best entry (key())
  unsigned wmax[R_WARPS];             // ord() of each warp's largest value
  unsigned long long cand[R_THREADS]; // exact bound: thread maxima at or above it
  unsigned long long surv[R_SURV];    // survivors (key())
  float red[R_WARPS], shi[R_WARPS], slo[R_WARPS];
  float lse[3];                       // the row's log-sum-exp as hi + mid + lo
  unsigned long long tau;
  int nc, ns, ns2;                    // candidates; survivors (value bound, exact bound)
  // rank 0: the request's rows * k candidates in flat order, as keys (ord() of the
  // cumulative score above the complemented flat index: larger is better) and tokens
  alignas(16) unsigned long long jkey[R_MAX_ROWS * KMAX];
  int jtok[R_MAX_ROWS * KMAX];
};

__device__ __forceinline__ float comp(const float4& a, int q) {
  return q == 0 ? a.x : (q == 1 ? a.y : (q == 2 ? a.z : a.w));
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of this CTA's shared-memory object p in the shared memory of cluster rank r.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, int r) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(out)
               : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(r));
  return out;
}
__device__ __forceinline__ void st_cluster(uint32_t a, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cluster(uint32_t a, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}

// Appends the entries of group g (first index e) that the predicate keeps; out of line so
// that the sixteen call sites stay small.
__device__ __noinline__ void row_push(RowSmem& sm, int* count, float4 g, int e, int V, float tv,
                                      unsigned long long tau) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float v = comp(g, q);
    const unsigned long long u = key(v, e + q);
    if (e + q < V && v >= tv && u >= tau) {
      const int at = atomicAdd(count, 1);
      if (at < R_SURV) sm.surv[at] = u;
    }
  }
}

// The exact bound (rare): every thread's best entry as a key, the k-th best warp maximum,
// the thread maxima at or above it, their k-th best tau, and the entries at or above tau
// (at most k threads' entries). Called by the whole CTA; leaves the sm.ns2 survivors in
// sm.surv (sm.nc, sm.ns2 and sm.tau start at zero).
__device__ __forceinline__ void row_exact(RowSmem& sm, const float4 (&a)[R_NF], int V, int k) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float m = a[0].x;
  int am = 0;
#pragma unroll
  for (int t = 1; t < 4 * R_NF; ++t) {
    const float v = comp(a[t >> 2], t & 3);
    if (v > m) { m = v; am = t; }
  }
  const int mi = 4 * tid + 4 * R_THREADS * (am >> 2) + (am & 3);
  const unsigned long long kt = 4 * tid < V ? key(m, mi) : 0ull;
  {
    const unsigned h = __reduce_max_sync(FULL, (unsigned)(kt >> 32));
    const unsigned l = __reduce_max_sync(FULL, (unsigned)(kt >> 32) == h ? (unsigned)kt : 0u);
    if (lane == 0) sm.wkey[warp] = ((unsigned long long)h << 32) | l;
  }
  __syncthreads();
  unsigned long long tau1;
  {
    const unsigned long long mine = lane < R_WARPS ? sm.wkey[lane] : 0ull;
    int rank = 0;
#pragma unroll
    for (int o = 0; o < R_WARPS; ++o) {
      const unsigned long long w = sm.wkey[o];
      rank += (w > mine || (w == mine && o < lane)) ? 1 : 0;
    }
    const unsigned sel = __ballot_sync(FULL, lane < R_WARPS && rank == k - 1);
    tau1 = __shfl_sync(FULL, mine, __ffs(sel) - 1);
  }
  {
    const bool c = kt != 0ull && kt >= tau1;
    const unsigned bal = __ballot_sync(FULL, c);
    if (bal) {
      const int leader = __ffs(bal) - 1;
      int at = 0;
      if (lane == leader) at = atomicAdd(&sm.nc, __popc(bal));
      at = __shfl_sync(FULL, at, leader);
      if (c) sm.cand[at + __popc(bal & ((1u << lane) - 1u))] = kt;
    }
  }
  __syncthreads();
  const int nc = sm.nc;  // 0 < nc: fewer than k means every entry survives (tau stays 0)
  for (int c = tid; c < nc; c += R_THREADS) {
    const unsigned long long u = sm.cand[c];
    int rank = 0;
    for (int o = 0; o < nc; ++o) rank += sm.cand[o] > u ? 1 : 0;
    if (rank == k - 1) sm.tau = u;
  }
  __syncthreads();
  const unsigned long long tau = sm.tau;
  if (kt != 0ull && kt >= tau) {
    const float tv = tau != 0ull ? unord((unsigned)(tau >> 32)) : -INFINITY;
#pragma unroll
    for (int j = 0; j < R_NF; ++j)
      if (fmaxf(fmaxf(a[j].x, a[j].y), fmaxf(a[j].z, a[j].w)) >= tv)
        row_push(sm, &sm.ns2, a[j], 4 * (tid + R_THREADS * j), V, tv, tau);
  }
  __syncthreads();
}

// grid (rows, batch), cluster (rows, 1, 1): blockIdx.x is the frontier row and the rank in
// the request's cluster. VEC: 16-byte aligned rows (128-bit loads), else scalar loads.
template <bool VEC>
__global__ void __launch_bounds__(R_THREADS, 1) topk_row_kernel(const LevelArgs p) {
  __shared__ RowSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s = blockIdx.x, b = blockIdx.y;
  const int rows = p.rows, k = p.k, V = p.vocab;
  const int r0 = b * rows + s;
  // every CTA of the cluster has started before the first store into rank 0's memory
  cluster_arrive_relaxed();
  if (tid == 0) {
    sm.ns = 0;
    sm.ns2 = 0;
    sm.nc = 0;
    sm.tau = 0ull;
  }
  griddep_wait();
  griddep_launch();  // one wave of CTAs: the next kernel may be scheduled beside it
  const float pscore = p.level == 1 ? (p.product ? 1.0f : 0.0f) : p.front_score_in[r0];
  const int pstore = p.level == 1 ? -1 : p.front_store_in[r0];
  const float* x = p.logits + (int64_t)r0 * p.row_stride;

  // entry 4 (tid + R_THREADS j) + q of the row sits in a[j], component q; entries past
  // the row are -inf (never kept, zero exp-sum terms)
  const float4 none = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  float4 a[R_NF];
#pragma unroll
  for (int j = 0; j < R_NF; ++j) {
    const int e = 4 * (tid + R_THREADS * j);
    if (VEC) {
      a[j] = e + 3 < V ? ld_stream(reinterpret_cast<const float4*>(x + e)) : none;
    } else {
      a[j].x = e < V ? x[e] : -INFINITY;
      a[j].y = e + 1 < V ? x[e + 1] : -INFINITY;
      a[j].z = e + 2 < V ? x[e + 2] : -INFINITY;
      a[j].w = e + 3 < V ? x[e + 3] : -INFINITY;
    }
  }
  if (VEC && (V & 3)) {  // the group that straddles the row's end
#pragma unroll
    for (int j = 0; j < R_NF; ++j) {
      const int e = 4 * (tid + R_THREADS * j);
      if (e < V && e + 3 >= V) {
        a[j].x = x[e];
        a[j].y = e + 1 < V ? x[e + 1] : -INFINITY;
        a[j].z = e + 2 < V ? x[e + 2] : -INFINITY;
      }
    }
  }

  // group maxima and the thread's largest value
  float m4[R_NF];
#pragma unroll
  for (int j = 0; j < R_NF; ++j) m4[j] = fmaxf(fmaxf(a[j].x, a[j].y), fmaxf(a[j].z, a[j].w));
  float m;
  {
    float t8[R_NF / 2];
#pragma unroll
    for (int j = 0; j < R_NF / 2; ++j) t8[j] = fmaxf(m4[2 * j], m4[2 * j + 1]);
    const float t4a = fmaxf(fmaxf(t8[0], t8[1]), fmaxf(t8[2], t8[3]));
    const float t4b = fmaxf(fmaxf(t8[4], t8[5]), fmaxf(t8[6], t8[7]));
    m = fmaxf(t4a, t4b);
  }
  {
    const unsigned wm = __reduce_max_sync(FULL, ord(m));
    if (lane == 0) sm.wmax[warp] = wm;
  }
  // exp-sum against the thread's largest entry
  {
    const float ref = fmaxf(m, -1e30f), rl = ref * L2E;  // finite: x = -inf gives 0
    float hi = 0.f, lo = 0.f;
#pragma unroll
    for (int g = 0; g < R_NF / 4; ++g) {
      float gs = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 c = a[4 * g + u];
        gs += (ex2(fmaf(c.x, L2E, -rl)) + ex2(fmaf(c.y, L2E, -rl))) +
              (ex2(fmaf(c.z, L2E, -rl)) + ex2(fmaf(c.w, L2E, -rl)));
      }
      pair_add(hi, lo, gs, 0.f);
    }
    float R = ref;
    warp_combine(R, hi, lo);
    if (lane == 0) { sm.red[warp] = R; sm.shi[warp] = hi; sm.slo[warp] = lo; }
  }
  __syncthreads();

  // t1: the k-th largest warp maximum (every warp computes it; ties by warp)
  float tv;
  {
    const unsigned mine = lane < R_WARPS ? sm.wmax[lane] : 0u;
    int rank = 0;
#pragma unroll
    for (int o = 0; o < R_WARPS; ++o) {
      const unsigned w = sm.wmax[o];
      rank += (w > mine || (w == mine && o < lane)) ? 1 : 0;
    }
    const unsigned sel = __ballot_sync(FULL, lane < R_WARPS && rank == k - 1);
    tv = unord(__shfl_sync(FULL, mine, __ffs(sel) - 1));
  }
  // survivors: entries of value tv or more
  if (m >= tv) {
#pragma unroll
    for (int j = 0; j < R_NF; ++j)
      if (m4[j] >= tv) row_push(sm, &sm.ns, a[j], 4 * (tid + R_THREADS * j), V, tv, 0ull);
  }
  if (warp == R_WARPS - 1) {  // the row's exp-sum
    float rr = lane < R_WARPS ? sm.red[lane] : -INFINITY;
    float hh = lane < R_WARPS ? sm.shi[lane] : 0.f, ll = lane < R_WARPS ? sm.slo[lane] : 0.f;
    warp_combine(rr, hh, ll);
    // log(hi + lo) = log(hi) + log1p(lo / hi); |lo / hi| is below an ulp
    if (lane == 0) { sm.lse[0] = rr; sm.lse[1] = logf(hh); sm.lse[2] = ll / hh; }
  }
  __syncthreads();
  int S = sm.ns;
  if (S > R_SURV) {  // block-uniform
    row_exact(sm, a, V, k);
    S = sm.ns2;
  }

  // the row's top k by rank among the survivors (one warp with shuffles when they fit a
  // warp), stored into rank 0's shared memory as joint keys
  const int off = p.level == 1 ? 0 : k + (p.level - 2) * k * k;
  if (s == 0 && tid >= rows * k && tid < (rows * k + 7) / 8 * 8) sm.jkey[tid] = 0ull;  // padding
  cluster_wait();  // every CTA of the cluster has started
  float cu = 0.f;
  int tok = -1, flat = -1;
  auto take = [&](unsigned long long u, int rank) {
    if (flat >= 0) {  // a second candidate of this thread (more than R_THREADS survivors)
      const int64_t at = (int64_t)b * p.store_cap + off + flat;
      p.store_token[at] = tok;
      p.store_score[at] = cu;
      p.store_parent[at] = pstore;
    }
    const float v = unord((unsigned)(u >> 32));
    const float logp = ((v - sm.lse[0]) - sm.lse[1]) - sm.lse[2];
    cu = p.product ? pscore * expf(logp) : pscore + logp;
    tok = (int)~(unsigned)u;
    flat = s * k + rank;
    const float cz = cu == 0.f ? 0.f : cu;  // -0 and +0 tie, as the comparison of scores has it
    st_cluster(cluster_addr(&sm.jkey[flat], 0), ((unsigned long long)ord(cz) << 32) | ~(unsigned)flat);
    st_cluster(cluster_addr(&sm.jtok[flat], 0), tok);
  };
  if (S <= 32) {
    if (warp == 0) {
      const unsigned long long u = lane < S ? sm.surv[lane] : 0ull;
      int rank = 0;
#pragma unroll
      for (int o = 0; o < 32; ++o) rank += __shfl_sync(FULL, u, o) > u ? 1 : 0;
      if (lane < S && rank < k) take(u, rank);
    }
  } else {
    for (int t = tid; t < S; t += R_THREADS) {
      const unsigned long long u = sm.surv[t];
      int rank = 0;
      for (int o = 0; o < S; ++o) rank += sm.surv[o] > u ? 1 : 0;
      if (rank < k) take(u, rank);
    }
  }
  cluster_arrive_release();
  if (flat >= 0) {  // the row's candidates (after the release: it does not wait for them)
    const int64_t at = (int64_t)b * p.store_cap + off + flat;
    p.store_token[at] = tok;
    p.store_score[at] = cu;
    p.store_parent[at] = pstore;
  }
  cluster_wait();  // rank 0: every row's keys have landed
  if (s != 0) return;

  // Joint top-K over the rows * K candidates: a candidate's rank is the number of larger
  // keys (larger cumulative score, then lower flat index). Four lanes per candidate count
  // a quarter of the keys each (two keys per 128-bit load; the padding keys are zero).
  const int nf = rows * k, n2 = (nf + 7) / 8 * 4;  // key pairs
  const ulonglong2* kp = reinterpret_cast<const ulonglong2*>(sm.jkey);
  for (int f0 = 0; f0 < nf; f0 += R_THREADS / 4) {
    if (f0 + 8 * warp >= nf) break;  // warp-uniform: the warp's eight candidates are past the end
    const int f = f0 + (tid >> 2), part = tid & 3;
    const unsigned long long kf = f < nf ? sm.jkey[f] : ~0ull;
    int rank = 0;
#pragma unroll 4
    for (int u = part; u < n2; u += 4) {
      const ulonglong2 x = kp[u];
      rank += (x.x > kf ? 1 : 0) + (x.y > kf ? 1 : 0);
    }
    rank += __shfl_xor_sync(FULL, rank, 1);
    rank += __shfl_xor_sync(FULL, rank, 2);
    if (part == 0 && f < nf && rank < k) {
      p.front_token_out[b * k + rank] = sm.jtok[f];
      p.front_score_out[b * k + rank] = unord((unsigned)(kf >> 32));
      p.front_store_out[b * k + rank] = off + f;
    }
  }
}

// ---- final selection --------------------------------------------------------------
// The total_tokens best candidates by key (ord() of the score; -0 taken as +0), ties to
// the lower store index. One 12-bit histogram pass finds the bin that holds the
// total_tokens-th best key; the candidates of that bin (a few dozen on spread scores) are
// ranked exactly by counting. When a bin holds more than F_BIN_MAX candidates (heavily
// tied scores) a radix select over the full key in three passes (11, 11 and 10 bits)
// gives the threshold key and the number of its equal keys to keep, in ascending store
// index. Node numbers (ascending store index) come from a block prefix sum. With
// tsv_draft_select_tree one warp then builds the selected trees' metadata.
constexpr int F_THREADS = 512;
constexpr int F_WARPS = F_THREADS / 32;
constexpr int F_MAX = 4096;                 // candidates per request
constexpr int F_PER = F_MAX / F_THREADS;    // candidates per thread
constexpr int F_TOP_BITS = 12;              // first pass: the key's top 12 bits
constexpr int F_TOP_BINS = 1 << F_TOP_BITS;
constexpr int F_BIN_MAX = 512;              // threshold-bin candidates ranked directly
constexpr int F_BINS = 2048;                // histogram bins of the fallback's widest pass

__device__ __forceinline__ unsigned score_key(float x) { return ord(x == 0.f ? 0.f : x); }

// Exclusive prefix sum of x over the block (thread order); s_warp holds F_WARPS
// partials. One barrier: two calls on the same s_warp need a barrier between them.
__device__ __forceinline__ int block_exclusive_scan(int x, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  const int ws = lane < F_WARPS && lane < warp ? s_warp[lane] : 0;
  return __reduce_add_sync(FULL, ws) + incl - x;
}

// Fallback radix select over the full keys: the total-th largest key and the number of
// candidates with exactly that key that are kept (the lowest store indices).
__device__ __noinline__ void radix_threshold(const unsigned* s_key, int C, int total,
                                             unsigned* s_hist, int* s_warp, unsigned* s_sel,
                                             unsigned& prefix_out, int& need_out) {
  const int tid = threadIdx.x;
  unsigned prefix = 0;
  int need = total;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int bits = pass == 2 ? 10 : 11;
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = 1 << bits, per = nb / F_THREADS;
    __syncthreads();  // the previous users of s_hist, s_sel and s_warp are done
    for (int i = tid; i < nb; i += F_THREADS) s_hist[i] = 0u;
    __syncthreads();
    for (int c = tid; c < C; c += F_THREADS) {
      const unsigned key = s_key[c];
      if (pass == 0 || (key >> (shift + bits)) == prefix) atomicAdd(&s_hist[(key >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    // thread t holds `per` bins from the top: nb - 1 - t * per downwards
    int local = 0;
    for (int q = 0; q < per; ++q) local += (int)s_hist[nb - 1 - (tid * per + q)];
    int acc = block_exclusive_scan(local, s_warp);  // candidates in the bins above
    if (acc < need && need <= acc + local) {
      for (int q = 0; q < per; ++q) {
        const int bin = nb - 1 - (tid * per + q);
        const int n = (int)s_hist[bin];
        if (acc + n >= need) {
          s_sel[0] = (unsigned)bin;
          s_sel[1] = (unsigned)acc;
          break;
        }
        acc += n;
      }
    }
    __syncthreads();
    prefix = (prefix << bits) | s_sel[0];
    need -= (int)s_sel[1];
  }
  prefix_out = prefix;
  need_out = need;
  __syncthreads();
}

__global__ void __launch_bounds__(F_THREADS)
select_final_kernel(const int32_t* __restrict__ store_token, const float* __restrict__ store_score,
                    const int32_t* __restrict__ store_parent, int C, int store_cap,
                    int total, const int32_t* __restrict__ root_token, int max_nodes,
                    int32_t* __restrict__ tokens, int32_t* __restrict__ parents,
                    int32_t* __restrict__ num_nodes, const int32_t* __restrict__ prefix_len,
                    int max_depth, MetaOut meta) {
  __shared__ unsigned s_key[F_MAX];
  // the histogram until the threshold is known, then the kept flags and node numbers
  static_assert(F_TOP_BINS == F_MAX && F_BINS <= F_TOP_BINS, "one array for both");
  __shared__ unsigned s_hist[F_TOP_BINS];
  int* s_node = reinterpret_cast<int*>(s_hist);
  __shared__ unsigned long long s_bin[F_BIN_MAX];  // key above the complemented index
  __shared__ int s_warp[2][F_WARPS];
  __shared__ unsigned s_sel[2];
  __shared__ int s_nbin;
  // the tree's metadata (meta.mask set): parents by node, the builder's scratch
  __shared__ int32_t s_tpar[TSV_MAX_NODES], s_dep[TSV_MAX_NODES], s_first[TSV_MAX_NODES],
      s_last[TSV_MAX_NODES];
  const int b = blockIdx.x, tid = threadIdx.x;
  const int64_t srow = (int64_t)b * store_cap;
  for (int i = tid; i < F_TOP_BINS; i += F_THREADS) s_hist[i] = 0u;
  if (tid == 0) s_nbin = 0;
  griddep_wait();
  griddep_launch();
  unsigned kr[F_PER];
#pragma unroll
  for (int i = 0; i < F_PER; ++i) {
    const int c = tid + i * F_THREADS;
    kr[i] = c < C ? score_key(store_score[srow + c]) : 0u;
  }
  __syncthreads();  // the histogram is clear
#pragma unroll
  for (int i = 0; i < F_PER; ++i) {
    const int c = tid + i * F_THREADS;
    if (c < C) {
      s_key[c] = kr[i];
      atomicAdd(&s_hist[kr[i] >> (32 - F_TOP_BITS)], 1u);
    }
  }
  __syncthreads();
  // the threshold bin: thread t holds bins F_TOP_BINS - 1 - 8t downwards
  static_assert(F_TOP_BINS == 8 * F_THREADS, "eight bins per thread");
  unsigned hv[8];
  int local = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    hv[q] = s_hist[F_TOP_BINS - 1 - (tid * 8 + q)];
    local += (int)hv[q];
  }
  int acc = block_exclusive_scan(local, s_warp[0]);  // candidates in the bins above
  if (acc < total && total <= acc + local) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (acc < total && total <= acc + (int)hv[q]) {
        s_sel[0] = (unsigned)(F_TOP_BINS - 1 - (tid * 8 + q));
        s_sel[1] = (unsigned)acc;
      }
      acc += (int)hv[q];
    }
  }
  __syncthreads();
  const unsigned bin = s_sel[0];
  const int need = total - (int)s_sel[1];  // candidates kept from the threshold bin
#pragma unroll
  for (int i = 0; i < F_PER; ++i) {
    const int c = tid + i * F_THREADS;
    if (c < C && (kr[i] >> (32 - F_TOP_BITS)) == bin) {
      const int at = atomicAdd(&s_nbin, 1);
      if (at < F_BIN_MAX) s_bin[at] = ((unsigned long long)kr[i] << 32) | ~(unsigned)c;
    }
  }
  __syncthreads();
  const int nbin = s_nbin;
  if (nbin <= F_BIN_MAX) {  // block-uniform
    // kept: the bins above; in the threshold bin, the `need` best by (key, lower index)
#pragma unroll
    for (int i = 0; i < F_PER; ++i) {
      const int c = tid + i * F_THREADS;
      if (c < C && (kr[i] >> (32 - F_TOP_BITS)) != bin)
        s_node[c] = (kr[i] >> (32 - F_TOP_BITS)) > bin ? 1 : 0;
    }
    for (int t = tid; t < nbin; t += F_THREADS) {
      const unsigned long long u = s_bin[t];
      int rank = 0;
#pragma unroll 4
      for (int o = 0; o < nbin; ++o) rank += s_bin[o] > u ? 1 : 0;
      s_node[~(unsigned)u] = rank < need ? 1 : 0;
    }
  } else {
    unsigned prefix;
    int need2;
    radix_threshold(s_key, C, total, s_hist, s_warp[1], s_sel, prefix, need2);
    // equal keys kept in ascending store index: contiguous per-thread segments
    const int seg = (C + F_THREADS - 1) / F_THREADS;
    const int c0 = min(C, tid * seg), c1 = min(C, c0 + seg);
    int eq = 0;
    for (int c = c0; c < c1; ++c) eq += s_key[c] == prefix ? 1 : 0;
    int e = block_exclusive_scan(eq, s_warp[0]);
    for (int c = c0; c < c1; ++c) {
      const unsigned key = s_key[c];
      s_node[c] = key > prefix || (key == prefix && e++ < need2) ? 1 : 0;
    }
  }
  __syncthreads();

  // node numbers in ascending store index, over contiguous per-thread segments
  const int seg = (C + F_THREADS - 1) / F_THREADS;
  const int c0 = min(C, tid * seg), c1 = min(C, c0 + seg);
  int mine = 0;
  for (int c = c0; c < c1; ++c) mine += s_node[c];
  int before = block_exclusive_scan(mine, s_warp[1]);
  for (int c = c0; c < c1; ++c)
    if (s_node[c]) s_node[c] = 1 + before++;
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
    const int pn = (p >= 0 && p < C) ? s_node[p] : 0;
    parents[trow + node] = pn;
    s_tpar[node] = pn;
  }
  if (meta.mask) {  // the tree's metadata, from the parents in shared memory
    if (tid == 0) s_tpar[0] = -1;
    __syncthreads();
    if (tid < 32)
      build_meta_warp(b, s_tpar, total + 1, prefix_len[b], max_nodes, max_depth, meta, s_tpar,
                      s_dep, s_first, s_last);
  }
}

// Clusters of `rows` row CTAs that can be resident at once (0 when the device or the
// runtime cannot run them), cached per device and cluster size.
int row_cluster_capacity(int rows) {
  static int cache[64][R_MAX_ROWS + 1];
  static bool known[64][R_MAX_ROWS + 1] = {};
  int dev = 0;
  if (rows < 1 || rows > R_MAX_ROWS || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  if (known[dev][rows]) return cache[dev][rows];
  int n = 0;
  if (device_cc() >= 90 &&
      cudaFuncSetAttribute(topk_row_kernel<true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
          cudaSuccess &&
      cudaFuncSetAttribute(topk_row_kernel<false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
          cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rows, 1);
    cfg.blockDim = dim3(R_THREADS);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = rows;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, topk_row_kernel<true>, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  cache[dev][rows] = n;
  known[dev][rows] = true;
  return n;
}

}  // namespace

TopkPlan plan_topk(int batch, int rows, int vocab, int top_k) {
  TopkPlan p{};
  const int64_t rows_total = (int64_t)batch * rows;
  // Small batches: one CTA per row and a cluster per request, when the row fits the CTA's
  // registers and the clusters run in at most two waves.
  if (vocab <= R_MAX_VOCAB && rows <= R_MAX_ROWS && rows_total <= 2 * device_sm_count() &&
      batch <= 2 * row_cluster_capacity(rows)) {
    p.cluster = true;
    p.chunks = 1;
    p.chunk_len = (int)round_up(vocab, 4);
    p.ws_bytes = align256((size_t)batch * sizeof(unsigned));
    return p;
  }
  // Large batches: the persistent kernel, one CTA per SM, when every share is at least a
  // row long (with room for the rounding to four entries) and rows are whole groups of
  // four entries; chunks = 2 gives each row two workspace slots (its at most two pieces),
  // and chunk_len lets the per-unit kernel use the same layout should the logits turn
  // out not to be 16-byte aligned.
  const int64_t shares = (int64_t)P_CTAS_PER_SM * device_sm_count();
  if (vocab % 4 == 0 && vocab >= RING_MIN && shares > 0 &&
      rows_total * vocab / shares - 8 >= vocab) {
    p.persistent = true;
    p.chunks = 2;
    p.chunk_len = (int)round_up(ceil_div(vocab, 2), 4);
    const size_t n = (size_t)rows_total * p.chunks;
    p.ws_bytes = align256((size_t)batch * sizeof(unsigned)) + align256(n * sizeof(ChunkStat)) +
                 align256(n * top_k * sizeof(float)) + align256(n * top_k * sizeof(int32_t));
    return p;
  }
  // Chunks per row: the count with the shortest estimated makespan, waves of resident CTAs
  // x (chunk length + a fixed cost per unit of about FIX_ENTRIES entries' streaming time:
  // start, finish and merge).
  constexpr int64_t FIX_ENTRIES = 16384;
  const int64_t slots = (int64_t)CTAS_PER_SM * device_sm_count();
  const int64_t cmax = std::max<int64_t>(1, std::min<int64_t>(MAX_CHUNKS, ceil_div(vocab, MIN_CHUNK)));
  int64_t best_c = 1, best_cost = INT64_MAX;
  for (int64_t c = 1; c <= cmax; ++c) {
    const int64_t len = round_up(ceil_div(vocab, c), 4);
    const int64_t waves = ceil_div(rows_total * ceil_div(vocab, len), slots);
    const int64_t cost = waves * (len + FIX_ENTRIES);
    if (cost < best_cost) { best_cost = cost; best_c = c; }
  }
  int chunks = (int)best_c;
  int chunk_len = (int)round_up(ceil_div(vocab, chunks), 4);
  chunks = (int)ceil_div(vocab, chunk_len);
  p.chunks = chunks;
  p.chunk_len = chunk_len;
  const size_t n = (size_t)rows_total * chunks;
  p.ws_bytes = align256((size_t)batch * sizeof(unsigned)) + align256(n * sizeof(ChunkStat)) +
               align256(n * top_k * sizeof(float)) + align256(n * top_k * sizeof(int32_t));
  return p;
}

int launch_topk_expand(const float* logits, int batch, int rows, int64_t row_stride, int vocab,
                       int top_k, int level, const float* front_score_in,
                       const int32_t* front_store_in, int store_cap, int32_t* store_token,
                       float* store_score, int32_t* store_parent, int32_t* front_token_out,
                       float* front_score_out, int32_t* front_store_out, void* ws,
                       const TopkPlan& plan, bool product, cudaStream_t stream) {
  const int rows_total = batch * rows;
  LevelArgs p;
  p.logits = logits;
  p.row_stride = row_stride;
  p.vocab = vocab;
  p.rows = rows;
  p.k = top_k;
  p.chunks = plan.chunks;
  p.chunk_len = plan.chunk_len;
  p.level = level;
  p.product = product;
  p.ws = carve(ws, batch, rows_total, plan.chunks, top_k);
  p.front_score_in = front_score_in;
  p.front_store_in = front_store_in;
  p.store_cap = store_cap;
  p.store_token = store_token;
  p.store_score = store_score;
  p.store_parent = store_parent;
  p.front_token_out = front_token_out;
  p.front_score_out = front_score_out;
  p.front_store_out = front_store_out;
  const bool vec = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) && (row_stride % 4 == 0);
  p.ring = vec && plan.chunk_len >= RING_MIN;
  p.rows_total = rows_total;
  int dev = 0;
  cudaGetDevice(&dev);
  if (plan.cluster) {
    if (row_cluster_capacity(rows) < 1) return TSV_ERR_UNSUPPORTED;  // sets the cluster attribute
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rows, batch);
    cfg.blockDim = dim3(R_THREADS);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = rows;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    void (*kern)(const LevelArgs) = vec ? topk_row_kernel<true> : topk_row_kernel<false>;
    if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) {
      cudaGetLastError();  // no programmatic serialization here: a plain cluster launch
      cfg.numAttrs = 1;
      cudaLaunchKernelEx(&cfg, kern, p);
    }
    return launch_status();
  }
  if (plan.persistent && vec) {
    // ring, survivors, and the request merge's staging for two slots per row
    constexpr size_t P_MERGE_MAX = (size_t)TSV_MAX_TOPK * 3 * TSV_MAX_TOPK * 8;
    constexpr size_t P_SMEM_MAX = (size_t)P_RING_BYTES + (size_t)P_SURV * 8 + P_MERGE_MAX;
    const size_t psmem = (size_t)P_RING_BYTES + (size_t)P_SURV * 8;
    static bool pattr_set[64] = {};
    if (dev < 0 || dev >= 64) return TSV_ERR_UNSUPPORTED;
    if (!pattr_set[dev]) {
      if (cudaFuncSetAttribute(topk_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)P_SMEM_MAX) != cudaSuccess)
        return launch_status();
      pattr_set[dev] = true;
    }
    const int st = launch_pdl(topk_stream_kernel, dim3(P_CTAS_PER_SM * device_sm_count()),
                              dim3(A_THREADS), psmem, stream, p);
    if (st != TSV_OK) return st;
    return launch_pdl(topk_merge_kernel, dim3(batch), dim3(A_THREADS),
                      (size_t)rows * (plan.chunks + 1) * top_k * 8, stream, p);
  }
  dim3 grid(plan.chunks, rows_total);
  const size_t smem = std::max<size_t>({(size_t)SURV_MAX * 8,
                                        (size_t)rows * (plan.chunks + 1) * top_k * 8,
                                        p.ring ? (size_t)RING_BYTES : (size_t)0});
  static bool attr_set[64] = {};
  if (smem > 48 * 1024 && dev >= 0 && dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(topk_level_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             std::max({MERGE_SMEM_MAX, SURV_MAX * 8, RING_BYTES})) != cudaSuccess)
      return launch_status();
    attr_set[dev] = true;
  }
  return launch_pdl(topk_level_kernel, grid, dim3(A_THREADS), smem, stream, p, vec);
}

int launch_select_final(const int32_t* store_token, const float* store_score,
                        const int32_t* store_parent, int batch, int num_candidates,
                        int store_cap, int total_tokens, const int32_t* root_token,
                        int max_nodes, int32_t* tokens, int32_t* parents, int32_t* num_nodes,
                        const int32_t* prefix_len, int max_depth, const MetaOut* meta,
                        cudaStream_t stream) {
  if (num_candidates > F_MAX) return TSV_ERR_INVALID_ARG;
  const MetaOut none{};
  return launch_pdl(select_final_kernel, dim3(batch), dim3(F_THREADS), 0, stream, store_token,
                    store_score, store_parent, num_candidates, store_cap, total_tokens,
                    root_token, max_nodes, tokens, parents, num_nodes, prefix_len, max_depth,
                    meta ? *meta : none);
}

}  // namespace tsv
