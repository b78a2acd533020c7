// Tree-verification attention on the 5th-generation tensor cores (tcgen05 + TMEM), bf16 in,
// fp32 accumulate, head_dim 128, with K/V brought into shared memory by cp.async.
//
// Pages: "推理系统手册 · 投机解码进阶：树形草稿与 EAGLE", section 实现 (forward_with_mask:
// each node attends to the whole prefix and, among the tree nodes, to its ancestors and
// itself; GQA heads share a KV head) and "TensorRT-LLM 源码完全拆解(二十二)", section
// CUDA Graph 里的掩码重排 (the attention reads the padded bit mask directly).
//
// One CTA = (request b, KV head h, one M tile of 128 query rows, split of the keys). The
// query rows of a KV head are every (node, query head of the group) pair, so each K/V
// tile serves all of them.
//
//   warps 4-5   loaders: 16-byte cp.async copies of 128-key K and V tiles into a 3-stage
//               K ring and a 4-stage V ring, K two tiles ahead of V, written in the
//               128-byte-swizzled K-major panel layout the MMAs read (rows at or past the
//               zero-padded end of the tree are zero-filled, never read). A loader thread
//               keeps at most three tiles of its own in flight; once a tile's copies have
//               landed it makes them visible to the tensor cores (proxy fence) and
//               arrives on the tile's FULL barrier (64 arrivals complete it). Before it
//               would block on a ring slot it signals every tile it still holds, so no
//               wait of the MMA warp can depend on a blocked loader.
//   warp 6      TMEM allocator + MMA issuer (warp-uniform descriptors, one elected lane
//               per instruction). After S_0 and S_1, step j issues
//                 O     += P_j V_j          A = P_j in TMEM, B = V (shared, MN-major)
//                 S_{j+2} = Q K_{j+2}^T     A = Q in TMEM, B = K (shared, K-major)
//               P_j V_j once the softmax has written P_j (GO phase j) and V_j is in; S_{j+2}
//               once P_j V_j has completed (S_{j+2} overwrites P_j's buffer, and only
//               MMAs into the same accumulator are ordered) and K_{j+2} is in.
//   warps 0-3   softmax warpgroup; thread = query row = TMEM lane. Each thread first
//               copies its rotated query row into TMEM (zeros for rows past the tree).
//               Per tile: one x128 TMEM load of S_j, the row max over 8 chains,
//               P = exp2(s * scale * log2e - m) rounded to bf16 and stored over S_j. The
//               running max m is raised only when a tile's max exceeds it by more than 8
//               (log2 units), and O in TMEM is rescaled then (after P_{j-1} V_{j-1} has
//               finished), otherwise never.
// TMEM (512 columns allocated): S/P[0] [0,128) S/P[1] [128,256) O [256,384) Q [384,448).
// A CTA that covers every key of its rows writes the normalised bf16 output itself;
// otherwise it writes its unnormalised O rows plus (m, l) for the split merge.
//
// Every mbarrier wait is bounded; on a timeout the CTA records TSV_REQ_TIMEOUT for the
// request, stops issuing work, waits for its copies and MMAs and frees its TMEM.
#include <stdint.h>

#include "attn_common.cuh"
#include "common.cuh"

namespace tsv {
namespace {

#include "tc_ptx.cuh"

constexpr int KEYS = 128;                 // keys per tile
constexpr int KST = 3, VST = 4;           // K and V ring depths (V tiles live two steps longer)
constexpr int LOAD_WARP0 = 4, MMA_WARP = 6;
constexpr int LOADERS = 64;               // loader threads
// seven warps: a sub-partition holds at most two, so ~200 registers per thread fit
constexpr int THREADS = 7 * 32;
constexpr uint32_t HALF = 128 * 128;      // 128 rows x 64 bf16 (one 128-byte-swizzled panel)
constexpr uint32_t TILE = 2 * HALF;       // 128 rows x 128 bf16
constexpr uint32_t SMEM_K = 0;            // KST K tiles
constexpr uint32_t SMEM_V = SMEM_K + KST * TILE;  // VST V tiles
constexpr uint32_t SMEM_BAR = SMEM_V + VST * TILE;
constexpr uint32_t SMEM_BYTES = SMEM_BAR + 256 + 1024;  // + alignment slack
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_S = 0;    // two S buffers of 128 columns; P_j is written over the
                                  // first 64 columns of S_j's buffer (128 bf16 per row)
constexpr uint32_t TMEM_O = 256;
constexpr uint32_t TMEM_Q = 384;  // 64 columns: the row's 128 rotated query values
constexpr float RESCALE_LOG2 = 8.f;
constexpr int CHUNKS_PER_THREAD = KEYS * 16 / LOADERS;  // 16-byte copies per tile

// barrier slots (8 bytes each) after SMEM_BAR
constexpr int BAR_Q = 0, BAR_K_FULL = 1, BAR_K_EMPTY = BAR_K_FULL + KST,
              BAR_V_FULL = BAR_K_EMPTY + KST, BAR_V_EMPTY = BAR_V_FULL + VST,
              BAR_S_FULL = BAR_V_EMPTY + VST, BAR_PV_DONE = BAR_S_FULL + 2,
              BAR_O_DONE = BAR_PV_DONE + 2,
              BAR_DRAIN = BAR_O_DONE + 1, BAR_GO = BAR_DRAIN + 1, NUM_BARS = BAR_GO + 2;
static_assert(8 * NUM_BARS + 12 <= 256, "barrier area");
static_assert(SMEM_BYTES <= 232448, "shared memory per block");
static_assert(CHUNKS_PER_THREAD * LOADERS == KEYS * 16, "a tile splits evenly over the loaders");

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool fill) {
  // src-size 0 writes sixteen zero bytes and reads nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(fill ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// the copies this thread has seen land become visible to the tensor cores' reads
__device__ __forceinline__ void fence_to_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

struct UmmaParams {
  AttnArgs a;
  float scale_log2;
  __nv_bfloat16* out;  // [B, max_nodes, Hq, D]: written here when a request has one split
};

__global__ void __launch_bounds__(THREADS, 1) attn_umma_kernel(const UmmaParams prm) {
  extern __shared__ uint8_t smem_raw[];
  const AttnArgs& a = prm.a;
  const int split = blockIdx.x, mt = blockIdx.y;
  const int b = blockIdx.z / a.hkv, h = blockIdx.z % a.hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();  // the prep kernel's rotated queries, cache appends and flags

  // ---- the CTA's work (uniform) --------------------------------------------------------
  const int valid = a.valid[b], T = a.num_nodes[b], P = a.prefix_len[b];
  if (!valid) return;
  const int rows = T * a.group;
  const int row0 = mt * 128;
  if (row0 >= rows) return;
  const int keys = P + T;
  const int kload = (keys + 15) & ~15;  // cache rows past the tree up to here are zeros
  const int n_tiles = (keys + KEYS - 1) / KEYS;
  const int t0 = split * a.tiles_per_split;
  const int t1 = min(n_tiles, t0 + a.tiles_per_split);
  if (t0 >= t1) return;
  const int n = t1 - t0;
  // this CTA covers every key of its rows: it writes the final output itself
  const bool single = n_tiles <= a.tiles_per_split;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + SMEM_BAR;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + SMEM_BAR + 8 * NUM_BARS);
  volatile uint32_t* abort = tmem_slot + 1;

  // softmax warps: this row's rotated query (256 bytes), zeros past the tree
  uint4 qreg[16];
  if (warp < 4) {
    const int r = row0 + warp * 32 + lane;
    const uint4* src = reinterpret_cast<const uint4*>(
        static_cast<const __nv_bfloat16*>(a.q_rot) + (((int64_t)b * a.hkv + h) * a.rows_pad + r) * 128);
#pragma unroll
    for (int i = 0; i < 16; ++i) qreg[i] = r < rows ? src[i] : make_uint4(0u, 0u, 0u, 0u);
  }
  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_Q), 4);  // one arrival per softmax warp (Q rows in TMEM)
    for (int s = 0; s < KST; ++s) {
      mbar_init(bar(BAR_K_FULL + s), LOADERS);
      mbar_init(bar(BAR_K_EMPTY + s), 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(bar(BAR_V_FULL + s), LOADERS);
      mbar_init(bar(BAR_V_EMPTY + s), 1);
    }
    mbar_init(bar(BAR_S_FULL + 0), 1);
    mbar_init(bar(BAR_S_FULL + 1), 1);
    mbar_init(bar(BAR_PV_DONE + 0), 1);
    mbar_init(bar(BAR_PV_DONE + 1), 1);
    mbar_init(bar(BAR_O_DONE), 1);
    mbar_init(bar(BAR_DRAIN), 1);
    // step j uses GO[j % 2]: the softmax can finish P_{j+1} before the MMA warp has seen
    // GO phase j complete
    mbar_init(bar(BAR_GO + 0), 4);  // the four softmax warps
    mbar_init(bar(BAR_GO + 1), 4);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == MMA_WARP) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= LOAD_WARP0 && warp < MMA_WARP) {
    // ---- loaders ---------------------------------------------------------------------
    const int lt = threadIdx.x - LOAD_WARP0 * 32;
    const char* kcache = static_cast<const char*>(a.k_cache);
    const char* vcache = static_cast<const char*>(a.v_cache);
    // tiles copied but not yet signalled, oldest first (FULL barrier addresses)
    uint32_t pend0 = 0, pend1 = 0;
    int npend = 0;
    auto signal_all = [&]() {
      cp_wait<0>();
      fence_to_async();
      if (npend > 0) mbar_arrive(pend0);
      if (npend > 1) mbar_arrive(pend1);
      npend = 0;
    };
    // one K or V tile j (of this CTA's range) into ring slot dst; full = its FULL barrier.
    // Thread lt copies 16-byte chunk c16 of rows rr + 4 i (i < 32): its global addresses
    // step by 1 KB and its shared ones by 512 bytes, and row (rr + 4 i) & 7 takes two
    // values, so every copy is one instruction with constant offsets.
    const int rr = lt >> 4, c16 = lt & 15;
    const uint32_t sw_even = (uint32_t)((c16 & 7) ^ (rr & 7)) << 4;
    const uint32_t sw_odd = (uint32_t)((c16 & 7) ^ ((rr + 4) & 7)) << 4;
    const uint32_t dlane = (uint32_t)(c16 >> 3) * HALF + (uint32_t)rr * 128u;
    auto copy_tile = [&](const char* cache, uint32_t dst, uint32_t full, int j) {
      const int k0 = (t0 + j) * KEYS;
      int64_t rb0, rb1;  // cache rows of keys k0 and k0 + 64
      if (a.layout == TSV_KV_CONTIGUOUS) {
        rb0 = ((int64_t)b * a.hkv + h) * a.capacity + k0;
        rb1 = rb0 + 64;
      } else {
        const int32_t* bt = a.block_table + (int64_t)b * a.max_blocks;
        const int blk0 = k0 < kload ? bt[k0 / TSV_KV_BLOCK] : 0;
        const int blk1 = k0 + 64 < kload ? bt[(k0 + 64) / TSV_KV_BLOCK] : 0;
        rb0 = ((int64_t)blk0 * a.hkv + h) * TSV_KV_BLOCK;
        rb1 = ((int64_t)blk1 * a.hkv + h) * TSV_KV_BLOCK;
      }
      const char* s0 = cache + (rb0 + rr) * 256 + c16 * 16;  // rows rr + 4 i, i < 16
      const char* s1 = cache + (rb1 + rr) * 256 + c16 * 16;  // rows 64 + rr + 4 i
      const uint32_t d0 = dst + dlane;
      const int lim = kload - k0 - rr;  // row rr + 4 i holds data when 4 i < lim
      if (lim >= 128) {  // every row of the tile
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t sw = (i & 1) ? sw_odd : sw_even;
          cp_async16(d0 + 512u * i + sw, s0 + 1024 * i, true);
          cp_async16(d0 + 8192u + 512u * i + sw, s1 + 1024 * i, true);
        }
      } else {  // the tile that ends the tree: rows past it are zero-filled, never read
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t sw = (i & 1) ? sw_odd : sw_even;
          const bool in0 = 4 * i < lim, in1 = 64 + 4 * i < lim;
          cp_async16(d0 + 512u * i + sw, in0 ? s0 + 1024 * i : cache, in0);
          cp_async16(d0 + 8192u + 512u * i + sw, in1 ? s1 + 1024 * i : cache, in1);
        }
      }
      cp_commit();
      if (npend == 2) {  // three tiles in flight: the oldest has landed
        cp_wait<2>();
        fence_to_async();
        mbar_arrive(pend0);
        pend0 = pend1;
        pend1 = full;
      } else if (npend == 1) {
        pend1 = full;
        npend = 2;
      } else {
        pend0 = full;
        npend = 1;
      }
    };
    // a ring slot is free once the MMAs that read its previous tile have completed
    auto slot_free = [&](uint32_t empty, uint32_t parity) {
      if (mbar_test(empty, parity)) return true;
      signal_all();  // never block while holding tiles the MMA warp may be waiting for
      // the ring's slack absorbs the wake-up latency: poll with short sleeps, leaving
      // the issue slots to the softmax warps sharing this sub-partition
      return mbar_wait(empty, parity, abort, false);
    };
    bool ok = true;
    for (int j = 0; ok && j <= n + 1; ++j) {  // K_j, then V_{j-2}
      if (j < n) {
        const int st = j % KST;
        if (j >= KST && !(ok = slot_free(bar(BAR_K_EMPTY + st), ((j / KST) - 1) & 1))) break;
        copy_tile(kcache, base + SMEM_K + st * TILE, bar(BAR_K_FULL + st), j);
      }
      if (j >= 2 && j - 2 < n) {
        const int jv = j - 2, st = jv % VST;
        if (jv >= VST && !(ok = slot_free(bar(BAR_V_EMPTY + st), ((jv / VST) - 1) & 1))) break;
        copy_tile(vcache, base + SMEM_V + st * TILE, bar(BAR_V_FULL + st), jv);
      }
    }
    signal_all();  // every copy this thread started has landed before the CTA can exit
  } else if (warp == MMA_WARP) {
    // ---- MMA issuer: the whole warp walks the loop with warp-uniform descriptors; one
    // elected lane issues each instruction
    constexpr uint32_t ID_QK = idesc(0), ID_PV = idesc(1);
    constexpr uint32_t TILE_D = TILE >> 4;  // descriptor address units are 16 bytes
    const uint64_t dk = sdesc(base + SMEM_K, 16, 1024);
    const uint64_t dv = sdesc(base + SMEM_V, HALF, 1024);
    // k-step ks of a K-major operand: 16 columns = 32 bytes inside a 64-column panel
    auto kmaj = [](int ks) -> uint64_t { return (uint64_t)((ks >> 2) * (HALF >> 4) + (ks & 3) * 2); };
    // S_j = Q K_j^T into S buffer j % 2; A = Q in TMEM (8 columns = 16 bf16 per k-step).
    // The buffer held P_{j-2}: the caller has seen P_{j-2} V_{j-2} complete.
    auto qk = [&](int j) {
      const uint64_t kd = dk + (uint64_t)((j % KST) * TILE_D);
      const uint32_t sd = tmem + TMEM_S + (j & 1) * 128;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        if (elect_one()) mma_ts(sd, tmem + TMEM_Q + ks * 8, kd + kmaj(ks), ID_QK, ks > 0);
      if (elect_one()) {
        mma_commit(bar(BAR_S_FULL + (j & 1)));
        mma_commit(bar(BAR_K_EMPTY + j % KST));
      }
      __syncwarp();
    };
    // O += P_j V_j over ksteps of 16 keys (V rows 16 ks .. 16 ks + 15: MN-major, 16
    // rows of 128 bytes per k-step)
    auto pv = [&](int j, int ksteps) {
      const uint64_t vd = dv + (uint64_t)((j % VST) * TILE_D);
      const uint32_t pa = tmem + TMEM_S + (j & 1) * 128;  // P_j over S_j's buffer
      const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        if (ks < ksteps && elect_one())
          mma_ts(tmem + TMEM_O, pa + ks * 8, vd + (uint64_t)(ks * 128), ID_PV, ks > 0 ? 1u : acc0);
      if (elect_one()) {
        mma_commit(bar(BAR_V_EMPTY + j % VST));
        mma_commit(bar(BAR_PV_DONE + (j & 1)));
      }
      __syncwarp();
    };
    bool ok = warp_wait(bar(BAR_Q), 0, abort) && warp_wait(bar(BAR_K_FULL), 0, abort, true);
    if (ok) {
      tc_fence_after();
      qk(0);
      if (n > 1 && (ok = warp_wait(bar(BAR_K_FULL + 1), 0, abort, true))) {
        tc_fence_after();
        qk(1);
      }
    }
    for (int j = 0; ok && j < n; ++j) {
      // GO phase j: P_j written by the softmax; V_j landed
      if (!(ok = warp_wait(bar(BAR_GO + (j & 1)), (j >> 1) & 1, abort, true))) break;
      if (!(ok = warp_wait(bar(BAR_V_FULL + j % VST), (j / VST) & 1, abort, true))) break;
      tc_fence_after();
      pv(j, (min(KEYS, keys - (t0 + j) * KEYS) + 15) >> 4);
      if (j + 2 < n) {
        // S_{j+2} goes into the buffer that holds P_j, and MMAs into different
        // accumulators are not ordered: P_j V_j has finished reading P_j first
        if (!(ok = warp_wait(bar(BAR_PV_DONE + (j & 1)), (j >> 1) & 1, abort, true))) break;
        if (!(ok = warp_wait(bar(BAR_K_FULL + (j + 2) % KST), ((j + 2) / KST) & 1, abort, true)))
          break;
        tc_fence_after();
        qk(j + 2);
      }
    }
    const bool issuer = lane == 0;
    if (issuer) {
      if (ok) mma_commit(bar(BAR_O_DONE));
      // drain: every MMA issued above has finished before TMEM is released
      mma_commit(bar(BAR_DRAIN));
      mbar_wait(bar(BAR_DRAIN), 0, nullptr);
    }
    __syncwarp();
  } else {
    // ---- softmax warpgroup -----------------------------------------------------------
    const int r = row0 + warp * 32 + lane;
    const bool live = r < rows;
    const int node = r / a.group;
    // rows past the tree read node 0's mask (their results are never stored)
    const uint32_t* mrow = a.mask + ((int64_t)b * a.max_nodes + (live ? node : 0)) * a.mask_words;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t o_addr = tmem + lane_base + TMEM_O;
    const float sl2 = prm.scale_log2;
    {
      // this row's rotated query (bf16 pairs, low half first) -> TMEM columns of Q
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 x = qreg[4 * c + i];
          w[4 * i] = x.x; w[4 * i + 1] = x.y; w[4 * i + 2] = x.z; w[4 * i + 3] = x.w;
        }
        tmem_st16(tmem + lane_base + TMEM_Q + 16 * c, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_Q));
    }
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      // S_j, and then P_j over its first 64 columns, in S buffer j % 2
      const uint32_t s_addr = tmem + lane_base + TMEM_S + (j & 1) * 128;
      if (!(ok = warp_wait(bar(BAR_S_FULL + (j & 1)), (j >> 1) & 1, abort, true))) break;
      tc_fence_after();
      const int k0 = (t0 + j) * KEYS;
      float v[128];
      tmem_ld128(s_addr, v);
      if (k0 + KEYS > P) {  // tile holds tree keys (or keys past the end): mask to -inf
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t vis = visible32(k0 + 32 * c, P, T, mrow, a.mask_words);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[32 * c + i] = ((vis >> i) & 1u) ? v[32 * c + i] : -INFINITY;
        }
      }
      // row max with 8 independent chains
      float m8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = v[i];
#pragma unroll
      for (int i = 8; i < 128; ++i) m8[i & 7] = fmaxf(m8[i & 7], v[i]);
      const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      const float mxs = mx * sl2;
      const bool need = mxs > m_used + RESCALE_LOG2;  // also true on the first visible tile
      const float factor = need ? ex2(m_used - mxs) : 1.f;
      if (need) m_used = mxs;
      // a row with nothing visible so far has only -inf scores: any finite offset works
      const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
      float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t pk[4][16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c0 = q * 32 + 2 * i;
          const float p0 = ex2(fmaf(v[c0], sl2, neg_m));
          const float p1 = ex2(fmaf(v[c0 + 1], sl2, neg_m));
          l8[(2 * i) & 7] += p0;
          l8[(2 * i + 1) & 7] += p1;
          __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
          pk[q][i] = *reinterpret_cast<uint32_t*>(&b2);
        }
      }
      l = l * factor + (((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7])));
      if (__any_sync(FULL, need) && j > 0) {
        // O must be quiescent: P_{j-1} V_{j-1} (and with it every earlier MMA) finished
        // (the next completion on that barrier, P_{j+1} V_{j+1}, needs P_{j+1}, so the
        // parity is unambiguous)
        if (!(ok = warp_wait(bar(BAR_PV_DONE + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort, true)))
          break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32(o_addr + 32 * c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= factor;
          tmem_st32(o_addr + 32 * c, o);
        }
      }
      // P_j over S_j (already in registers); this warp's share of GO phase j
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_st16(s_addr + 16 * q, pk[q]);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_GO + (j & 1)));
    }
    // epilogue: the CTA's share of the key loop is done; the stream's next kernel may be
    // scheduled (it waits for this grid to complete before touching memory)
    griddep_launch();
    if (ok) ok = warp_wait(bar(BAR_O_DONE), 0, abort);
    tc_fence_after();
    if (single) {
      // normalised bf16 output: out[b, node, h * G + g, :]
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* dst = prm.out + (((int64_t)b * a.max_nodes + node) * a.hq + h * a.group +
                                      r % a.group) * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[32];
        tmem_ld32(o_addr + 32 * c, o);
        if (live && ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn(o[8 * i + 2 * e] * inv, o[8 * i + 2 * e + 1] * inv);
              w[e] = *reinterpret_cast<uint32_t*>(&b2);
            }
            d4[i] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    } else {
      const int64_t prow = (((int64_t)b * a.hkv + h) * a.nsplit + split) * a.rows_pad + r;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[32];
        tmem_ld32(o_addr + 32 * c, o);
        if (live && ok) {
          float4* dst = reinterpret_cast<float4*>(a.o_part + prow * 128 + 32 * c);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
      }
      if (live && ok) {
        a.ml[prow * 2 + 0] = m_used;
        a.ml[prow * 2 + 1] = l;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort && threadIdx.x == 0 && a.err) a.err[b] = TSV_REQ_TIMEOUT;
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

bool umma_supported(const AttnPlan& p) {
  return p.dtype == TSV_DTYPE_BF16 && p.head_dim == 128 && device_cc() >= 100;
}

int launch_attn_umma(const AttnPlan& p, const AttnArgs& a, float scale_log2, void* out,
                     cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return TSV_ERR_UNSUPPORTED;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(attn_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return launch_status();
    attr_set[dev] = true;
  }
  UmmaParams prm{a, scale_log2, static_cast<__nv_bfloat16*>(out)};
  dim3 grid(p.nsplit, (unsigned)ceil_div(p.rows, 128), p.batch * p.hkv);  // M tiles of 128 rows
  const int st = launch_pdl(attn_umma_kernel, grid, dim3(THREADS), SMEM_BYTES, stream, prm);
  if (st != TSV_OK || p.nsplit == 1) return st;
  return launch_split_merge(p, a, out, stream);
}

}  // namespace tsv
