// Tree-verification attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA),
// bf16 in, fp32 accumulate, head_dim 128.
//
// NOT DISPATCHED: tree_verify_attn runs attn_mma.cu. With one 128-row M tile per KV head
// and every K/V byte streamed from HBM (B = 64, P = 1024, 9-node trees) right after a
// large write, about one call in a hundred ended in an unspecified launch failure, one
// CTA stopping in the middle of its key loop with K/V copies in flight; the cause is
// not known, so this kernel is kept for reference only.
//
// Pages: "推理系统手册 · 投机解码进阶：树形草稿与 EAGLE", section 实现 (forward_with_mask:
// each node attends to the whole prefix and, among the tree nodes, to its ancestors and
// itself; GQA heads share a KV head) and "TensorRT-LLM 源码完全拆解(二十二)", section
// CUDA Graph 里的掩码重排 (the Blackwell attention reads the padded bit mask directly).
//
// One CTA = (request b, KV head h, one M tile of 128 query rows, split of the keys). The
// query rows of a KV head are every (node, query head of the group) pair, so each K/V
// tile serves all of them (a second M tile of the same head reads it again, mostly
// from L2).
//
//   warp 4      TMA producer: K/V tiles of 128 keys (64-key boxes, 128-byte swizzle)
//               into a 3-stage K ring and a 4-stage V ring; K runs two tiles ahead of V
//   warp 5      TMEM allocator + MMA issuer (warp-uniform descriptors, one elected lane
//               per instruction). After S_0 and S_1, step j (j = 0 .. n - 1) issues
//                 O     += P_j V_j          A = P_j in TMEM, B = V (shared, MN-major)
//                 S_{j+2} = Q K_{j+2}^T     A = Q in TMEM, B = K (shared, K-major)
//               once the softmax has written P_j. S is double-buffered and P_j is
//               written over the first half of S_j's buffer, so the softmax always finds
//               the next S computed while it works on the current tile. Only MMAs into
//               the same accumulator are guaranteed to execute in issue order: S_{j+2}
//               (accumulator S) may otherwise overlap P_j V_j (accumulator O) and write
//               over P_j while it is being read, so the warp waits for P_j V_j's
//               completion before it issues S_{j+2} (hidden: S_{j+2} is needed a whole
//               tile later). Q and P come from TMEM: the shared-memory port carries only
//               the K and V tiles.
//   warp 6      relay: arrives on GO for step j once V_j and K_{j+2} have landed (a step
//               ahead of the softmax: GO alternates between two barriers by step
//               parity); the four softmax warps arrive on it once P_j is written. The
//               MMA warp tests that one barrier per step, between steps: a test's round
//               trip behind the shared-memory operand traffic (a few hundred cycles)
//               stalls the warp's issue, so none sits between the MMAs of a step.
//   warps 0-3   softmax warpgroup; thread = query row = TMEM lane. Each thread first
//               copies its rotated query row into TMEM. Per tile: one x128 TMEM load of
//               S_j, the row max over 8 chains, P = exp2(s * scale * log2e - m) rounded to
//               bf16 and stored over S_j. The running max m is raised only when a tile's
//               max exceeds it by more than 8 (log2 units), and O in TMEM is rescaled
//               then (after P_{j-1} V_{j-1} has finished), otherwise never.
// TMEM (512 columns allocated): S/P[0] [0,128) S/P[1] [128,256) O [256,384) Q [384,448).
// A CTA that covers every key of its rows writes the normalised bf16 output itself;
// otherwise it writes its unnormalised O rows plus (m, l), and the merge kernel (one warp
// per query row, launched after this grid) combines the splits with their log-sum-exp
// weights. (Merging inside the last split to finish cost more: one SM then reads every
// partial of its 128 rows while the rest of the GPU idles.)
//
// The ancestor bitmask is applied from a 32-bit visibility word per 32-key chunk,
// funnel-shifted out of the row's node mask (read only on tiles that hold tree keys).
//
// Every mbarrier wait is bounded; on a timeout the CTA records TSV_REQ_TIMEOUT for the
// request, stops issuing work, drains its MMAs and copies and frees its TMEM.
#include <cuda.h>

#include "attn_common.cuh"
#include "common.cuh"

namespace tsv {
namespace {

#include "tc_ptx.cuh"

constexpr int KEYS = 128;                 // keys per tile
constexpr int KST = 3, VST = 4;           // K and V ring depths (V tiles live two steps longer)
constexpr int THREADS = 224;
constexpr int TMA_WARP = 4, MMA_WARP = 5, RELAY_WARP = 6;
constexpr uint32_t HALF = 128 * 128;      // 128 rows x 64 bf16 (one 128-byte-swizzled panel)
constexpr uint32_t TILE = 2 * HALF;       // 128 rows x 128 bf16
constexpr uint32_t BOX64 = 64 * 128;      // one 64-row TMA box of a panel
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

// barrier slots (8 bytes each) after SMEM_BAR
constexpr int BAR_Q = 0, BAR_K_FULL = 1, BAR_K_EMPTY = BAR_K_FULL + KST,
              BAR_V_FULL = BAR_K_EMPTY + KST, BAR_V_EMPTY = BAR_V_FULL + VST,
              BAR_S_FULL = BAR_V_EMPTY + VST, BAR_PV_DONE = BAR_S_FULL + 2,
              BAR_O_DONE = BAR_PV_DONE + 2,
              BAR_DRAIN = BAR_O_DONE + 1, BAR_GO = BAR_DRAIN + 1, NUM_BARS = BAR_GO + 2;
static_assert(8 * NUM_BARS + 12 <= 256, "barrier area");
static_assert(SMEM_BYTES <= 232448, "shared memory per block");

struct TcParams {
  AttnArgs a;
  float scale_log2;
  __nv_bfloat16* out;  // [B, max_nodes, Hq, D]: written here when a request has one split
};


__global__ void __launch_bounds__(THREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const TcParams prm) {
  extern __shared__ uint8_t smem_raw[];
  const AttnArgs& a = prm.a;
  const int split = blockIdx.x, mt = blockIdx.y;
  const int b = blockIdx.z / a.hkv, h = blockIdx.z % a.hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();  // the prep kernel's rotated queries, cache appends and flags

  // ---- the CTA's work (uniform; the three loads in one round trip) -------------------
  const int valid = a.valid[b], T = a.num_nodes[b], P = a.prefix_len[b];
  if (!valid) return;
  const int rows = T * a.group;
  const int row0 = mt * 128;
  if (row0 >= rows) return;
  const int keys = P + T;
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

  // The producer warp initialises the barriers and starts loading at once; the other
  // warps meet at a named barrier (after the TMEM allocation, with the softmax warps'
  // query rows already on their way into registers) that the producer only arrives at.
  uint4 qreg[16];  // softmax warps: this row's rotated query (256 bytes)
  if (warp < 4) {
    const uint4* src = reinterpret_cast<const uint4*>(
        static_cast<const __nv_bfloat16*>(a.q_rot) +
        (((int64_t)b * a.hkv + h) * a.rows_pad + row0 + warp * 32 + lane) * 128);
#pragma unroll
    for (int i = 0; i < 16; ++i) qreg[i] = src[i];
  }
  if (threadIdx.x == TMA_WARP * 32) {
    mbar_init(bar(BAR_Q), 4);  // one arrival per softmax warp (Q rows in TMEM)
    for (int s = 0; s < KST; ++s) {
      mbar_init(bar(BAR_K_FULL + s), 1);
      mbar_init(bar(BAR_K_EMPTY + s), 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(bar(BAR_V_FULL + s), 1);
      mbar_init(bar(BAR_V_EMPTY + s), 1);
    }
    mbar_init(bar(BAR_S_FULL + 0), 1);
    mbar_init(bar(BAR_S_FULL + 1), 1);
    mbar_init(bar(BAR_PV_DONE + 0), 1);
    mbar_init(bar(BAR_PV_DONE + 1), 1);
    mbar_init(bar(BAR_O_DONE), 1);
    mbar_init(bar(BAR_DRAIN), 1);
    // step j uses GO[j % 2]: the last step needs no MMA work after step n - 1, so with
    // one barrier its phase could complete before the MMA warp has seen step n - 1's
    mbar_init(bar(BAR_GO + 0), 5);  // four softmax warps + the relay
    mbar_init(bar(BAR_GO + 1), 5);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  uint32_t tmem = 0;  // the producer does not use TMEM
  if (warp == TMA_WARP) {
    __syncwarp();
    asm volatile("bar.arrive 1, %0;" ::"n"(THREADS) : "memory");
  } else {
    if (warp == MMA_WARP) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory");
    tc_fence_after();
    tmem = *tmem_slot;
  }

  if (warp == TMA_WARP) {
    // ---- producer: the whole warp walks the loop, lane 0 issues. K runs two tiles ahead
    // of V (order K0 K1 K2 V0 K3 V1 ...), as Q K^T does ahead of P V.
    // Paged caches: the block ids of 32 consecutive 64-key boxes sit in the lanes'
    // registers (one load round trip per 16 tiles instead of one per box).
    const int box0 = t0 * (KEYS / TSV_KV_BLOCK);
    int win = -1;  // first box of the loaded window
    int blk_reg = 0;
    auto row_of = [&](int key) -> int {  // warp-uniform call
      if (a.layout == TSV_KV_CONTIGUOUS) return (int)(((int64_t)b * a.hkv + h) * a.capacity + key);
      const int box = key / TSV_KV_BLOCK;
      const int w = box0 + ((box - box0) & ~31);
      if (w != win) {
        win = w;
        const int nb = (keys + TSV_KV_BLOCK - 1) / TSV_KV_BLOCK;
        blk_reg = w + lane < nb ? a.block_table[(int64_t)b * a.max_blocks + w + lane] : 0;
      }
      const int blk = __shfl_sync(FULL, blk_reg, box - win);
      return (blk * a.hkv + h) * TSV_KV_BLOCK;
    };
    // one K or V tile: 1 or 2 boxes of 64 keys (a box past the last key is not loaded)
    auto load = [&](const CUtensorMap* map, uint32_t dst, uint32_t full, int j) {
      const int k0 = (t0 + j) * KEYS;
      const int chunks = (k0 + 64 < keys) ? 2 : 1;
      int row[2];
      for (int c = 0; c < 2; ++c) row[c] = c < chunks ? row_of(k0 + 64 * c) : 0;
      if (lane != 0) return;
      mbar_expect_tx(full, chunks * 2 * BOX64);
      for (int c = 0; c < chunks; ++c)
        for (int hf = 0; hf < 2; ++hf)
          tma_load_2d(dst + hf * HALF + c * BOX64, map, hf * 64, row[c], full);
    };
    int issued_k = 0, issued_v = 0;
    bool ok = true;
    for (int j = 0; ok && j <= n + 1; ++j) {
      if (j < n) {
        const int st = j % KST;
        if (j >= KST && !(ok = warp_wait(bar(BAR_K_EMPTY + st), ((j / KST) - 1) & 1, abort, true)))
          break;
        load(&tm_k, base + SMEM_K + st * TILE, bar(BAR_K_FULL + st), j);
        issued_k = j + 1;
      }
      if (j >= 2 && j - 2 < n) {
        const int jv = j - 2, st = jv % VST;
        if (jv >= VST && !(ok = warp_wait(bar(BAR_V_EMPTY + st), ((jv / VST) - 1) & 1, abort, true)))
          break;
        load(&tm_v, base + SMEM_V + st * TILE, bar(BAR_V_FULL + st), jv);
        issued_v = jv + 1;
      }
    }
    // Before the CTA can exit, every copy it started has landed (immediate unless a
    // wait above gave up).
    if (lane == 0) {
      for (int j = issued_k > KST ? issued_k - KST : 0; j < issued_k; ++j)
        mbar_wait(bar(BAR_K_FULL + j % KST), (j / KST) & 1, nullptr);
      for (int j = issued_v > VST ? issued_v - VST : 0; j < issued_v; ++j)
        mbar_wait(bar(BAR_V_FULL + j % VST), (j / VST) & 1, nullptr);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ---- MMA issuer: the whole warp walks the loop with warp-uniform descriptors; one
    // elected lane issues each instruction (a lane-0 branch that builds descriptors per
    // MMA was measured to issue about 30% slower than the tensor pipe drains).
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
    // rows of 128 bytes per k-step). (Testing the next step's barrier between these
    // MMAs was measured to slow their issue: its shared-memory round trip stalls the
    // warp.)
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
    // S_0 and S_1 first; then step j issues P_j V_j and S_{j+2} = Q K_{j+2}^T, so the
    // softmax always finds the next S computed while it works on the current one
    bool ok = warp_wait(bar(BAR_Q), 0, abort) && warp_wait(bar(BAR_K_FULL), 0, abort);
    if (ok) {
      tc_fence_after();
      qk(0);
      if (n > 1 && (ok = warp_wait(bar(BAR_K_FULL + 1), 0, abort, true))) {
        tc_fence_after();
        qk(1);
      }
    }
    for (int j = 0; ok && j < n; ++j) {
      // GO phase j: P_j written by the softmax, V_j and K_{j+2} landed
      if (!(ok = warp_wait(bar(BAR_GO + (j & 1)), (j >> 1) & 1, abort, true))) break;
      tc_fence_after();
      pv(j, (min(KEYS, keys - (t0 + j) * KEYS) + 15) >> 4);
      if (j + 2 < n) {
        // S_{j+2} goes into the buffer that holds P_j, and MMAs into different
        // accumulators are not ordered: P_j V_j has finished reading P_j first
        if (!(ok = warp_wait(bar(BAR_PV_DONE + (j & 1)), (j >> 1) & 1, abort, true))) break;
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
  } else if (warp == RELAY_WARP) {
    // ---- relay: its share of GO phase j once V_j and K_{j+2} have landed. GO is
    // double-buffered by step parity, so the relay only waits for phase j - 2 (the last
    // one on the same barrier) to have completed before arriving: it runs a step ahead
    // of the softmax instead of after it.
    bool ok = true;
    for (int j = 0; ok && j < n; ++j) {
      if (j >= 2 && !(ok = warp_wait(bar(BAR_GO + (j & 1)), ((j - 2) >> 1) & 1, abort, true))) break;
      if (j + 2 < n &&
          !(ok = warp_wait(bar(BAR_K_FULL + (j + 2) % KST), ((j + 2) / KST) & 1, abort, true)))
        break;
      if (!(ok = warp_wait(bar(BAR_V_FULL + j % VST), (j / VST) & 1, abort, true))) break;
      if (lane == 0) mbar_arrive(bar(BAR_GO + (j & 1)));
      __syncwarp();
    }
  } else if (warp < 4) {
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
      // this row's rotated query (bf16 pairs, low half first, loaded before the setup
      // barrier) -> TMEM columns of Q; rows past the tree copy whatever the workspace
      // holds (their results are never stored)
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

// ---- split merge: one warp per query row -------------------------------------------
// Combines the key splits of the rows whose request took more than one split: lane s
// holds split s's (m, l) (m in log2 units), the warp forms the log-sum-exp weights
// w_s = 2^(m_s - M) / L, and lane c accumulates output columns 4c .. 4c + 3 over the splits
// (eight partial loads in flight), written as bf16. Rows of a single-split request were
// written by the attention kernel itself; rows past the tree were zeroed by the prep.
constexpr int MERGE_ROWS = 8;  // warps (query rows) per CTA

__global__ void __launch_bounds__(MERGE_ROWS * 32)
tc_merge_kernel(const AttnArgs a, __nv_bfloat16* __restrict__ out) {
  griddep_wait();
  griddep_launch();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = blockIdx.x * MERGE_ROWS + warp;
  const int b = blockIdx.y / a.hkv, h = blockIdx.y % a.hkv;
  if (!a.valid[b]) return;
  const int T = a.num_nodes[b], P = a.prefix_len[b];
  if (r >= T * a.group) return;
  const int n_tiles = (P + T + 127) / 128;
  const int nsp = (n_tiles + a.tiles_per_split - 1) / a.tiles_per_split;
  if (nsp <= 1) return;
  const int64_t pbase = ((int64_t)b * a.hkv + h) * a.nsplit;
  float2 ml = make_float2(-INFINITY, 0.f);
  if (lane < nsp) ml = reinterpret_cast<const float2*>(a.ml)[(pbase + lane) * a.rows_pad + r];
  float M = ml.x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, o));
  float e = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
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

bool tc_supported(const AttnPlan& p) {
  return p.dtype == TSV_DTYPE_BF16 && p.head_dim == 128 && device_cc() >= 100 &&
         encode_fn() != nullptr;
}

int launch_attn_tc(const AttnPlan& p, const AttnArgs& a, float scale_log2, void* out,
                   cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return TSV_ERR_UNSUPPORTED;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return launch_status();
    attr_set[dev] = true;
  }
  CUtensorMap mk, mv;
  const uint64_t kv_rows = a.layout == TSV_KV_CONTIGUOUS
                               ? (uint64_t)p.batch * p.hkv * a.capacity
                               : (uint64_t)a.num_blocks * p.hkv * TSV_KV_BLOCK;
  if (!make_map(&mk, a.k_cache, kv_rows, 64) || !make_map(&mv, a.v_cache, kv_rows, 64))
    return TSV_ERR_UNSUPPORTED;
  TcParams prm{a, scale_log2, static_cast<__nv_bfloat16*>(out)};
  dim3 grid(p.nsplit, (unsigned)ceil_div(p.rows, TC_M_GROUP), p.batch * p.hkv);  // M tiles of 128 rows
  const int st = launch_pdl(attn_tc_kernel, grid, dim3(THREADS), SMEM_BYTES, stream, mk, mv, prm);
  if (st != TSV_OK || p.nsplit == 1) return st;
  // the split merge (its warps return at once for rows of single-split requests)
  dim3 gm((unsigned)ceil_div(p.rows, MERGE_ROWS), p.batch * p.hkv);
  return launch_pdl(tc_merge_kernel, gm, dim3(MERGE_ROWS * 32), 0, stream, a,
                    static_cast<__nv_bfloat16*>(out));
}

}  // namespace tsv
