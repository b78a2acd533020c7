// Tree-verification attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA),
// bf16 in, fp32 accumulate, head_dim 128.
//
// Pages: "推理系统手册 · 投机解码进阶：树形草稿与 EAGLE", section 实现 (forward_with_mask:
// each node attends to the whole prefix and, among the tree nodes, to its ancestors and
// itself; GQA heads share a KV head) and "TensorRT-LLM 源码完全拆解(二十二)", section
// CUDA Graph 里的掩码重排 (the Blackwell attention reads the padded bit mask directly).
//
// One CTA = (request b, KV head h, group of 256 query rows, split of the keys). The
// query rows of a KV head are every (node, query head of the group) pair, so the KV
// tiles of the split are read from HBM once for all of them.
//
//   warp 8      TMA producer: Q tiles once, then K/V tiles of 128 keys (64-key boxes,
//               128-byte swizzle) into a 2-stage shared-memory ring
//   warp 9      TMEM allocator + MMA issuer (one elected lane):
//                 S_mt = Q_mt K^T       A, B = shared memory, both K-major
//                 O_mt += P_mt V        A = P in TMEM, B = V in shared memory, MN-major
//   warps 0-7   two softmax warpgroups, one per 128-row M tile; thread = query row =
//               TMEM lane. Pass 1 takes the row max of the masked scores, pass 2 writes
//               P = exp2(s * scale * log2e - m) as bf16 over the S columns. The running
//               max m is only raised when the tile max exceeds it by more than 8 (log2
//               units); O in TMEM is rescaled then, otherwise never.
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512).
// Each CTA writes its unnormalised O rows plus (m, l) to the split workspace; the merge
// kernel (attn.cu) combines the splits with a warp-shuffle log-sum-exp reduction.
//
// The ancestor bitmask is applied from registers: every row keeps its node's mask words
// and builds a 32-bit visibility word per 32-column chunk with a funnel shift.
//
// Every mbarrier wait is bounded; on a timeout the CTA records TSV_REQ_TIMEOUT for the
// request, stops issuing work, drains its MMAs and frees its TMEM.
#include <cuda.h>

#include "attn_common.cuh"
#include "common.cuh"

namespace tsv {
namespace {

constexpr int KEYS = 128;                 // keys per tile
constexpr int STAGES = 2;
constexpr int THREADS = 320;
constexpr int TMA_WARP = 8, MMA_WARP = 9;
constexpr uint32_t HALF = 128 * 128;      // 128 rows x 64 bf16 (one 128-byte-swizzled panel)
constexpr uint32_t TILE = 2 * HALF;       // 128 rows x 128 bf16
constexpr uint32_t BOX64 = 64 * 128;      // one 64-row TMA box of a panel
constexpr uint32_t SMEM_Q = 0;            // 2 M tiles
constexpr uint32_t SMEM_KV = 2 * TILE;    // STAGES x (K tile, V tile)
constexpr uint32_t SMEM_BAR = SMEM_KV + STAGES * 2 * TILE;
constexpr uint32_t SMEM_BYTES = SMEM_BAR + 256 + 1024;  // + alignment slack
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.f;
constexpr uint32_t WAIT_LIMIT = 1u << 22;  // try_wait polls before a wait gives up
constexpr uint64_t WAIT_NS = 1000000000ull;  // and at most one second

// barrier slots (8 bytes each) after SMEM_BAR
constexpr int BAR_Q = 0, BAR_KV_FULL = 1, BAR_KV_EMPTY = BAR_KV_FULL + STAGES,
              BAR_S_FULL = BAR_KV_EMPTY + STAGES, BAR_P_FULL = BAR_S_FULL + 2,
              BAR_O_DONE = BAR_P_FULL + 2, BAR_DRAIN = BAR_O_DONE + 1, NUM_BARS = BAR_DRAIN + 1;

// ---- PTX wrappers ----------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: false when the limit ran out (the CTA then aborts) or, if `abort` is
// given, when another role of the CTA has given up already.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort) {
  const uint64_t t0 = now_ns();
  for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (abort && *abort) return false;
    if ((i & 1023u) == 1023u && now_ns() - t0 > WAIT_NS) break;
  }
  if (abort) *abort = 1;
  return false;
}
// The whole warp waits; every lane gets the same answer.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort) {
  bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 columns of 32 bits; the wait sits in the same asm so no use of the
// registers can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory matrix descriptor: 128-byte swizzle, tcgen05 descriptor version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: D f32, A/B bf16, M = 128, N = 128.
constexpr uint32_t idesc(uint32_t b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major << 16) | ((128u >> 3) << 17) |
         ((128u >> 4) << 24);
}

struct TcParams {
  AttnArgs a;
  float scale_log2;
};

__device__ __forceinline__ uint32_t pick(const uint32_t (&w)[9], int i) {
  uint32_t r = 0;
#pragma unroll
  for (int k = 0; k < 9; ++k) r = (i == k) ? w[k] : r;
  return r;
}

// Visibility of the 32 keys k .. k+31 for a row whose node has mask words mw.
__device__ __forceinline__ uint32_t visible32(int k, int P, int T, const uint32_t (&mw)[9]) {
  if (k + 32 <= P) return 0xffffffffu;
  const int t = k - P;  // tree index of column 0
  uint32_t pre = 0;
  if (t < 0) pre = (1u << (-t)) - 1u;  // -t in [1, 31]
  uint32_t tr = 0;
  const int ts = t < 0 ? 0 : t;
  if (ts < T) {
    const int idx = ts >> 5, off = ts & 31;
    uint32_t bits = __funnelshift_r(pick(mw, idx), pick(mw, idx + 1), off);
    if (T - ts < 32) bits &= (1u << (T - ts)) - 1u;
    tr = bits << (ts - t);
  }
  return pre | tr;
}

__global__ void __launch_bounds__(THREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const TcParams prm) {
  extern __shared__ uint8_t smem_raw[];
  const AttnArgs& a = prm.a;
  const int split = blockIdx.x, mg = blockIdx.y;
  const int b = blockIdx.z / a.hkv, h = blockIdx.z % a.hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- the CTA's work (uniform) ------------------------------------------------------
  if (!a.valid[b]) return;
  const int T = a.num_nodes[b], P = a.prefix_len[b];
  const int rows = T * a.group;
  const int row0 = mg * 256;
  if (row0 >= rows) return;
  const int n_mt = rows - row0 > 128 ? 2 : 1;
  const int keys = P + T;
  const int n_tiles = (keys + KEYS - 1) / KEYS;
  const int t0 = split * a.tiles_per_split;
  const int t1 = min(n_tiles, t0 + a.tiles_per_split);
  if (t0 >= t1) return;
  const int n = t1 - t0;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + SMEM_BAR;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + SMEM_BAR + 8 * NUM_BARS);
  volatile uint32_t* abort = tmem_slot + 1;

  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_Q), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(BAR_KV_FULL + s), 1);
      mbar_init(bar(BAR_KV_EMPTY + s), 1);
    }
    for (int m = 0; m < 2; ++m) {
      mbar_init(bar(BAR_S_FULL + m), 1);
      mbar_init(bar(BAR_P_FULL + m), 128);
    }
    mbar_init(bar(BAR_O_DONE), 1);
    mbar_init(bar(BAR_DRAIN), 1);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == MMA_WARP) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == TMA_WARP) {
    // ---- producer: the whole warp walks the loop, lane 0 issues ----------------------
    const int qrow = (b * a.hkv + h) * a.rows_pad + row0;
    if (lane == 0) {
      mbar_expect_tx(bar(BAR_Q), n_mt * TILE);
      for (int mt = 0; mt < n_mt; ++mt)
        for (int hf = 0; hf < 2; ++hf)
          tma_load_2d(base + SMEM_Q + mt * TILE + hf * HALF, &tm_q, hf * 64, qrow + mt * 128,
                      bar(BAR_Q));
    }
    int issued = 0;
    for (int j = 0; j < n; ++j) {
      const int st = j % STAGES;
      if (j >= STAGES && !warp_wait(bar(BAR_KV_EMPTY + st), ((j / STAGES) - 1) & 1, abort)) break;
      if (lane == 0) {
        const int k0 = (t0 + j) * KEYS;
        const int chunks = (k0 + 64 < keys) ? 2 : 1;
        mbar_expect_tx(bar(BAR_KV_FULL + st), chunks * 4 * BOX64);
        const uint32_t kdst = base + SMEM_KV + st * 2 * TILE;
        const uint32_t vdst = kdst + TILE;
        for (int c = 0; c < chunks; ++c) {
          const int key = k0 + 64 * c;
          int row;
          if (a.layout == TSV_KV_CONTIGUOUS) {
            row = (int)(((int64_t)b * a.hkv + h) * a.capacity + key);
          } else {
            const int blk = a.block_table[(int64_t)b * a.max_blocks + key / TSV_KV_BLOCK];
            row = (blk * a.hkv + h) * TSV_KV_BLOCK;
          }
          for (int hf = 0; hf < 2; ++hf) {
            tma_load_2d(kdst + hf * HALF + c * BOX64, &tm_k, hf * 64, row, bar(BAR_KV_FULL + st));
            tma_load_2d(vdst + hf * HALF + c * BOX64, &tm_v, hf * 64, row, bar(BAR_KV_FULL + st));
          }
        }
      }
      issued = j + 1;
    }
    // Before the CTA can exit, every copy it started has landed (immediate unless a
    // wait above gave up).
    if (lane == 0) {
      mbar_wait(bar(BAR_Q), 0, nullptr);
      for (int j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j)
        mbar_wait(bar(BAR_KV_FULL + j % STAGES), (j / STAGES) & 1, nullptr);
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ---- MMA issuer: the whole warp walks the loop, lane 0 issues --------------------
    constexpr uint32_t ID_QK = idesc(0), ID_PV = idesc(1);
    const bool issuer = lane == 0;
    auto qk = [&](int mt, int st) {
      if (!issuer) return;
      const uint32_t qa = base + SMEM_Q + mt * TILE;
      const uint32_t ka = base + SMEM_KV + st * 2 * TILE;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks >> 2) * HALF + (ks & 3) * 32;
        mma_ss(tmem + mt * 128, sdesc(qa + off, 16, 1024), sdesc(ka + off, 16, 1024), ID_QK,
               ks > 0);
      }
      mma_commit(bar(BAR_S_FULL + mt));
    };
    auto pv = [&](int mt, int st, int ksteps, bool acc) {
      if (!issuer) return;
      const uint32_t va = base + SMEM_KV + st * 2 * TILE + TILE;
      for (int ks = 0; ks < ksteps; ++ks)
        mma_ts(tmem + 256 + mt * 128, tmem + mt * 128 + ks * 8,
               sdesc(va + ks * 16 * 128, HALF, 1024), ID_PV, (acc || ks > 0) ? 1u : 0u);
    };
    bool ok = warp_wait(bar(BAR_Q), 0, abort) && warp_wait(bar(BAR_KV_FULL), 0, abort);
    if (ok) {
      tc_fence_after();
      for (int mt = 0; mt < n_mt; ++mt) qk(mt, 0);
    }
    for (int j = 0; ok && j < n; ++j) {
      const int st = j % STAGES;
      const int valid = min(KEYS, keys - (t0 + j) * KEYS);
      const int ksteps = (valid + 15) >> 4;
      for (int mt = 0; ok && mt < n_mt; ++mt) {
        if (!(ok = warp_wait(bar(BAR_P_FULL + mt), j & 1, abort))) break;
        tc_fence_after();
        pv(mt, st, ksteps, j > 0);
        if (mt == n_mt - 1 && issuer) mma_commit(bar(BAR_KV_EMPTY + st));
        if (j + 1 < n) {
          const int st2 = (j + 1) % STAGES;
          if (mt == 0) {
            if (!(ok = warp_wait(bar(BAR_KV_FULL + st2), ((j + 1) / STAGES) & 1, abort))) break;
            tc_fence_after();
          }
          qk(mt, st2);
        }
      }
    }
    if (issuer) {
      if (ok) mma_commit(bar(BAR_O_DONE));
      // drain: every MMA issued above has finished before TMEM is released
      mma_commit(bar(BAR_DRAIN));
      mbar_wait(bar(BAR_DRAIN), 0, nullptr);
    }
    __syncwarp();
  } else if (warp / 4 < n_mt) {
    // ---- softmax warpgroups ----------------------------------------------------------
    const int mt = warp / 4, quad = warp & 3;
    const int r = row0 + mt * 128 + quad * 32 + lane;
    const bool live = r < rows;
    const int node = r / a.group;
    uint32_t mw[9];
#pragma unroll
    for (int k = 0; k < 9; ++k) mw[k] = 0;
    if (live) {
      const uint32_t* mrow = a.mask + ((int64_t)b * a.max_nodes + node) * a.mask_words;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < a.mask_words) mw[k] = mrow[k];
    }
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + mt * 128;
    const uint32_t o_addr = tmem + lane_base + 256 + mt * 128;
    const float sl2 = prm.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!(ok = warp_wait(bar(BAR_S_FULL + mt), j & 1, abort))) break;
      tc_fence_after();
      const int k0 = (t0 + j) * KEYS;
      const bool tail = k0 + KEYS > P;
      float v[32];
      // pass 1: row max of the visible scores
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tmem_ld32(s_addr + 32 * c, v);
        const uint32_t vis = tail ? visible32(k0 + 32 * c, P, T, mw) : 0xffffffffu;
#pragma unroll
        for (int i = 0; i < 32; ++i) mx = fmaxf(mx, ((vis >> i) & 1u) ? v[i] : -INFINITY);
      }
      const float mxs = mx * sl2;
      const bool need = mxs > m_used + RESCALE_LOG2;  // also true on the first visible tile
      const float factor = need ? ex2(m_used - mxs) : 1.f;
      if (__any_sync(FULL, need) && j > 0) {
        // O is quiescent: this tile's S was committed after the previous P V finished.
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          tmem_ld32(o_addr + 32 * c, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= factor;
          tmem_st32(o_addr + 32 * c, v);
        }
        tmem_wait_st();
      }
      if (need) {
        l *= factor;
        m_used = mxs;
      }
      // pass 2: P = exp2(s * scale_log2 - m) in bf16 over the first 64 S columns
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tmem_ld32(s_addr + 32 * c, v);
        const uint32_t vis = tail ? visible32(k0 + 32 * c, P, T, mw) : 0xffffffffu;
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float p0 = ((vis >> i) & 1u) ? ex2(fmaf(v[i], sl2, -m_used)) : 0.f;
          const float p1 = ((vis >> (i + 1)) & 1u) ? ex2(fmaf(v[i + 1], sl2, -m_used)) : 0.f;
          l += p0 + p1;
          __nv_bfloat162 pk = __floats2bfloat162_rn(p0, p1);
          packed[i >> 1] = *reinterpret_cast<uint32_t*>(&pk);
        }
        tmem_st16(s_addr + 16 * c, packed);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(BAR_P_FULL + mt));
    }
    // epilogue: unnormalised O row and (m, l) of this split
    if (ok) ok = warp_wait(bar(BAR_O_DONE), 0, abort);
    tc_fence_after();
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

  tc_fence_before();
  __syncthreads();
  if (*abort && threadIdx.x == 0 && a.err) a.err[b] = TSV_REQ_TIMEOUT;
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---- host side -----------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
  }
  return fn;
}

bool make_map(CUtensorMap* m, void* base, uint64_t rows, uint32_t box_rows) {
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {128 * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_supported(const AttnPlan& p) {
  return p.dtype == TSV_DTYPE_BF16 && p.head_dim == 128 && device_cc() >= 100 &&
         encode_fn() != nullptr;
}

int launch_attn_tc(const AttnPlan& p, const AttnArgs& a, float scale_log2, void* out,
                   cudaStream_t stream) {
  (void)out;
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
  CUtensorMap mq, mk, mv;
  const uint64_t kv_rows = a.layout == TSV_KV_CONTIGUOUS
                               ? (uint64_t)p.batch * p.hkv * a.capacity
                               : (uint64_t)a.num_blocks * p.hkv * TSV_KV_BLOCK;
  if (!make_map(&mq, a.q_rot, (uint64_t)p.batch * p.hkv * p.rows_pad, 128) ||
      !make_map(&mk, a.k_cache, kv_rows, 64) || !make_map(&mv, a.v_cache, kv_rows, 64))
    return TSV_ERR_UNSUPPORTED;
  TcParams prm{a, scale_log2};
  dim3 grid(p.nsplit, (unsigned)ceil_div(p.rows, TC_M_GROUP), p.batch * p.hkv);
  attn_tc_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(mq, mk, mv, prm);
  return launch_status();
}

}  // namespace tsv
