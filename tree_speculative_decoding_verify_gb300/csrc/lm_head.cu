// The target model's greedy token at every tree node: argmax over the vocabulary of the
// lm_head logits, with the logits never written to memory.
//
// Pages: "推理系统手册 · 投机解码进阶：树形草稿与 EAGLE", section 实现 (the verifier's forward
// returns lm_head(norm(x)) for every tree node and the walk takes
// pred = logits[node].argmax()); the EAGLE v2 dynamic-tree walkthrough, section 5
// (evaluate_posterior compares each candidate with torch.argmax(logits) at its parent);
// "TensorRT-LLM 源码完全拆解(二十二)", section 验证:在树上走一条路径 (target_predict, the
// target's argmax at every node, is the input of the greedy verification kernel).
//
// logits[m, v] = sum_k hidden[m, k] * weight[v, k]: a GEMM of the node rows (M) against
// the vocabulary (N) over the hidden size (K) on the 5th-generation tensor cores, bf16 in,
// fp32 accumulate in TMEM. One CTA = one M tile of 128 rows x one vocabulary range; the
// ranges are whole 32-entry chunks, as equal as the chunk count allows, so every CTA of a
// wave streams the same number of weight bytes. A range is walked in 256-entry tiles from
// its first entry; its last tile may be narrower (then N = its width rounded up to 32).
//   warp 4      TMA producer: 64-column panels of the row tile (128 x 64) and of the
//               vocabulary tile (256 x 64 in one copy, or 32-row copies for a narrow
//               tile), 128-byte swizzle, into a 4-stage ring
//   warp 5      TMEM allocator + MMA issuer: tcgen05.mma M=128 N<=256 K=16, A and B from
//               shared memory (K-major), four per panel, into one of two TMEM
//               accumulators (256 columns each) so the next tile's MMAs overlap the
//               epilogue of this one
//   warps 0-3   epilogue; thread = row = TMEM lane: x128 TMEM loads, the first maximum
//               of the tile's valid columns, folded into the row's running best as a
//               64-bit key (larger value first, then lower index)
// Each CTA writes its best key per row; a second kernel takes the largest key of every
// row over the vocabulary ranges. Every mbarrier wait is bounded (a timeout marks the
// row keys invalid through the abort path and the CTA drains and frees its TMEM).
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace tsv {
namespace {

#include "tc_ptx.cuh"

constexpr int LM_THREADS = 192;  // warps 0-3 epilogue, 4 producer, 5 MMA
constexpr int LM_TMA_WARP = 4, LM_MMA_WARP = 5;
constexpr int BM = 128, BN = 256, BK = 64;  // rows, vocabulary entries, hidden per panel
constexpr int VCHUNK = 32;                   // granularity of the vocabulary ranges
constexpr int STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 2;  // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;  // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t LM_SMEM_BAR = STAGES * STAGE_BYTES;
constexpr uint32_t LM_SMEM_BYTES = LM_SMEM_BAR + 256 + 1024;  // barriers; alignment slack
constexpr int LB_FULL = 0, LB_EMPTY = STAGES, LB_DFULL = 2 * STAGES, LB_DFREE = LB_DFULL + 2,
              LB_DRAIN = LB_DFREE + 2, LB_NUM = LB_DRAIN + 1;
static_assert(8 * LB_NUM + 8 <= 256, "barrier area");
static_assert(LM_SMEM_BYTES <= 232448, "shared memory per block");

// instruction descriptor: D f32, A and B bf16, both K-major, M = 128, N = n (16 | n <= 256)
__device__ __forceinline__ uint32_t lm_idesc(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}

// Order-preserving 64-bit image of (logit, vocabulary index): larger logit first, then the
// lower index.
__device__ __forceinline__ unsigned long long lm_key(float v, int i) {
  unsigned u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned)(~(unsigned)i);
}

struct LmParams {
  int rows, hidden, vocab, chunks, splits;  // chunks: VCHUNK-entry pieces of the vocabulary
  unsigned long long* keys;  // [splits, rows]
};

__global__ void __launch_bounds__(LM_THREADS, 1)
lm_head_argmax_kernel(const __grid_constant__ CUtensorMap tm_a,
                      const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_b32, const LmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const int mt = blockIdx.x, split = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // split s takes the vocabulary chunks [s * C / S, (s + 1) * C / S) (counts differ by one
  // at most), as BN-entry tiles from its first entry; the last tile may be narrower
  const int r0 = (int)((int64_t)split * p.chunks / p.splits) * VCHUNK;
  const int r1 = min(p.vocab, (int)((int64_t)(split + 1) * p.chunks / p.splits) * VCHUNK);
  const int nt = (r1 - r0 + BN - 1) / BN;
  const int kp = p.hidden / BK;  // panels per vocabulary tile
  griddep_wait();
  if (nt <= 0) return;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + LM_SMEM_BAR;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + LM_SMEM_BAR + 8 * LB_NUM);
  volatile uint32_t* abort = tmem_slot + 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(LB_FULL + s), 1);
      mbar_init(bar(LB_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(LB_DFULL + b), 1);
      mbar_init(bar(LB_DFREE + b), 4);  // one arrival per epilogue warp
    }
    mbar_init(bar(LB_DRAIN), 1);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == LM_MMA_WARP) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == LM_TMA_WARP) {
    // ---- producer: panels in the order the MMAs take them --------------------------
    int issued = 0;
    bool ok = true;
    for (int j = 0; ok && j < nt; ++j) {
      for (int q = 0; q < kp; ++q) {
        const int g = j * kp + q, st = g % STAGES;
        if (g >= STAGES &&
            !(ok = warp_wait(bar(LB_EMPTY + st), ((g / STAGES) - 1) & 1, abort, true)))
          break;
        if (lane == 0) {
          const uint32_t sa = base + st * STAGE_BYTES, sb = sa + A_BYTES;
          const int v0 = r0 + j * BN, w = min(BN, r1 - v0);
          const int pieces = w == BN ? 1 : (w + VCHUNK - 1) / VCHUNK;
          mbar_expect_tx(bar(LB_FULL + st),
                         A_BYTES + (w == BN ? B_BYTES : pieces * (B_BYTES / (BN / VCHUNK))));
          tma_load_2d(sa, &tm_a, q * BK, mt * BM, bar(LB_FULL + st));
          if (w == BN) {
            tma_load_2d(sb, &tm_b, q * BK, v0, bar(LB_FULL + st));
          } else {  // a narrow tile: VCHUNK rows at a time, 4 KB apart in shared memory
            for (int c = 0; c < pieces; ++c)
              tma_load_2d(sb + c * (B_BYTES / (BN / VCHUNK)), &tm_b32, q * BK, v0 + c * VCHUNK,
                          bar(LB_FULL + st));
          }
        }
        __syncwarp();
        issued = g + 1;
      }
    }
    // every copy this CTA started has landed before it may exit
    if (lane == 0)
      for (int g = issued > STAGES ? issued - STAGES : 0; g < issued; ++g)
        mbar_wait(bar(LB_FULL + g % STAGES), (g / STAGES) & 1, nullptr);
    __syncwarp();
  } else if (warp == LM_MMA_WARP) {
    // ---- MMA issuer: warp-uniform descriptors, one elected lane per instruction ------
    const uint64_t da = sdesc(base, 16, 1024);
    constexpr uint32_t STAGE_D = STAGE_BYTES >> 4, A_D = A_BYTES >> 4;  // 16-byte units
    bool ok = true;
    for (int j = 0; ok && j < nt; ++j) {
      const int buf = j & 1;
      // the accumulator's previous tile (j - 2) has been read by the epilogue
      if (j >= 2 && !(ok = warp_wait(bar(LB_DFREE + buf), ((j - 2) >> 1) & 1, abort, true))) break;
      tc_fence_after();
      const uint32_t d = tmem + buf * BN;
      const int w = min(BN, r1 - (r0 + j * BN));
      const uint32_t id = lm_idesc(w == BN ? BN : ((w + VCHUNK - 1) / VCHUNK) * VCHUNK);
      for (int q = 0; ok && q < kp; ++q) {
        const int g = j * kp + q, st = g % STAGES;
        if (!(ok = warp_wait(bar(LB_FULL + st), (g / STAGES) & 1, abort, true))) break;
        tc_fence_after();
        const uint64_t a = da + (uint64_t)(st * STAGE_D), b = a + A_D;
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks)  // 16 columns = 32 bytes per k-step
          if (elect_one()) mma_ss(d, a + ks * 2, b + ks * 2, id, (q > 0 || ks > 0) ? 1u : 0u);
        if (elect_one()) mma_commit(bar(LB_EMPTY + st));
        __syncwarp();
      }
      if (ok && elect_one()) mma_commit(bar(LB_DFULL + buf));
      __syncwarp();
    }
    if (lane == 0) {
      // drain: every MMA issued above has finished before TMEM is released
      mma_commit(bar(LB_DRAIN));
      mbar_wait(bar(LB_DRAIN), 0, nullptr);
    }
    __syncwarp();
  } else {
    // ---- epilogue: thread = row ------------------------------------------------------
    const int r = mt * BM + warp * 32 + lane;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    unsigned long long best = 0ull;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int buf = j & 1;
      if (!(ok = warp_wait(bar(LB_DFULL + buf), (j >> 1) & 1, abort, true))) break;
      tc_fence_after();
      const int v0 = r0 + j * BN;
      const int valid = min(BN, r1 - v0);  // columns past the split's range are stale
      float bv = -INFINITY;
      int bi = v0;
#pragma unroll
      for (int c = 0; c < BN / 128; ++c) {
        if (c * 128 >= valid) break;
        float v[128];
        tmem_ld128(tmem + lane_base + buf * BN + c * 128, v);
        if (valid >= (c + 1) * 128) {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (v[i] > bv) { bv = v[i]; bi = v0 + c * 128 + i; }
        } else {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (c * 128 + i < valid && v[i] > bv) { bv = v[i]; bi = v0 + c * 128 + i; }
        }
      }
      // the accumulator may take the tile after next
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(LB_DFREE + buf));
      if (bv > -INFINITY || best == 0ull) best = max(best, lm_key(bv, bi));
    }
    if (r < p.rows) p.keys[(size_t)split * p.rows + r] = ok ? best : 0ull;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == LM_MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// The largest key of every row over the vocabulary ranges -> argmax (and its logit); one
// warp per row, the lanes striding over the ranges (the loads of a row are independent,
// so they overlap). A key of 0 (a range whose bounded wait gave up) gives -1.
constexpr int FIN_THREADS = 256;
__global__ void __launch_bounds__(FIN_THREADS)
lm_head_finalize_kernel(const unsigned long long* __restrict__ keys, int rows, int splits,
                        int32_t* __restrict__ argmax, float* __restrict__ max_logit) {
  griddep_wait();
  griddep_launch();
  const int r = (int)((blockIdx.x * (unsigned)FIN_THREADS + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;  // whole warps leave together
  unsigned long long k = 0ull;
  bool bad = false;
  for (int s = lane; s < splits; s += 32) {
    const unsigned long long x = keys[(size_t)s * rows + r];
    bad |= x == 0ull;
    k = max(k, x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) k = max(k, __shfl_xor_sync(FULL, k, o));
  bad = __any_sync(FULL, bad);
  if (lane != 0) return;
  if (bad) {
    argmax[r] = -1;
    if (max_logit) max_logit[r] = __int_as_float(0x7fc00000);
    return;
  }
  argmax[r] = (int32_t)(~(unsigned)(k & 0xffffffffu));
  const unsigned u = (unsigned)(k >> 32);
  if (max_logit) max_logit[r] = __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

bool make_map_rows(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                   uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

LmPlan plan_lm_head(int rows, int vocab) {
  LmPlan p{};
  p.m_tiles = (int)ceil_div(rows, BM);
  p.chunks = (int)ceil_div(vocab, VCHUNK);
  // One CTA per SM at a time. The splits S minimise waves(S) x (chunks per split + 1):
  // the CTAs of one wave take equal shares, and the +1 stands for a CTA's fixed cost.
  const int64_t sms = device_sm_count();
  int64_t best_s = 1, best_cost = INT64_MAX;
  const int64_t s_max = std::min<int64_t>(p.chunks, 8 * sms);
  for (int64_t s = 1; s <= s_max; ++s) {
    const int64_t waves = ceil_div((int64_t)p.m_tiles * s, sms);
    const int64_t cost = waves * (ceil_div(p.chunks, s) + 1);
    if (cost <= best_cost) best_cost = cost, best_s = s;  // ties: more CTAs
  }
  p.splits = (int)best_s;
  p.ws_bytes = align256((size_t)p.splits * rows * sizeof(unsigned long long));
  return p;
}

bool lm_head_supported() { return device_cc() >= 100 && encode_fn() != nullptr; }

int launch_lm_head_argmax(const LmPlan& plan, const void* hidden, const void* weight, int rows,
                          int hidden_size, int vocab, int32_t* argmax, float* max_logit,
                          void* ws, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return TSV_ERR_UNSUPPORTED;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(lm_head_argmax_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             LM_SMEM_BYTES) != cudaSuccess)
      return launch_status();
    attr_set[dev] = true;
  }
  CUtensorMap ma, mb, mb32;
  if (!make_map_rows(&ma, hidden, (uint64_t)hidden_size, (uint64_t)rows, BM) ||
      !make_map_rows(&mb, weight, (uint64_t)hidden_size, (uint64_t)vocab, BN) ||
      !make_map_rows(&mb32, weight, (uint64_t)hidden_size, (uint64_t)vocab, VCHUNK))
    return TSV_ERR_UNSUPPORTED;
  LmParams prm{rows, hidden_size, vocab, plan.chunks, plan.splits,
               static_cast<unsigned long long*>(ws)};
  int st = launch_pdl(lm_head_argmax_kernel, dim3(plan.m_tiles, plan.splits), dim3(LM_THREADS),
                      LM_SMEM_BYTES, stream, ma, mb, mb32, prm);
  if (st != TSV_OK) return st;
  return launch_pdl(lm_head_finalize_kernel,
                    dim3((unsigned)ceil_div((int64_t)rows * 32, FIN_THREADS)), dim3(FIN_THREADS), 0,
                    stream, static_cast<const unsigned long long*>(ws), rows, plan.splits,
                    argmax, max_logit);
}

}  // namespace tsv
