// Tree-verification attention on warp-level tensor-core MMAs (mma.sync m16n8k16, bf16 in,
// fp32 accumulate), head_dim 128, K/V streamed through a cp.async ring in shared memory.
//
// Pages: "推理系统手册 · 投机解码进阶：树形草稿与 EAGLE", section 实现 (forward_with_mask:
// each node attends to the whole prefix and, among the tree nodes, to its ancestors and
// itself; GQA heads share a KV head) and "TensorRT-LLM 源码完全拆解(二十二)", section
// CUDA Graph 里的掩码重排 (the attention reads the padded bit mask directly).
//
// One CTA = (request b, KV head h, 128 query rows, split of the keys); eight warps of 16
// rows each. The query rows of a KV head are every (node, query head of the group) pair,
// so each K/V tile in shared memory serves all of them.
//   loads      every thread copies its share of each 64-key K and V tile with 16-byte
//              cp.async into a STAGES-deep ring (rows at or past the zero-padded end of
//              the tree are zero-filled, never read); row-chunk c of key row r sits at
//              chunk c ^ (r & 7), so the 8-row ldmatrix reads below are conflict-free
//   S = Q K^T  Q is held as A fragments in registers (loaded once); K fragments come
//              from ldmatrix (keys are the rows of the B = K^T operand)
//   softmax    per row, in log2 units: tile maximum over the four lanes that share a row,
//              running max m and sum l, O rescaled by 2^(m_old - m_new); tree keys are
//              masked with the row's node mask, keys past the tree with -inf
//   O += P V   P is rebuilt in registers as A fragments straight from the S accumulators
//              (the C layout of two n8 tiles is the A layout of one k16 step); V
//              fragments come from ldmatrix.trans
// A CTA that covers every key of its rows writes the normalised bf16 output; otherwise it
// writes its unnormalised rows and (m, l) for the split merge. Warps whose 16 rows are all
// past the tree only help with the loads.
#include <stdint.h>

#include "attn_common.cuh"
#include "common.cuh"

namespace tsv {
namespace {

constexpr int BM = 128, BN = 64, D = 128;     // query rows, keys per tile, head dim
constexpr int WARPS = 8, THREADS = WARPS * 32;
constexpr int STAGES = 4;
constexpr int ROW_BYTES = D * 2;              // one K or V row, bf16
constexpr int TILE_BYTES = BN * ROW_BYTES;    // 16 KB
constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // K tile, then V tile
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES;
constexpr int CHUNKS = TILE_BYTES / 16;       // 16-byte copies per tile
static_assert(CHUNKS % THREADS == 0, "every thread copies the same number of chunks");
static_assert(BN == TSV_KV_BLOCK, "a tile is one block of a paged cache");

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// byte offset of 16-byte chunk c of row r inside a tile
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * ROW_BYTES + ((c ^ (r & 7)) << 4));
}
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
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// d += a b (m16n8k16, row-major A, column-major B, bf16 in, fp32 accumulate)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

struct MmaParams {
  AttnArgs a;
  float scale_log2;
  __nv_bfloat16* out;  // [B, max_nodes, Hq, D]
};

__global__ void __launch_bounds__(THREADS, 1) attn_mma_kernel(const MmaParams prm) {
  extern __shared__ __align__(128) uint8_t smem[];
  const AttnArgs& a = prm.a;
  const int split = blockIdx.x, mt = blockIdx.y;
  const int b = blockIdx.z / a.hkv, h = blockIdx.z % a.hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;  // row group and column pair of the fragments
  griddep_wait();  // the prep kernel's rotated queries, cache appends and flags

  const int valid = a.valid[b], T = a.num_nodes[b], P = a.prefix_len[b];
  if (!valid) return;
  const int rows = T * a.group;
  const int row0 = mt * BM;
  if (row0 >= rows) return;
  const int keys = P + T;
  const int kload = (keys + 15) & ~15;  // rows past the tree up to here are zeros
  const int n_tiles = (keys + BN - 1) / BN;
  const int t0 = split * a.tiles_per_split;
  const int t1 = min(n_tiles, t0 + a.tiles_per_split);
  if (t0 >= t1) return;
  const int n = t1 - t0;
  const bool single = n_tiles <= a.tiles_per_split;

  // ---- loads: thread tid copies chunks tid, tid + THREADS, ... of each tile -----------
  const char* kbase = static_cast<const char*>(a.k_cache);
  const char* vbase = static_cast<const char*>(a.v_cache);
  const uint32_t sbase = smem_addr(smem);
  auto issue = [&](int i) {  // tile t0 + i into stage i % STAGES
    const int key0 = (t0 + i) * BN;
    int64_t rowbase;  // cache row of key0 (a tile never crosses a paged block)
    if (a.layout == TSV_KV_CONTIGUOUS) {
      rowbase = ((int64_t)b * a.hkv + h) * a.capacity + key0;
    } else {
      const int blk = key0 < kload ? a.block_table[(int64_t)b * a.max_blocks + key0 / BN] : 0;
      rowbase = ((int64_t)blk * a.hkv + h) * TSV_KV_BLOCK;
    }
    const uint32_t st = sbase + (uint32_t)((i % STAGES) * STAGE_BYTES);
#pragma unroll
    for (int q = 0; q < CHUNKS / THREADS; ++q) {
      const int idx = tid + q * THREADS, r = idx >> 4, c = idx & 15;
      const bool in = key0 + r < kload;
      const int64_t off = in ? (rowbase + r) * ROW_BYTES + c * 16 : 0;
      cp_async16(st + swz(r, c), kbase + off, in);
      cp_async16(st + TILE_BYTES + swz(r, c), vbase + off, in);
    }
  };
#pragma unroll
  for (int i = 0; i < STAGES - 1; ++i) {
    if (i < n) issue(i);
    cp_commit();
  }

  // ---- this warp's 16 rows: Q fragments, masks --------------------------------------
  const int wr0 = row0 + warp * 16;
  const bool active = wr0 < rows;
  const int ra = wr0 + g, rb = ra + 8;  // the thread's two rows
  uint32_t qf[8][4];
  {
    const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(a.q_rot) +
                              ((int64_t)b * a.hkv + h) * a.rows_pad * D;
    const uint32_t* qa = reinterpret_cast<const uint32_t*>(qb + (int64_t)ra * D);
    const uint32_t* qc = reinterpret_cast<const uint32_t*>(qb + (int64_t)rb * D);
    const bool la = active && ra < rows, lb = active && rb < rows;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int w = kk * 8 + t4;  // 32-bit word of dims kk*16 + 2 t4
      qf[kk][0] = la ? qa[w] : 0u;
      qf[kk][1] = lb ? qc[w] : 0u;
      qf[kk][2] = la ? qa[w + 4] : 0u;
      qf[kk][3] = lb ? qc[w + 4] : 0u;
    }
  }
  // node masks of the two rows (rows past the tree read node 0's; never stored)
  const uint32_t* mra = a.mask + ((int64_t)b * a.max_nodes + (ra < rows ? ra / a.group : 0)) * a.mask_words;
  const uint32_t* mrb = a.mask + ((int64_t)b * a.max_nodes + (rb < rows ? rb / a.group : 0)) * a.mask_words;

  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  const float sl2 = prm.scale_log2;

  for (int i = 0; i < n; ++i) {
    if (i + STAGES - 1 < n) issue(i + STAGES - 1);
    cp_commit();
    cp_wait<STAGES - 1>();  // this thread's copies of tile i have landed
    __syncthreads();        // and everyone's
    if (active) {
      const uint32_t ks = sbase + (uint32_t)((i % STAGES) * STAGE_BYTES);
      const uint32_t vs = ks + TILE_BYTES;
      const int key0 = (t0 + i) * BN;
      // S = Q K^T: 8 n-tiles of 8 keys; ldmatrix x4 gives B for two n-tiles per k-step
      float s[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {
          // matrices: (keys 16jp.., dims 16kk..), (keys 16jp.., dims 16kk+8..),
          //           (keys 16jp+8.., dims 16kk..), (keys 16jp+8.., dims 16kk+8..)
          const int mat = lane >> 3;
          const int kr = 16 * jp + ((mat >> 1) << 3) + (lane & 7);
          uint32_t bf[4];
          ldsm4(ks + swz(kr, 2 * kk + (mat & 1)), bf);
          mma16816(s[2 * jp], qf[kk], bf[0], bf[1]);
          mma16816(s[2 * jp + 1], qf[kk], bf[2], bf[3]);
        }
      }
      // mask and scale (log2 units); columns 2 t4 and 2 t4 + 1 of each n-tile
      const bool tree_tile = key0 + BN > P;
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kidx = key0 + 8 * j + 2 * t4 + (e & 1);
          float x = s[j][e] * sl2;
          if (tree_tile && kidx >= P) {
            const int tt = kidx - P;
            const uint32_t* mr = e < 2 ? mra : mrb;
            const bool vis = kidx < keys && ((mr[tt >> 5] >> (tt & 31)) & 1u);
            x = vis ? x : -INFINITY;
          }
          s[j][e] = x;
        }
      // row maxima over the tile (rows ra: e = 0, 1; rb: e = 2, 3)
      float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        mx_a = fmaxf(mx_a, fmaxf(s[j][0], s[j][1]));
        mx_b = fmaxf(mx_b, fmaxf(s[j][2], s[j][3]));
      }
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        mx_a = fmaxf(mx_a, __shfl_xor_sync(FULL, mx_a, off));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(FULL, mx_b, off));
      }
      const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
      // a row with nothing visible so far keeps O = 0, l = 0 (any finite reference works)
      const float ref_a = mn_a == -INFINITY ? 0.f : mn_a;
      const float ref_b = mn_b == -INFINITY ? 0.f : mn_b;
      const float al_a = exp2f(m_a - ref_a), al_b = exp2f(m_b - ref_b);
      m_a = mn_a;
      m_b = mn_b;
      float sum_a = 0.f, sum_b = 0.f;
      uint32_t pf[4][4];  // P as A fragments, one per k-step of 16 keys
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float p0 = exp2f(s[j][0] - ref_a), p1 = exp2f(s[j][1] - ref_a);
        const float p2 = exp2f(s[j][2] - ref_b), p3 = exp2f(s[j][3] - ref_b);
        sum_a += p0 + p1;
        sum_b += p2 + p3;
        pf[j >> 1][(j & 1) * 2 + 0] = pack_bf16(p0, p1);
        pf[j >> 1][(j & 1) * 2 + 1] = pack_bf16(p2, p3);
      }
      l_a = l_a * al_a + sum_a;
      l_b = l_b * al_b + sum_b;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] *= al_a;
        o[j][1] *= al_a;
        o[j][2] *= al_b;
        o[j][3] *= al_b;
      }
      // O += P V: 16 n-tiles of 8 dims, 4 k-steps of 16 keys; ldmatrix.trans x4 gives B
      // for two n-tiles of one k-step
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int jp = 0; jp < 8; ++jp) {
          // matrices: (keys 16kk.., dims 16jp..), (keys 16kk+8.., dims 16jp..),
          //           (keys 16kk.., dims 16jp+8..), (keys 16kk+8.., dims 16jp+8..)
          const int mat = lane >> 3;
          const int vr = 16 * kk + ((mat & 1) << 3) + (lane & 7);
          uint32_t bf[4];
          ldsm4t(vs + swz(vr, 2 * jp + (mat >> 1)), bf);
          mma16816(o[2 * jp], pf[kk], bf[0], bf[1]);
          mma16816(o[2 * jp + 1], pf[kk], bf[2], bf[3]);
        }
      }
    }
    __syncthreads();  // stage i % STAGES is free for tile i + STAGES
  }
  cp_wait<0>();
  griddep_launch();  // the next kernel may be scheduled (it waits for this grid to finish)
  if (!active) return;

  // ---- epilogue: the thread's rows ra (o[.][0..1]) and rb (o[.][2..3]) ---------------
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l_a += __shfl_xor_sync(FULL, l_a, off);
    l_b += __shfl_xor_sync(FULL, l_b, off);
  }
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? rb : ra;
    if (r >= rows) continue;
    const float l = half ? l_b : l_a;
    const int node = r / a.group;
    if (single) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint32_t* dst = reinterpret_cast<uint32_t*>(
          prm.out + (((int64_t)b * a.max_nodes + node) * a.hq + h * a.group + r % a.group) * D);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        dst[4 * j + t4] = pack_bf16(o[j][2 * half] * inv, o[j][2 * half + 1] * inv);
    } else {
      const int64_t prow = (((int64_t)b * a.hkv + h) * a.nsplit + split) * a.rows_pad + r;
      float2* dst = reinterpret_cast<float2*>(a.o_part + prow * D);
#pragma unroll
      for (int j = 0; j < 16; ++j) dst[4 * j + t4] = make_float2(o[j][2 * half], o[j][2 * half + 1]);
      if (t4 == 0) {
        a.ml[prow * 2 + 0] = half ? m_b : m_a;
        a.ml[prow * 2 + 1] = l;
      }
    }
  }
}

}  // namespace

int launch_attn_mma(const AttnPlan& p, const AttnArgs& a, float scale_log2, void* out,
                    cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return TSV_ERR_UNSUPPORTED;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(attn_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return launch_status();
    attr_set[dev] = true;
  }
  MmaParams prm{a, scale_log2, static_cast<__nv_bfloat16*>(out)};
  dim3 grid(p.nsplit, (unsigned)ceil_div(p.rows, BM), p.batch * p.hkv);
  const int st = launch_pdl(attn_mma_kernel, grid, dim3(THREADS), SMEM_BYTES, stream, prm);
  if (st != TSV_OK || p.nsplit == 1) return st;
  return launch_split_merge(p, a, out, stream);
}

}  // namespace tsv
