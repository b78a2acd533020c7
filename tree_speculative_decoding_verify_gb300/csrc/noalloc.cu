// tsv_tree_verify_attn_noalloc: tree-verification attention for callers that cannot
// allocate device memory (see include/tsv.h). The scratch that tsv_tree_verify_attn
// takes from the caller lives here instead, in a fixed file-scope device array.
//
// Who needs this: a caller whose device memory is entirely owned by its own pool or
// arena (so a cudaMalloc would fail or break its accounting), or one running in a
// latency-critical loop that must not call cudaMalloc (which can synchronize the device)
// and that cannot size and keep a workspace itself. The array costs every GPU that loads
// the library TSV_NOALLOC_SCRATCH_BYTES of memory until the process exits.
#include <mutex>

#include "attn_common.cuh"
#include "common.cuh"
#include "kernels.h"

namespace tsv {
namespace {

// The scratch. Host code must not use this name as an address: on the host it is only a
// stand-in for the symbol; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TSV_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
void* g_scratch_addr[MAX_DEVICES];
std::mutex g_scratch_mu;

// Device address of the scratch on the current device (looked up once per device, with
// that device current). nullptr if the lookup failed.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

bool shape_ok(const tsv_attn_shape* s, const tsv_kv_cache* c) {
  if (!s || !c || !c->k || !c->v) return false;
  if (c->dtype != TSV_DTYPE_F32 && c->dtype != TSV_DTYPE_BF16) return false;
  if (c->num_kv_heads < 1 || (c->head_dim != 64 && c->head_dim != 128)) return false;
  if (c->layout == TSV_KV_CONTIGUOUS) {
    if (c->capacity < TSV_KV_BLOCK || c->capacity % TSV_KV_BLOCK) return false;
  } else if (c->layout == TSV_KV_PAGED) {
    if (!c->block_table || c->max_blocks < 1 || c->num_blocks < 1) return false;
  } else {
    return false;
  }
  if ((reinterpret_cast<uintptr_t>(c->k) | reinterpret_cast<uintptr_t>(c->v)) % 16) return false;
  if (s->batch < 0 || s->max_nodes < 1 || s->max_nodes > TSV_MAX_NODES || s->max_prefix < 0)
    return false;
  if (s->num_q_heads < 1 || s->num_q_heads % c->num_kv_heads) return false;
  if ((int64_t)s->batch * c->num_kv_heads > 65535) return false;
  if ((int64_t)s->max_nodes * (s->num_q_heads / c->num_kv_heads) > 1024) return false;
  return true;
}

}  // namespace
}  // namespace tsv

using namespace tsv;

extern "C" int tsv_tree_verify_attn_noalloc(const tsv_attn_shape* shape, const void* q,
                                            const void* k_new, const void* v_new,
                                            const tsv_kv_cache* cache, const int32_t* prefix_len,
                                            const int32_t* num_nodes, const int32_t* position_ids,
                                            const uint32_t* mask, float rope_theta,
                                            float softmax_scale, void* out, int32_t* err,
                                            tsv_stream_t stream) {
  if (!shape_ok(shape, cache)) return TSV_ERR_INVALID_ARG;
  if (!(rope_theta > 0.f) || !(softmax_scale > 0.f)) return TSV_ERR_INVALID_ARG;
  if (shape->batch == 0) return TSV_OK;
  if (!q || !k_new || !v_new || !prefix_len || !num_nodes || !position_ids || !mask || !out)
    return TSV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_new) |
       reinterpret_cast<uintptr_t>(v_new) | reinterpret_cast<uintptr_t>(out)) % 16)
    return TSV_ERR_INVALID_ARG;
  const AttnPlan plan = plan_attn(shape, cache);
  if (plan.ws_bytes > (size_t)TSV_NOALLOC_SCRATCH_BYTES) return TSV_ERR_WORKSPACE;
  void* ws = scratch_address();
  if (!ws) return TSV_ERR_CUDA;
  // Nothing in the scratch has to start at zero: every region the kernels read
  // (rotated queries, split partials, request flags) is written earlier in this call.
  return launch_attn(plan, q, k_new, v_new, cache, prefix_len, num_nodes, position_ids, mask,
                     rope_theta, softmax_scale, out, ws, err, (cudaStream_t)stream);
}
