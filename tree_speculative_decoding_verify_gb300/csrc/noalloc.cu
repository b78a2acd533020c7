// tsv_tree_verify_attn_noalloc: tree-verification attention for callers that cannot
// allocate device memory (see include/tsv.h). The scratch that tsv_tree_verify_attn
// takes from the caller lives here instead, in a fixed file-scope device array.
//
// Who needs this: a caller whose device memory is entirely owned by its own pool or
// arena (so a cudaMalloc would fail or break its accounting), or one running in a
// latency-critical loop that must not call cudaMalloc (which can synchronize the device)
// and that cannot size and keep a workspace itself. The array costs every GPU that loads
// the library TSV_NOALLOC_SCRATCH_BYTES of memory until the process exits.
#include <cuda.h>

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
// Device address of the scratch per device, with the CUDA context it was looked up in: a
// device reset (or any new context on the device) loads the module again at another
// address, so a lookup from another context is not reused.
struct ScratchAddr {
  CUcontext ctx;
  void* addr;
};
ScratchAddr g_scratch[MAX_DEVICES];
std::mutex g_scratch_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
    cudaGetLastError();
  }
  return fn;
}

CUcontext current_context() {
  CUcontext c = nullptr;
  const CtxGetCurrentFn fn = ctx_get_current();
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of the scratch on the current device, looked up with that device current
// the first time a context uses it. nullptr if the lookup failed.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  CUcontext ctx = current_context();
  if (ctx && g_scratch[dev].addr && g_scratch[dev].ctx == ctx) return g_scratch[dev].addr;
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    cudaGetLastError();
    return nullptr;
  }
  // the lookup made the device's primary context current if none was
  g_scratch[dev].ctx = ctx ? ctx : current_context();
  g_scratch[dev].addr = p;
  return p;
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
  // the same host checks as tsv_tree_verify_attn
  bool empty = false;
  const int st = attn_call_check(shape, cache, q, k_new, v_new, prefix_len, num_nodes,
                                 position_ids, mask, rope_theta, softmax_scale, out, &empty);
  if (st != TSV_OK || empty) return st;
  const AttnPlan plan = plan_attn(shape, cache);
  if (plan.ws_bytes > (size_t)TSV_NOALLOC_SCRATCH_BYTES) return TSV_ERR_WORKSPACE;
  void* ws = scratch_address();
  if (!ws) return TSV_ERR_CUDA;
  // Nothing in the scratch has to start at zero: every region the kernels read
  // (rotated queries, split partials, request flags) is written earlier in this call.
  return launch_attn(plan, q, k_new, v_new, cache, prefix_len, num_nodes, position_ids, mask,
                     rope_theta, softmax_scale, out, ws, err, (cudaStream_t)stream);
}
