// Internal helpers shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/tsv.h"

namespace tsv {

// ---- host side ---------------------------------------------------------------
void record_cuda_error(cudaError_t e);
int launch_status();                    // TSV_OK or TSV_ERR_CUDA after a launch
int device_sm_count();                  // cached per device
int device_cc();                        // 10 * major + minor, cached per device

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Every kernel is launched with programmatic stream serialization: the launch may be
// scheduled while the previous kernel of the stream is finishing, and the kernel waits
// (griddep_wait) before it touches memory that earlier work writes or reads, so stream
// order still holds for every access; only the launch latency is hidden.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
               cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) != cudaSuccess) {
    cudaGetLastError();  // no programmatic serialization here: a plain launch
    cfg.numAttrs = 0;
    cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  }
  return launch_status();
}

// ---- device side -------------------------------------------------------------
constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Programmatic dependent launch: wait for the previous grid of the stream to complete (its
// memory visible); let the next grid of the stream be scheduled.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// (value, index) order used by every selection: larger value first, then lower index.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

}  // namespace tsv
