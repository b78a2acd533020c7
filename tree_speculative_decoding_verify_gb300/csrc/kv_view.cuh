// Device view of a KV cache for the kernels that move accepted rows (internal).
#pragma once

#include "common.cuh"

namespace tsv {

struct CacheView {
  char* k;
  char* v;
  const int32_t* block_table;
  int64_t capacity, layer_stride_bytes;
  int hkv, row_bytes, layout, max_blocks, num_blocks, num_layers;
};

// Byte offset of (request b, kv head h, slot) in one layer's K or V; *ok = false for a
// block-table entry outside [0, num_blocks).
__device__ __forceinline__ int64_t slot_offset(const CacheView& c, int b, int h, int slot,
                                               bool* ok) {
  if (c.layout == TSV_KV_CONTIGUOUS) {
    return (((int64_t)b * c.hkv + h) * c.capacity + slot) * c.row_bytes;
  }
  const int blk = c.block_table[(int64_t)b * c.max_blocks + slot / TSV_KV_BLOCK];
  if (blk < 0 || blk >= c.num_blocks) { *ok = false; return 0; }
  return (((int64_t)blk * c.hkv + h) * TSV_KV_BLOCK + slot % TSV_KV_BLOCK) * c.row_bytes;
}

// Slots a request may use: the contiguous capacity or its block-table reach.
__device__ __forceinline__ int64_t cache_slots(const CacheView& c) {
  return c.layout == TSV_KV_CONTIGUOUS ? c.capacity : (int64_t)c.max_blocks * TSV_KV_BLOCK;
}

inline CacheView make_cache_view(const tsv_kv_cache* cache) {
  CacheView cv{};
  if (!cache) return cv;
  const int esize = cache->dtype == TSV_DTYPE_BF16 ? 2 : 4;
  cv.k = static_cast<char*>(cache->k);
  cv.v = static_cast<char*>(cache->v);
  cv.block_table = cache->block_table;
  cv.capacity = cache->capacity;
  cv.layer_stride_bytes = cache->layer_stride * esize;
  cv.hkv = cache->num_kv_heads;
  cv.row_bytes = cache->head_dim * esize;
  cv.layout = cache->layout;
  cv.max_blocks = cache->max_blocks;
  cv.num_blocks = cache->num_blocks;
  cv.num_layers = cache->num_layers;
  return cv;
}

}  // namespace tsv
