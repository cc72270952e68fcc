// Host-side helpers shared by the libpkv entry points.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Streaming multiprocessors of the current device (cached per device).
int device_sm_count();

// Status of the launches just issued on this thread.
inline int launch_status() { return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// An NVTX range over an entry point's call when tracing is on (pkv_set_nvtx).
struct NvtxRange {
  bool on;
  explicit NvtxRange(const char* name);
  ~NvtxRange();
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Tensor map over a [rows, heads, dim] array of `elt_bytes`-byte elements
// (bf16 = 2, e4m3 = 1), boxes of box_inner elements x 1 head x box_rows rows,
// swizzle of 128 or 64 bytes (or 0 for none).  False if the driver refuses it.
bool make_tmap_3d(CUtensorMap* map, const void* base, int elt_bytes, int64_t rows, int heads, int dim,
                  int box_inner, int box_rows, int swizzle_bytes);

// Varlen sequences with few queries are served by the decode kernels, one
// item per query row (coded b * kRouteCode + qi): those with one query always,
// and those with up to kRouteMaxQ when no sequence of the batch has more
// (speculative verification); longer ones by the prefill tiles.
constexpr int kRouteMaxQ = 8;
constexpr int kRouteCode = 16;
static_assert(kRouteMaxQ < kRouteCode, "query index must fit the item code");

// When no sequence has more than kRouteMaxQ queries and max_len_q * group
// query rows fit kMultiRows, one decode CTA per (split, kv head, sequence)
// serves every (query, head) row of the sequence, so its K/V is read once;
// otherwise each routed query row is a decode item of its own.
constexpr int kMultiRows = 16;
inline bool multi_query_items(int max_len_q, int group) {
  return max_len_q >= 1 && max_len_q <= kRouteMaxQ && max_len_q * group <= kMultiRows;
}
// Blocks of 8 (query, head) rows on the decode MMAs' N side for items of
// multi_q queries (multi_q = 0: one query row per item).
inline int multi_query_row_blocks(int multi_q, int group) { return multi_q > 0 && multi_q * group > 8 ? 2 : 1; }

// Decode kernels serving the routed query rows of a paged varlen batch
// (at most item_bound items; splits planned for `batch` sequences).  multi_q:
// 0 (an item is one query row) or the bound on queries per item (an item is a
// sequence, see multi_query_items).  after_primary: launch the split kernel as
// a programmatic dependent of the kernel just before it on the stream, which
// must not write anything the decode kernels read.

size_t varlen_decode_workspace(int batch, int items, int num_heads, int num_kv_heads, int head_dim, int max_len_k,
                               int cache_dtype, int multi_q);
int launch_varlen_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* items,
                         const int32_t* item_count, const int32_t* cu_q, const int32_t* cu_k,
                         const int32_t* block_table, int32_t max_blocks_per_seq, int32_t batch, int32_t item_bound,
                         int32_t num_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                         int32_t max_len_k, int64_t total_q, float scale, int cache_dtype, float k_scale,
                         float v_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                         int32_t* err_flag, int32_t multi_q, bool after_primary, cudaStream_t st);

}  // namespace pkv
