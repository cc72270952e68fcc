// Copy-on-write of shared cache blocks.
//
// Source: "KV cache / batching / paged attention" (1s.xyz, chapter 15), section
// "PagedAttention：メモリを「ページ」で貸し出す": several answers generated from
// one prompt share the blocks of their common part, and a shared block is
// copied only once one of them has to write into it.  This call makes those
// copies: for each (src, dst) pair, block dst of each cache becomes a copy of
// block src, byte for byte (bf16, FP8 or INT8 codes alike).
//
// Design: an HBM-bound copy.  Each CTA takes whole pairs (grid-stride over the
// pair list) and moves a block of each cache in 16-byte vectors, every thread
// issuing all of its loads of a round before its stores.  The pair is read
// once per CTA and checked; offsets are 64-bit.
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__device__ __forceinline__ void copy_block(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t chunks) {
  for (int64_t base = threadIdx.x; base < chunks; base += (int64_t)kCopyThreads * kCopyUnroll) {
    uint4 r[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t c = base + (int64_t)u * kCopyThreads;
      if (c < chunks) r[u] = __ldg(src + c);
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t c = base + (int64_t)u * kCopyThreads;
      if (c < chunks) dst[c] = r[u];
    }
  }
}

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(uint8_t* __restrict__ k_cache,
                                                                   uint8_t* __restrict__ v_cache, int64_t block_bytes,
                                                                   int32_t num_blocks,
                                                                   const int32_t* __restrict__ pairs,
                                                                   int32_t num_pairs, int32_t* err) {
  const int64_t chunks = block_bytes >> 4;
  for (int32_t i = blockIdx.x; i < num_pairs; i += gridDim.x) {
    const int32_t src = __ldg(pairs + 2 * (int64_t)i);
    const int32_t dst = __ldg(pairs + 2 * (int64_t)i + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (threadIdx.x == 0) flag_error(err, PKV_DEVERR_BLOCK);
      continue;  // never dereferenced
    }
    copy_block(reinterpret_cast<const uint4*>(k_cache + src * block_bytes),
               reinterpret_cast<uint4*>(k_cache + dst * block_bytes), chunks);
    if (v_cache != nullptr)
      copy_block(reinterpret_cast<const uint4*>(v_cache + src * block_bytes),
                 reinterpret_cast<uint4*>(v_cache + dst * block_bytes), chunks);
  }
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_copy_blocks(void* k_cache, void* v_cache, int64_t block_bytes, int32_t num_blocks,
                               const int32_t* block_pairs, int32_t num_pairs, int32_t* err_flag, void* stream) {
  const pkv::NvtxRange nvtx_range("pkv_copy_blocks");
  using namespace pkv;
  if (num_pairs < 0 || num_blocks <= 0 || block_bytes <= 0) return PKV_ERR_INVALID_ARG;
  if (block_bytes % 16 != 0) return PKV_ERR_INVALID_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (k_cache == nullptr || block_pairs == nullptr) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || (v_cache != nullptr && !aligned16(v_cache))) return PKV_ERR_INVALID_ARG;
  const int sms = device_sm_count();
  if (sms <= 0) return PKV_ERR_CUDA;
  // enough CTAs per SM to keep several 16-byte loads per thread in flight
  const int64_t cap = (int64_t)sms * 8;
  const int grid = (int)(num_pairs < cap ? num_pairs : cap);
  copy_blocks_kernel<<<grid, kCopyThreads, 0, as_stream(stream)>>>(
      static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), block_bytes, num_blocks, block_pairs,
      num_pairs, err_flag);
  return launch_status();
}
