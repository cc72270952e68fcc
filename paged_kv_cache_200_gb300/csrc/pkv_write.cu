// Slot-mapped KV-cache write (bf16 copy, or FP8 E4M3 / INT8 quantise-on-write).
//
// Source: "効率的な KV キャッシュ管理と Attention 計算" (itan.pw), section "Triton
// カーネルによる KV キャッシュ書き込み": every new token's K and V row
// (num_kv_heads*head_dim contiguous elements) is stored at row slot_mapping[t]
// of the flat cache; section "Python 層からのカーネル呼び出し" fixes the layout
// checks (inner dims contiguous, free row stride, one slot per token).
//
// Design: one warp per (tensor, token) row.  The row is moved in 16-byte
// vectors (8 bf16), all loads of a lane issued before its stores; the slot is
// read once per warp.  Destination offsets are 64-bit (a 4 GB pool overflows
// 32-bit element offsets).  FP8: each element becomes
// e4m3_rne_satfinite(float(x) * inv_scale) -- one fp32 multiply and the
// hardware's round-to-nearest-even saturating conversion.
#include <cuda_fp8.h>

#include <cmath>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int kWriteThreads = 256;
constexpr int kWriteUnroll = 4;

template <int kMode>  // 0: bf16 copy, 1: FP8 E4M3, 2: INT8
__global__ void __launch_bounds__(kWriteThreads) kv_cache_write_kernel(
    const uint16_t* __restrict__ k, int64_t k_stride, const uint16_t* __restrict__ v, int64_t v_stride,
    int32_t num_tokens, int32_t row_elems, void* __restrict__ k_cache, void* __restrict__ v_cache,
    int64_t num_slots, const int32_t* __restrict__ slot_mapping, float k_inv, float v_inv, int32_t* err) {
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (kWriteThreads / 32);
  const int chunks = row_elems >> 3;  // 16-byte vectors per row
  for (int64_t row = (int64_t)blockIdx.x * (kWriteThreads / 32) + (threadIdx.x >> 5); row < 2 * (int64_t)num_tokens;
       row += warps_total) {
    const bool is_v = row >= num_tokens;
    const int64_t t = is_v ? row - num_tokens : row;
    const int32_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;  // padding token
    if ((int64_t)slot >= num_slots) {
      if (lane == 0) flag_error(err, PKV_DEVERR_SLOT);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>((is_v ? v : k) + t * (is_v ? v_stride : k_stride));
    const float inv = is_v ? v_inv : k_inv;
    for (int c0 = lane; c0 < chunks; c0 += 32 * kWriteUnroll) {
      uint4 buf[kWriteUnroll];
#pragma unroll
      for (int u = 0; u < kWriteUnroll; ++u) {
        const int c = c0 + u * 32;
        if (c < chunks) buf[u] = __ldg(src + c);
      }
#pragma unroll
      for (int u = 0; u < kWriteUnroll; ++u) {
        const int c = c0 + u * 32;
        if (c >= chunks) break;
        if constexpr (kMode == 0) {
          uint4* dst = reinterpret_cast<uint4*>(is_v ? v_cache : k_cache) + (int64_t)slot * chunks + c;
          *dst = buf[u];
        } else {
          uint2* dst = reinterpret_cast<uint2*>(is_v ? v_cache : k_cache) + (int64_t)slot * chunks + c;
          *dst = kMode == 1 ? quantize8_e4m3(buf[u], inv) : quantize8_int8(buf[u], inv);
        }
      }
    }
  }
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_kv_cache_write(const void* k, int64_t k_row_stride, const void* v, int64_t v_row_stride,
                                  int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim, void* k_cache,
                                  void* v_cache, int32_t cache_dtype, int64_t num_slots,
                                  const int32_t* slot_mapping, float k_inv_scale, float v_inv_scale,
                                  int32_t* err_flag, void* stream) {
  const pkv::NvtxRange nvtx_range("pkv_kv_cache_write");
  using namespace pkv;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_slots <= 0) return PKV_ERR_INVALID_ARG;
  if (cache_dtype != PKV_BF16 && cache_dtype != PKV_FP8_E4M3 && cache_dtype != PKV_INT8) return PKV_ERR_UNSUPPORTED;
  const int64_t row_elems = (int64_t)num_kv_heads * head_dim;
  if (row_elems % 8 != 0 || row_elems > (1 << 20)) return PKV_ERR_UNSUPPORTED;
  // a one-byte cache needs finite positive inverse scales (0, a negative value, inf or NaN
  // would store codes that stand for no value of the input)
  if (cache_dtype != PKV_BF16 && (!(k_inv_scale > 0.f) || !(v_inv_scale > 0.f) || !std::isfinite(k_inv_scale) ||
                                  !std::isfinite(v_inv_scale)))
    return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
  if (k_row_stride < row_elems || v_row_stride < row_elems || k_row_stride % 8 || v_row_stride % 8)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID_ARG;
  const int64_t rows = 2 * (int64_t)num_tokens;
  const int warps_per_block = kWriteThreads / 32;
  int64_t blocks = (rows + warps_per_block - 1) / warps_per_block;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  cudaStream_t st = as_stream(stream);
  auto kern = cache_dtype == PKV_BF16 ? kv_cache_write_kernel<0>
               : cache_dtype == PKV_FP8_E4M3 ? kv_cache_write_kernel<1> : kv_cache_write_kernel<2>;
  kern<<<(unsigned)blocks, kWriteThreads, 0, st>>>(static_cast<const uint16_t*>(k), k_row_stride,
                                                   static_cast<const uint16_t*>(v), v_row_stride, num_tokens,
                                                   (int32_t)row_elems, k_cache, v_cache, num_slots, slot_mapping,
                                                   k_inv_scale, v_inv_scale, err_flag);
  return launch_status();
}
