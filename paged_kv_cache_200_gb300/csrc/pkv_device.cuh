// Device-side helpers shared by the libpkv kernels (sm_103a).
//
// Inline PTX wrappers for the instructions the kernels are built from:
// cp.async (16-byte, zero-fill), ldmatrix / movmatrix, mma.sync bf16, ex2.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

__device__ __forceinline__ void flag_error(int32_t* err, int32_t bit) {
  if (err != nullptr) atomicOr(err, bit);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared copy; copies `src_bytes` (0 or 16) bytes and fills the rest with zeros.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Transpose an 8x8 matrix of 16-bit elements held in the mma/ldmatrix fragment layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
  return d;
}

// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D (16x8 fp32) += A (16x16 f16, row) * B (16x8 f16, col)
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two E4M3 codes (bits 0..7 and 8..15 of the low, resp. high, half of w) -> f16x2,
// exactly (every E4M3 value is an f16 value), with the hardware conversion.
__device__ __forceinline__ uint32_t e4m3x2_lo_to_f16x2(uint32_t w) {
  uint32_t d;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n}\n" : "=r"(d) : "r"(w));
  return d;
}
__device__ __forceinline__ uint32_t e4m3x2_hi_to_f16x2(uint32_t w) {
  uint32_t d;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.rn.f16x2.e4m3x2 %0, hi;\n}\n" : "=r"(d) : "r"(w));
  return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}

// Eight bf16 values (one 16-byte vector) -> eight OCP E4M3 codes, each
// e4m3_rne_satfinite(float(x) * inv): one fp32 multiply and the hardware's
// round-to-nearest-even saturating conversion.
__device__ __forceinline__ uint2 quantize8_e4m3(uint4 v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t packed[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t bytes = 0;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const uint32_t word = w[h * 2 + p];
      const float lo = __uint_as_float(word << 16);
      const float hi = __uint_as_float(word & 0xFFFF0000u);
      const __nv_fp8x2_storage_t two =
          __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(lo, inv), __fmul_rn(hi, inv)), __NV_SATFINITE, __NV_E4M3);
      bytes |= (uint32_t)two << (16 * p);
    }
    packed[h] = bytes;
  }
  return make_uint2(packed[0], packed[1]);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Eight bf16 values -> eight INT8 codes, each
// clamp(round_half_even(float(x) * inv), -127, 127); a NaN product gives 0
// (the float-to-int conversion's rule), an infinity saturates.
__device__ __forceinline__ uint2 quantize8_int8(uint4 v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t packed[2] = {0u, 0u};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const uint32_t word = w[e >> 1];
    const float x = __uint_as_float((e & 1) ? (word & 0xFFFF0000u) : (word << 16));
    int r = __float2int_rn(__fmul_rn(x, inv));
    r = r > 127 ? 127 : (r < -127 ? -127 : r);
    packed[e >> 2] |= ((uint32_t)r & 0xFFu) << (8 * (e & 3));
  }
  return make_uint2(packed[0], packed[1]);
}

// INT8 codes to f16, exactly, by a byte permute: with its sign bit flipped a
// code c is the unsigned byte c + 128; placed as the low mantissa byte of an
// f16 whose exponent field gives 2^10 (high byte 0x64) it reads
// 1024 + c + 128 = 1152 + c.  The decode kernel feeds these biased values to
// its MMAs and takes the excess (1152 times the sum of the other factor) off
// once: from the logits for K, from the output for V.
constexpr float kInt8Bias = 1152.f;

// Packed fp32 pairs (sm_100+): two lanes of arithmetic per instruction.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three floats in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 2^x with the hardware approximation (ex2.approx, relative error ~2^-22).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}


// ---------------------------------------------------------------------------
// mbarrier, TMA and timer helpers
// ---------------------------------------------------------------------------

#ifdef PKV_TEST_WAIT_NS
constexpr uint64_t kWaitNs = PKV_TEST_WAIT_NS;  // test builds: a short limit
#else
constexpr uint64_t kWaitNs = 2000000000ull;  // every bounded wait gives up after 2 s
#endif

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of parity `parity`: false when the deadline
// passes or (when given) another role of the CTA has set *abort_flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (abort_flag != nullptr && *abort_flag) return false;
      const uint64_t now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kWaitNs) {
        return false;
      }
    }
  }
}

// 3-D tiled TMA load (box given by the tensor map) completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* map, int c0, int c1, int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// Prefetch the box of a 3-D tensor map at these coordinates into L2 (no
// shared memory written, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_3d(const void* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace pkv
