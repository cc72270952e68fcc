// Paged decode attention: split-KV kernel + log-sum-exp combine kernel.
//
// Source: "ページド・アテンション" (transformers docs), section "デコードパス": one
// query token per sequence; its keys are the first cache_seqlens[b] positions,
// found through row b of block_table (shape (batch, max_blocks_per_seq));
// blocks need not be contiguous.  "効率的な KV キャッシュ管理と Attention 計算"
// (itan.pw), "Attention モジュールの実装": the decode branch attends after the
// new token was written.  "KV cache / batching / paged attention" (1s.xyz ch. 15),
// "FlashAttention：注意計算そのものを速く": tiling with a running max and sum
// gives exactly ordinary attention.
//
// Design (GB300):
// * Grid (split, kv_head, seq).  A CTA owns one kv head of one sequence over a
//   contiguous range of positions, and serves every query head of that GQA
//   group, so each K/V page row is read from HBM once per group.
// * 4 warps; each warp streams its own 16-position groups (positions
//   16*(warp + 4*i)) through a private ring of shared-memory stages, filled by
//   one lane with TMA boxes of 16 rows (128- or 64-byte swizzle) that complete
//   on a per-stage mbarrier; V rows past the sequence end are zeroed after
//   the copy lands.  A bad block id issues no copy and is flagged.
// * Scores on tensor cores with the operands swapped: S^T[16 tok x 8 heads] =
//   K[16 x D] * Q^T[D x 8] (mma.sync m16n8k16), so a group of up to 8 heads
//   fills the N=8 side and no token row is padding.  P is transposed in
//   registers (movmatrix) into the B operand of O^T[D x 8] += V^T * P^T.
// * Online softmax in the log2 domain, fp32; the running max moves only when
//   it grows by more than 2^8; masked positions get -inf (never
//   multiply-by-zero, so stale or NaN cache rows cannot leak in).
// * FP8 E4M3 or INT8 cache: codes widen exactly to f16 (the hardware
//   conversion, resp. byte permutes and one f16 subtract) and the MMAs run in
//   f16; Q is scaled by a power of two into f16 range, k_scale folds into the
//   logit scale and v_scale into the output.  One-byte caches run 4 CTAs per
//   SM (bf16: 2), which hides the widening work behind more warps.
// * Split sizes come from the host: few long sequences are cut so that their
//   CTAs fill whole waves of resident CTAs; mixed batches get about 32 CTAs
//   per SM at the longest length.
// * Per-CTA partials (O/l, log2-sum-exp) go to the caller's workspace; a
//   second kernel, launched as a programmatic dependent of the first, merges
//   the splits of each (seq, head).  A sequence that fits one split is written
//   directly by the split kernel.
// * Append mode (decode with the step's cache update): the warp whose copies
//   read the new position stores the new K/V rows first.
#include <cmath>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int kDecWarps = 4;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kGroupTok = 16;       // positions per warp step
constexpr int kMaxGroup = 8;        // query heads per kv head handled by one CTA
constexpr int kResidentBf16 = 2;    // split-kernel CTAs per SM with a bf16 cache (3 stages)
constexpr int kResidentCoded = 4;   // ... with one-byte codes (3 stages)
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
  const uint16_t* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* seqlens;
  const int32_t* block_table;
  int32_t max_blocks;
  int32_t num_heads;
  int32_t num_kv_heads;
  int32_t group;
  int32_t block_size;
  int32_t num_blocks;
  int32_t split_tokens;
  int32_t max_splits;
  int32_t split_major;  // grid order: (items, kv heads, splits) instead of (splits, kv heads, items)
  float scale_log2;
  float v_mul;
  uint16_t* out;
  float* lse;
  float* ws_o;
  float* ws_lse;
  int32_t* err;
  // Varlen routing (all null for a plain decode call): CTA z serves sequence
  // items[z] when z < *item_count; its q/out row is cu_q[b] and its length
  // cu_k[b+1]-cu_k[b].  lse[b, h] lives at lse[h*lse_head_stride + row*lse_row_stride].
  const int32_t* items;
  const int32_t* item_count;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int64_t lse_head_stride;
  int64_t lse_row_stride;
  // Multi-query items (varlen routing): 0, or the bound on queries per item;
  // then items[z] is a sequence and its (query, head) rows fill the N side.
  int32_t multi_q;
  // Append (decode with an in-place cache update): seqlens hold the lengths
  // before this step's token, which takes position seqlens[b]; its K/V rows
  // (k_new/v_new row b, quantised for an FP8 cache) are stored there by the
  // CTA whose positions end with it, before that CTA's copies read them, and
  // the sequence attends seqlens[b] + 1 positions.  k_new == null: no append.
  const uint16_t* k_new;
  const uint16_t* v_new;
  int64_t k_new_stride, v_new_stride;  // elements between rows
  float k_inv, v_inv;                  // FP8: 1 / scale of each cache
#ifdef PKV_TEST_HOOKS
  int32_t test_skip_group;             // test builds: CTA (0,0,0), warp 0 withholds this group's copies (-1: none)
#endif
};

// Sequence served by grid index z (or -1) and, in varlen mode, which of its
// queries (qi): a routed item is b * kRouteCode + qi.
__device__ __forceinline__ int item_sequence(const DecodeParams& p, int z, int& qi) {
  qi = 0;
  if (p.items == nullptr) return z;
  if (z >= __ldg(p.item_count)) return -1;
  const int code = __ldg(p.items + z);
  qi = code % kRouteCode;
  return code / kRouteCode;
}
__device__ __forceinline__ int64_t item_row(const DecodeParams& p, int b, int qi) {
  return p.cu_q != nullptr ? (int64_t)__ldg(p.cu_q + b) + qi : (int64_t)b;
}

// Attended length of sequence b (query qi of a varlen sequence sees the keys
// up to qi + Lk - Lq, bottom-right causal), clamped to what the block table and
// the workspace can hold (violations are flagged by the caller thread).
__device__ __forceinline__ int attended_length(const DecodeParams& p, int b, int qi, bool report) {
  int len;
  if (p.cu_k != nullptr) {
    const int lk = __ldg(p.cu_k + b + 1) - __ldg(p.cu_k + b);
    const int lq = __ldg(p.cu_q + b + 1) - __ldg(p.cu_q + b);
    len = qi + lk - lq + 1;
    if (len < 0 && lk >= 0) len = 0;  // a query that sees no key (not an error)
    if (len > lk) len = lk;
  } else {
    len = __ldg(p.seqlens + b);
  }
  if (p.k_new != nullptr && len >= 0) len += 1;  // the appended token
  const int64_t cap_bt = (int64_t)p.max_blocks * p.block_size;
  const int64_t cap_ws = (int64_t)p.max_splits * p.split_tokens;
  bool bad = false;
  if (len < 0) { len = 0; bad = true; }
  if ((int64_t)len > cap_bt) { len = (int)cap_bt; bad = true; }
  if ((int64_t)len > cap_ws) { len = (int)cap_ws; bad = true; }
  if (bad && report) flag_error(p.err, PKV_DEVERR_LENGTH);
  return len;
}

// Shared-memory layout of one staged 16-position tile of K or V (one kv head):
// TMA boxes of 16 rows x kBoxRow bytes, 128-byte swizzle for 128-byte rows
// (16-byte chunk c of row r at chunk c ^ (r & 7)), 64-byte swizzle for
// 64-byte rows (chunk c ^ ((r >> 1) & 3)); a 256-byte bf16 row is two boxes.
template <int kRowBytes>
struct TileLayout {
  static constexpr int kBoxRow = kRowBytes >= 128 ? 128 : kRowBytes;
  static constexpr int kBoxes = kRowBytes / kBoxRow;
  static constexpr int kBoxBytes = kGroupTok * kBoxRow;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  static constexpr int kChunksPerBox = kBoxRow / 16;
  static constexpr int kSwizzle = kBoxRow;  // 128 or 64 bytes
  __device__ __forceinline__ static int offset(int row, int chunk) {
    const int box = chunk / kChunksPerBox;
    const int cc = chunk % kChunksPerBox;
    const int sw = kChunksPerBox == 8 ? (cc ^ (row & 7)) : (cc ^ ((row >> 1) & 3));
    return box * kBoxBytes + row * kBoxRow + sw * 16;
  }
};

// kFp8: one-byte codes (E4M3, or INT8 when kInt8) widened to f16 for f16 MMAs.
// kNB: blocks of 8 rows on the MMAs' N side.  A row is a query head of the
// GQA group (plain decode: kNB = 1) or, for multi-query items (p.multi_q > 0),
// a (query, head) pair of the sequence: row r is query r / group, head
// r % group, and sees the positions up to its own bottom-right causal limit.
// Two row blocks need more registers: those kernels run 2 CTAs per SM.
template <int D, bool kFp8, int kStages, bool kInt8 = false, int kNB = 1>
__global__ void __launch_bounds__(kDecThreads, kFp8 && kNB == 1 ? kResidentCoded : kResidentBf16)
    paged_decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                              const DecodeParams p) {
  constexpr int kRowBytes = D * (kFp8 ? 1 : 2);  // one position, one kv head
  using TL = TileLayout<kRowBytes>;
  constexpr int kTileBytes = TL::kTileBytes;
  constexpr int kStageBytes = 2 * kTileBytes;     // K then V
  constexpr int kWarpBytes = kStages * kStageBytes;
  constexpr int kDT = D / 16;
  constexpr int kRows = 8 * kNB;                  // rows served by this CTA (at most)
  constexpr int kBoxElems = TL::kBoxRow / (kFp8 ? 1 : 2);
  // two one-byte codes (bytes 0..1, resp. 2..3, of a word) -> f16x2: E4M3
  // exactly; INT8 as 1152 + c (the permute alone), the excess taken off the
  // logits below (K) and the output in the merge (V)
  auto code_lo = [](uint32_t w) {
    return kInt8 ? prmt(w ^ 0x80808080u, 0x64646464u, 0x4140u) : e4m3x2_lo_to_f16x2(w);
  };
  auto code_hi = [](uint32_t w) {
    return kInt8 ? prmt(w ^ 0x80808080u, 0x64646464u, 0x4342u) : e4m3x2_hi_to_f16x2(w);
  };

  // The combine kernel may be scheduled as soon as every CTA of this grid has
  // started; it waits for this grid's completion before it reads anything.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = p.split_major ? blockIdx.z : blockIdx.x;
  const int kvh = blockIdx.y;
  const int z = p.split_major ? blockIdx.x : blockIdx.z;
  int qi;
  const int b = item_sequence(p, z, qi);
  if (b < 0) return;
  // multi-query item: the sequence's lq queries, each with its own limit
  const int lq = p.multi_q ? __ldg(p.cu_q + b + 1) - __ldg(p.cu_q + b) : 1;
  if (lq <= 0) return;
  const int64_t qrow_idx = item_row(p, b, qi);  // the item's first query row

  // the CTA's positions: those of its last query (the whole prefix)
  const int len = attended_length(p, b, p.multi_q ? lq - 1 : qi, split == 0 && kvh == 0 && threadIdx.x == 0);
  const int n_splits = (len + p.split_tokens - 1) / p.split_tokens;
  if (split >= (n_splits > 0 ? n_splits : 1)) return;
  const int t_begin = split * p.split_tokens;
#ifdef PKV_TEST_HOOKS
  const bool skip_lane = p.test_skip_group >= 0 && split == 0 && kvh == 0 && z == 0;
#endif
  const int t_end = min(t_begin + p.split_tokens, len);
  const int n_groups = t_end > t_begin ? (t_end - t_begin + kGroupTok - 1) / kGroupTok : 0;
  const int my_groups = n_groups > warp ? (n_groups - warp + kDecWarps - 1) / kDecWarps : 0;
  const int32_t* bt = p.block_table + (int64_t)b * p.max_blocks;
  const int n_rows = p.multi_q ? lq * p.group : p.group;  // rows of this item (<= kRows)

  uint8_t* wsm = smem + warp * kWarpBytes;
  const uint32_t wsm_u32 = smem_u32(wsm);
  // one mbarrier per stage of this warp, after all warps' stages
  const uint32_t bar0 = smem_u32(smem + kDecWarps * kWarpBytes) + warp * kStages * 8;
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  // ---- Q as the B operand (n = row lane/4 of each block, k = head dim) ----
  uint32_t qf[kNB][kDT][2];
  // positions this thread's rows see: rows 2j and 2j+1 of each block (masks of the S^T fragments)
  int lim_a[kNB], lim_b[kNB];
#pragma unroll
  for (int bk = 0; bk < kNB; ++bk) {
    const int r = bk * 8 + (lane >> 2);
    const int j = lane & 3;
    const int qr = p.multi_q ? r / p.group : 0;
    const int hh = p.multi_q ? r % p.group : r;
    const bool hv = r < n_rows;
    const uint16_t* qrow =
        p.q + ((qrow_idx + (hv ? qr : 0)) * p.num_heads + (int64_t)kvh * p.group + (hv ? hh : 0)) * D;
#pragma unroll
    for (int kk = 0; kk < kDT; ++kk) {
      if constexpr (!kFp8) {
        qf[bk][kk][0] = hv ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * j) : 0u;
        qf[bk][kk][1] = hv ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * j) : 0u;
      } else {
        // FP8 K fragments carry head dims 4j..4j+3 of each 16-wide slice in
        // k-slots {2j,2j+1,2j+8,2j+9}; Q uses the same permutation.
        const uint2 w = hv ? *reinterpret_cast<const uint2*>(qrow + kk * 16 + 4 * j) : make_uint2(0u, 0u);
        qf[bk][kk][0] = w.x;
        qf[bk][kk][1] = w.y;
      }
    }
    // row (query qr) sees positions < len - (lq - 1 - qr); rows past the item see none
    auto row_lim = [&](int rr) {
      if (rr >= n_rows) return 0;
      const int q_of = p.multi_q ? rr / p.group : 0;
      return len - (lq - 1 - q_of);
    };
    lim_a[bk] = min(t_end, row_lim(bk * 8 + 2 * j));
    lim_b[bk] = min(t_end, row_lim(bk * 8 + 2 * j + 1));
  }
  // FP8 cache: the MMAs run in f16 (E4M3 widens to f16 exactly).  Q goes from
  // bf16 to f16 scaled by a power of two 2^-e chosen so that its largest
  // magnitude stays below 2^14 (no overflow); 2^e is folded into the logit scale.
  float scale_log2 = p.scale_log2;
  if constexpr (kFp8) {
    float qmax = 0.f;
#pragma unroll
    for (int bk = 0; bk < kNB; ++bk)
#pragma unroll
      for (int kk = 0; kk < kDT; ++kk)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          qmax = fmaxf(qmax, fabsf(__uint_as_float(qf[bk][kk][h2] << 16)));
          qmax = fmaxf(qmax, fabsf(__uint_as_float(qf[bk][kk][h2] & 0xFFFF0000u)));
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
    int e = 0;
    if (qmax > 16384.f) e = (int)ceilf(log2f(qmax / 16384.f));  // qmax <= 2^14 * 2^e
    const float qs = exp2f((float)-e);
    scale_log2 *= exp2f((float)e);
#pragma unroll
    for (int bk = 0; bk < kNB; ++bk)
#pragma unroll
      for (int kk = 0; kk < kDT; ++kk)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
          qf[bk][kk][h2] = pack_f16x2(__uint_as_float(qf[bk][kk][h2] << 16) * qs,
                                      __uint_as_float(qf[bk][kk][h2] & 0xFFFF0000u) * qs);
  }
  // INT8: K codes widen to 1152 + c, so a score exceeds the one over the codes
  // by 1152 times the row's sum of (f16) Q; that excess, in logit units, per
  // row of this thread's S^T fragment (rows 2j, 2j+1 of each block)
  float kx_a[kNB], kx_b[kNB];
#pragma unroll
  for (int bk = 0; bk < kNB; ++bk) kx_a[bk] = kx_b[bk] = 0.f;
  if constexpr (kInt8) {
#pragma unroll
    for (int bk = 0; bk < kNB; ++bk) {
      float qsum = 0.f;  // this lane's head dims of row lane/4
#pragma unroll
      for (int kk = 0; kk < kDT; ++kk)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&qf[bk][kk][h2]));
          qsum += f.x + f.y;
        }
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);  // whole row, in every lane of its quad
      const int j = lane & 3;
      kx_a[bk] = kInt8Bias * __shfl_sync(0xffffffffu, qsum, 8 * j) * scale_log2;
      kx_b[bk] = kInt8Bias * __shfl_sync(0xffffffffu, qsum, 8 * j + 4) * scale_log2;
    }
  }

  auto block_of = [&](int pos0, bool report) -> int {
    const int blk = __ldg(bt + pos0 / p.block_size);
    if (blk < 0 || blk >= p.num_blocks) {
      if (report) flag_error(p.err, PKV_DEVERR_BLOCK);
      return -1;
    }
    return blk;
  };

  // Block ids of this warp's tiles: lane l holds that of tile blk_base + l,
  // loaded and checked 32 tiles at a time, so that a stage's copies wait on no
  // global load.  Bit s of stage_ok: the tile in stage s has a valid block.
  int blk_base = -32, blk_lane = -1;
  uint32_t stage_ok = 0;
  auto tile_block = [&](int i) -> int {  // (warp-uniform i, increasing)
    if (i >= blk_base + 32) {
      blk_base = i & ~31;
      const int ti = blk_base + lane;
      blk_lane = ti < my_groups ? block_of(t_begin + (warp + ti * kDecWarps) * kGroupTok, true) : -1;
    }
    return __shfl_sync(0xffffffffu, blk_lane, i & 31);
  };

  // Stage i's copies: one TMA box per 128-byte (or 64-byte) column slice of K
  // and of V; a bad block id issues nothing and just completes the phase.
  auto issue = [&](int i) {
    if (i >= my_groups) return;
    const int g = warp + i * kDecWarps;
    const int pos0 = t_begin + g * kGroupTok;
    const int blk = tile_block(i);
    const int st = i % kStages;
    stage_ok = blk >= 0 ? (stage_ok | (1u << st)) : (stage_ok & ~(1u << st));
    if (lane == 0) {
      const uint32_t bar = bar0 + 8 * st;
      const uint32_t dst = wsm_u32 + st * kStageBytes;
      fence_proxy_async_smem();  // order earlier generic writes (V tail zeroing) before the async copies
#ifdef PKV_TEST_HOOKS
      // test builds only: withhold this stage's copies and arrival, so that its wait runs out
      if (skip_lane && warp == 0 && i == p.test_skip_group) return;
#endif
      if (blk >= 0) {
        const int slot0 = blk * p.block_size + pos0 % p.block_size;
        mbar_expect_tx(bar, kStageBytes);
#pragma unroll
        for (int bx = 0; bx < TL::kBoxes; ++bx) {
          tma_load_3d(dst + bx * TL::kBoxBytes, &tm_k, bx * kBoxElems, kvh, slot0, bar);
          tma_load_3d(dst + kTileBytes + bx * TL::kBoxBytes, &tm_v, bx * kBoxElems, kvh, slot0, bar);
        }
      } else {
        mbar_arrive(bar);
      }
    }
  };

  float o[kNB][kDT][4];
  float m0[kNB], m1[kNB], l0[kNB], l1[kNB];
#pragma unroll
  for (int bk = 0; bk < kNB; ++bk) {
#pragma unroll
    for (int t = 0; t < kDT; ++t) o[bk][t][0] = o[bk][t][1] = o[bk][t][2] = o[bk][t][3] = 0.f;
    m0[bk] = m1[bk] = -INFINITY;
    l0[bk] = l1[bk] = 0.f;
  }

  // Append: the warp whose copies read the new position stores its K/V rows
  // for this kv head first (a generic write, then a proxy fence so the TMA
  // reads see it).  Skipped when the length was clamped (flagged above).
  if (p.k_new != nullptr && t_end == len && len > 0 && __ldg(p.seqlens + b) == len - 1) {
    const int pos = len - 1;
    if (warp == ((pos - t_begin) / kGroupTok) % kDecWarps) {
      const int blk = block_of(pos, lane == 0);
      constexpr int kChunks = D / 8;  // 16-byte bf16 vectors per head row
      if (blk >= 0 && lane < 2 * kChunks) {
        const bool is_v = lane >= kChunks;
        const int c = lane % kChunks;
        const int64_t slot = (int64_t)blk * p.block_size + pos % p.block_size;
        const uint16_t* src = (is_v ? p.v_new + b * p.v_new_stride : p.k_new + b * p.k_new_stride) + kvh * D;
        const uint4 w = *reinterpret_cast<const uint4*>(src + c * 8);
        uint8_t* row = const_cast<uint8_t*>(is_v ? p.v_cache : p.k_cache) +
                       (slot * p.num_kv_heads + kvh) * (int64_t)kRowBytes;
        if constexpr (kFp8)
          reinterpret_cast<uint2*>(row)[c] =
              kInt8 ? quantize8_int8(w, is_v ? p.v_inv : p.k_inv) : quantize8_e4m3(w, is_v ? p.v_inv : p.k_inv);
        else
          reinterpret_cast<uint4*>(row)[c] = w;
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      __syncwarp();
    }
  }

#pragma unroll
  for (int i = 0; i < kStages - 1; ++i) issue(i);

  int consumed = 0;
  for (int i = 0; i < my_groups; ++i) {
    const int st = i % kStages;
    if (!mbar_wait(bar0 + 8 * st, (i / kStages) & 1, nullptr)) {
      if (lane == 0) flag_error(p.err, PKV_DEVERR_TIMEOUT);
      break;
    }
    consumed = i + 1;
    // Many sequences (the sequence-major grid): refill now the stage this warp
    // finished with in the previous iteration (its lanes passed the __syncwarp
    // at that iteration's end), so that two tiles are in flight while this one
    // is computed (decode batch step +0.3 %, multi-query +0.2 %, same box).
    // Few long sequences (split-major) stream at the copy peak already and
    // lose 1-5 % with the extra copies in flight: they refill after the compute.
    if (!p.split_major) issue(i + kStages - 1);
    const int g = warp + i * kDecWarps;
    const int pos0 = t_begin + g * kGroupTok;
    const bool blk_ok = (stage_ok >> st) & 1u;
    uint8_t* stp = wsm + st * kStageBytes;
    const uint32_t ks = smem_u32(stp);
    const uint32_t vs = ks + kTileBytes;
    const int valid = t_end - pos0;  // rows of this group inside the sequence (may exceed 16)
    if (blk_ok && valid < kGroupTok) {
      // rows past the sequence end hold other positions' (or stale) values: zero V there
      for (int idx = lane; idx < kGroupTok * (kRowBytes / 16); idx += 32) {
        const int row = idx / (kRowBytes / 16);
        const int ch = idx % (kRowBytes / 16);
        if (row >= valid) *reinterpret_cast<uint4*>(stp + kTileBytes + TL::offset(row, ch)) = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }

    if (blk_ok) {
      // ---- S^T = K Q^T (16 positions x 8 rows per block) ----
      // two independent accumulator chains (even / odd 16-wide slices of the head dim)
      float s[kNB][4], s2[kNB][4];
#pragma unroll
      for (int bk = 0; bk < kNB; ++bk)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[bk][e] = s2[bk][e] = 0.f;
      {
        const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int csel = lane >> 4;
        if constexpr (!kFp8) {
#pragma unroll
          for (int kk = 0; kk < kDT; ++kk) {
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(ks + TL::offset(row, 2 * kk + csel), a0, a1, a2, a3);
#pragma unroll
            for (int bk = 0; bk < kNB; ++bk)
              mma_bf16_16816((kk & 1) ? s2[bk] : s[bk], a0, a1, a2, a3, qf[bk][kk][0], qf[bk][kk][1]);
          }
        } else {
#pragma unroll
          for (int pp = 0; pp < kDT / 2; ++pp) {
            uint32_t r0, r1, r2, r3;
            ldmatrix_x4(ks + TL::offset(row, 2 * pp + csel), r0, r1, r2, r3);
            const uint32_t e0 = code_lo(r0), e1 = code_lo(r1), e2 = code_hi(r0), e3 = code_hi(r1);
            const uint32_t f0 = code_lo(r2), f1 = code_lo(r3), f2 = code_hi(r2), f3 = code_hi(r3);
#pragma unroll
            for (int bk = 0; bk < kNB; ++bk) {
              mma_f16_16816(s[bk], e0, e1, e2, e3, qf[bk][2 * pp][0], qf[bk][2 * pp][1]);
              mma_f16_16816(s2[bk], f0, f1, f2, f3, qf[bk][2 * pp + 1][0], qf[bk][2 * pp + 1][1]);
            }
          }
        }
#pragma unroll
        for (int bk = 0; bk < kNB; ++bk)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[bk][e] += s2[bk][e];
      }

      // ---- online softmax (log2 domain); this thread: positions lane/4 (+8), rows 2j, 2j+1 ----
      // The reference max m moves only when the tile max exceeds it by more
      // than 2^8, so O is rescaled rarely; P stays below 2^8.
      const int tok0 = pos0 + (lane >> 2);
      uint32_t pb0[kNB], pb1[kNB];
#pragma unroll
      for (int bk = 0; bk < kNB; ++bk) {
        const float x0 = tok0 < lim_a[bk] ? fmaf(s[bk][0], scale_log2, -kx_a[bk]) : -INFINITY;
        const float x1 = tok0 < lim_b[bk] ? fmaf(s[bk][1], scale_log2, -kx_b[bk]) : -INFINITY;
        const float x2 = tok0 + 8 < lim_a[bk] ? fmaf(s[bk][2], scale_log2, -kx_a[bk]) : -INFINITY;
        const float x3 = tok0 + 8 < lim_b[bk] ? fmaf(s[bk][3], scale_log2, -kx_b[bk]) : -INFINITY;
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mu0 = (mx0 > m0[bk] + 8.f || (m0[bk] == -INFINITY && mx0 != -INFINITY)) ? mx0 : m0[bk];
        const float mu1 = (mx1 > m1[bk] + 8.f || (m1[bk] == -INFINITY && mx1 != -INFINITY)) ? mx1 : m1[bk];
        const bool live0 = mu0 != -INFINITY, live1 = mu1 != -INFINITY;
        const float p0 = live0 ? fast_exp2(x0 - mu0) : 0.f;
        const float p1 = live1 ? fast_exp2(x1 - mu1) : 0.f;
        const float p2 = live0 ? fast_exp2(x2 - mu0) : 0.f;
        const float p3 = live1 ? fast_exp2(x3 - mu1) : 0.f;
        if (__any_sync(0xffffffffu, (mu0 != m0[bk] && m0[bk] != -INFINITY) || (mu1 != m1[bk] && m1[bk] != -INFINITY))) {
          const float al0 = (mu0 != m0[bk] && m0[bk] != -INFINITY) ? fast_exp2(m0[bk] - mu0) : 1.f;
          const float al1 = (mu1 != m1[bk] && m1[bk] != -INFINITY) ? fast_exp2(m1[bk] - mu1) : 1.f;
          l0[bk] *= al0;
          l1[bk] *= al1;
#pragma unroll
          for (int t = 0; t < kDT; ++t) {
            o[bk][t][0] *= al0;
            o[bk][t][1] *= al1;
            o[bk][t][2] *= al0;
            o[bk][t][3] *= al1;
          }
        }
        m0[bk] = mu0;
        m1[bk] = mu1;
        l0[bk] += p0 + p2;
        l1[bk] += p1 + p3;
        // P as the B operand (k = position, n = row): positions 0..7, then 8..15
        pb0[bk] = movmatrix_trans(kFp8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1));
        pb1[bk] = movmatrix_trans(kFp8 ? pack_f16x2(p2, p3) : pack_bf16x2(p2, p3));
      }

      // ---- O^T += V^T P^T (V fragments shared by the row blocks) ----
      {
        const int row = (lane & 7) + (lane >> 4) * 8;
        const int csel = (lane >> 3) & 1;
        if constexpr (!kFp8) {
#pragma unroll
          for (int t = 0; t < kDT; ++t) {
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4_trans(vs + TL::offset(row, 2 * t + csel), a0, a1, a2, a3);
#pragma unroll
            for (int bk = 0; bk < kNB; ++bk) mma_bf16_16816(o[bk][t], a0, a1, a2, a3, pb0[bk], pb1[bk]);
          }
        } else {
#pragma unroll
          for (int pp = 0; pp < kDT / 2; ++pp) {
            uint32_t r0, r1, r2, r3;
            ldmatrix_x4_trans(vs + TL::offset(row, 2 * pp + csel), r0, r1, r2, r3);
            // r: bytes (pos 2j, dim 2u), (2j, 2u+1), (2j+1, 2u), (2j+1, 2u+1); widen
            // bytes {0, 2} (even dim, both positions), then {1, 3} (odd dim).  INT8
            // picks them in its widening permute; E4M3 reorders the word first.
            uint32_t ev[4], od[4];
            if constexpr (kInt8) {
              // V codes widen to 1152 + c (no subtract): O then exceeds the sum
              // over the codes by 1152 l, since O and l are always scaled
              // together; the merge below takes 1152 L off once
              const uint32_t x0 = r0 ^ 0x80808080u, x1 = r1 ^ 0x80808080u;
              const uint32_t x2 = r2 ^ 0x80808080u, x3 = r3 ^ 0x80808080u;
              ev[0] = prmt(x0, 0x64646464u, 0x4240u); ev[1] = prmt(x1, 0x64646464u, 0x4240u);
              ev[2] = prmt(x2, 0x64646464u, 0x4240u); ev[3] = prmt(x3, 0x64646464u, 0x4240u);
              od[0] = prmt(x0, 0x64646464u, 0x4341u); od[1] = prmt(x1, 0x64646464u, 0x4341u);
              od[2] = prmt(x2, 0x64646464u, 0x4341u); od[3] = prmt(x3, 0x64646464u, 0x4341u);
            } else {
              const uint32_t t0 = prmt(r0, 0u, 0x3120u), t1 = prmt(r1, 0u, 0x3120u);
              const uint32_t t2 = prmt(r2, 0u, 0x3120u), t3 = prmt(r3, 0u, 0x3120u);
              ev[0] = code_lo(t0); ev[1] = code_lo(t1); ev[2] = code_lo(t2); ev[3] = code_lo(t3);
              od[0] = code_hi(t0); od[1] = code_hi(t1); od[2] = code_hi(t2); od[3] = code_hi(t3);
            }
#pragma unroll
            for (int bk = 0; bk < kNB; ++bk) {
              mma_f16_16816(o[bk][2 * pp], ev[0], ev[1], ev[2], ev[3], pb0[bk], pb1[bk]);
              mma_f16_16816(o[bk][2 * pp + 1], od[0], od[1], od[2], od[3], pb0[bk], pb1[bk]);
            }
          }
        }
      }
    }
    __syncwarp();  // every lane is done with this stage before it is refilled
    if (p.split_major) issue(i + kStages - 1);
  }
  // copies issued but never consumed (only after a timeout) land before the
  // shared memory is reused; if one of them does not land in time either, the
  // CTA writes nothing (its results are undefined, PKV_DEVERR_TIMEOUT is set)
  bool drained = true;
  for (int i = consumed; i < min(my_groups, consumed + kStages - 1); ++i)
    if (!mbar_wait(bar0 + 8 * (i % kStages), (i / kStages) & 1, nullptr)) drained = false;
  if (__syncthreads_or(!drained)) return;

  // ---- merge the four warps of the CTA ----
#pragma unroll
  for (int bk = 0; bk < kNB; ++bk)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0[bk] += __shfl_xor_sync(0xffffffffu, l0[bk], off);
      l1[bk] += __shfl_xor_sync(0xffffffffu, l1[bk], off);
    }
  float* m_s = reinterpret_cast<float*>(smem);           // [warps][rows]
  float* l_s = m_s + kDecWarps * kRows;                   // [warps][rows]
  float* o_s = l_s + kDecWarps * kRows;                   // [warps][rows][D]
  {
    const int j = lane & 3;
    const int r = lane >> 2;
#pragma unroll
    for (int bk = 0; bk < kNB; ++bk) {
      if (lane < 4) {
        m_s[warp * kRows + bk * 8 + 2 * j] = m0[bk];
        m_s[warp * kRows + bk * 8 + 2 * j + 1] = m1[bk];
        l_s[warp * kRows + bk * 8 + 2 * j] = l0[bk];
        l_s[warp * kRows + bk * 8 + 2 * j + 1] = l1[bk];
      }
      float* ow = o_s + (warp * kRows + bk * 8) * D;
#pragma unroll
      for (int t = 0; t < kDT; ++t) {
        int d0, d1;
        if constexpr (!kFp8) {
          d0 = 16 * t + r;
          d1 = d0 + 8;
        } else {
          d0 = 32 * (t >> 1) + 2 * r + (t & 1);
          d1 = d0 + 16;
        }
        ow[(2 * j) * D + d0] = o[bk][t][0];
        ow[(2 * j + 1) * D + d0] = o[bk][t][1];
        ow[(2 * j) * D + d1] = o[bk][t][2];
        ow[(2 * j + 1) * D + d1] = o[bk][t][3];
      }
    }
  }
  __syncthreads();
  const bool single = n_splits <= 1;
  const int qpi = p.multi_q ? p.multi_q : 1;  // query rows per item in the partials
  for (int idx = threadIdx.x; idx < n_rows * D; idx += kDecThreads) {
    const int r = idx / D;
    const int d = idx % D;
    float ms = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) ms = fmaxf(ms, m_s[w * kRows + r]);
    float L = 0.f, acc = 0.f;
    if (ms != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float mw = m_s[w * kRows + r];
        const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - ms);
        L += l_s[w * kRows + r] * f;
        acc += o_s[(w * kRows + r) * D + d] * f;
      }
    }
    const bool any = L > 0.f;
    if constexpr (kInt8) acc -= kInt8Bias * L;  // the V codes were widened to 1152 + c
    const float val = any ? acc * p.v_mul / L : 0.f;
    const float lse2 = any ? ms + log2f(L) : -INFINITY;
    const int qr = p.multi_q ? r / p.group : 0;
    const int hq = kvh * p.group + (p.multi_q ? r % p.group : r);
    const int64_t orow = qrow_idx + qr;
    // partials are indexed by grid item, query of the item and head
    const int64_t bh = ((int64_t)z * qpi + qr) * p.num_heads + hq;
    if (single) {
      p.out[(orow * p.num_heads + hq) * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
      if (p.lse != nullptr && d == 0)
        p.lse[hq * p.lse_head_stride + orow * p.lse_row_stride] = any ? lse2 * kLn2 : -INFINITY;
    } else {
      p.ws_o[(bh * p.max_splits + split) * D + d] = val;
      if (d == 0) p.ws_lse[bh * p.max_splits + split] = lse2;
    }
  }
}

// One warp per (item, query of the item, query head): merge the splits by log-sum-exp.
template <int D>
__global__ void __launch_bounds__(128) paged_decode_combine_kernel(const DecodeParams p, int batch) {
  // launched as a programmatic dependent of the split kernel: wait until that
  // grid has completed and its partials are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qpi = p.multi_q ? p.multi_q : 1;
  const int64_t bh = (int64_t)blockIdx.x * 4 + warp;
  if (bh >= (int64_t)batch * qpi * p.num_heads) return;
  const int z = (int)(bh / ((int64_t)qpi * p.num_heads));
  const int qr = (int)((bh / p.num_heads) % qpi);
  const int hq = (int)(bh % p.num_heads);
  int qi;
  const int b = item_sequence(p, z, qi);
  if (b < 0) return;
  const int lq = p.multi_q ? __ldg(p.cu_q + b + 1) - __ldg(p.cu_q + b) : 1;
  if (qr >= lq) return;
  const int64_t row = item_row(p, b, qi) + qr;
  // the split kernel's CTAs cover the positions of the item's last query
  const int len = attended_length(p, b, p.multi_q ? lq - 1 : qi, false);
  const int n = (len + p.split_tokens - 1) / p.split_tokens;
  if (n <= 1) return;
  const float* ls = p.ws_lse + bh * p.max_splits;
  float mx = -INFINITY;
  for (int s = lane; s < n; s += 32) mx = fmaxf(mx, ls[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float sum = 0.f;
  if (mx != -INFINITY)
    for (int s = lane; s < n; s += 32) sum += fast_exp2(ls[s] - mx);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const bool any = mx != -INFINITY && sum > 0.f;
  const float lse2 = any ? mx + log2f(sum) : -INFINITY;
  constexpr int kPer = D / 32;
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  if (any) {
    const float* os = p.ws_o + bh * p.max_splits * D + lane * kPer;
    for (int s = 0; s < n; ++s) {
      const float w = fast_exp2(ls[s] - lse2);
      if constexpr (kPer == 4) {
        const float4 v = *reinterpret_cast<const float4*>(os + (int64_t)s * D);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
        acc[2] += w * v.z;
        acc[3] += w * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(os + (int64_t)s * D);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
      }
    }
  }
  uint16_t* orow = p.out + (row * p.num_heads + hq) * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; ++e) orow[e] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[e]));
  if (p.lse != nullptr && lane == 0)
    p.lse[hq * p.lse_head_stride + row * p.lse_row_stride] = any ? lse2 * kLn2 : -INFINITY;
}

struct SplitPlan {
  int split_tokens;
  int max_splits;
  size_t workspace;
  // launch the split kernel as a programmatic dependent of the kernel before
  // it on the stream (which reads nothing it writes): its CTAs then start on
  // SMs that kernel's CTAs have left
  bool after_primary = false;
  // grid order: split index slowest (few, long sequences: each wave then
  // spreads over every sequence; long-context decode +1 %), else fastest
  // (many sequences of mixed lengths: a sequence's splits run side by side)
  bool split_major = false;
};

// Positions per CTA (split_tokens), a multiple of 64 (4 warps x 16), at least
// 512.  A resident slot is one CTA on one SM (SMs x CTAs per SM for the cache's
// element size), and a wave fills every slot once.
//  * Fewer (sequence, kv head) units than SMs: the sequences are few and long,
//    taken as equally long.  Each candidate split count is costed as
//    waves x (split_tokens + a fixed per-CTA cost), which favours splits that
//    end on a whole wave and penalises many short CTAs (measured on 8 x 128K
//    contexts: bf16 6.47 -> 6.64 TB/s, FP8 5.82 -> 5.88 TB/s against 8 waves of
//    2 CTAs per SM).
//  * Otherwise the lengths are mixed and unknown on the host: about 16 CTAs
//    per SM at the longest length, which leaves the short sequences one CTA
//    (measured on 64 sequences of 1K..16K: 6.41 TB/s at 32, 6.47-6.50 at 16,
//    6.38 at 12; for 64 sequences x 4 queries, whose items carry two row
//    blocks, 0.383 ms at 16 and 0.395 at 8).
constexpr int64_t kCtaOverheadPos = 96;  // prologue + merge of one CTA, in positions of streaming time
constexpr int64_t kCtasPerSmMixed = 16;

int resident_ctas(int cache_dtype) { return cache_dtype == PKV_BF16 ? kResidentBf16 : kResidentCoded; }

SplitPlan plan_split(int batch, int num_heads, int num_kv_heads, int head_dim, int max_seqlen_k, int cache_dtype) {
  SplitPlan pl{64, 1, 0};
  if (batch <= 0 || max_seqlen_k <= 0) return pl;
  const int64_t units = (int64_t)batch * num_kv_heads;
  const int64_t sms = device_sm_count();
  const int64_t L = max_seqlen_k;
  const int64_t whole = (L + 63) / 64 * 64;
  auto clamp_split = [&](int64_t c) {  // multiple of 64, at least 512, at most the whole sequence
    c = (c + 63) / 64 * 64;
    if (c < 512) c = 512;
    return c < whole ? c : whole;
  };
  int64_t c;
  if (whole <= 512) {
    c = whole;
  } else if (units < sms) {
    pl.split_major = true;
    const int64_t slots = sms * resident_ctas(cache_dtype);
    const int64_t n_max = 8 * slots / units + 1;  // beyond 8 waves' worth of splits nothing is gained
    c = whole;
    int64_t best = INT64_MAX;
    for (int64_t n = 1; n <= n_max; ++n) {
      const int64_t cn = clamp_split((L + n - 1) / n);
      const int64_t splits = (L + cn - 1) / cn;
      const int64_t waves = (units * splits + slots - 1) / slots;
      const int64_t cost = waves * (cn + kCtaOverheadPos);
      if (cost < best) {
        best = cost;
        c = cn;
      }
      if (cn == 512) break;  // every larger n gives the same split
    }
  } else {
    const int64_t target = sms * kCtasPerSmMixed;
    c = clamp_split((L * units + target - 1) / target);
  }
  pl.split_tokens = (int)c;
  pl.max_splits = (int)((max_seqlen_k + c - 1) / c);
  if (pl.max_splits > 1) {
    const size_t rows = (size_t)batch * num_heads * pl.max_splits;
    pl.workspace = rows * head_dim * sizeof(float) + ((rows * sizeof(float) + 255) / 256) * 256;
  }
  return pl;
}

template <int D, bool kFp8, bool kInt8 = false, int kNB = 1>
int launch_decode(const DecodeParams& p, int batch, const SplitPlan& pl, int64_t num_slots, cudaStream_t st) {
  constexpr int kStages = 3;  // shared memory for kResidentCoded (one-byte codes) or kResidentBf16 CTAs per SM
  constexpr int kRowBytes = D * (kFp8 ? 1 : 2);
  using TL = TileLayout<kRowBytes>;
  constexpr int kSmemPipe = kDecWarps * kStages * 2 * TL::kTileBytes + kDecWarps * kStages * 8;
  constexpr int kRows = 8 * kNB;
  constexpr int kSmemMerge = (2 * kDecWarps * kRows + kDecWarps * kRows * D) * (int)sizeof(float);
  constexpr int kSmem = (kSmemPipe > kSmemMerge ? kSmemPipe : kSmemMerge) + 1024;
  CUtensorMap mk, mv;
  const int box_elems = TL::kBoxRow / (kFp8 ? 1 : 2);
  if (!make_tmap_3d(&mk, p.k_cache, kFp8 ? 1 : 2, num_slots, p.num_kv_heads, D, box_elems, kGroupTok, TL::kSwizzle) ||
      !make_tmap_3d(&mv, p.v_cache, kFp8 ? 1 : 2, num_slots, p.num_kv_heads, D, box_elems, kGroupTok, TL::kSwizzle))
    return PKV_ERR_CUDA;
  auto kern = paged_decode_split_kernel<D, kFp8, kStages, kInt8, kNB>;
  static bool attr_set[64] = {false};  // per instantiation and device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= 64) dev = 63;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
      return PKV_ERR_CUDA;
    attr_set[dev] = true;
  }
  const dim3 grid = pl.split_major ? dim3(batch, p.num_kv_heads, pl.max_splits)
                                   : dim3(pl.max_splits, p.num_kv_heads, batch);
  if (pl.after_primary) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, mk, mv, p) != cudaSuccess) return PKV_ERR_CUDA;
  } else {
    kern<<<grid, kDecThreads, kSmem, st>>>(mk, mv, p);
  }
  if (pl.max_splits > 1) {
    // programmatic dependent launch: the combine grid's launch overlaps the
    // split kernel's last wave instead of following its completion
    const int64_t rows = (int64_t)batch * (p.multi_q ? p.multi_q : 1) * p.num_heads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, paged_decode_combine_kernel<D>, p, batch) != cudaSuccess) return PKV_ERR_CUDA;
  }
  return launch_status();
}

template <int kNB>
int dispatch_decode_rows(int cache_dtype, int head_dim, const DecodeParams& p, int batch, const SplitPlan& pl,
                         int64_t ns, cudaStream_t st) {
  if (head_dim == 128) {
    if (cache_dtype == PKV_FP8_E4M3) return launch_decode<128, true, false, kNB>(p, batch, pl, ns, st);
    if (cache_dtype == PKV_INT8) return launch_decode<128, true, true, kNB>(p, batch, pl, ns, st);
    return launch_decode<128, false, false, kNB>(p, batch, pl, ns, st);
  }
  if (cache_dtype == PKV_FP8_E4M3) return launch_decode<64, true, false, kNB>(p, batch, pl, ns, st);
  if (cache_dtype == PKV_INT8) return launch_decode<64, true, true, kNB>(p, batch, pl, ns, st);
  return launch_decode<64, false, false, kNB>(p, batch, pl, ns, st);
}

int dispatch_decode(int cache_dtype, int head_dim, const DecodeParams& p, int batch, const SplitPlan& pl,
                    int64_t ns, cudaStream_t st) {
  if (head_dim == 128) {
    if (cache_dtype == PKV_FP8_E4M3) return launch_decode<128, true>(p, batch, pl, ns, st);
    if (cache_dtype == PKV_INT8) return launch_decode<128, true, true>(p, batch, pl, ns, st);
    return launch_decode<128, false>(p, batch, pl, ns, st);
  }
  if (cache_dtype == PKV_FP8_E4M3) return launch_decode<64, true>(p, batch, pl, ns, st);
  if (cache_dtype == PKV_INT8) return launch_decode<64, true, true>(p, batch, pl, ns, st);
  return launch_decode<64, false>(p, batch, pl, ns, st);
}

}  // namespace
}  // namespace pkv

extern "C" size_t pkv_paged_attn_decode_workspace(int32_t batch, int32_t num_heads, int32_t num_kv_heads,
                                                  int32_t head_dim, int32_t max_seqlen_k) {
  if (batch <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_seqlen_k <= 0) return 0;
  // enough for every cache element type (their plans differ in CTAs per SM)
  const size_t a = pkv::plan_split(batch, num_heads, num_kv_heads, head_dim, max_seqlen_k, PKV_BF16).workspace;
  const size_t b = pkv::plan_split(batch, num_heads, num_kv_heads, head_dim, max_seqlen_k, PKV_INT8).workspace;
  return a > b ? a : b;
}

namespace pkv {
namespace {

#ifdef PKV_TEST_HOOKS
int g_test_skip_group = -1;
#endif

struct AppendArgs {
  const void* k_new;
  int64_t k_new_stride;
  const void* v_new;
  int64_t v_new_stride;
  float k_inv, v_inv;
};

int decode_impl(const void* q, const void* k_cache, const void* v_cache, int32_t cache_dtype,
                                     const int32_t* cache_seqlens, const int32_t* block_table,
                                     int32_t max_blocks_per_seq, int32_t batch, int32_t num_heads,
                                     int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                     int32_t num_blocks, int32_t max_seqlen_k, float scale, float k_scale,
                                     float v_scale, void* out, float* lse, void* workspace,
                                     size_t workspace_bytes, int32_t* err_flag, void* stream, const AppendArgs* app) {
  if (batch < 0 || num_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
      max_seqlen_k < 0 || block_size <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (num_heads / num_kv_heads > kMaxGroup) return PKV_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (block_size % 16 != 0) return PKV_ERR_UNSUPPORTED;
  if (cache_dtype != PKV_BF16 && cache_dtype != PKV_FP8_E4M3 && cache_dtype != PKV_INT8) return PKV_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (cache_dtype != PKV_BF16 && (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) ||
                                  !std::isfinite(v_scale)))
    return PKV_ERR_INVALID_ARG;
  if (batch == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !cache_seqlens || !block_table || !out) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || (reinterpret_cast<uintptr_t>(q) & 7u) ||
      (reinterpret_cast<uintptr_t>(out) & 7u))
    return PKV_ERR_INVALID_ARG;
  const int mlen = max_seqlen_k > 0 ? max_seqlen_k : 1;
  const SplitPlan pl = plan_split(batch, num_heads, num_kv_heads, head_dim, mlen, cache_dtype);
  if (pl.workspace > 0 && (workspace == nullptr || workspace_bytes < pl.workspace ||
                           (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return PKV_ERR_WORKSPACE;

  DecodeParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.seqlens = cache_seqlens;
  p.block_table = block_table;
  p.max_blocks = max_blocks_per_seq;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.split_tokens = pl.split_tokens;
  p.max_splits = pl.max_splits;
  p.split_major = pl.split_major ? 1 : 0;
  const bool coded = cache_dtype != PKV_BF16;  // one-byte codes with per-tensor scales
  p.scale_log2 = scale * kLog2e * (coded ? k_scale : 1.f);
  p.v_mul = coded ? v_scale : 1.f;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  if (pl.max_splits > 1) {
    const size_t rows = (size_t)batch * num_heads * pl.max_splits;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + rows * head_dim * sizeof(float));
  }
  p.err = err_flag;
  p.lse_head_stride = 1;
  p.lse_row_stride = num_heads;
  if (app != nullptr) {
    p.k_new = static_cast<const uint16_t*>(app->k_new);
    p.v_new = static_cast<const uint16_t*>(app->v_new);
    p.k_new_stride = app->k_new_stride;
    p.v_new_stride = app->v_new_stride;
    p.k_inv = app->k_inv;
    p.v_inv = app->v_inv;
  }
  cudaStream_t st = as_stream(stream);
  const int64_t ns = (int64_t)num_blocks * block_size;
#ifdef PKV_TEST_HOOKS
  p.test_skip_group = g_test_skip_group;
#endif
  return dispatch_decode(cache_dtype, head_dim, p, batch, pl, ns, st);
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_paged_attn_decode(const void* q, const void* k_cache, const void* v_cache, int32_t cache_dtype,
                                     const int32_t* cache_seqlens, const int32_t* block_table,
                                     int32_t max_blocks_per_seq, int32_t batch, int32_t num_heads,
                                     int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                     int32_t num_blocks, int32_t max_seqlen_k, float scale, float k_scale,
                                     float v_scale, void* out, float* lse, void* workspace,
                                     size_t workspace_bytes, int32_t* err_flag, void* stream) {
  const pkv::NvtxRange nvtx_range("pkv_paged_attn_decode");
  return pkv::decode_impl(q, k_cache, v_cache, cache_dtype, cache_seqlens, block_table, max_blocks_per_seq, batch,
                          num_heads, num_kv_heads, head_dim, block_size, num_blocks, max_seqlen_k, scale, k_scale,
                          v_scale, out, lse, workspace, workspace_bytes, err_flag, stream, nullptr);
}

extern "C" int pkv_paged_attn_decode_with_kvcache(const void* q, const void* k_new, int64_t k_new_row_stride,
                                                  const void* v_new, int64_t v_new_row_stride, void* k_cache,
                                                  void* v_cache, int32_t cache_dtype, const int32_t* cache_seqlens,
                                                  const int32_t* block_table, int32_t max_blocks_per_seq,
                                                  int32_t batch, int32_t num_heads, int32_t num_kv_heads,
                                                  int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                                  int32_t max_seqlen_k, float scale, float k_scale, float v_scale,
                                                  float k_inv_scale, float v_inv_scale, void* out, float* lse,
                                                  void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                                  void* stream) {
  const pkv::NvtxRange nvtx_range("pkv_paged_attn_decode_with_kvcache");
  using namespace pkv;
  // a one-byte cache needs finite positive inverse scales, even when there is nothing to do
  if (cache_dtype != PKV_BF16 && (!(k_inv_scale > 0.f) || !(v_inv_scale > 0.f) || !std::isfinite(k_inv_scale) ||
                                  !std::isfinite(v_inv_scale)))
    return PKV_ERR_INVALID_ARG;
  if (batch > 0) {
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (!k_new || !v_new) return PKV_ERR_INVALID_ARG;
    if (k_new_row_stride < row || v_new_row_stride < row || k_new_row_stride % 8 || v_new_row_stride % 8)
      return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_INVALID_ARG;
  }
  const AppendArgs app{k_new, k_new_row_stride, v_new, v_new_row_stride, k_inv_scale, v_inv_scale};
  return decode_impl(q, k_cache, v_cache, cache_dtype, cache_seqlens, block_table, max_blocks_per_seq, batch,
                     num_heads, num_kv_heads, head_dim, block_size, num_blocks, max_seqlen_k, scale, k_scale, v_scale,
                     out, lse, workspace, workspace_bytes, err_flag, stream, &app);
}

namespace pkv {

// Partials of `items` routed rows, split as a decode batch of `batch` sequences would be.
size_t varlen_decode_workspace(int batch, int items, int num_heads, int num_kv_heads, int head_dim, int max_len_k,
                               int cache_dtype, int multi_q) {
  if (batch <= 0 || items <= 0 || max_len_k <= 0) return 0;
  const SplitPlan pl = plan_split(batch, num_heads, num_kv_heads, head_dim, max_len_k, cache_dtype);
  if (pl.max_splits <= 1) return 0;
  const size_t rows = (size_t)items * (multi_q > 0 ? multi_q : 1) * num_heads * pl.max_splits;
  return rows * head_dim * sizeof(float) + ((rows * sizeof(float) + 255) / 256) * 256;
}

// Decode kernels over the routed query rows of a paged varlen batch
// (items[0..*item_count) on the device, at most `items` of them); the split
// size is planned for `batch` sequences.
int launch_varlen_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* items,
                         const int32_t* item_count, const int32_t* cu_q, const int32_t* cu_k,
                         const int32_t* block_table, int32_t max_blocks_per_seq, int32_t batch, int32_t item_bound,
                         int32_t num_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                         int32_t max_len_k, int64_t total_q, float scale, int cache_dtype, float k_scale,
                         float v_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                         int32_t* err_flag, int32_t multi_q, bool after_primary, cudaStream_t st) {
  const bool fp8 = cache_dtype != PKV_BF16;  // one-byte codes
  if (num_heads / num_kv_heads > kMaxGroup || block_size % 16 != 0) return PKV_ERR_UNSUPPORTED;
  SplitPlan pl = plan_split(batch, num_heads, num_kv_heads, head_dim, max_len_k > 0 ? max_len_k : 1, cache_dtype);
  pl.after_primary = after_primary;
  if (varlen_decode_workspace(batch, item_bound, num_heads, num_kv_heads, head_dim, max_len_k > 0 ? max_len_k : 1,
                              cache_dtype, multi_q) > workspace_bytes)
    return PKV_ERR_WORKSPACE;
  DecodeParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_table = block_table;
  p.max_blocks = max_blocks_per_seq;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.split_tokens = pl.split_tokens;
  p.max_splits = pl.max_splits;
  p.split_major = pl.split_major ? 1 : 0;
  p.scale_log2 = scale * kLog2e * (fp8 ? k_scale : 1.f);
  p.v_mul = fp8 ? v_scale : 1.f;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  if (pl.max_splits > 1) {
    const size_t rows = (size_t)item_bound * (multi_q > 0 ? multi_q : 1) * num_heads * pl.max_splits;
    p.ws_o = static_cast<float*>(workspace);
    p.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + rows * head_dim * sizeof(float));
  }
  p.err = err_flag;
  p.items = items;
  p.item_count = item_count;
  p.cu_q = cu_q;
  p.cu_k = cu_k;
  p.lse_head_stride = total_q;
  p.lse_row_stride = 1;
  p.multi_q = multi_q;
  const int64_t ns = (int64_t)num_blocks * block_size;
  if (multi_q > 0) {
    // (query, head) rows of a sequence in blocks of 8 on the MMAs' N side
    const int rows = multi_q * p.group;
    if (rows > kMultiRows) return PKV_ERR_UNSUPPORTED;
    if (multi_query_row_blocks(multi_q, p.group) > 1)
      return dispatch_decode_rows<2>(cache_dtype, head_dim, p, item_bound, pl, ns, st);
    return dispatch_decode_rows<1>(cache_dtype, head_dim, p, item_bound, pl, ns, st);
  }
  return dispatch_decode(cache_dtype, head_dim, p, item_bound, pl, ns, st);
}

}  // namespace pkv

// ---------------------------------------------------------------------------
// Decode for callers that cannot allocate device memory.
//
// The split-KV partials live in one file-scope device array of fixed size
// instead of a caller workspace.  Every GPU that loads this library holds the
// array until the process exits.  Its device address is looked up once per
// device (cudaGetSymbolAddress, with that device current) by the first call
// made on that device; make that first call before any stream capture.  The
// cached address is valid while the device's primary context lives (a
// cudaDeviceReset ends it, and the module may then load at another address).
// Every call shares the array and finds the previous call's partials in it;
// nothing in it needs to start at zero (each call writes every partial it
// reads), but two calls that overlap on the GPU, on different streams,
// overwrite each other's partials.
// ---------------------------------------------------------------------------

#include <mutex>

static constexpr size_t kPkvFixedScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char pkv_decode_fixed_scratch[kPkvFixedScratchBytes];

namespace {

std::mutex g_fixed_scratch_mu;
void* g_fixed_scratch_addr[64] = {nullptr};

int fixed_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= 64) return PKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_fixed_scratch_mu);
  if (g_fixed_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, pkv_decode_fixed_scratch) != cudaSuccess || p == nullptr) return PKV_ERR_CUDA;
    g_fixed_scratch_addr[dev] = p;
  }
  *out = g_fixed_scratch_addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" size_t pkv_paged_attn_decode_noalloc_max_scratch(void) { return kPkvFixedScratchBytes; }

extern "C" int pkv_paged_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                             int32_t cache_dtype, const int32_t* cache_seqlens,
                                             const int32_t* block_table, int32_t max_blocks_per_seq, int32_t batch,
                                             int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                             int32_t block_size, int32_t num_blocks, int32_t max_seqlen_k,
                                             float scale, float k_scale, float v_scale, void* out, float* lse,
                                             int32_t* err_flag, void* stream) {
  const size_t need = pkv_paged_attn_decode_workspace(batch, num_heads, num_kv_heads, head_dim, max_seqlen_k);
  if (need > kPkvFixedScratchBytes) return PKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = fixed_scratch_address(&scratch);
  if (st != PKV_OK) return st;
  return pkv_paged_attn_decode(q, k_cache, v_cache, cache_dtype, cache_seqlens, block_table, max_blocks_per_seq,
                               batch, num_heads, num_kv_heads, head_dim, block_size, num_blocks, max_seqlen_k, scale,
                               k_scale, v_scale, out, lse, scratch, kPkvFixedScratchBytes, err_flag, stream);
}

#ifdef PKV_TEST_HOOKS
// Test builds only: the next decode calls withhold the copies of 16-position
// group `group` of warp 0 in CTA (split 0, kv head 0, sequence 0), so that its
// bounded wait runs out (-1 restores normal operation).
extern "C" PKV_API void pkv_test_decode_skip_group(int group) { pkv::g_test_skip_group = group; }
#endif
