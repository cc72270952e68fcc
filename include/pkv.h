/*
 * pkv.h -- C ABI of libpkv, paged KV-cache attention for one NVIDIA GB300 (sm_103a).
 *
 * The operations, in the order a serving layer calls them for one step:
 *
 *   pkv_kv_cache_write      scatter each new token's K/V row into the paged cache
 *   pkv_paged_attn_decode   one query token per sequence over its paged cache
 *   pkv_paged_attn_decode_with_kvcache  the write and the decode in one launch
 *   pkv_paged_attn_varlen   causal GQA attention over packed variable-length
 *                           sequences, K/V packed or read from the paged cache
 *   pkv_copy_blocks         copy-on-write of shared cache blocks
 *
 * Sources (web pages, by title and section):
 *   [KVM]  "効率的な KV キャッシュ管理と Attention 計算" (itan.pw): "Triton カーネルによる
 *          KV キャッシュ書き込み" (the write), "Python 層からのカーネル呼び出し" (its shape
 *          and stride checks), "Attention モジュールの実装" (write first, then varlen
 *          attention for prefill or paged attention for decode).
 *   [PA]   "ページド・アテンション" (transformers docs): "Varlen パス" (cu_seq_lens,
 *          max lengths) and "デコードパス" (block_table, cache_seqlens).
 *   [CH15] "KV cache / batching / paged attention" (1s.xyz, chapter 15): FP8 KV
 *          halves the cache ("KVキャッシュはどれくらいメモリを食う？"), GQA, PagedAttention,
 *          prefix caching / chunked prefill, FlashAttention (tiling is exact).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument is a DEVICE pointer owned by the caller, except
 *   where a comment says "host".  The library allocates no memory; scratch
 *   space ("workspace") is passed in and sized by the matching *_workspace call.
 * - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *   NULL = the legacy default stream).  No call synchronises the device or
 *   reads device data on the host, so calls can be captured in a CUDA graph.
 * - Head layout: q/k/v rows are [heads, head_dim] contiguous, head_dim innermost.
 *   A cache is [num_blocks, block_size, num_kv_heads, head_dim] contiguous,
 *   i.e. a flat array of num_slots = num_blocks*block_size rows of
 *   num_kv_heads*head_dim elements; slot = block*block_size + offset.
 * - GQA: query head h reads kv head h / (num_heads / num_kv_heads).
 * - Supported: head_dim 64 or 128; num_heads a multiple of num_kv_heads with
 *   num_heads/num_kv_heads <= 8 for decode; block_size a multiple of 16 for
 *   the paged attention calls (any >= 1 for the write).
 * - Return value: a pkv_status.  Host-visible argument problems return
 *   PKV_ERR_INVALID_ARG / PKV_ERR_UNSUPPORTED / PKV_ERR_WORKSPACE before any
 *   launch; a failed launch returns PKV_ERR_CUDA.
 * - Device metadata (slots, block ids, lengths) is never trusted blindly:
 *   a slot >= num_slots, a block id outside [0, num_blocks) or a length that
 *   does not fit the block table is skipped (never dereferenced) and, when
 *   `err_flag` is non-NULL, sets bits of *err_flag (an int32 in device memory,
 *   OR-ed atomically; PKV_DEVERR_* below).  Clear it before the call to read it.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad stride */
  PKV_ERR_UNSUPPORTED = 2, /* dtype, head_dim, group size or block size not built */
  PKV_ERR_WORKSPACE = 3,   /* workspace pointer NULL or smaller than required */
  PKV_ERR_CUDA = 4         /* a kernel launch or a driver call failed */
} pkv_status;

/* Element types.  Queries, outputs and bf16 caches are bfloat16, the type the
 * method is stated in; float16 is not built (code 1 is left unassigned, and any
 * dtype code other than those below returns PKV_ERR_UNSUPPORTED). */
typedef enum {
  PKV_BF16 = 0,      /* bfloat16 */
  PKV_FP8_E4M3 = 2,  /* OCP FP8 E4M3 (cache only), per-tensor scale */
  PKV_INT8 = 3       /* symmetric INT8 codes -127..127 (cache only), per-tensor scale */
} pkv_dtype;

/* bits of *err_flag */
#define PKV_DEVERR_SLOT 1        /* a slot_mapping entry >= num_slots (row skipped) */
#define PKV_DEVERR_BLOCK 2       /* a block_table entry outside [0, num_blocks) was needed */
#define PKV_DEVERR_LENGTH 4      /* a length is negative or needs more than max_blocks_per_seq blocks */
#define PKV_DEVERR_TIMEOUT 8     /* a bounded wait inside a kernel gave up (the tile was abandoned);
                                    the call's out and lse are then undefined, while the context,
                                    the caches and later calls stay valid */

/* Human-readable name of a pkv_status. */
PKV_API const char* pkv_status_string(int status);

/* Library ABI version (increases when a signature changes). */
PKV_API int pkv_abi_version(void);

/*
 * Tracing (no counterpart on the source pages; a profiling aid of this library).
 * on != 0: the compute entry points below (write, decode, decode with append,
 * varlen, block copy; not the decode without a workspace, which must allocate
 * nothing, and an attached tool may) open an NVTX range named after themselves
 * for the host-side span of the call, which holds its launches, so that a
 * timeline tool shows the library's calls; on == 0 (the default): no range, one
 * relaxed atomic load per call.  Without a tool attached, a range is a no-op.
 * Process-wide; thread-safe.
 */
PKV_API void pkv_set_nvtx(int on);

/*
 * KV-cache write ([KVM] "Triton カーネルによる KV キャッシュ書き込み"; checks from
 * "Python 層からのカーネル呼び出し").
 *
 * For every token t in [0, num_tokens) with s = slot_mapping[t]:
 *   k_cache row s := k row t,  v_cache row s := v row t   (a row is num_kv_heads*head_dim elements)
 * s < 0 marks a padding token: nothing is written.  s >= num_slots is skipped
 * and flagged (PKV_DEVERR_SLOT).  Two tokens with the same slot race (the
 * caller must not pass duplicates).
 *
 * k, v:          bf16, token t's row starts at element t*k_row_stride (resp.
 *                v_row_stride) and holds [num_kv_heads, head_dim] contiguous
 *                elements; the row strides are free (K and V may be views of a
 *                fused QKV projection) but must be multiples of 8 elements and
 *                the pointers 16-byte aligned.
 * k_cache, v_cache: [num_slots, num_kv_heads, head_dim] of cache_dtype, 16-byte aligned.
 * cache_dtype:   PKV_BF16 (bits copied), PKV_FP8_E4M3: each element is stored as
 *                e4m3_rne_satfinite(float(x) * inv_scale), one fp32 multiply
 *                and one round-to-nearest-even saturating conversion, or
 *                PKV_INT8: clamp(round_half_even(float(x) * inv_scale), -127, 127)
 *                ([CH15] KV size: FP8 or INT8 halve the cache; NaN stores 0).
 * k_inv_scale, v_inv_scale: 1/scale of each FP8 / INT8 cache, finite and positive
 *                (checked even when num_tokens == 0; ignored for PKV_BF16).
 * num_kv_heads*head_dim must be a multiple of 8.
 */
PKV_API int pkv_kv_cache_write(const void* k, int64_t k_row_stride, const void* v, int64_t v_row_stride,
                       int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                       void* k_cache, void* v_cache, int32_t cache_dtype, int64_t num_slots,
                       const int32_t* slot_mapping, float k_inv_scale, float v_inv_scale,
                       int32_t* err_flag, void* stream);

/*
 * Copy-on-write of shared blocks ([CH15] "PagedAttention：メモリを「ページ」で貸し出す":
 * answers generated from one prompt share the blocks of their common part, and
 * a shared block is copied only once one of them must write into it).
 *
 * For each i in [0, num_pairs), with (src, dst) = (block_pairs[2i], block_pairs[2i+1]):
 *   block dst of k_cache := block src of k_cache, and the same for v_cache,
 * byte for byte.  A block is block_bytes bytes (block_size*num_kv_heads*head_dim
 * elements of the cache's type); block b starts at byte b*block_bytes.
 *
 * k_cache, v_cache: the pools, 16-byte aligned; v_cache may be NULL (K only).
 * block_bytes:   a positive multiple of 16.
 * block_pairs:   int32 [num_pairs][2] (src, dst).  A pair with a block id outside
 *                [0, num_blocks) is skipped and flagged (PKV_DEVERR_BLOCK).  Every
 *                copy must read a block no pair of the same call writes (no dst
 *                is also a src, no two pairs share a dst); otherwise the result
 *                is unspecified.  num_pairs == 0 does nothing.
 */
PKV_API int pkv_copy_blocks(void* k_cache, void* v_cache, int64_t block_bytes, int32_t num_blocks,
                            const int32_t* block_pairs, int32_t num_pairs, int32_t* err_flag, void* stream);

/*
 * Workspace bytes pkv_paged_attn_decode (and pkv_paged_attn_decode_with_kvcache)
 * needs for these sizes on the current device, whatever the cache type (0 is a
 * valid answer; the split plan depends on the SM count and on the cache type,
 * and the larger plan is sized).  max_seqlen_k is a host upper bound of
 * cache_seqlens.  Returns 0 for invalid sizes as well; the call itself then
 * reports the error.
 */
PKV_API size_t pkv_paged_attn_decode_workspace(int32_t batch, int32_t num_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t max_seqlen_k);

/*
 * Paged decode attention ([PA] "デコードパス"; [KVM] "Attention モジュールの実装",
 * decode branch).  Each sequence b has one query token q[b] ([batch, num_heads,
 * head_dim] bf16) and attends to its first cache_seqlens[b] cached positions
 * (the count AFTER this step's token was written): position p of sequence b is
 * slot block_table[b*max_blocks_per_seq + p/block_size]*block_size + p%block_size.
 *
 *   out[b,h,:] = sum_p softmax_p(scale * <q[b,h], k_p>) * v_p       (bf16, RNE)
 *   lse[b,h]   = log sum_p exp(scale * <q[b,h], k_p>)               (fp32, natural log; nullable)
 * with k_p, v_p taken from kv head h/(num_heads/num_kv_heads).  A sequence
 * with cache_seqlens[b] == 0 outputs zeros and lse = -inf.
 *
 * cache_dtype PKV_BF16, or a one-byte cache where the cached code c stands for
 * c's value times k_scale (resp. v_scale): PKV_FP8_E4M3 (OCP E4M3) or
 * PKV_INT8 (symmetric codes -127..127).  k_scale and v_scale must be finite
 * and positive for a one-byte cache (ignored for PKV_BF16).  Long sequences
 * are split across CTAs and merged by log-sum-exp; workspace holds the
 * partial results.
 * max_seqlen_k: host upper bound of cache_seqlens (it sizes the split).
 */
PKV_API int pkv_paged_attn_decode(const void* q, const void* k_cache, const void* v_cache, int32_t cache_dtype,
                          const int32_t* cache_seqlens, const int32_t* block_table,
                          int32_t max_blocks_per_seq, int32_t batch, int32_t num_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t num_blocks, int32_t max_seqlen_k, float scale, float k_scale,
                          float v_scale, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, int32_t* err_flag, void* stream);

/*
 * Decode attention with an in-place cache append ([PA] "デコードパス": the
 * example's cache_seqlens count the tokens cached BEFORE this step, and the
 * new token goes to the next position, in a held block or a new one; [KVM]
 * "Attention モジュールの実装": write the step's K/V, then attend).  One call does
 * both: for each sequence b, position pos = cache_seqlens[b] is
 *   slot = block_table[b*max_blocks_per_seq + pos/block_size]*block_size + pos%block_size,
 * k_cache row slot := k_new row b and v_cache row slot := v_new row b (bf16
 * copied, or FP8 as e4m3_rne_satfinite(float(x)*inv_scale) like
 * pkv_kv_cache_write), and then q[b] attends cache_seqlens[b] + 1 positions
 * exactly as pkv_paged_attn_decode does.  The row is stored by the CTA that
 * reads that position, before it reads it, so no separate write launch is
 * needed.
 *
 * k_new, v_new:  bf16 [batch, num_kv_heads, head_dim] rows at k_new_row_stride /
 *                v_new_row_stride elements (multiples of 8), 16-byte aligned.
 * cache_dtype:   PKV_BF16, PKV_FP8_E4M3 or PKV_INT8 (stored as pkv_kv_cache_write does).
 * k_inv_scale, v_inv_scale: 1/scale of each one-byte cache, finite and positive
 *                (checked even when batch == 0; ignored for PKV_BF16).
 * max_seqlen_k:  host upper bound of cache_seqlens + 1 (the attended length);
 *                the workspace is pkv_paged_attn_decode_workspace(..., max_seqlen_k).
 * Other arguments as for pkv_paged_attn_decode.  A position whose block id is
 * outside [0, num_blocks) is flagged (PKV_DEVERR_BLOCK) and not written.
 */
PKV_API int pkv_paged_attn_decode_with_kvcache(const void* q, const void* k_new, int64_t k_new_row_stride,
                                               const void* v_new, int64_t v_new_row_stride, void* k_cache,
                                               void* v_cache, int32_t cache_dtype, const int32_t* cache_seqlens,
                                               const int32_t* block_table, int32_t max_blocks_per_seq,
                                               int32_t batch, int32_t num_heads, int32_t num_kv_heads,
                                               int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                               int32_t max_seqlen_k, float scale, float k_scale, float v_scale,
                                               float k_inv_scale, float v_inv_scale, void* out, float* lse,
                                               void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                               void* stream);

/*
 * Workspace bytes pkv_paged_attn_varlen needs for these arguments on the
 * current device (0 is a valid answer).  `paged` is non-zero when a block table
 * will be passed; total_k, kv_dtype and block_size are the values the call will
 * get (they decide whether the paged K/V are gathered first, see below).
 * Returns 0 for invalid sizes as well.
 */
PKV_API size_t pkv_paged_attn_varlen_workspace(int32_t batch, int32_t total_q, int32_t total_k, int32_t num_heads,
                                               int32_t num_kv_heads, int32_t head_dim, int32_t max_len_q,
                                               int32_t max_len_k, int32_t paged, int32_t kv_dtype,
                                               int32_t block_size);

/*
 * Variable-length causal attention ([PA] "Varlen パス"; [KVM] "Attention モジュールの実装",
 * prefill branch; [CH15] prefix caching and chunked prefill).
 *
 * Sequence b has Lq_b = cu_seqlens_q[b+1]-cu_seqlens_q[b] queries, packed as
 * rows cu_seqlens_q[b].. of q ([total_q, num_heads, head_dim] bf16), and
 * Lk_b = cu_seqlens_k[b+1]-cu_seqlens_k[b] keys:
 *   - block_table == NULL: k, v are packed [total_k, num_kv_heads, head_dim] bf16
 *     and key j of sequence b is row cu_seqlens_k[b]+j;
 *   - otherwise k, v are the paged caches [num_blocks*block_size, num_kv_heads,
 *     head_dim] bf16 and key j is slot block_table[b*max_blocks_per_seq + j/block_size]
 *     *block_size + j%block_size (prefix reuse: the keys of a shared prefix are
 *     the same blocks in several rows of the table).
 * Causal alignment is bottom-right: query i of sequence b sees key j iff
 * j <= i + Lk_b - Lq_b (the queries are the last Lq_b of the Lk_b positions).
 *   out[row, h, :] = softmax_j(scale * <q[row,h], k_j>) . v_j      (bf16, RNE)
 *   lse[h, row]    = log sum_j exp(scale * <q[row,h], k_j>)        (fp32; nullable)
 * with kv head h/(num_heads/num_kv_heads).  A query that sees no key outputs
 * zeros and lse = -inf.
 *
 * max_len_q, max_len_k: host upper bounds of the lengths (grid sizing).
 * total_k: packed mode: rows of the packed k/v.  Paged mode: 0, or an upper
 *          bound on the summed key counts of the sequences the prefill tiles
 *          serve (see routing below).  With total_k > 0 and a one-byte cache or
 *          block_size < 64, those sequences' K/V are first gathered through the
 *          block table into a packed bf16 buffer in the workspace (one-byte
 *          codes widened exactly), and the packed tile loop runs on it: one
 *          small copy box per page and head-dim half would bound the paged
 *          loop.  Keys past the bound are not gathered and flagged
 *          (PKV_DEVERR_LENGTH).
 * kv_dtype: PKV_BF16; or, in paged mode, PKV_FP8_E4M3 or PKV_INT8, where a
 *          cached code c stands for c's value times k_scale (resp. v_scale).
 *          With total_k > 0 the tiles read a bf16 copy gathered into the
 *          workspace; with total_k == 0 and head_dim 128 they read the pages
 *          themselves, widen the codes to f16 in shared memory and run f16
 *          MMAs, the query then also taken as f16 (|q| must stay below 65504);
 *          with total_k == 0 and head_dim 64 (and some sequence with more
 *          queries than the routing bound below) the call returns
 *          PKV_ERR_UNSUPPORTED.
 * Supported: head_dim 64 or 128, causal != 0; paged block_size a multiple of 16
 * that divides 128 or is a multiple of 128.  All of q, k, v, out 16-byte aligned.
 * Routing (paged mode, num_heads/num_kv_heads <= 8): when no sequence has more
 * than 8 queries, every query row is computed by the decode kernels over its
 * own causal prefix (split-KV over the GQA group; speculative verification);
 * otherwise only the sequences with exactly one query are, and the others by
 * the 128-row tiles.
 */
PKV_API int pkv_paged_attn_varlen(const void* q, const void* k, const void* v, int32_t kv_dtype,
                                  const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
                                  int32_t total_q, int32_t total_k, int32_t max_len_q, int32_t max_len_k,
                                  const int32_t* block_table, int32_t max_blocks_per_seq, int32_t block_size,
                                  int32_t num_blocks, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                  float scale, int32_t causal, float k_scale, float v_scale, void* out,
                                  float* lse, void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                  void* stream);

/*
 * Paged decode attention without a caller workspace (no counterpart on the
 * source pages; an addition of this library).
 *
 * Some callers cannot allocate device memory: a plugin hosted by an engine
 * that has already reserved all of the device's memory for its own pool, or a
 * latency-critical loop where cudaMalloc's implicit device synchronisation is
 * not allowed.  They cannot supply the workspace pkv_paged_attn_decode needs.
 * This entry point computes the same result as pkv_paged_attn_decode (same
 * arguments, same kernels, same status codes) but keeps the split-KV partials
 * in a fixed 32 MiB array that the library declares in device memory; it
 * allocates nothing itself.
 *
 * - Limit: requests whose pkv_paged_attn_decode_workspace(...) exceeds
 *   pkv_paged_attn_decode_noalloc_max_scratch() (32 MiB) are rejected with
 *   PKV_ERR_WORKSPACE before any launch.
 * - Every GPU that loads the library holds the 32 MiB array until the process exits.
 * - The first call on each device looks up the array's device address once
 *   (with that device current); make that first call before any stream capture.
 *   The address is kept for the life of the process and stays valid while the
 *   device's primary context lives: after a cudaDeviceReset (or anything else
 *   that destroys and recreates that context) do not call this entry point again
 *   in the same process.
 * - All calls share the array.  Nothing in it must start at zero, but calls that
 *   overlap on the GPU (e.g. on two streams) race on it and corrupt each other.
 * The caller still passes inputs and outputs (q, caches, metadata, out, lse).
 */
PKV_API int pkv_paged_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                          int32_t cache_dtype, const int32_t* cache_seqlens,
                                          const int32_t* block_table, int32_t max_blocks_per_seq,
                                          int32_t batch, int32_t num_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                          int32_t max_seqlen_k, float scale, float k_scale, float v_scale,
                                          void* out, float* lse, int32_t* err_flag, void* stream);

/* Bytes of the fixed scratch array pkv_paged_attn_decode_noalloc uses (its size limit). */
PKV_API size_t pkv_paged_attn_decode_noalloc_max_scratch(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
