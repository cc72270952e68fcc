// Causal GQA varlen prefill on tcgen05 tensor cores (TMEM accumulators, TMA-fed).
//
// Source: "ページド・アテンション" (transformers docs), section "Varlen パス": packed
// variable-length sequences indexed by cumulative lengths cu_seq_lens_q/k and
// their maxima; "効率的な KV キャッシュ管理と Attention 計算" (itan.pw), section
// "Attention モジュールの実装": causal prefill, reading K/V from the paged cache
// through block_tables when prefixes are shared; "KV cache / batching / paged
// attention" (1s.xyz ch. 15), "FlashAttention：注意計算そのものを速く": tiles in
// on-chip memory give exactly ordinary attention.
//
// Causal alignment: query i of a sequence with Lq queries and Lk keys sees key
// j iff j <= i + Lk - Lq (the queries are the last Lq positions; prefix reuse).
//
// Persistent kernel, one 352-thread CTA per SM (384 with one-byte pages).  A
// work item is a pair of 128-row query tiles (A, B) of one sequence that read
// the same K/V tiles, so each K/V tile is loaded once for 256 query rows: one
// query tile of two heads of a GQA group when the group is even (both see the
// same keys), else two adjacent tiles of one head, paired from the sequence's
// end (tile A stops at its own last visible K/V tile, one before B's).  Items
// are claimed through a global counter, longest first, and published to the
// CTA's warps through a shared ring.
//   warp 0      producer: Q of both tiles (TMA), then K/V tiles of 128 keys
//               (2 stages each), K one tile ahead of V.  Packed K/V: one TMA
//               box per head-dim half.  Paged K/V: one box per page and
//               half, each issued by its own lane, the block ids read two
//               tiles ahead.
//   warps 1, 2  MMA issuers, one thread each: warp 1 for tile A, warp 2 for
//               tile B.  Per K/V tile j a thread issues O += P(j-1) V(j-1),
//               then S(j) = Q K(j)^T.  One thread issues an M=128 MMA only
//               every ~120-140 cycles, whatever N is, so the two tiles' MMAs
//               come from two threads and interleave in the tensor core.
//   warps 3..6  softmax of tile A, warps 7..10 of tile B: one thread per query
//               row, all 128 keys of each tile.  The two groups take turns
//               tile by tile while both have tiles left.  The running max
//               moves only when it grows by more than 2^8, so O is rescaled
//               rarely (by the same thread, in TMEM).  P (bf16 pairs)
//               overwrites half of its S columns.  After the tile's last PV
//               the group reads O, releases it, and stores the normalised rows.
//   warp 11     (FP8 / INT8 pages only) widening: each landed one-byte K/V
//               tile becomes the f16 tile in place, each Q tile f16, and the
//               MMAs run f16 x f16.
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A at 256, O_B at 384.
// Every mbarrier wait is bounded by a deadline; on expiry the CTA flags
// PKV_DEVERR_TIMEOUT, waits (bounded) for its own copies and MMAs, frees TMEM
// and returns.
#include <cmath>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int kBM = 128;          // query rows per query tile
constexpr int kPairRows = 2 * kBM;  // query rows per work item (tiles A and B)
constexpr int kBN = 128;          // keys per K/V tile
constexpr int kThreads = 352;     // producer warp, 2 MMA warps, 2 softmax warp groups
constexpr int kThreadsCoded = 384;  // one-byte caches: + a widening warp
constexpr int kWidenWarp = 11;
constexpr int kSoftmaxWarp0 = 3;  // first softmax warp (tile A: warps 3..6, tile B: 7..10)
constexpr int kGroupThreads = 128;  // a softmax warp group: one thread per row of its tile
constexpr int kSoftmaxThreads = 256;  // all softmax warps (one group per tile, or all on one tile)
constexpr int kUnifiedKeys = 4096;    // key bound from which the one-tile-at-a-time softmax runs
constexpr uint32_t kTmemCols = 512;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;    // log2 units

struct PrefillParams {
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* block_table;
  int32_t max_blocks;
  int32_t block_size;
  int32_t box_rows;      // rows per paged TMA box: min(block_size, 128)
  int32_t num_blocks;
  int32_t num_heads;
  int32_t group;
  int32_t n_pairs;       // tile pairs (or, with head_pairs, query tiles) of the longest sequence
  int32_t head_pairs;    // 1: a pair is one query tile of two heads of a GQA group (even groups); 0: two tiles of one head
  int32_t item_heads;    // items per (pair, sequence): num_heads / 2 with head_pairs, else num_heads
  int32_t batch;
  int32_t route_decode;  // sequences with at most this many queries are left to the decode kernels (0: none)
  int32_t* item_counter; // work-item counter, zero at launch
  const int32_t* unit_order;  // units (sequence b, pair pe) coded b * n_pairs + pe, most K/V tiles first
  const int4* unit_seq;       // per unit: its sequence's cu_q[b], cu_q[b+1], cu_k[b], cu_k[b+1]
  const int32_t* n_units;     // units in unit_order
  const int32_t* active_ctas; // CTAs that run (the others leave their SMs to the decode kernels of the call)
  float scale_log2;
  float v_mul;           // output factor (FP8 V scale of a gathered cache, else 1)
  int64_t total_q;
  uint16_t* out;
  int32_t out_v8;        // out is 32-byte aligned: rows are stored 32 bytes per instruction
#ifdef PKV_TEST_HOOKS
  int32_t test_skip_k;   // test builds: CTA 0 withholds the copy of this K tile (its count in the CTA; -1: none)
#endif
  float* lse;
  int32_t* err;
};

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier, TMA, tcgen05
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 format).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16: bf16 x bf16 (or f16 x f16) -> f32, A K-major.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n, bool b_mn_major, bool f16 = false) {
  return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D (TMEM) (+)= A (TMEM, M x K, 16-bit pairs per column) * B (shared memory descriptor).
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

#define PKV_TMEM_LD32(taddr, r)                                                                                    \
  asm volatile(                                                                                                    \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%" \
      "19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                                                 \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),            \
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),      \
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),    \
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])     \
      : "r"(taddr))

#define PKV_TMEM_ST32(taddr, r)                                                                                   \
  asm volatile(                                                                                                   \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%" \
      "18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),                                 \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),          \
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),  \
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), \
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])                                                   \
      : "memory")

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }


// ---------------------------------------------------------------------------
// shared-memory plan
// ---------------------------------------------------------------------------

template <int D, bool kUnified = false>  // kUnified: the one-tile softmax's larger per-thread areas
struct Smem {
  static constexpr int kAtoms = D / 64;                 // 64-element (128-byte) column groups
  static constexpr int kTileBytes = 128 * D * 2;        // a [128 x D] bf16 tile
  static constexpr int kAtomBytes = 128 * 128;          // [128 rows x 128 B]
  static constexpr int kQ = 0;                          // query tiles A and B
  static constexpr int kK = kQ + 2 * kTileBytes;        // 2 stages
  static constexpr int kV = kK + 2 * kTileBytes;        // 2 stages
  static constexpr int kBar = kV + 2 * kTileBytes;
  static constexpr int kNumBars = 40;
  static constexpr int kMisc = kBar + kNumBars * 8;     // tmem holder, abort flag
  static constexpr int kRingData = kMisc + 16;          // 4 ring slots x 8 ints (item, q0, Lq, k0, Lk)
  static constexpr int kEpi = kRingData + 4 * 32;       // per tile and softmax thread: output and lse offsets, rows (32 B)
  static constexpr int kXch = kEpi + 2 * (kUnified ? kSoftmaxThreads : kGroupThreads) * 32;
  static constexpr int kTotal = kXch + (kUnified ? 2 * kSoftmaxThreads * 4 : 0);  // 2 rounds x 256 floats swapped by row halves
  static constexpr int kAlloc = kTotal + 1024;          // slack to align the base to 1024
};
static_assert(Smem<128, true>::kAlloc <= 227 * 1024, "shared memory plan exceeds a CTA's limit");

constexpr int kRing = 4;  // work-item ring slots

// mbarrier indices (each one distinct; checked below).  "X" is the query
// tile of the pair (0: A, 1: B).  Every barrier below can only be one phase
// ahead of its waiter (each role's next arrival depends on the waiter having
// seen the previous one), so single parity waits are unambiguous.
enum Bar {
  kQFull0 = 0,       // +X: Q tile landed (producer -> MMA)
  kQEmpty0 = 2,      // +X: last S of the item's tile X done, Q buffer free (MMA -> producer)
  kKFull0 = 4,       // +stage: K tile landed
  kKEmpty0 = 6,      // +stage: every S reading the K stage done (one arrival per MMA thread)
  kVFull0 = 8,       // +stage: V tile landed
  kVEmpty0 = 10,     // +stage: every PV reading the V stage done (one arrival per MMA thread)
  kSFull0 = 12,      // +X: S of the next tile done (MMA -> softmax X); also means PV_X of the tile before is done
  kPFull0 = 14,      // +X: P of that tile written (softmax X, 128 arrivals -> MMA)
  kODone0 = 16,      // +X: the item's last PV_X done (MMA -> softmax X epilogue)
  kOFree0 = 18,      // +X: softmax X has read O_X (128 arrivals -> MMA, before the next item's first PV_X)
  kRingFull0 = 20,   // +slot (4): a work item index published by the producer
  kRingEmpty0 = 24,  // +slot (4): both MMA threads, the 8 softmax warps (and the widening warp) have read it
  kDrain0 = 28,      // +X: every MMA of issuer X done (end of the kernel)
  kTurn0 = 30,       // +X: the other softmax group finished its tile; group X may start its next one
  kQReady0 = 32,     // +X: one-byte caches: Q converted to f16 in place (producer -> MMA)
  kKReady0 = 34,     // +stage: one-byte caches: K widened to f16 in place (producer -> MMA)
  kVReady0 = 36,     // +stage: one-byte caches: V widened to f16 in place (producer -> MMA)
  kXch0 = 38,        // row halves: a round of swapped values written (256 arrivals; one-tile softmax)
  kBarCount = 39
};
static_assert(kQEmpty0 == kQFull0 + 2 && kKFull0 == kQEmpty0 + 2 && kKEmpty0 == kKFull0 + 2 &&
                  kVFull0 == kKEmpty0 + 2 && kVEmpty0 == kVFull0 + 2 && kSFull0 == kVEmpty0 + 2 &&
                  kPFull0 == kSFull0 + 2 && kODone0 == kPFull0 + 2 && kOFree0 == kODone0 + 2 &&
                  kRingFull0 == kOFree0 + 2 && kRingEmpty0 == kRingFull0 + kRing && kDrain0 == kRingEmpty0 + kRing &&
                  kTurn0 == kDrain0 + 2 && kQReady0 == kTurn0 + 2 && kKReady0 == kQReady0 + 2 &&
                  kVReady0 == kKReady0 + 2 && kXch0 == kVReady0 + 2 && kBarCount == kXch0 + 1,
              "mbarrier index ranges must not overlap");
static_assert(Smem<128>::kNumBars >= kBarCount && Smem<64>::kNumBars >= kBarCount, "too few mbarrier slots");

// A sequence's query/key offsets and (checked) lengths.  The producer warp
// reads them from global memory once per work item and hands them to the
// other roles through the work-item ring, so only one warp waits on those loads.
struct SeqBase {
  int q0, Lq, k0, Lk;
};
// One work item: the pair's two query tiles X = 0 (A), 1 (B), each with its
// first row, rows inside the sequence and K/V tiles it attends (n[X]).
struct Seq {
  int q0, Lq, k0, Lk, diag;
  int row0[2], rows[2], n[2];
  int n_kv;  // K/V tiles the pair reads: max(n[0], n[1])
  bool skip;
};

// Unit u of the list: its code and its sequence's cumulative offsets q0, q1,
// k0, k1 (two independent loads; the offsets are checked by seq_check).
__device__ __forceinline__ void unit_load(const PrefillParams& p, int u, int (&raw)[4], int& code) {
  const int4 r = __ldg(p.unit_seq + u);
  code = __ldg(p.unit_order + u);
  raw[0] = r.x;
  raw[1] = r.y;
  raw[2] = r.z;
  raw[3] = r.w;
}
__device__ __forceinline__ SeqBase seq_check(const PrefillParams& p, const int (&raw)[4], bool report) {
  SeqBase s;
  s.q0 = raw[0];
  s.Lq = raw[1] - raw[0];
  s.k0 = raw[2];
  s.Lk = raw[3] - raw[2];
  bool bad = false;
  if (s.Lq < 0) { s.Lq = 0; bad = true; }
  if (s.Lk < 0) { s.Lk = 0; bad = true; }
  if (p.block_table != nullptr && (int64_t)s.Lk > (int64_t)p.max_blocks * p.block_size) {
    s.Lk = p.max_blocks * p.block_size;
    bad = true;
  }
  if (bad && report) flag_error(p.err, PKV_DEVERR_LENGTH);
  return s;
}
// Pair pe of a sequence, counted from its end.  With head pairs (even GQA
// groups) it is query tile T-1-pe, T = ceil(Lq/128), of two heads of the same
// group: A and B see the same keys and read the same K/V tiles.  Otherwise it
// holds query tiles T-2-2pe (A) and T-1-2pe (B) of one head: the last tiles,
// which see the most keys, pair up, and a sequence with an odd tile count
// leaves tile 0 alone (it sees one K/V tile); tile B sees the most keys, and
// tile A stops at its own last visible K/V tile (one before B's when the query
// and key lengths match) and releases the stages it does not read.
__device__ __forceinline__ void pair_tiles(int Lq, int pe, bool head_pairs, int& tA, int& tB) {
  const int T = (Lq + kBM - 1) / kBM;
  tB = head_pairs ? T - 1 - pe : T - 1 - 2 * pe;
  tA = head_pairs ? tB : tB - 1;
}
// K/V tiles that pair pe of a sequence with Lq queries and Lk keys reads:
// those its tile B attends (B sees at least as many keys as A).
__device__ __forceinline__ int unit_kv_tiles(int Lq, int Lk, int pe, bool head_pairs) {
  int tA, tB;
  pair_tiles(Lq, pe, head_pairs, tA, tB);
  const int rows = min(kBM, Lq - tB * kBM);
  const int kmax = tB * kBM + rows - 1 + Lk - Lq;  // last key tile B's last row sees
  return kmax < 0 ? 0 : min(kmax / kBN + 1, (Lk + kBN - 1) / kBN);
}
// Query head of tile X of an item whose head slot is hs.
__device__ __forceinline__ int tile_head(const PrefillParams& p, int hs, int x) {
  return p.head_pairs ? 2 * hs + x : hs;
}
__device__ __forceinline__ Seq seq_derive(const PrefillParams& p, const SeqBase& b0, int pair) {
  Seq s;
  s.q0 = b0.q0;
  s.Lq = b0.Lq;
  s.k0 = b0.k0;
  s.Lk = b0.Lk;
  s.diag = s.Lk - s.Lq;
  const int kv_tiles = (s.Lk + kBN - 1) / kBN;
  int t[2];
  pair_tiles(s.Lq, pair, p.head_pairs != 0, t[0], t[1]);
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    if (t[x] < 0) {
      s.row0[x] = 0;
      s.rows[x] = 0;
      s.n[x] = 0;
    } else {
      s.row0[x] = t[x] * kBM;
      s.rows[x] = min(kBM, s.Lq - s.row0[x]);
      const int kmax = s.row0[x] + s.rows[x] - 1 + s.diag;  // last key the tile's last row sees
      s.n[x] = kmax < 0 ? 0 : min(kmax / kBN + 1, kv_tiles);
    }
  }
  // tile B's rows see at least as many keys as tile A's: the pair reads B's K/V tiles
  s.n_kv = max(s.n[0], s.n[1]);
  s.skip = s.rows[1] <= 0 || s.Lq <= p.route_decode;
  return s;
}

// Work item -> (sequence, pair, head slot: the head, or with head pairs the
// pair of heads 2 hs, 2 hs + 1).  Items run through the units (sequence, pair)
// in the order the prep kernel writes (the pairs that read the most K/V tiles
// first), the head slots of a unit one after another, so CTAs running side by
// side share K/V through L2.
struct Item {
  int b, pair, head;
  int head_b;  // (ring consumers) the query head of tile B; tile A's is tile_head(p, head, 0)
};
__device__ __forceinline__ Item item_of(const PrefillParams& p, int it, int code) {
  Item x;
  x.b = code / p.n_pairs;
  x.pair = code % p.n_pairs;
  x.head = it % p.item_heads;
  return x;
}

// ---------------------------------------------------------------------------
// one-byte caches read by the tile loop: widening to f16 in shared memory
// ---------------------------------------------------------------------------
// With an FP8 or INT8 cache the tile loop runs f16 x f16 MMAs: every E4M3 code
// and every INT8 code (-127..127) is exactly an f16 value, so the producer warp
// widens each landed K/V tile in place, and converts each Q tile from bf16 to
// f16 once per item (exact for |q| in f16's normal range; |q| > 65504 would
// become infinite).  The per-tensor scales act as in the gathered path: k_scale
// joins the logit scale and v_scale the output factor.

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// A [128 rows x 128] bf16 tile (two 128-byte atoms), converted to f16 in
// place, 16 bytes per lane and access (elementwise: the swizzle does not matter).
__device__ __forceinline__ void widen_q_f16(uint8_t* tile, int lane) {
  uint4* v = reinterpret_cast<uint4*>(tile);
#pragma unroll 4
  for (int i = lane; i < 2 * kBM * 8; i += 32) {
    uint4 w = v[i];
    w.x = bf16x2_to_f16x2(w.x);
    w.y = bf16x2_to_f16x2(w.y);
    w.z = bf16x2_to_f16x2(w.z);
    w.w = bf16x2_to_f16x2(w.w);
    v[i] = w;
  }
}

// Codes 4k..4k+1 (lo) or 4k+2..4k+3 (hi) of a 32-bit word of one-byte codes -> f16x2.
template <int kCode>
__device__ __forceinline__ uint32_t code2_to_f16x2(uint32_t w, bool hi) {
  if constexpr (kCode == 1) {
    return hi ? e4m3x2_hi_to_f16x2(w) : e4m3x2_lo_to_f16x2(w);
  } else {
    // INT8: with its sign bit flipped, code c is the low mantissa byte of the
    // f16 1152 + c (exponent byte 0x64); 1152 is then taken off exactly
    const uint32_t b = prmt(w ^ 0x80808080u, 0x64646464u, hi ? 0x4342u : 0x4140u);
    __half2 h = *reinterpret_cast<const __half2*>(&b);
    h = __hsub2(h, __half2half2(__ushort_as_half((unsigned short)0x6480u)));  // 1152
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// The one-byte [128 rows x 128 B] tile that TMA landed (128-byte swizzle) in
// the second half of a K/V stage, widened in place to the f16 tile the MMAs
// read (two 128-byte atoms of 128 rows, 128-byte swizzle).  Lane l takes rows
// l, l+32, l+64, l+96 and reads a whole row before writing: the one-byte row r
// occupies exactly the bytes of f16 row r of the second atom, and no other lane
// reads or writes them.
template <int kCode>
__device__ __forceinline__ void widen_kv_f16(uint8_t* stage, int lane) {
  const uint8_t* src = stage + kBM * 128;
#pragma unroll 1
  for (int i = 0; i < kBN / 32; ++i) {
    const int r = lane + 32 * i;
    const int sw = r & 7;
    uint4 in[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) in[c] = *reinterpret_cast<const uint4*>(src + r * 128 + ((c ^ sw) << 4));
#pragma unroll
    for (int c = 0; c < 8; ++c) {  // codes 16c..16c+15 -> f16 chunks 2c, 2c+1 of atom c / 4
      const uint32_t w[4] = {in[c].x, in[c].y, in[c].z, in[c].w};
      uint32_t h[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        h[2 * k] = code2_to_f16x2<kCode>(w[k], false);
        h[2 * k + 1] = code2_to_f16x2<kCode>(w[k], true);
      }
      uint8_t* row = stage + (c >> 2) * (kBM * 128) + r * 128;
      *reinterpret_cast<uint4*>(row + ((((2 * c) & 7) ^ sw) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(row + ((((2 * c + 1) & 7) ^ sw) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
}

// Persistent kernel: one CTA per SM takes work items from the global counter.
// All roles walk the same published list and keep running counters (items,
// tiles) so the barriers' phases continue across items.
// kCode: 0 bf16 K/V (packed or paged); 1 E4M3, 2 INT8 codes (paged, d128),
// widened to f16 in shared memory by the producer warp.
template <int D, bool kPaged, int kCode, bool kUnified = false>
__global__ void __launch_bounds__(kCode ? kThreadsCoded : kThreads, 1)
    varlen_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using L = Smem<D, kUnified>;
  constexpr bool kCoded = kCode != 0;
  static_assert(!kCoded || (kPaged && D == 128), "one-byte K/V tiles: paged, head dim 128");
  // the MMA threads wait for a landed tile (bf16) or for its widening (one-byte codes)
  constexpr int kQWait0 = kCoded ? kQReady0 : kQFull0;
  constexpr int kKWait0 = kCoded ? kKReady0 : kKFull0;
  constexpr int kVWait0 = kCoded ? kVReady0 : kVFull0;
  // Launched as a programmatic dependent of the kernel before it: wait until
  // that grid has completed and its writes (the unit list, the work counter;
  // the gathered K/V, when a gather ran before, which lets this grid launch
  // only at its end) are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if ((int)blockIdx.x >= __ldg(p.active_ctas)) return;
  // The decode kernels of the same call (the routed query rows) may start as
  // soon as SMs free up: they read nothing this kernel writes, and the routed
  // row list they read is complete (the prep grid has completed).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_items = __ldg(p.n_units) * p.item_heads;

  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8 * i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(kQFull0 + x), 1);
      mbar_init(bar(kQEmpty0 + x), 1);
      mbar_init(bar(kKFull0 + x), 1);
      mbar_init(bar(kKEmpty0 + x), 2);
      mbar_init(bar(kVFull0 + x), 1);
      mbar_init(bar(kVEmpty0 + x), 2);
      mbar_init(bar(kSFull0 + x), 1);
      mbar_init(bar(kPFull0 + x), kUnified ? kSoftmaxThreads : kGroupThreads);
      mbar_init(bar(kODone0 + x), 1);
      mbar_init(bar(kOFree0 + x), kUnified ? kSoftmaxThreads : kGroupThreads);
    }
    mbar_init(bar(kXch0), kSoftmaxThreads);
    mbar_init(bar(kDrain0), 1);
    mbar_init(bar(kDrain0 + 1), 1);
    mbar_init(bar(kTurn0), kGroupThreads / 32);
    mbar_init(bar(kTurn0 + 1), kGroupThreads / 32);
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(kQReady0 + x), 1);
      mbar_init(bar(kKReady0 + x), 1);
      mbar_init(bar(kVReady0 + x), 1);
    }
    for (int r = 0; r < kRing; ++r) {
      mbar_init(bar(kRingFull0 + r), 1);
      mbar_init(bar(kRingEmpty0 + r), 2 + 2 * kGroupThreads / 32 + (kCoded ? 1 : 0));
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // TMEM columns: S of tile X at 128 X (P of that tile, bf16 pairs: keys 0..63
  // over its columns 0..31, keys 64..127 over 64..95), O of tile X at 256 + 128 X.
  auto tS = [&](int x) -> uint32_t { return tmem + 128 * x; };
  auto tO = [&](int x) -> uint32_t { return tmem + 256 + 128 * x; };

  auto fail = [&]() {
    *abort_flag = 1;
    flag_error(p.err, PKV_DEVERR_TIMEOUT);
  };
  // Work items are handed out dynamically, longest first (item_of orders
  // them), through a global counter; the producer warp claims them and
  // publishes each one that has work into a 4-slot ring that the MMA and
  // softmax warps read in order.  -1 ends the list.
  volatile int* ring = reinterpret_cast<volatile int*>(smem + L::kRingData);
  // Consumer side: item of the u-th ring entry (or -1, also on timeout), its
  // pair and head (decoded by the producer) and its sequence.
  auto ring_get = [&](int u, SeqBase& sb, Item& x) -> int {
    const int slot = u & (kRing - 1);
    if (!mbar_wait(bar(kRingFull0 + slot), (u / kRing) & 1, abort_flag)) return -1;
    const volatile int* e = ring + 8 * slot;
    const int it = e[0];
    sb.q0 = e[1];
    sb.Lq = e[2];
    sb.k0 = e[3];
    sb.Lk = e[4];
    x.pair = e[5];
    x.head = e[6];
    x.head_b = e[7];
    x.b = 0;
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kRingEmpty0 + slot));
    return it;
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    int last_k[2] = {-1, -1}, last_v[2] = {-1, -1}, last_q[2] = {-1, -1};
    int g = 0, ur = 0;        // K/V tiles, ring entries
    int qc[2] = {0, 0};       // Q loads per tile slot
    bool ok = true;
    auto publish = [&](int it, const SeqBase& sb, const Item& x) -> bool {
      const int slot = ur & (kRing - 1);
      if (ur >= kRing && !mbar_wait(bar(kRingEmpty0 + slot), ((ur / kRing) - 1) & 1, abort_flag)) return false;
      if (lane == 0) {
        volatile int* e = ring + 8 * slot;
        e[0] = it;
        e[1] = sb.q0;
        e[2] = sb.Lq;
        e[3] = sb.k0;
        e[4] = sb.Lk;
        e[5] = x.pair;
        e[6] = x.head;
        e[7] = tile_head(p, x.head, 1);
        mbar_arrive(bar(kRingFull0 + slot));
      }
      __syncwarp();
      ++ur;
      return true;
    };
    // The next item is claimed from the global counter a few tiles before
    // the current one's last, and its offsets are loaded while those tiles
    // are issued: neither latency then sits between two items, and a claimed
    // item waits only a few tiles (dynamic balance is kept).  The unit list
    // holds only pairs with rows of sequences this kernel serves; an item that
    // turns out empty all the same is passed over.
    int claim = 0;  // lane 0: atomic result for the next item
    bool claimed = false, resolved = false;
    int it = 0, next = n_items;
    int it_code = 0, next_code = 0;  // unit codes of it and next
    int raw[4] = {0, 0, 0, 0};
    auto claim_next = [&]() {
      if (claimed) return;
      if (lane == 0) claim = atomicAdd(p.item_counter, 1);
      claimed = true;
    };
    auto resolve_next = [&]() {
      claim_next();
      if (resolved) return;
      next = __shfl_sync(0xffffffffu, claim, 0);
      if (next < n_items) unit_load(p, next / p.item_heads, raw, next_code);
      resolved = true;
    };
    resolve_next();
    it = next;
    it_code = next_code;
    while (ok && it < n_items) {
      claimed = resolved = false;
      const Item x = item_of(p, it, it_code);
      const SeqBase si = seq_check(p, raw, x.pair == 0 && x.head == 0 && lane == 0);
      const Seq sq = seq_derive(p, si, x.pair);
      if (sq.skip) {
        resolve_next();
        it = next;
        it_code = next_code;
        continue;
      }
      if (!publish(it, si, x)) { ok = false; break; }
      if (sq.n_kv == 0) {
        resolve_next();
        it = next;
        it_code = next_code;
        continue;
      }
      const int kvh = tile_head(p, x.head, 0) / p.group;  // (both heads of a head pair share it)
      const int32_t* bt = kPaged ? p.block_table + (int64_t)x.b * p.max_blocks : nullptr;
      // Q of tile X (only when it attends keys), into its buffer once the
      // previous item's last S of that tile is done
      auto load_q = [&](int xq) -> bool {
        if (sq.n[xq] == 0) return true;
        if (qc[xq] > 0 && !mbar_wait(bar(kQEmpty0 + xq), (qc[xq] - 1) & 1, abort_flag)) return false;
        if (lane == 0) {
          mbar_expect_tx(bar(kQFull0 + xq), L::kTileBytes);
          for (int a = 0; a < L::kAtoms; ++a)
            tma_load_3d(sbase + L::kQ + xq * L::kTileBytes + a * L::kAtomBytes, &tm_q, a * 64, tile_head(p, x.head, xq),
                        sq.q0 + sq.row0[xq], bar(kQFull0 + xq));
        }
        last_q[xq] = qc[xq];
        ++qc[xq];
        return true;
      };
      const int br = kPaged ? p.box_rows : kBN;
      const int npages = kBN / br;
      // Paged tiles: lane (page pg, head-dim atom at) issues one box; at most
      // 8 pages x 2 atoms, as block sizes are multiples of 16.  A one-byte
      // row (128 codes) is one 128-byte box row: one box per page, landing in
      // the second half of the stage.
      constexpr int kLoadAtoms = kCoded ? 1 : L::kAtoms;
      const int pg = lane % npages, at = lane / npages;
      const bool box_lane = lane < npages * kLoadAtoms;
      // Block id of this lane's page of local tile j (0 past the keys).  The
      // table is read two tiles before the id is used, so the load's latency
      // overlaps the waits in between; tile_slot checks and converts it.
      auto tile_blk = [&](int j) -> int {
        int blk = 0;
        if (kPaged && box_lane && j < sq.n_kv) {
          const int pos = j * kBN + pg * br;
          if (pos < sq.Lk) blk = __ldg(bt + pos / p.block_size);
        }
        return blk;
      };
      auto tile_slot = [&](int j, int blk) -> int {
        if (!kPaged || !box_lane) return 0;
        if (blk < 0 || blk >= p.num_blocks) {
          flag_error(p.err, PKV_DEVERR_BLOCK);
          blk = 0;  // never dereference a bad id; the sequence's result is unspecified
        }
        return blk * p.block_size + (j * kBN + pg * br) % p.block_size;
      };
      auto issue = [&](int t, int j, int my_slot) -> bool {  // t = 0: K, 1: V; local tile j
        const int gg = g + j;
        const int s = gg & 1, u = gg >> 1;
        const uint32_t empty = bar((t ? kVEmpty0 : kKEmpty0) + s);
        const uint32_t full = bar((t ? kVFull0 : kKFull0) + s);
        if (u > 0 && !mbar_wait(empty, (u - 1) & 1, abort_flag)) return false;
        const uint32_t dst = sbase + (t ? L::kV : L::kK) + s * L::kTileBytes;
        const CUtensorMap* map = t ? &tm_v : &tm_k;
        const int key0 = j * kBN;
#ifdef PKV_TEST_HOOKS
        // test builds only: withhold this K tile's copy and arrival, so that the waits on it run out
        if (t == 0 && blockIdx.x == 0 && gg == p.test_skip_k) {
          last_k[s] = u;
          return true;
        }
#endif
        if constexpr (!kPaged) {
          if (lane == 0) {
            mbar_expect_tx(full, L::kTileBytes);
            for (int a = 0; a < L::kAtoms; ++a)
              tma_load_3d(dst + a * L::kAtomBytes, map, a * 64, kvh, sq.k0 + key0, full);
          }
        } else {
          int loaded = 0;
          for (int q = 0; q < npages; ++q)
            if (key0 + q * br < sq.Lk) ++loaded;
          // one lane per (page, atom) issues that box, after the byte count is registered
          if (lane == 0) mbar_expect_tx(full, (uint32_t)(loaded * br * 128 * kLoadAtoms));
          __syncwarp();
          if (box_lane && pg < loaded)
            tma_load_3d(dst + (kCoded ? L::kAtomBytes : at * L::kAtomBytes) + pg * br * 128, map,
                        kCoded ? 0 : at * 64, kvh, my_slot, full);
          __syncwarp();
        }
        (t ? last_v : last_k)[s] = u;
        return true;
      };
      // The next item's Q rows, prefetched into L2 once it is known, so that
      // its Q loads (which wait for this item's last S of each tile) hit L2.
      auto prefetch_next_q = [&]() {
        if (lane != 0 || next >= n_items) return;
        const Item y = item_of(p, next, next_code);
        const int lq = raw[1] - raw[0];
        if (lq <= p.route_decode) return;
        int tq[2];
        pair_tiles(lq, y.pair, p.head_pairs != 0, tq[0], tq[1]);
        for (int xq = 0; xq < 2; ++xq)
          if (tq[xq] >= 0)
            for (int a = 0; a < L::kAtoms; ++a)
              tma_prefetch_3d(&tm_q, a * 64, tile_head(p, y.head, xq), raw[0] + tq[xq] * kBM);
      };
      // K(0), Q_A, Q_B (the K stage frees up before the Q buffers do), then K
      // one tile ahead of V
      int slot_cur = tile_slot(0, tile_blk(0));
      int blk_next = tile_blk(1);
      if (!issue(0, 0, slot_cur)) { ok = false; break; }
      if (!load_q(0) || !load_q(1)) { ok = false; break; }
      const int claim_at = sq.n_kv > 3 ? sq.n_kv - 3 : 0;  // tiles ahead of the item's end
      const int resolve_at = min(claim_at + 1, sq.n_kv - 1);
      for (int j = 0; j < sq.n_kv && ok; ++j) {
        if (j == claim_at) claim_next();
        const int blk_after = tile_blk(j + 2);
        const int slot_next = (j + 1 < sq.n_kv) ? tile_slot(j + 1, blk_next) : 0;
        if (j + 1 < sq.n_kv && !issue(0, j + 1, slot_next)) { ok = false; break; }
        if (!issue(1, j, slot_cur)) { ok = false; break; }
        if (j == resolve_at) {
          resolve_next();
          prefetch_next_q();
        }
        slot_cur = slot_next;
        blk_next = blk_after;
      }
      if (!ok) break;
      resolve_next();
      it = next;
      it_code = next_code;
      g += sq.n_kv;
    }
    if (ok && !publish(-1, SeqBase{0, 0, 0, 0}, Item{0, 0, 0})) ok = false;
    if (!ok) fail();
    // Every copy this CTA issued has landed before shared memory is released.
    // These waits ignore the abort flag (a copy in flight always lands); a
    // copy that was never issued leaves its phase pending until the deadline.
    for (int s = 0; s < 2; ++s) {
      if (last_q[s] >= 0) mbar_wait(bar(kQFull0 + s), last_q[s] & 1, nullptr);
      if (last_k[s] >= 0) mbar_wait(bar(kKFull0 + s), last_k[s] & 1, nullptr);
      if (last_v[s] >= 0) mbar_wait(bar(kVFull0 + s), last_v[s] & 1, nullptr);
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------------ MMA issuers
    // Thread 0 of warp 1 issues tile A's MMAs, thread 0 of warp 2 tile B's.
    // One thread issues an M=128 MMA only every ~120-140 cycles (its own
    // issue latency, whatever N is), well below the tensor core's rate, so
    // the two tiles' MMAs come from two threads and interleave in the tensor
    // core.  Each thread runs its own tile's S and PV in issue order; the K/V
    // stages are released by one arrival of each thread.  Lanes 1..31 idle.
    const int xq = warp - 1;
    if (lane == 0) {
      constexpr uint32_t kIdescQK = make_idesc(kBM, kBN, false, kCoded);
      constexpr uint32_t kIdescPV = make_idesc(kBM, D, true, kCoded);
      bool ok = true, issued = false;
      int g = 0;   // K/V tiles consumed
      int qc = 0;  // items whose tile attends keys (Q buffer uses)
      int pc = 0;  // P tiles consumed
      int oc = 0;  // O accumulations completed (items)
      for (int u = 0; ok; ++u) {
        const int slot = u & (kRing - 1);
        if (!mbar_wait(bar(kRingFull0 + slot), (u / kRing) & 1, abort_flag)) break;
        const volatile int* e = ring + 8 * slot;
        const int it = e[0];
        const SeqBase si{e[1], e[2], e[3], e[4]};
        const int pair = e[5];
        mbar_arrive(bar(kRingEmpty0 + slot));
        if (it < 0) break;
        const Seq sq = seq_derive(p, si, pair);
        const int nkv = sq.n_kv;
        if (nkv == 0) continue;
        const int nx = xq ? sq.n[1] : sq.n[0];  // this tile's K/V tiles: 0..nkv
        if (nx == 0) {
          // this tile has no rows: release each K/V stage of the item once it is
          // loaded (K and V each on its own: with one-byte caches V(j) is widened
          // only after the producer has seen K(j-1) released)
          for (int j = 0; j < nkv && ok; ++j) {
            const int gg = g + j, s = gg & 1;
            if (!mbar_wait(bar(kKWait0 + s), (gg >> 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive(bar(kKEmpty0 + s));
            if (!mbar_wait(bar(kVWait0 + s), (gg >> 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive(bar(kVEmpty0 + s));
          }
          g += nkv;
          continue;
        }
        // S(j) = Q K(j)^T overwrites the S/P columns that the PV issued just
        // before reads: tcgen05.mma operations from one thread execute in issue
        // order, so no wait for that PV's completion is needed; the softmax
        // threads' reads of S(j-1) were ordered before that PV by its P wait.
        auto issue_s = [&](int j) -> bool {
          const int gg = g + j, s = gg & 1;
          if (!mbar_wait(bar(kKWait0 + s), (gg >> 1) & 1, abort_flag)) return false;
          if (j == 0 && !mbar_wait(bar(kQWait0 + xq), qc & 1, abort_flag)) return false;
          tc_fence_after();  // (one-byte caches: the producer's widening writes are ordered before the MMAs)
          const uint64_t qdesc = sw128_desc(sbase + L::kQ + xq * L::kTileBytes, 16, 1024);
          const uint64_t kdesc = sw128_desc(sbase + L::kK + s * L::kTileBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * L::kAtomBytes + (kk & 3) * 32) >> 4);
            mma_bf16(tS(xq), qdesc + off, kdesc + off, kIdescQK, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(kSFull0 + xq));
          mma_commit(bar(kKEmpty0 + s));
          if (j == nx - 1) mma_commit(bar(kQEmpty0 + xq));
          issued = true;
          return true;
        };
        // O += P(jt) V(jt)
        auto issue_pv = [&](int jt) -> bool {
          const int gg = g + jt, s = gg & 1;
          if (!mbar_wait(bar(kVWait0 + s), (gg >> 1) & 1, abort_flag)) return false;
          // keys at or beyond Lk (only in a sequence's last K/V tile): zero their
          // V rows, so that stale or foreign data never meets P = 0.  Both MMA
          // threads do this, each before its own PV; they only ever write zeros.
          const int valid = sq.Lk - jt * kBN;
          if (valid < kBN) {
            uint8_t* vs = smem + L::kV + s * L::kTileBytes;
            const int first = valid > 0 ? valid : 0;
            for (int a = 0; a < L::kAtoms; ++a)
              for (int row = first; row < kBN; ++row) {
                uint4* dst = reinterpret_cast<uint4*>(vs + a * L::kAtomBytes + row * 128);
#pragma unroll
                for (int c = 0; c < 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
              }
            fence_proxy_async_smem();
          }
          // the item's first PV overwrites O: the previous item's epilogue must have read it
          if (jt == 0 && oc > 0 && !mbar_wait(bar(kOFree0 + xq), (oc - 1) & 1, abort_flag)) return false;
          if (!mbar_wait(bar(kPFull0 + xq), pc & 1, abort_flag)) return false;
          tc_fence_after();  // P written (and O read) by the softmax threads before these MMAs
          // descriptors differ only in their start-address field (bits 0..13, address >> 4)
          const uint64_t vdesc = sw128_desc(sbase + L::kV + s * L::kTileBytes, L::kAtomBytes, 1024);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)  // P: 8 columns of bf16 pairs per 16 keys, keys 64.. at column 64
            mma_bf16_ts(tO(xq), tS(xq) + 8 * kk + (kk >= 4 ? 32 : 0), vdesc + (uint64_t)((16 * kk * 128) >> 4),
                        kIdescPV, (jt > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(kVEmpty0 + s));
          if (jt == nx - 1) mma_commit(bar(kODone0 + xq));
          ++pc;
          if (jt == nx - 1) ++oc;
          return true;
        };
        // K/V tiles past this tile's last visible one (tile A only): released once loaded
        auto pass = [&](int bar0, int full0, int jt) -> bool {
          const int gg = g + jt, s = gg & 1;
          if (!mbar_wait(bar(full0 + s), (gg >> 1) & 1, abort_flag)) return false;
          mbar_arrive(bar(bar0 + s));
          return true;
        };
        for (int j = 0; j <= nkv && ok; ++j) {
          if (j >= 1 && !(j - 1 < nx ? issue_pv(j - 1) : pass(kVEmpty0, kVWait0, j - 1))) ok = false;
          if (ok && j < nkv && !(j < nx ? issue_s(j) : pass(kKEmpty0, kKWait0, j))) ok = false;
        }
        if (!ok) break;
        ++qc;
        g += nkv;
      }
      if (!ok) fail();
      // drain: all MMAs this thread issued have completed before TMEM is
      // released (an issued MMA always completes, so the abort flag is ignored)
      if (issued) {
        mma_commit(bar(kDrain0 + xq));
        mbar_wait(bar(kDrain0 + xq), 0, nullptr);
      }
    }
    __syncwarp();  // the warp reconverges before the CTA barrier below
  } else if (!kCoded || warp < kWidenWarp) {
    if constexpr (!kUnified) {
      // ------------------------------------------------------------------ softmax warps
      const int xq = (warp - kSoftmaxWarp0) >> 2;  // query tile of this warp group
      const int quarter = warp & 3;       // TMEM lanes this warp may access
      const int r = quarter * 32 + lane;  // TMEM lane == query row in the tile
      const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
      const float c = p.scale_log2;
      bool ok = true;
      int sc = 0, oc = 0;  // S tiles and items (with keys) processed
      int tc = 0;          // tiles processed in turn with the other group
      for (int u = 0; ok; ++u) {
        SeqBase si;
        Item x;
        const int it = ring_get(u, si, x);
        if (it < 0) break;
        // Only a few values live across the tile loop (the 128 scores need the
        // registers): the output offsets, the row limits and the loop counts.
        int rows, nkv, vis0, jm;
        int64_t obase, lse_idx;  // this tile's first output element; this row's lse index
        int nturn;  // tiles taken in turn with the other group: the first n[0]
        {
          const Seq sq = seq_derive(p, si, x.pair);
          // (selects, not an indexed load: xq differs between warps but the arrays stay in registers)
          rows = xq ? sq.rows[1] : sq.rows[0];
          const int row0 = xq ? sq.row0[1] : sq.row0[0];
          nkv = xq ? sq.n[1] : sq.n[0];
          const int head = xq ? x.head_b : x.head * (1 + p.head_pairs);  // tile_head(p, x.head, xq)
          obase = ((int64_t)(sq.q0 + row0) * p.num_heads + head) * D;
          lse_idx = (int64_t)head * p.total_q + sq.q0 + row0 + r;
          // key limit of this row (bottom-right causal, inside the keys); tiles
          // before jm need no mask for any row of the tile (its first row has
          // the smallest limit)
          vis0 = min(row0 + r + sq.diag, sq.Lk - 1);
          const int first = row0 + sq.diag;  // limit of the tile's first row
          jm = min(first < kBN - 1 ? 0 : (first + 1) / kBN, sq.Lk / kBN);
          // While both tiles have K/V tiles left, the two groups take turns, tile
          // by tile (A0, B0, A1, B1, ...): each softmax then has the SM's
          // sub-partitions to itself, and while one group works the other tile's
          // MMAs run.  Tile B's tiles past A's last one run without turns.
          nturn = sq.n[0];
        }
        if (rows <= 0) continue;
        // the offsets wait in shared memory while the tile loop runs (registers)
        int64_t* epi = reinterpret_cast<int64_t*>(smem + L::kEpi) + 4 * (threadIdx.x - kSoftmaxWarp0 * 32);
        epi[0] = obase;
        epi[1] = lse_idx;
        epi[2] = rows;
        if (nkv == 0) {
          const bool row_valid = r < rows;
          // rows that see no key: zeros and lse = -inf
          if (row_valid) {
            uint16_t* orow = p.out + obase + (int64_t)r * p.num_heads * D;
            for (int cc = 0; cc < D / 8; ++cc) reinterpret_cast<uint4*>(orow)[cc] = make_uint4(0, 0, 0, 0);
            if (p.lse) p.lse[lse_idx] = -INFINITY;
          }
          continue;
        }
        float m = -INFINITY, l = 0.f;
        for (int j = 0; j < nkv; ++j) {
          if (!mbar_wait(bar(kSFull0 + xq), sc & 1, abort_flag)) { ok = false; break; }
          ++sc;
          if (j < nturn) {  // tile A waits for B's previous tile, tile B for A's current one
            const int need = xq == 0 ? tc - 1 : tc;
            if (need >= 0 && !mbar_wait(bar(kTurn0 + xq), need & 1, abort_flag)) { ok = false; break; }
          }
          tc_fence_after();
          // All 128 scores of the row in one TMEM round trip; P of keys 64..127
          // goes to columns 64..95 and of keys 0..63 to columns 0..31 (each half
          // over S columns already read; columns 32..63 and 96..127 are unused).
          const int key0 = j * kBN;
          uint32_t sr[kBN];
          PKV_TMEM_LD32(tS(xq) + lane_off + 0, (sr + 0));
          PKV_TMEM_LD32(tS(xq) + lane_off + 32, (sr + 32));
          PKV_TMEM_LD32(tS(xq) + lane_off + 64, (sr + 64));
          PKV_TMEM_LD32(tS(xq) + lane_off + 96, (sr + 96));
          tmem_wait_ld();
          if (j >= jm) {
            const int vis = vis0 - key0;  // columns 0..vis are visible
  #pragma unroll
            for (int k = 0; k < kBN; ++k) sr[k] = (k <= vis) ? sr[k] : __float_as_uint(-INFINITY);
          }
          float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  #pragma unroll
          for (int k = 0; k < kBN; k += 2)
            mx4[(k >> 1) & 3] = fmax3(mx4[(k >> 1) & 3], __uint_as_float(sr[k]), __uint_as_float(sr[k + 1]));
          const float mt = fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3])) * c;
          float m_use = m;
          if (mt > m + kRescaleThreshold || (m == -INFINITY && mt != -INFINITY)) m_use = mt;
          const bool live = m_use != -INFINITY;
          const bool moved = m_use != m;
          const float alpha = (moved && m != -INFINITY) ? fast_exp2(m - m_use) : (moved ? 0.f : 1.f);
          // p = 2^(s*c - m) on fp32 pairs; a row that saw no key yet (m = -inf) gives 0
          const float nm = live ? -m_use : -INFINITY;
          const uint64_t c2 = f32x2_pack(c, c), nm2 = f32x2_pack(nm, nm);
          uint64_t sum2[2] = {0ull, 0ull};
  #pragma unroll
          for (int h = 1; h >= 0; --h) {
            // P of keys 64h..64h+63 as bf16 pairs, packed in place over the scores just used
            uint32_t* pk = sr + 64 * h;
  #pragma unroll
            for (int k = 0; k < 64; k += 2) {
              float x0, x1;
              f32x2_unpack(ffma2(f32x2_pack(__uint_as_float(pk[k]), __uint_as_float(pk[k + 1])), c2, nm2), x0, x1);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              sum2[(k >> 1) & 1] = fadd2(sum2[(k >> 1) & 1], f32x2_pack(p0, p1));
              pk[k >> 1] = kCoded ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
            }
            PKV_TMEM_ST32(tS(xq) + lane_off + 64 * h, pk);
          }
          float s00, s01, s10, s11;
          f32x2_unpack(sum2[0], s00, s01);
          f32x2_unpack(sum2[1], s10, s11);
          l = l * alpha + ((s00 + s01) + (s10 + s11));
          m = m_use;
          // rescale O_X when this row's reference max moved (warp-collective TMEM
          // access).  PV_X of the previous tile is done: it was issued before this
          // tile's S, whose completion was just waited for.
          if (j > 0 && __any_sync(0xffffffffu, moved && alpha != 1.f)) {
  #pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
              uint32_t o[32];
              PKV_TMEM_LD32(tO(xq) + lane_off + ch * 32, o);
              tmem_wait_ld();
  #pragma unroll
              for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
              PKV_TMEM_ST32(tO(xq) + lane_off + ch * 32, o);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(kPFull0 + xq));
          if (j < nturn) {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kTurn0 + (xq ^ 1)));
            ++tc;
          }
        }
        if (!ok) break;
        // ---- epilogue: O_X / l, released as soon as it is read, then stored ----
        if (!mbar_wait(bar(kODone0 + xq), oc & 1, abort_flag)) {
          ok = false;
          break;
        }
        ++oc;
        tc_fence_after();
        const float inv = l > 0.f ? p.v_mul / l : 0.f;
        obase = epi[0];
        lse_idx = epi[1];
        const bool row_valid = r < (int)epi[2];
        // O, normalised, packed to bf16 and stored 32 columns at a time; O is
        // released once read.  Head dim 64: the whole row in one TMEM round trip
        // (64 registers).  Head dim 128: chunk by chunk, so that no 128-register
        // row is live (that spilled and cost 2-6 %).
        uint4* orow = reinterpret_cast<uint4*>(p.out + obase + (int64_t)r * p.num_heads * D);
        constexpr int kOneTrip = D <= 64;
        uint32_t o_all[kOneTrip ? D : 32];
        if constexpr (kOneTrip) {
  #pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) PKV_TMEM_LD32(tO(xq) + lane_off + ch * 32, (o_all + ch * 32));
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(bar(kOFree0 + xq));
        }
  #pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          const uint32_t* o = o_all + (kOneTrip ? ch * 32 : 0);
          if constexpr (!kOneTrip) {
            PKV_TMEM_LD32(tO(xq) + lane_off + ch * 32, o_all);
            tmem_wait_ld();
            if (ch == D / 32 - 1) {
              tc_fence_before();
              mbar_arrive(bar(kOFree0 + xq));
            }
          }
          if (row_valid) {
            uint32_t w[16];
  #pragma unroll
            for (int k = 0; k < 16; ++k)
              w[k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv, __uint_as_float(o[2 * k + 1]) * inv);
            if (p.out_v8) {  // whole 32-byte sectors, half the store instructions
  #pragma unroll
              for (int h = 0; h < 2; ++h)
                asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(orow + ch * 4 + 2 * h),
                             "r"(w[8 * h]), "r"(w[8 * h + 1]), "r"(w[8 * h + 2]), "r"(w[8 * h + 3]), "r"(w[8 * h + 4]),
                             "r"(w[8 * h + 5]), "r"(w[8 * h + 6]), "r"(w[8 * h + 7])
                             : "memory");
            } else {
  #pragma unroll
              for (int q = 0; q < 4; ++q) orow[ch * 4 + q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            }
          }
        }
        if (row_valid && p.lse != nullptr) p.lse[lse_idx] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
      }
      if (!ok) fail();
      tc_fence_before();
    } else {
      // ------------------------------------------------------------------ softmax warps
      // All eight warps work on one tile at a time, A then B, K/V tile by K/V
      // tile (A0, B0, A1, B1, ...): while they run one tile's softmax the other
      // tile's MMAs run.  Warps 3..6 take keys 0..63 of their rows, warps 7..10
      // keys 64..127 (TMEM lanes (warp % 4) * 32 + lane in both): two warps per
      // sub-partition share each row, swapping the row maxima through shared
      // memory; the row sums are combined once, at the epilogue.
      const int tid = threadIdx.x - kSoftmaxWarp0 * 32;  // 0..255
      const int hk = tid >> 7;                            // key half of this thread
      const int quarter = warp & 3;       // TMEM lanes this warp may access
      const int r = quarter * 32 + lane;  // TMEM lane == query row in the tile
      const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
      const float c = p.scale_log2;
      volatile float* xch = reinterpret_cast<volatile float*>(smem + L::kXch);  // [2][256]
      bool ok = true;
      int sc[2] = {0, 0}, oc[2] = {0, 0};  // S tiles and items (with keys) processed, per tile
      int xc = 0;                          // exchanges with the other half
      // this thread's value v for exchange round xc, plus the partner's
      auto exchange = [&](float v) -> float {
        xch[(xc & 1) * kSoftmaxThreads + tid] = v;
        mbar_arrive(bar(kXch0));
        if (!mbar_wait(bar(kXch0), xc & 1, abort_flag)) ok = false;
        const float o = xch[(xc & 1) * kSoftmaxThreads + (tid ^ 128)];
        ++xc;
        return o;
      };
      for (int u = 0; ok; ++u) {
        SeqBase si;
        Item x;
        const int it = ring_get(u, si, x);
        if (it < 0) break;
        int rows[2], nkv[2], vis0[2], jm[2];
        float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
        {
          const Seq sq = seq_derive(p, si, x.pair);
  #pragma unroll
          for (int xq = 0; xq < 2; ++xq) {
            rows[xq] = sq.rows[xq];
            nkv[xq] = sq.n[xq];
            const int row0 = sq.row0[xq];
            const int head = xq ? x.head_b : x.head * (1 + p.head_pairs);  // tile_head(p, x.head, xq)
            // the offsets wait in shared memory while the tile loop runs (registers)
            int64_t* epi = reinterpret_cast<int64_t*>(smem + L::kEpi) + 4 * (xq * kSoftmaxThreads + tid);
            epi[0] = ((int64_t)(sq.q0 + row0) * p.num_heads + head) * D;  // the tile's first output element
            epi[1] = (int64_t)head * p.total_q + sq.q0 + row0 + r;         // this row's lse index
            // key limit of this row (bottom-right causal, inside the keys); tiles
            // before jm need no mask for any row of the tile (its first row has
            // the smallest limit)
            vis0[xq] = min(row0 + r + sq.diag, sq.Lk - 1);
            const int first = row0 + sq.diag;  // limit of the tile's first row
            jm[xq] = min(first < kBN - 1 ? 0 : (first + 1) / kBN, sq.Lk / kBN);
          }
        }
        // rows that see no key: zeros and lse = -inf (each half its 64 columns)
  #pragma unroll
        for (int xq = 0; xq < 2; ++xq) {
          if (rows[xq] <= 0 || nkv[xq] != 0 || r >= rows[xq]) continue;
          const int64_t* epi = reinterpret_cast<const int64_t*>(smem + L::kEpi) + 4 * (xq * kSoftmaxThreads + tid);
          uint16_t* orow = p.out + epi[0] + (int64_t)r * p.num_heads * D;
          for (int cc = hk * (D / 16); cc < (hk + 1) * (D / 16); ++cc)
            reinterpret_cast<uint4*>(orow)[cc] = make_uint4(0, 0, 0, 0);
          if (p.lse && hk == 0) p.lse[epi[1]] = -INFINITY;
        }
        const bool live_a = rows[0] > 0 && nkv[0] > 0, live_b = rows[1] > 0 && nkv[1] > 0;
        const int nmax = max(live_a ? nkv[0] : 0, live_b ? nkv[1] : 0);
        // one softmax step of tile xq over its K/V tile j
        auto step = [&](const int xq, const int j) {
          if (!mbar_wait(bar(kSFull0 + xq), sc[xq] & 1, abort_flag)) {
            ok = false;
            return;
          }
          ++sc[xq];
          tc_fence_after();
          // this half's 64 scores of the row in one TMEM round trip; P of its keys
          // goes, as bf16 pairs, over the first 32 of its S columns (already read)
          const int key0 = j * kBN + hk * 64;
          uint32_t sr[64];
          PKV_TMEM_LD32(tS(xq) + lane_off + hk * 64, (sr + 0));
          PKV_TMEM_LD32(tS(xq) + lane_off + hk * 64 + 32, (sr + 32));
          tmem_wait_ld();
          if (j >= jm[xq]) {
            const int vis = vis0[xq] - key0;  // columns 0..vis of this half are visible
  #pragma unroll
            for (int k = 0; k < 64; ++k) sr[k] = (k <= vis) ? sr[k] : __float_as_uint(-INFINITY);
          }
          float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  #pragma unroll
          for (int k = 0; k < 64; k += 2)
            mx4[(k >> 1) & 3] = fmax3(mx4[(k >> 1) & 3], __uint_as_float(sr[k]), __uint_as_float(sr[k + 1]));
          const float mine = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
          const float mt = fmaxf(mine, exchange(mine)) * c;
          if (!ok) return;
          const float mo = m[xq];
          float m_use = mo;
          if (mt > mo + kRescaleThreshold || (mo == -INFINITY && mt != -INFINITY)) m_use = mt;
          const bool live = m_use != -INFINITY;
          const bool moved = m_use != mo;
          const float alpha = (moved && mo != -INFINITY) ? fast_exp2(mo - m_use) : (moved ? 0.f : 1.f);
          // p = 2^(s*c - m) on fp32 pairs; a row that saw no key yet (m = -inf) gives 0
          const float nm = live ? -m_use : -INFINITY;
          const uint64_t c2 = f32x2_pack(c, c), nm2 = f32x2_pack(nm, nm);
          uint64_t sum2[2] = {0ull, 0ull};
  #pragma unroll
          for (int k = 0; k < 64; k += 2) {
            float x0, x1;
            f32x2_unpack(ffma2(f32x2_pack(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), c2, nm2), x0, x1);
            const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
            sum2[(k >> 1) & 1] = fadd2(sum2[(k >> 1) & 1], f32x2_pack(p0, p1));
            sr[k >> 1] = kCoded ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
          }
          PKV_TMEM_ST32(tS(xq) + lane_off + hk * 64, sr);
          float s00, s01, s10, s11;
          f32x2_unpack(sum2[0], s00, s01);
          f32x2_unpack(sum2[1], s10, s11);
          l[xq] = l[xq] * alpha + ((s00 + s01) + (s10 + s11));
          m[xq] = m_use;
          // rescale this half's columns of O_X when the row's reference max moved
          // (warp-collective TMEM access).  PV_X of the previous tile is done: it
          // was issued before this tile's S, whose completion was just waited for.
          if (j > 0 && __any_sync(0xffffffffu, moved && alpha != 1.f)) {
  #pragma unroll
            for (int ch = 0; ch < D / 64; ++ch) {
              uint32_t o[32];
              PKV_TMEM_LD32(tO(xq) + lane_off + hk * (D / 2) + ch * 32, o);
              tmem_wait_ld();
  #pragma unroll
              for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
              PKV_TMEM_ST32(tO(xq) + lane_off + hk * (D / 2) + ch * 32, o);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(kPFull0 + xq));
        };
        for (int j = 0; j < nmax && ok; ++j) {
          if (live_a && j < nkv[0]) step(0, j);
          if (ok && live_b && j < nkv[1]) step(1, j);
        }
        if (!ok) break;
        // ---- epilogue of each tile with keys: O_X / l, released once read, then stored ----
  #pragma unroll
        for (int xq = 0; xq < 2; ++xq) {
          if (!(xq ? live_b : live_a)) continue;
          const float lt = l[xq] + exchange(l[xq]);  // the whole row's sum
          if (!ok) break;
          if (!mbar_wait(bar(kODone0 + xq), oc[xq] & 1, abort_flag)) {
            ok = false;
            break;
          }
          ++oc[xq];
          tc_fence_after();
          const float inv = lt > 0.f ? p.v_mul / lt : 0.f;
          const int64_t* epi = reinterpret_cast<const int64_t*>(smem + L::kEpi) + 4 * (xq * kSoftmaxThreads + tid);
          const bool row_valid = r < rows[xq];
          uint4* orow = reinterpret_cast<uint4*>(p.out + epi[0] + (int64_t)r * p.num_heads * D);
          // this half's D/2 columns of O, 32 at a time, normalised, packed to bf16
          // and stored; O is released once every chunk is read
  #pragma unroll
          for (int cl = 0; cl < D / 64; ++cl) {
            const int ch = hk * (D / 64) + cl;  // 32-column chunk of the row
            uint32_t o[32];
            PKV_TMEM_LD32(tO(xq) + lane_off + ch * 32, o);
            tmem_wait_ld();
            if (cl == D / 64 - 1) {
              tc_fence_before();
              mbar_arrive(bar(kOFree0 + xq));
            }
            if (row_valid) {
              uint32_t w[16];
  #pragma unroll
              for (int k = 0; k < 16; ++k)
                w[k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv, __uint_as_float(o[2 * k + 1]) * inv);
              if (p.out_v8) {  // whole 32-byte sectors, half the store instructions
  #pragma unroll
                for (int h = 0; h < 2; ++h)
                  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(orow + ch * 4 + 2 * h),
                               "r"(w[8 * h]), "r"(w[8 * h + 1]), "r"(w[8 * h + 2]), "r"(w[8 * h + 3]),
                               "r"(w[8 * h + 4]), "r"(w[8 * h + 5]), "r"(w[8 * h + 6]), "r"(w[8 * h + 7])
                               : "memory");
              } else {
  #pragma unroll
                for (int q = 0; q < 4; ++q)
                  orow[ch * 4 + q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
              }
            }
          }
          if (row_valid && hk == 0 && p.lse != nullptr)
            p.lse[epi[1]] = lt > 0.f ? (m[xq] + log2f(lt)) * kLn2 : -INFINITY;
        }
      }
      if (!ok) fail();
      tc_fence_before();
    }
  } else {
    // ------------------------------------------------------------------ widening warp
    // One-byte caches: each landed Q, K and V tile of the published items, in
    // the order the MMA threads use them, is widened in place to f16 and
    // released to them (the whole warp converts; lane 0 signals).
    if constexpr (kCoded) {
      bool ok = true;
      int g = 0;                // K/V tiles
      int qc[2] = {0, 0};       // Q loads per tile slot
      auto widen = [&](int full, uint32_t parity, int ready, uint8_t* buf, bool q) -> bool {
        int wok = 1;
        if (lane == 0) wok = mbar_wait(bar(full), parity, abort_flag);
        if (!__shfl_sync(0xffffffffu, wok, 0)) return false;
        mbar_wait(bar(full), parity, abort_flag);  // every lane acquires the landed bytes (complete)
        if (q)
          widen_q_f16(buf, lane);
        else
          widen_kv_f16<kCode>(buf, lane);
        fence_proxy_async_smem();  // the generic writes, before the tensor core reads them
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(ready));
        return true;
      };
      for (int u = 0; ok; ++u) {
        SeqBase si;
        Item x;
        if (__any_sync(0xffffffffu, ring_get(u, si, x) < 0)) break;  // (every lane reads the entry)
        const Seq sq = seq_derive(p, si, x.pair);
        if (sq.n_kv == 0) continue;
        for (int xq = 0; xq < 2 && ok; ++xq) {
          if (sq.n[xq] == 0) continue;
          if (!widen(kQFull0 + xq, (uint32_t)qc[xq] & 1u, kQReady0 + xq, smem + L::kQ + xq * L::kTileBytes, true))
            ok = false;
          ++qc[xq];
        }
        for (int j = 0; j < sq.n_kv && ok; ++j) {
          const int gg = g + j, s = gg & 1;
          const uint32_t par = (uint32_t)(gg >> 1) & 1u;
          if (!widen(kKFull0 + s, par, kKReady0 + s, smem + L::kK + s * L::kTileBytes, false) ||
              !widen(kVFull0 + s, par, kVReady0 + s, smem + L::kV + s * L::kTileBytes, false))
            ok = false;
        }
        g += sq.n_kv;
      }
      if (!ok && lane == 0) fail();
      __syncwarp();
    }
  }

  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// Tile-count buckets of the unit order (counts past the last share it).
constexpr int kOrderBuckets = 1024;

// Exclusive prefix sum of v over the CTA's threads (in thread order) and the
// CTA's total: a shuffle scan within each warp, then one warp scans the warp
// totals.  ws: 33 shared slots; every thread of the CTA calls it.
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* ws, T& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  T x = v;  // inclusive within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const T w = lane < nw ? ws[lane] : T(0);
    T wx = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T y = __shfl_up_sync(0xffffffffu, wx, o);
      if (lane >= o) wx += y;
    }
    if (lane < nw) ws[lane] = wx - w;  // warps before this one
    if (lane == 31) ws[32] = wx;
  }
  __syncthreads();
  const T r = ws[warp] + x - v;
  total = ws[32];
  __syncthreads();  // (ws is free for the next call)
  return r;
}

// SM split of a mixed batch.  The prefill CTAs hold one SM each for the whole
// call, and the decode kernels that serve the routed rows start on the SMs the
// prefill leaves free, then take the prefill's SMs as its CTAs finish.  The
// prep kernel models the call's time for every prefill CTA count K and runs
// the best K (all SMs when no row is routed):
// - a prefill work item takes kItemNs plus kStepNs per K/V step at head dim
//   128 (measured on this kernel: about 1.3 and 2.1 us; head dim 64 steps take
//   0.8 of that, one-byte pages widened in the tile loop 1.4x);
// - the prefill on K CTAs ends at max(P / K, t_1, t_K + t_(K+1)), P the summed
//   item times and t_i the i-th longest item: the longest-first order puts the
//   first K items on their own CTAs, and the next one after the shortest of them;
// - the routed rows' K/V bytes stream at kDecodeBytesPerNs per SM (about 45 GB/s
//   measured per SM of the split-KV kernel), on the S - K free SMs until the
//   prefill ends and on all S after, at most at kDecodeChipBytesPerNs.
constexpr float kItemNs = 1300.f;
constexpr float kStepNs = 2100.f;
constexpr float kDecodeBytesPerNs = 45.f;
constexpr float kDecodeChipBytesPerNs = 5800.f;
constexpr float kSplitSlack = 0.02f;

struct PrepArgs {
  const int32_t* cu_q;
  const int32_t* cu_k;
  int batch;
  // routed rows (items == nullptr: none)
  int32_t* items;
  int32_t* count;
  int route_cap;
  int route_max_q;   // sequences with up to this many queries are routed (0: none)
  int per_sequence;  // one item per routed sequence (else one per query row)
  // prefill work items and unit list (unit_order == nullptr: no prefill kernel)
  int32_t* item_counter;
  int32_t* unit_order;
  int4* unit_seq;
  int32_t* n_units;
  int units_cap;
  int n_pairs;
  int head_pairs;
  int item_heads;
  // SM split: prefill CTAs that run (of sms)
  int32_t* active_ctas;
  int sms;
  float step_ns;          // kStepNs scaled to the head dim and page format
  float decode_pos_bytes; // K/V bytes of one routed position (all kv heads)
  // gathered sequences' packed offsets (cu_g == nullptr: no gather)
  int32_t* cu_g;
  int64_t gather_cap;
  int32_t* err;
};

// Varlen prep (one CTA of 1024 threads): compacts the sequences the decode
// kernels serve (one query, or up to route_max_q) into items[0..*count),
// resets the prefill kernel's work-item counter, writes the packed offsets of
// a gathered batch, then the prefill unit list (with each unit's sequence
// offsets, so that a claimed item needs one round of loads) and the SM split.
__global__ void __launch_bounds__(1024) varlen_prep_kernel(const PrepArgs a) {
  // the kernel after this one (the gather, or the prefill when no gather runs)
  // may launch now: it waits for this grid's completion before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ int n;
  __shared__ int64_t carry;
  __shared__ unsigned long long routed_pos;  // positions the routed items read (decode load)
  __shared__ unsigned long long unit_tiles;  // K/V tile steps of all prefill units
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // Every section below visits sequence b = threadIdx.x first: its offsets are
  // loaded once, here (later sequences of a batch above blockDim load again).
  int f_q0 = 0, f_q1 = 0, f_k0 = 0, f_k1 = 0;
  if ((int)threadIdx.x < a.batch) {
    f_q0 = __ldg(a.cu_q + threadIdx.x);
    f_q1 = __ldg(a.cu_q + threadIdx.x + 1);
    f_k0 = __ldg(a.cu_k + threadIdx.x);
    f_k1 = __ldg(a.cu_k + threadIdx.x + 1);
  }
  auto offsets = [&](int b, int& q0, int& q1, int& k0, int& k1) {
    if (b == (int)threadIdx.x) {
      q0 = f_q0, q1 = f_q1, k0 = f_k0, k1 = f_k1;
    } else {
      q0 = __ldg(a.cu_q + b), q1 = __ldg(a.cu_q + b + 1), k0 = __ldg(a.cu_k + b), k1 = __ldg(a.cu_k + b + 1);
    }
  };
  if (threadIdx.x == 0) {
    n = 0;
    carry = 0;
    routed_pos = 0;
    unit_tiles = 0;
    *a.item_counter = 0;
  }
  __syncthreads();
  if (a.items != nullptr) {
    // every query row of a sequence with 1..route_max_q queries (item codes
    // b * kRouteCode + qi; the bound route_cap holds them all), or, with
    // per_sequence, one item per such sequence (code b * kRouteCode)
    // (slots claimed once per warp: the lanes' counts scanned, one atomic)
    unsigned long long pos = 0;
    for (int b0 = 0; b0 < a.batch; b0 += blockDim.x) {
      const int b = b0 + threadIdx.x;
      int nq = 0, lk = 0;
      if (b < a.batch) {
        int q0, q1, k0, k1;
        offsets(b, q0, q1, k0, k1);
        const int lq = q1 - q0;
        if (lq >= 1 && lq <= a.route_max_q) nq = a.per_sequence ? 1 : lq;
        lk = k1 - k0;
      }
      int x = nq;  // inclusive warp scan of the counts
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      int wbase = 0;
      if (lane == 31 && x > 0) wbase = atomicAdd(&n, x);
      const int base = __shfl_sync(0xffffffffu, wbase, 31) + x - nq;
      for (int i = 0; i < nq; ++i)
        if (base + i < a.route_cap) a.items[base + i] = b * kRouteCode + i;
      if (nq > 0 && lk > 0) pos += (unsigned long long)lk * nq;
    }
    for (int o = 16; o > 0; o >>= 1) pos += __shfl_xor_sync(0xffffffffu, pos, o);
    if (lane == 0 && pos) atomicAdd(&routed_pos, pos);
    __syncthreads();
    if (threadIdx.x == 0) *a.count = n < a.route_cap ? n : a.route_cap;
  }
  if (a.cu_g != nullptr) {
    // Packed offsets of the gathered sequences (those the prefill kernel
    // serves: more than one query, or any query when nothing is routed):
    // cu_g[b] = sum of their key counts before b.  An exclusive scan over the
    // CTA per chunk of blockDim sequences, carried across chunks.
    __shared__ int64_t scan_ws[33];
    for (int base = 0; base < a.batch; base += blockDim.x) {
      const int b = base + threadIdx.x;
      int64_t v = 0;
      if (b < a.batch) {
        int q0, q1, k0, k1;
        offsets(b, q0, q1, k0, k1);
        const int lq = q1 - q0, lk = k1 - k0;
        const bool gathered = lq > a.route_max_q;
        v = gathered && lk > 0 ? lk : 0;
      }
      int64_t chunk = 0;
      const int64_t before = block_exclusive_scan(v, scan_ws, chunk);
      if (b < a.batch) a.cu_g[b] = (int32_t)(carry + before);
      __syncthreads();  // (every thread has read carry)
      if (threadIdx.x == 0) carry += chunk;
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      a.cu_g[a.batch] = (int32_t)carry;
      if (carry > a.gather_cap) flag_error(a.err, PKV_DEVERR_LENGTH);  // rows past the buffer are not gathered
    }
    __syncthreads();  // (the unit list below reads cu_g)
  }
  if (a.unit_order != nullptr) {
    // The prefill kernel's units (sequence b, pair pe, for the sequences it
    // serves) in longest-processing-time order: by the K/V tiles the pair
    // reads, most first, so that the longest items start at once and the
    // short ones fill in at the end.  A counting sort over the tile counts;
    // units with equal counts land in any order, which changes no result.
    // blockDim.x (1024) divides kOrderBuckets.
    __shared__ int hist[kOrderBuckets];
    __shared__ int wtot[33];
    __shared__ float wbest_t[33];  // per-warp minima, then (slot 32) the CTA's
    __shared__ int wbest_k[32];    // per-warp picks
    __shared__ int s_units;
    for (int i = threadIdx.x; i < kOrderBuckets; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    // a group of lps lanes per sequence (a power of two, up to a warp: more
    // lanes for fewer sequences), the group's lanes taking the units in turn
    int lps = 1;
    while (lps < 32 && lps * 2 * a.batch <= (int)blockDim.x) lps *= 2;
    const int grp = threadIdx.x / lps, sub = threadIdx.x % lps, ngrp = blockDim.x / lps;
    for (int pass = 0; pass < 2; ++pass) {
      unsigned long long tiles = 0;
      for (int b = grp; b < a.batch; b += ngrp) {
        int q0, q1, ck0, ck1;
        offsets(b, q0, q1, ck0, ck1);
        const int lq = q1 - q0;
        const int lk = ck1 - ck0;
        if (lq < 0 || lk < 0) {
          if (pass == 0) flag_error(a.err, PKV_DEVERR_LENGTH);
          continue;
        }
        if (lq <= a.route_max_q) continue;  // no rows, or left to the decode kernels
        const int T = (lq + kBM - 1) / kBM;
        const int all = a.head_pairs ? T : (T + 1) / 2;
        if (pass == 0 && all > a.n_pairs) flag_error(a.err, PKV_DEVERR_LENGTH);  // more queries than max_len_q
        const int nu = min(all, a.n_pairs);
        // the offsets the prefill kernel reads K/V at: the packed copy's when gathered
        // (cu_g is written above by other threads of this CTA: plain loads)
        const int k0 = pass == 1 ? (a.cu_g != nullptr ? a.cu_g[b] : ck0) : 0;
        const int k1 = pass == 1 ? (a.cu_g != nullptr ? a.cu_g[b + 1] : ck1) : 0;
        for (int pe = sub; pe < nu; pe += lps) {
          const int t = unit_kv_tiles(lq, lk, pe, a.head_pairs != 0);
          const int c = min(t, kOrderBuckets - 1);
          if (pass == 0) {
            atomicAdd(&hist[c], 1);
            tiles += t;
          } else {
            const int pos = atomicAdd(&hist[c], 1);
            if (pos < a.units_cap) {
              a.unit_order[pos] = b * a.n_pairs + pe;
              a.unit_seq[pos] = make_int4(q0, q1, k0, k1);
            } else
              flag_error(a.err, PKV_DEVERR_LENGTH);  // more query rows than total_q
          }
        }
      }
      for (int o = 16; o > 0; o >>= 1) tiles += __shfl_xor_sync(0xffffffffu, tiles, o);
      if (lane == 0 && tiles) atomicAdd(&unit_tiles, tiles);
      __syncthreads();
      if (pass == 1) break;
      // bucket c -> first position of its units: the units with more tiles
      // come before it.  Thread t owns the buckets kOrderBuckets-1-t*per-i.
      const int per = kOrderBuckets / blockDim.x;
      int local = 0;
      for (int i = 0; i < per; ++i) local += hist[kOrderBuckets - 1 - threadIdx.x * per - i];
      int all_units = 0;
      int run = block_exclusive_scan(local, wtot, all_units);
      for (int i = 0; i < per; ++i) {
        const int c = kOrderBuckets - 1 - threadIdx.x * per - i;
        const int h = hist[c];
        hist[c] = run;
        run += h;
      }
      if (threadIdx.x == blockDim.x - 1) {
        s_units = run < a.units_cap ? run : a.units_cap;
        *a.n_units = s_units;
      }
      __syncthreads();
      // SM split (hist holds each bucket's first position): thread K-1 models K
      // prefill CTAs; the largest K whose modelled time is within kSplitSlack
      // of the smallest runs (near the best K the model is flat, while one CTA
      // too few for the longest items costs a whole item)
      const int units = s_units;
      if (routed_pos == 0 || units == 0) {  // (uniform) nothing routed: every CTA
        if (threadIdx.x == 0) *a.active_ctas = a.sms;
        continue;
      }
      float t_mine = INFINITY;
      const int K = threadIdx.x + 1;
      if (K <= a.sms) {
        // time of the j-th longest item: its unit's bucket is the lowest one
        // whose first position is at most the unit's rank
        auto item_t = [&](int j) -> float {  // (item numbers fit int32: checked on the host)
          const int r = j / a.item_heads;
          int lo = 0, hi = kOrderBuckets - 1;  // hist[kOrderBuckets - 1] == 0 <= r
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (hist[mid] <= r) hi = mid; else lo = mid + 1;
          }
          return kItemNs + a.step_ns * (float)lo;
        };
        const int n_items = units * a.item_heads;
        const float P = (float)a.item_heads * ((float)units * kItemNs + (float)unit_tiles * a.step_ns);
        const float D = (float)routed_pos * a.decode_pos_bytes;  // bytes
        float tp = fmaxf(P / (float)K, item_t(0));
        if (n_items > K) tp = fmaxf(tp, item_t(K - 1) + item_t(K));
        const float free_rate = (float)(a.sms - K) * kDecodeBytesPerNs;
        const float all_rate = fminf((float)a.sms * kDecodeBytesPerNs, kDecodeChipBytesPerNs);
        t_mine = D <= free_rate * tp ? tp : tp + (D - free_rate * tp) / all_rate;
      }
      // CTA-wide minimum of the modelled times, then the largest K within the slack
      // (warp shuffles, then warp 0 over the warps' results)
      const int nw = blockDim.x >> 5;
      float t_min = t_mine;
      for (int o = 16; o > 0; o >>= 1) t_min = fminf(t_min, __shfl_xor_sync(0xffffffffu, t_min, o));
      if (lane == 0) wbest_t[warp] = t_min;
      __syncthreads();
      if (warp == 0) {
        float v = lane < nw ? wbest_t[lane] : INFINITY;
        for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) wbest_t[32] = v;
      }
      __syncthreads();
      t_min = wbest_t[32];
      int k_pick = t_min < INFINITY && t_mine <= t_min * (1.f + kSplitSlack) ? K : 0;
      for (int o = 16; o > 0; o >>= 1) k_pick = max(k_pick, __shfl_xor_sync(0xffffffffu, k_pick, o));
      if (lane == 0) wbest_k[warp] = k_pick;
      __syncthreads();
      if (warp == 0) {
        int v = lane < nw ? wbest_k[lane] : 0;
        for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) *a.active_ctas = v > 0 ? v : a.sms;
      }
      __syncthreads();
    }
  }
}

// Gather (paged -> packed): key j of every gathered sequence b is copied from
// its cache slot to row cu_g[b] + j of a packed bf16 buffer, for K and V.  An
// FP8 cache is widened exactly (every E4M3 value is a bf16 value; the scales
// are applied by the attention).  Bad block ids are flagged and give zero rows;
// rows at or past `cap` are not written.  CTA t: packed rows
// [kGatherPos t, kGatherPos (t + 1)) (the grid covers the cap, so sequences
// left to the decode kernels, which have no rows, cost nothing), one warp per
// row at a time, which finds its sequence by a binary search over cu_g; a lane
// issues all of its loads of a round (K and V) before its stores.
constexpr int kGatherPos = 16;

__device__ __forceinline__ uint4 widen8_e4m3(uint2 codes) {
  const uint32_t cw[2] = {codes.x, codes.y};
  uint32_t o[4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t lo = e4m3x2_lo_to_f16x2(cw[h]), hi = e4m3x2_hi_to_f16x2(cw[h]);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
    const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&hi));
    o[2 * h] = pack_bf16x2(a.x, a.y);
    o[2 * h + 1] = pack_bf16x2(c.x, c.y);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint4 widen8_int8(uint2 codes) {
  const uint32_t cw[2] = {codes.x, codes.y};
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const int8_t c0 = (int8_t)(cw[e >> 2] >> (8 * (e & 3)));
    const int8_t c1 = (int8_t)(cw[e >> 2] >> (8 * ((e & 3) + 1)));
    o[e >> 1] = pack_bf16x2((float)c0, (float)c1);  // |c| <= 127: exact in bf16
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int kMode>  // 0: bf16 rows, 1: E4M3 codes, 2: INT8 codes
__global__ void __launch_bounds__(256) gather_kv_kernel(const uint8_t* __restrict__ k_cache,
                                                        const uint8_t* __restrict__ v_cache,
                                                        const int32_t* __restrict__ cu_g, int32_t batch,
                                                        const int32_t* __restrict__ block_table, int32_t max_blocks,
                                                        int32_t block_size, int32_t num_blocks, int32_t row_elems,
                                                        int64_t cap, uint16_t* __restrict__ k_out,
                                                        uint16_t* __restrict__ v_out, int32_t* err) {
  constexpr int kPer = 4;  // 16-byte output vectors per lane and tensor in one round
  // a programmatic dependent of the prep kernel: wait for its packed offsets
  // (cu_g: written by the prep; plain loads)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int64_t total = cu_g[batch];  // gathered rows; those at or past the buffer's cap are not
  if (total > cap) total = cap;   // written (the prep flagged them)
  const int chunks = row_elems >> 3;  // 16-byte bf16 vectors per row
  const int64_t cap_rows = (int64_t)max_blocks * block_size;
  for (int64_t row = (int64_t)blockIdx.x * kGatherPos + warp; row < (int64_t)(blockIdx.x + 1) * kGatherPos;
       row += 8) {
    if (row >= total) break;
    // the sequence of packed row `row`: the last b with cu_g[b] <= row (the
    // sequences the prefill tiles do not serve have no rows)
    int lo = 0, hi = batch;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)cu_g[mid] <= row) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int64_t j = row - cu_g[b];  // key j of sequence b
    if (j >= cap_rows) {  // more keys than the table holds: not gathered
      if (lane == 0) flag_error(err, PKV_DEVERR_LENGTH);
      continue;
    }
    const int blk = __ldg(block_table + (int64_t)b * max_blocks + j / block_size);
    const bool bad = blk < 0 || blk >= num_blocks;
    if (bad && lane == 0) flag_error(err, PKV_DEVERR_BLOCK);
    const int64_t slot = bad ? 0 : (int64_t)blk * block_size + j % block_size;
    uint4* kd = reinterpret_cast<uint4*>(k_out + row * row_elems);
    uint4* vd = reinterpret_cast<uint4*>(v_out + row * row_elems);
    for (int base = 0; base < chunks; base += 32 * kPer) {
      uint4 kr[kPer], vr[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int c = base + u * 32 + lane;
        kr[u] = vr[u] = make_uint4(0u, 0u, 0u, 0u);
        if (c < chunks && !bad) {
          if constexpr (kMode == 0) {
            kr[u] = __ldg(reinterpret_cast<const uint4*>(k_cache + slot * row_elems * 2) + c);
            vr[u] = __ldg(reinterpret_cast<const uint4*>(v_cache + slot * row_elems * 2) + c);
          } else {
            const uint2 kc2 = __ldg(reinterpret_cast<const uint2*>(k_cache + slot * row_elems) + c);
            const uint2 vc2 = __ldg(reinterpret_cast<const uint2*>(v_cache + slot * row_elems) + c);
            kr[u] = kMode == 1 ? widen8_e4m3(kc2) : widen8_int8(kc2);
            vr[u] = kMode == 1 ? widen8_e4m3(vc2) : widen8_int8(vc2);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int c = base + u * 32 + lane;
        if (c < chunks) {
          kd[c] = kr[u];
          vd[c] = vr[u];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

#ifdef PKV_TEST_HOOKS
int g_test_skip_k = -1;
#endif

struct VarlenWs {
  size_t count_off, items_off, decode_off, order_off, useq_off, cu_g_off, gk_off, gv_off, total;
};

// Paged K/V with blocks smaller than this (or FP8) are gathered into a packed
// bf16 buffer first when the caller sizes it (total_k > 0): one small TMA box
// per 16-token page and head-dim half bounds the paged loop, while the gather
// is a plain HBM copy and the packed loop runs at the full tile rate.
constexpr int kGatherBelowBlock = 64;

bool uses_gather(bool paged, int kv_dtype, int block_size, int64_t total_k) {
  return paged && total_k > 0 && (kv_dtype != PKV_BF16 || block_size < kGatherBelowBlock);
}

// [0, 256): the prefill work-item counter, the routed-row count, the prefill
// unit count and the prefill CTAs that run; then, when the prefill kernel
// runs, its unit list (int32 codes) and the units' sequence offsets (int4),
// each at most min(batch x n_pairs, total_q / 128 + batch) entries; then the
// routed row list and the decode partials (paged mode), then, when K/V are
// gathered, the packed offsets cu_g[batch+1] and the packed K and V buffers of
// total_k rows each.
constexpr size_t kUnitCountOff = 8;
constexpr size_t kActiveCtasOff = 12;
// Queries up to which a sequence is routed to the decode kernels: kRouteMaxQ
// when no sequence of the batch has more (then every query row is routed and
// there are total_q items), else 1 (then at most one item per sequence).
int route_max_q(int max_len_q) { return max_len_q <= kRouteMaxQ ? kRouteMaxQ : 1; }
// Queries per routed item: max_len_q when each item is a whole sequence
// (multi_query_items), else 0 (each item is one query row).
int route_multi_q(int max_len_q, int group) { return multi_query_items(max_len_q, group) ? max_len_q : 0; }
// Pairs of the longest sequence: query tiles with head pairs (even GQA
// groups), else pairs of tiles of one head.
int prefill_pairs(int max_len_q, int group) {
  return group % 2 == 0 ? (max_len_q + kBM - 1) / kBM : (max_len_q + kPairRows - 1) / kPairRows;
}
// Entries of the prefill unit list: none when every query row is routed,
// else at most one per pair of each sequence, no more than
// ceil(Lq_b / 128) <= Lq_b / 128 + 1 each.
int64_t prefill_units(int batch, int total_q, int max_len_q, int group, bool route) {
  if (route && max_len_q <= kRouteMaxQ) return 0;
  const int64_t all = (int64_t)batch * prefill_pairs(max_len_q, group);
  const int64_t by_rows = (int64_t)total_q / kBM + batch;
  return all < by_rows ? all : by_rows;
}
int route_items_bound(int batch, int total_q, int max_len_q, int group) {
  if (route_multi_q(max_len_q, group) > 0) return batch < total_q ? batch : total_q;
  return route_max_q(max_len_q) > 1 ? total_q : (batch < total_q ? batch : total_q);
}

VarlenWs varlen_ws_layout(int batch, int route_items, int num_heads, int num_kv_heads, int head_dim, int max_len_k,
                          bool route, bool gather, int64_t total_k, int kv_dtype, int multi_q, int64_t units) {
  VarlenWs w{0, 0, 0, 0, 0, 0, 0, 0, 256};
  if (batch <= 0) return w;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  if (units > 0) {
    w.order_off = w.total;
    w.useq_off = w.order_off + up((size_t)units * 4);
    w.total = w.useq_off + up((size_t)units * 16);
  }
  if (route && route_items > 0) {
    w.count_off = 4;
    w.items_off = w.total;
    w.decode_off = w.items_off + up((size_t)route_items * 4);
    w.total = w.decode_off +
              varlen_decode_workspace(batch, route_items, num_heads, num_kv_heads, head_dim, max_len_k, kv_dtype,
                                      multi_q);
  }
  if (gather) {
    w.cu_g_off = up(w.total);
    w.gk_off = w.cu_g_off + up(((size_t)batch + 1) * 4);
    const size_t buf = up((size_t)total_k * num_kv_heads * head_dim * 2);
    w.gv_off = w.gk_off + buf;
    w.total = w.gv_off + buf;
  }
  return w;
}

template <int D, bool kPaged, int kCode = 0>
int launch_prefill(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const PrefillParams& p,
                   int batch, cudaStream_t st, bool unified = false) {
  auto kern = varlen_prefill_kernel<D, kPaged, kCode, false>;
  if constexpr (D == 128 && kCode == 0) {
    if (unified) kern = varlen_prefill_kernel<D, kPaged, kCode, true>;
  } else {
    unified = false;
  }
  const int smem = unified ? Smem<D, true>::kAlloc : Smem<D>::kAlloc;
  static bool attr_set[2][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= 64) dev = 63;
  if (!attr_set[unified][dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return PKV_ERR_CUDA;
    attr_set[unified][dev] = true;
  }
  const int64_t items = (int64_t)p.n_pairs * batch * p.item_heads;
  const int64_t sms = device_sm_count();
  const int grid = (int)(items < sms ? items : sms);
  // a programmatic dependent of the kernel before it: after the prep, its CTAs
  // start as the prep runs and wait for its completion (the gather does not
  // trigger: its grid needs the SMs to itself)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kCode ? kThreadsCoded : kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, p) != cudaSuccess) return PKV_ERR_CUDA;
  return launch_status();
}

}  // namespace
}  // namespace pkv

// Single-query sequences go to the decode kernels in paged mode when the GQA
// group fits one decode CTA.
static bool routes_decode(bool paged, int num_heads, int num_kv_heads) {
  return paged && num_kv_heads > 0 && num_heads % num_kv_heads == 0 && num_heads / num_kv_heads <= 8;
}

extern "C" size_t pkv_paged_attn_varlen_workspace(int32_t batch, int32_t total_q, int32_t total_k,
                                                  int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                                  int32_t max_len_q, int32_t max_len_k, int32_t paged,
                                                  int32_t kv_dtype, int32_t block_size) {
  if (batch <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_len_k < 0 || total_k < 0 ||
      total_q < 0)
    return 0;
  const bool gather = pkv::uses_gather(paged != 0, kv_dtype, block_size, total_k);
  const int group = num_heads / num_kv_heads;
  const bool route = routes_decode(paged != 0, num_heads, num_kv_heads);
  return pkv::varlen_ws_layout(batch, pkv::route_items_bound(batch, total_q, max_len_q, group), num_heads,
                               num_kv_heads, head_dim, max_len_k, route, gather, total_k, kv_dtype,
                               pkv::route_multi_q(max_len_q, group),
                               pkv::prefill_units(batch, total_q, max_len_q, group, route))
      .total;
}

extern "C" int pkv_paged_attn_varlen(const void* q, const void* k, const void* v, int32_t kv_dtype,
                                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
                                     int32_t total_q, int32_t total_k, int32_t max_len_q, int32_t max_len_k,
                                     const int32_t* block_table, int32_t max_blocks_per_seq, int32_t block_size,
                                     int32_t num_blocks, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                     float scale, int32_t causal, float k_scale, float v_scale, void* out,
                                     float* lse, void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                     void* stream) {
  const pkv::NvtxRange nvtx_range("pkv_paged_attn_varlen");
  using namespace pkv;
  if (batch < 0 || total_q < 0 || total_k < 0 || max_len_q < 0 || max_len_k < 0 || num_heads <= 0 ||
      num_kv_heads <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (head_dim != 128 && head_dim != 64) return PKV_ERR_UNSUPPORTED;
  if (kv_dtype != PKV_BF16 && kv_dtype != PKV_FP8_E4M3 && kv_dtype != PKV_INT8) return PKV_ERR_UNSUPPORTED;
  const bool fp8 = kv_dtype != PKV_BF16;  // one-byte codes (E4M3 or INT8) with per-tensor scales
  const bool paged = block_table != nullptr;
  const bool route = routes_decode(paged, num_heads, num_kv_heads);
  // no sequence has more queries than the routing bound: every query row goes
  // to the decode kernels and no prefill tile runs
  const bool all_routed = route && max_len_q <= kRouteMaxQ;
  // the prefill tiles read a one-byte cache in paged mode only: through the
  // gather (total_k > 0) or, without a gather bound, widened in the tile loop
  // (head dim 128)
  if (fp8 && !all_routed && (!paged || (total_k <= 0 && head_dim != 128))) return PKV_ERR_UNSUPPORTED;
  if (fp8 && (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale)))
    return PKV_ERR_INVALID_ARG;
  if (!causal) return PKV_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (paged) {
    if (block_size <= 0 || block_size % 16 != 0 || (block_size < 128 && 128 % block_size != 0) ||
        (block_size > 128 && block_size % 128 != 0))
      return PKV_ERR_UNSUPPORTED;
    if (num_blocks <= 0 || max_blocks_per_seq <= 0) return PKV_ERR_INVALID_ARG;
  }
  if (batch == 0 || total_q == 0 || max_len_q == 0) return PKV_OK;
  if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !out) return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return PKV_ERR_INVALID_ARG;

  const bool gather = uses_gather(paged, kv_dtype, block_size, total_k);
  const int group = num_heads / num_kv_heads;
  const int route_items = route ? route_items_bound(batch, total_q, max_len_q, group) : 0;
  const int rmq = route ? route_max_q(max_len_q) : 0;  // queries up to which a sequence is routed
  const int multi_q = route ? route_multi_q(max_len_q, group) : 0;  // an item is a whole sequence
  const int64_t units = prefill_units(batch, total_q, max_len_q, group, route);
  // unit codes b * n_pairs + pe and item numbers are int32
  if ((int64_t)batch * prefill_pairs(max_len_q, group) > INT32_MAX || units * num_heads > INT32_MAX)
    return PKV_ERR_UNSUPPORTED;
  const VarlenWs wl = varlen_ws_layout(batch, route_items, num_heads, num_kv_heads, head_dim, max_len_k, route,
                                       gather, total_k, kv_dtype, multi_q, units);
  if (wl.total > 0 && (workspace == nullptr || workspace_bytes < wl.total ||
                       (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return PKV_ERR_WORKSPACE;
  char* wsb = static_cast<char*>(workspace);

  // Gathered mode runs the packed kernel on the gathered buffers, with the
  // packed offsets cu_g in place of cu_seqlens_k (same lengths for the
  // gathered sequences, zero for the ones the decode kernels take).
  const bool packed_tiles = !paged || gather;
  const bool coded_tiles = fp8 && !packed_tiles;  // one-byte pages widened by the tile loop
  const void* kt = gather ? static_cast<const void*>(wsb + wl.gk_off) : k;
  const void* vt = gather ? static_cast<const void*>(wsb + wl.gv_off) : v;
  CUtensorMap mq, mk, mv;
  const int64_t kv_rows = !paged ? (int64_t)total_k : gather ? (int64_t)total_k : (int64_t)num_blocks * block_size;
  const int kv_box = packed_tiles ? 128 : (block_size < 128 ? block_size : 128);
  // [rows, heads, dim] bf16, boxes of 64 elements x 1 head x box rows, 128-byte swizzle
  // (not needed when every query row goes to the decode kernels)
  // (one-byte pages: boxes of 128 codes, one 128-byte row per position)
  const int kv_elt = coded_tiles ? 1 : 2, kv_inner = coded_tiles ? 128 : 64;
  if (!all_routed && (!make_tmap_3d(&mq, q, 2, total_q, num_heads, head_dim, 64, 128, 128) ||
                      !make_tmap_3d(&mk, kt, kv_elt, kv_rows, num_kv_heads, head_dim, kv_inner, kv_box, 128) ||
                      !make_tmap_3d(&mv, vt, kv_elt, kv_rows, num_kv_heads, head_dim, kv_inner, kv_box, 128)))
    return PKV_ERR_CUDA;

  PrefillParams p{};
  p.cu_q = cu_seqlens_q;
  p.cu_k = gather ? reinterpret_cast<const int32_t*>(wsb + wl.cu_g_off) : cu_seqlens_k;
  p.block_table = packed_tiles ? nullptr : block_table;
  p.max_blocks = max_blocks_per_seq;
  p.block_size = block_size;
  p.box_rows = kv_box;
  p.num_blocks = num_blocks;
  p.num_heads = num_heads;
  p.group = num_heads / num_kv_heads;
  // even GQA groups pair two heads of a group on one query tile (same keys,
  // shared K/V); other groups pair two adjacent tiles of one head
  p.head_pairs = (p.group % 2 == 0) ? 1 : 0;
  p.item_heads = p.head_pairs ? num_heads / 2 : num_heads;
  p.n_pairs = prefill_pairs(max_len_q, p.group);
  p.batch = batch;
  p.route_decode = rmq;
  // FP8: the gathered codes are exact bf16 values; k_scale joins the logit
  // scale and v_scale the output factor
  p.scale_log2 = scale * kLog2e * (fp8 ? k_scale : 1.f);
  p.v_mul = fp8 ? v_scale : 1.f;
  p.total_q = total_q;
  p.out = static_cast<uint16_t*>(out);
  p.out_v8 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;
  p.lse = lse;
  p.err = err_flag;
#ifdef PKV_TEST_HOOKS
  p.test_skip_k = g_test_skip_k;
#endif
  cudaStream_t st = as_stream(stream);
  int32_t* count = nullptr;
  int32_t* items = nullptr;
  p.item_counter = static_cast<int32_t*>(workspace);
  int32_t* unit_order = units > 0 ? reinterpret_cast<int32_t*>(wsb + wl.order_off) : nullptr;
  p.unit_order = unit_order;
  p.unit_seq = units > 0 ? reinterpret_cast<const int4*>(wsb + wl.useq_off) : nullptr;
  p.n_units = reinterpret_cast<const int32_t*>(wsb + kUnitCountOff);
  p.active_ctas = reinterpret_cast<const int32_t*>(wsb + kActiveCtasOff);
  if (route && route_items > 0) {
    count = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + wl.count_off);
    items = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + wl.items_off);
  }
  int32_t* cu_g = gather ? reinterpret_cast<int32_t*>(wsb + wl.cu_g_off) : nullptr;
  PrepArgs pa{};
  pa.cu_q = cu_seqlens_q;
  pa.cu_k = cu_seqlens_k;
  pa.batch = batch;
  pa.items = items;
  pa.count = count;
  pa.route_cap = route_items;
  pa.route_max_q = rmq;
  pa.per_sequence = multi_q > 0 ? 1 : 0;
  pa.item_counter = p.item_counter;
  pa.unit_order = unit_order;
  pa.unit_seq = units > 0 ? reinterpret_cast<int4*>(wsb + wl.useq_off) : nullptr;
  pa.n_units = reinterpret_cast<int32_t*>(wsb + kUnitCountOff);
  pa.units_cap = (int)units;
  pa.n_pairs = p.n_pairs;
  pa.head_pairs = p.head_pairs;
  pa.item_heads = p.item_heads;
  pa.active_ctas = reinterpret_cast<int32_t*>(wsb + kActiveCtasOff);
  pa.sms = device_sm_count();
  pa.step_ns = kStepNs * (head_dim == 64 ? 0.8f : 1.f) * (coded_tiles ? 1.4f : 1.f);
  pa.decode_pos_bytes = (float)num_kv_heads * head_dim * 2.f * (fp8 ? 1.f : 2.f);
  pa.cu_g = cu_g;
  pa.gather_cap = (int64_t)total_k;
  pa.err = err_flag;
  varlen_prep_kernel<<<1, 1024, 0, st>>>(pa);
  if (gather) {
    const int64_t gx = ((int64_t)total_k + kGatherPos - 1) / kGatherPos;
    const dim3 ggrid((unsigned)(gx > 0 ? gx : 1), 1, 1);
    const int row_elems = num_kv_heads * head_dim;
    uint16_t* gk = reinterpret_cast<uint16_t*>(wsb + wl.gk_off);
    uint16_t* gv = reinterpret_cast<uint16_t*>(wsb + wl.gv_off);
    const auto* kc = static_cast<const uint8_t*>(k);
    const auto* vc = static_cast<const uint8_t*>(v);
    auto gk_kern = kv_dtype == PKV_FP8_E4M3 ? gather_kv_kernel<1>
                   : kv_dtype == PKV_INT8   ? gather_kv_kernel<2>
                                            : gather_kv_kernel<0>;
    // a programmatic dependent of the prep (which triggers at its start): its
    // launch and CTA start hide behind the prep
    cudaLaunchConfig_t gcfg = {};
    gcfg.gridDim = ggrid;
    gcfg.blockDim = dim3(256);
    gcfg.stream = st;
    cudaLaunchAttribute gattr[1];
    gattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    gattr[0].val.programmaticStreamSerializationAllowed = 1;
    gcfg.attrs = gattr;
    gcfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&gcfg, gk_kern, kc, vc, (const int32_t*)cu_g, (int32_t)batch, block_table,
                           max_blocks_per_seq, block_size, num_blocks, row_elems, (int64_t)total_k, gk, gv,
                           err_flag) != cudaSuccess)
      return PKV_ERR_CUDA;
  }
  // Long keys (a bound of kUnifiedKeys or more): all softmax warps work on one
  // tile at a time, two threads per row (faster K/V steps, costlier item ends)
  const bool unified = max_len_k >= kUnifiedKeys;
  int rc = PKV_OK;
  if (all_routed)
    rc = launch_status();
  else if (head_dim == 128)
    rc = packed_tiles                     ? launch_prefill<128, false>(mq, mk, mv, p, batch, st, unified)
         : !coded_tiles                   ? launch_prefill<128, true>(mq, mk, mv, p, batch, st, unified)
         : kv_dtype == PKV_FP8_E4M3       ? launch_prefill<128, true, 1>(mq, mk, mv, p, batch, st)
                                          : launch_prefill<128, true, 2>(mq, mk, mv, p, batch, st);
  else
    rc = packed_tiles ? launch_prefill<64, false>(mq, mk, mv, p, batch, st)
                      : launch_prefill<64, true>(mq, mk, mv, p, batch, st);
  if (rc != PKV_OK || items == nullptr) return rc;
  return launch_varlen_decode(q, k, v, items, count, cu_seqlens_q, cu_seqlens_k, block_table, max_blocks_per_seq,
                              batch, route_items, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                              max_len_k,
                              total_q,
                              scale, kv_dtype, k_scale, v_scale, out, lse, wsb + wl.decode_off,
                              (gather ? wl.cu_g_off : wl.total) - wl.decode_off, err_flag, multi_q, !all_routed,
                              st);
}

#ifdef PKV_TEST_HOOKS
// Test builds only: the next varlen calls withhold, in CTA 0 of the prefill
// kernel, the copy of its `tile`-th K tile, so that the waits on it run out
// (-1 restores normal operation).
extern "C" PKV_API void pkv_test_prefill_skip_k(int tile) { pkv::g_test_skip_k = tile; }
#endif
