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
// Persistent kernel, one 320-thread CTA per SM.  A work item is 128 query rows
// of one (sequence, query head); items are claimed through a global counter,
// longest first, and published to the CTA's warps through a shared ring.
//   warp 0      producer: Q once per item (TMA), then K/V tiles of 128 keys
//               (2 stages each), K one tile ahead of V.  Packed K/V: one TMA
//               box per head-dim half.  Paged K/V: one box per page and
//               half, each issued by its own lane, the block ids read two
//               tiles ahead.
//   warp 1      MMA issuer (one thread): S = Q K^T into TMEM, then for each
//               64-key half h of the tile O_h += P_h V_h with P read from TMEM.
//   warps 2..9  softmax, two warps per 32 rows: warps 2..5 own keys 0..63 of
//               every tile, warps 6..9 keys 64..127.  Each half is its own
//               online-softmax stream with its own O accumulator, so the halves
//               never synchronise inside the key loop; they are merged once in
//               the epilogue (log2-sum-exp weights), like two KV splits.  The
//               running max moves only when it grows by more than 2^8, so O is
//               rescaled rarely.  P (bf16 pairs) overwrites its S columns.
// TMEM (512 columns): S buffers [0,128) and [128,256); O_0 at 256, O_1 at 384.
// Every mbarrier wait is bounded by a deadline; on expiry the CTA flags
// PKV_DEVERR_TIMEOUT, drains its copies and MMAs, frees TMEM and returns.
#include <cmath>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int kBM = 128;          // query rows per CTA
constexpr int kBN = 128;          // keys per tile
constexpr int kThreads = 320;
constexpr int kSoftmaxThreads = 256;
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
  int32_t n_qtiles;
  int32_t batch;
  int32_t route_decode;  // sequences with at most this many queries are left to the decode kernels (0: none)
  int32_t* item_counter; // work-item counter, zero at launch
  float scale_log2;
  float v_mul;           // output factor (FP8 V scale of a gathered cache, else 1)
  int64_t total_q;
  uint16_t* out;
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

// Instruction descriptor, kind::f16: bf16 x bf16 -> f32, A K-major.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
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

template <int D>
struct Smem {
  static constexpr int kAtoms = D / 64;                 // 64-element (128-byte) column groups
  static constexpr int kTileBytes = 128 * D * 2;        // a [128 x D] bf16 tile
  static constexpr int kAtomBytes = 128 * 128;          // [128 rows x 128 B]
  static constexpr int kQ = 0;                          // 2 buffers (by work item)
  static constexpr int kK = kQ + 2 * kTileBytes;        // 2 stages
  static constexpr int kV = kK + 2 * kTileBytes;        // 2 stages
  static constexpr int kBar = kV + 2 * kTileBytes;
  static constexpr int kNumBars = 28;
  static constexpr int kMisc = kBar + kNumBars * 8;     // tmem holder, abort flag
  static constexpr int kRingData = kMisc + 16;          // 4 ring slots x 8 ints (item, q0, Lq, k0, Lk)
  static constexpr int kXchg = kRingData + 4 * 32;      // float m[2][128], l[2][128]
  static constexpr int kStage = kXchg + 4 * 128 * 4;    // output staging: 8 softmax warps x 16 half rows
  static constexpr int kTotal = kStage + 8 * 16 * D;
  static constexpr int kAlloc = kTotal + 1024;          // slack to align the base to 1024
};

constexpr int kRing = 4;  // work-item ring slots

// mbarrier indices (each one distinct; checked below).  K and V stages have
// no "empty" barriers of their own: a K stage is free once S of its tile is
// done (kSFull), a V stage once the tile's PV is (kPvDone).  Fewer commits
// and waits keep the MMA thread, which runs nearly in step with the tensor
// core, issuing MMAs.
enum Bar {
  kQFull0 = 0,       // +buffer (2)
  kQEmpty0 = 2,      // +buffer (2)
  kKFull0 = 4,       // +stage (2)
  kVFull0 = 6,       // +stage (2)
  kSFull0 = 8,       // +S buffer (2)
  kRingFull0 = 10,   // +slot (4): a work item index published by the producer
  kDrain = 14,
  kXchgA = 15,       // softmax threads: (m, l) of both halves published
  kXchgB = 16,       // softmax threads have read O and the exchange slots (MMA waits before the next item's PV)
  // The next two sets have one barrier per S buffer, i.e. per tile parity.
  // A parity wait can only tell "phase k done" from "phase k pending" when
  // the barrier is never two phases away from the waiter; with one barrier
  // per tile parity, tile t's phase has tile t-2's before it (known complete:
  // S(t) was issued after PV(t-2)) and tile t+2's after it (cannot have
  // started), so every wait below is unambiguous even when skipped tiles'
  // phases were never waited on.
  kPFull0 = 17,      // +buffer (2): P of that tile written, both halves (softmax -> MMA)
  kPvDone0 = 19,     // +buffer (2): O += P V of that tile landed (MMA -> softmax, producer)
  kRingEmpty0 = 21,  // +slot (4): the MMA warp and the 8 softmax warps have read the slot
  kBarCount = 25
};
static_assert(kQEmpty0 == kQFull0 + 2 && kKFull0 == kQEmpty0 + 2 && kVFull0 == kKFull0 + 2 &&
                  kSFull0 == kVFull0 + 2 && kRingFull0 == kSFull0 + 2 && kDrain == kRingFull0 + kRing &&
                  kXchgA == kDrain + 1 && kXchgB == kXchgA + 1 && kPFull0 == kXchgB + 1 &&
                  kPvDone0 == kPFull0 + 2 && kRingEmpty0 == kPvDone0 + 2 && kBarCount == kRingEmpty0 + kRing,
              "mbarrier index ranges must not overlap");

// A sequence's query/key offsets and (checked) lengths.  The producer warp
// reads them from global memory once per work item and hands them to the
// other roles through the work-item ring, so only one warp waits on those loads.
struct SeqBase {
  int q0, Lq, k0, Lk;
};
struct Seq {
  int q0, Lq, k0, Lk, row0, rows, diag, n_kv;
  bool skip;
};

// Cumulative offsets of sequence b: q0, q1, k0, k1 (loads only; checked by seq_check).
__device__ __forceinline__ void seq_load(const PrefillParams& p, int b, int (&raw)[4]) {
  raw[0] = __ldg(p.cu_q + b);
  raw[1] = __ldg(p.cu_q + b + 1);
  raw[2] = __ldg(p.cu_k + b);
  raw[3] = __ldg(p.cu_k + b + 1);
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
__device__ __forceinline__ Seq seq_derive(const PrefillParams& p, const SeqBase& b0, int qtile) {
  Seq s;
  s.q0 = b0.q0;
  s.Lq = b0.Lq;
  s.k0 = b0.k0;
  s.Lk = b0.Lk;
  s.row0 = qtile * kBM;
  s.rows = min(kBM, s.Lq - s.row0);
  s.diag = s.Lk - s.Lq;
  s.skip = s.rows <= 0 || s.Lq <= p.route_decode;
  const int kmax = s.row0 + s.rows - 1 + s.diag;  // last key the last row sees
  const int kv_tiles = (s.Lk + kBN - 1) / kBN;
  s.n_kv = kmax < 0 ? 0 : min(kmax / kBN + 1, kv_tiles);
  return s;
}

static_assert(Smem<128>::kNumBars >= kBarCount && Smem<64>::kNumBars >= kBarCount, "too few mbarrier slots");

// Work item -> (sequence, query tile, head).  Items are ordered by query tile,
// last tiles (most keys under causal masking) first, then sequence, then head,
// so CTAs running side by side share K/V through L2.
struct Item {
  int b, qtile, head;
};
__device__ __forceinline__ Item item_of(const PrefillParams& p, int it) {
  const int per = p.batch * p.num_heads;
  Item x;
  x.qtile = p.n_qtiles - 1 - it / per;
  const int rem = it % per;
  x.b = rem / p.num_heads;
  x.head = rem % p.num_heads;
  return x;
}

// Persistent kernel: one CTA per SM walks the work items blockIdx.x,
// blockIdx.x + gridDim.x, ...  All roles walk the same list and keep running
// counters (item, tile) so the barriers' phases continue across items.
template <int D, bool kPaged>
__global__ void __launch_bounds__(kThreads, 1)
    varlen_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_items = p.n_qtiles * p.batch * p.num_heads;

  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8 * i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kQFull0 + s), 1);
      mbar_init(bar(kQEmpty0 + s), 1);
      mbar_init(bar(kKFull0 + s), 1);
      mbar_init(bar(kVFull0 + s), 1);
      mbar_init(bar(kSFull0 + s), 1);
      mbar_init(bar(kPFull0 + s), kSoftmaxThreads);
      mbar_init(bar(kPvDone0 + s), 1);
    }
    mbar_init(bar(kDrain), 1);
    for (int r = 0; r < kRing; ++r) {
      mbar_init(bar(kRingFull0 + r), 1);
      mbar_init(bar(kRingEmpty0 + r), 1 + (kSoftmaxThreads / 32));
    }
    mbar_init(bar(kXchgA), kSoftmaxThreads);
    mbar_init(bar(kXchgB), kSoftmaxThreads);
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
  // TMEM columns: S buffers [0,128) and [128,256); O halves [256, 256+D) and [384, 384+D).
  // P of a tile (bf16 pairs) overwrites the first 32 columns of each half's S columns.
  auto tS = [&](int sb) -> uint32_t { return tmem + 128 * sb; };
  auto tO = [&](int h) -> uint32_t { return tmem + 256 + 128 * h; };

  auto fail = [&]() {
    *abort_flag = 1;
    flag_error(p.err, PKV_DEVERR_TIMEOUT);
  };
  // Work items are handed out dynamically, longest first (item_of orders
  // them), through a global counter; the producer warp claims them and
  // publishes each one that has work into a 4-slot ring that the MMA and
  // softmax warps read in order.  -1 ends the list.
  volatile int* ring = reinterpret_cast<volatile int*>(smem + L::kRingData);
  // Consumer side: item of the u-th ring entry (or -1, also on timeout) and its sequence.
  auto ring_get = [&](int u, SeqBase& sb) -> int {
    const int slot = u & (kRing - 1);
    if (!mbar_wait(bar(kRingFull0 + slot), (u / kRing) & 1, abort_flag)) return -1;
    const volatile int* e = ring + 8 * slot;
    const int it = e[0];
    sb.q0 = e[1];
    sb.Lq = e[2];
    sb.k0 = e[3];
    sb.Lk = e[4];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kRingEmpty0 + slot));
    return it;
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    int last_k[2] = {-1, -1}, last_v[2] = {-1, -1}, last_q[2] = {-1, -1};
    int g = 0, uq = 0, ur = 0;  // tiles, items with keys, ring entries
    bool ok = true;
    auto publish = [&](int it, const SeqBase& sb) -> bool {
      const int slot = ur & (kRing - 1);
      if (ur >= kRing && !mbar_wait(bar(kRingEmpty0 + slot), ((ur / kRing) - 1) & 1, abort_flag)) return false;
      if (lane == 0) {
        volatile int* e = ring + 8 * slot;
        e[0] = it;
        e[1] = sb.q0;
        e[2] = sb.Lq;
        e[3] = sb.k0;
        e[4] = sb.Lk;
        mbar_arrive(bar(kRingFull0 + slot));
      }
      __syncwarp();
      ++ur;
      return true;
    };
    // The next item is claimed from the global counter a few tiles before
    // the current one's last, and its offsets are loaded while those tiles
    // are issued: neither latency then sits between two items, and a claimed
    // item waits only a few tiles (dynamic balance is kept).  A skipped item
    // (a sequence left to the decode kernels, or a query tile past its end)
    // moves the counter past the other heads of its (tile, sequence), which
    // are skipped too.
    int claim = 0;  // lane 0: atomic result for the next item
    bool claimed = false, resolved = false;
    int it = 0, next = n_items;
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
      if (next < n_items) seq_load(p, item_of(p, next).b, raw);
      resolved = true;
    };
    resolve_next();
    it = next;
    while (ok && it < n_items) {
      claimed = resolved = false;
      const Item x = item_of(p, it);
      const SeqBase si = seq_check(p, raw, x.qtile == 0 && x.head == 0 && lane == 0);
      const Seq sq = seq_derive(p, si, x.qtile);
      if (sq.skip) {
        const int block_end = (it / p.num_heads + 1) * p.num_heads;  // first item of the next (tile, sequence)
        if (lane == 0 && block_end < n_items) atomicMax(p.item_counter, block_end);
        resolve_next();
        it = next;
        continue;
      }
      if (!publish(it, si)) { ok = false; break; }
      if (sq.n_kv == 0) {
        resolve_next();
        it = next;
        continue;
      }
      const int kvh = x.head / p.group;
      const int32_t* bt = kPaged ? p.block_table + (int64_t)x.b * p.max_blocks : nullptr;
      const int qb = uq & 1, qu = uq >> 1;
      if (qu > 0 && !mbar_wait(bar(kQEmpty0 + qb), (qu - 1) & 1, abort_flag)) { ok = false; break; }
      if (lane == 0) {
        mbar_expect_tx(bar(kQFull0 + qb), L::kTileBytes);
        for (int a = 0; a < L::kAtoms; ++a)
          tma_load_3d(sbase + L::kQ + qb * L::kTileBytes + a * L::kAtomBytes, &tm_q, a * 64, x.head,
                      sq.q0 + sq.row0, bar(kQFull0 + qb));
      }
      last_q[qb] = qu;
      const int br = kPaged ? p.box_rows : kBN;
      const int npages = kBN / br;
      // Paged tiles: lane (page pg, head-dim atom at) issues one box; at most
      // 8 pages x 2 atoms, as block sizes are multiples of 16.
      const int pg = lane % npages, at = lane / npages;
      const bool box_lane = lane < npages * L::kAtoms;
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
        // the stage is free once the MMAs that read it are done: S(gg-2) for K, PV(gg-2) for V
        const uint32_t empty = t ? bar(kPvDone0 + s) : bar(kSFull0 + s);
        const uint32_t full = bar((t ? kVFull0 : kKFull0) + s);
        if (u > 0 && !mbar_wait(empty, (u - 1) & 1, abort_flag)) return false;
        const uint32_t dst = sbase + (t ? L::kV : L::kK) + s * L::kTileBytes;
        const CUtensorMap* map = t ? &tm_v : &tm_k;
        const int key0 = j * kBN;
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
          if (lane == 0) mbar_expect_tx(full, (uint32_t)(loaded * br * 128 * L::kAtoms));
          __syncwarp();
          if (box_lane && pg < loaded)
            tma_load_3d(dst + at * L::kAtomBytes + pg * br * 128, map, at * 64, kvh, my_slot, full);
          __syncwarp();
        }
        (t ? last_v : last_k)[s] = u;
        return true;
      };
      // K runs one tile ahead of V within the item
      int slot_cur = tile_slot(0, tile_blk(0));
      int blk_next = tile_blk(1);
      if (!issue(0, 0, slot_cur)) { ok = false; break; }
      const int claim_at = sq.n_kv > 3 ? sq.n_kv - 3 : 0;  // tiles ahead of the item's end
      for (int j = 0; j < sq.n_kv && ok; ++j) {
        if (j == claim_at) claim_next();
        if (j > claim_at && j == sq.n_kv - 1) resolve_next();
        const int blk_after = tile_blk(j + 2);
        const int slot_next = (j + 1 < sq.n_kv) ? tile_slot(j + 1, blk_next) : 0;
        if (j + 1 < sq.n_kv && !issue(0, j + 1, slot_next)) { ok = false; break; }
        if (!issue(1, j, slot_cur)) { ok = false; break; }
        slot_cur = slot_next;
        blk_next = blk_after;
      }
      if (!ok) break;
      resolve_next();
      it = next;
      g += sq.n_kv;
      ++uq;
    }
    if (ok && !publish(-1, SeqBase{0, 0, 0, 0})) ok = false;
    if (!ok) fail();
    // every copy this CTA issued has landed before shared memory is released
    for (int s = 0; s < 2; ++s) {
      if (last_q[s] >= 0) mbar_wait(bar(kQFull0 + s), last_q[s] & 1, abort_flag);
      if (last_k[s] >= 0) mbar_wait(bar(kKFull0 + s), last_k[s] & 1, abort_flag);
      if (last_v[s] >= 0) mbar_wait(bar(kVFull0 + s), last_v[s] & 1, abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdescQK = make_idesc(kBM, kBN, false);
    constexpr uint32_t kIdescPV = make_idesc(kBM, D, true);
    bool ok = true, issued = false;
    int g = 0, uq = 0;
    // O_h += P_h V_h for global tile t (local index jt within its item, whose keys end at Lk)
    auto issue_pv = [&](int t, int jt, int Lk) -> bool {
      if (!mbar_wait(bar(kVFull0 + (t & 1)), (t >> 1) & 1, abort_flag)) return false;
      // the first PV of an item overwrites O: the previous item's epilogue must have read it
      if (jt == 0 && uq > 0 && !mbar_wait(bar(kXchgB), (uq - 1) & 1, abort_flag)) return false;
      const uint32_t vbase = sbase + L::kV + (t & 1) * L::kTileBytes;
      // keys at or beyond Lk: zero their V rows (stale or foreign data must not meet P = 0)
      const int valid = Lk - jt * kBN;
      if (valid < kBN) {
        uint8_t* vs = smem + L::kV + (t & 1) * L::kTileBytes;
        const int first = valid > 0 ? valid : 0;
        const int nchunks = (kBN - first) * 8;  // 16-byte chunks per atom
        for (int a = 0; a < L::kAtoms; ++a)
          for (int c = lane; c < nchunks; c += 32)
            *reinterpret_cast<uint4*>(vs + a * L::kAtomBytes + (first + c / 8) * 128 + (c % 8) * 16) =
                make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
        __syncwarp();
      }
      // descriptors differ only in their start-address field (bits 0..13, address >> 4)
      const uint64_t vdesc = sw128_desc(vbase, L::kAtomBytes, 1024);
      // both halves' P, then all eight PV MMAs and one commit: every wait and
      // commit the MMA thread runs between MMAs leaves the tensor core idle
      if (!mbar_wait(bar(kPFull0 + (t & 1)), (t >> 1) & 1, abort_flag)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t acc = jt > 0 ? 1u : 0u;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t pa = tS(t & 1) + 64 * h;  // P_h: 32 columns of bf16 pairs = 64 keys
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ts(tO(h), pa + 8 * kk, vdesc + (uint64_t)(((64 * h + 16 * kk) * 128) >> 4), kIdescPV,
                        kk > 0 ? 1u : acc);
        }
        mma_commit(bar(kPvDone0 + (t & 1)));  // also frees V stage t & 1
      }
      __syncwarp();
      return true;
    };
    for (int u = 0; ok; ++u) {
      SeqBase si;
      const int it = ring_get(u, si);
      if (it < 0) break;
      const Item x = item_of(p, it);
      const Seq sq = seq_derive(p, si, x.qtile);
      if (sq.n_kv == 0) continue;
      const int qb = uq & 1;
      if (!mbar_wait(bar(kQFull0 + qb), (uq >> 1) & 1, abort_flag)) { ok = false; break; }
      for (int j = 0; j < sq.n_kv; ++j) {
        const int gg = g + j, s = gg & 1;
        if (!mbar_wait(bar(kKFull0 + s), (gg >> 1) & 1, abort_flag)) { ok = false; break; }
        // S(gg) overwrites buffer s, whose P(gg-2) the PV issued just before
        // reads: tcgen05.mma operations from one thread execute in issue
        // order, so no wait for that PV's completion is needed here.
        tc_fence_after();
        if (lane == 0) {
          const uint64_t qdesc = sw128_desc(sbase + L::kQ + qb * L::kTileBytes, 16, 1024);
          const uint64_t kdesc = sw128_desc(sbase + L::kK + s * L::kTileBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * L::kAtomBytes + (kk & 3) * 32) >> 4);
            mma_bf16(tS(s), qdesc + off, kdesc + off, kIdescQK, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(kSFull0 + s));  // also frees K stage s
          if (j == sq.n_kv - 1) mma_commit(bar(kQEmpty0 + qb));
        }
        __syncwarp();
        issued = true;
        if (j > 0 && !issue_pv(gg - 1, j - 1, sq.Lk)) { ok = false; break; }
      }
      if (ok && !issue_pv(g + sq.n_kv - 1, sq.n_kv - 1, sq.Lk)) ok = false;
      g += sq.n_kv;
      ++uq;
    }
    if (!ok) fail();
    // drain: all MMAs this thread issued have completed before TMEM is released
    if (issued) {
      if (lane == 0) mma_commit(bar(kDrain));
      __syncwarp();
      mbar_wait(bar(kDrain), 0, abort_flag);
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;   // keys [64*half, 64*half + 64) of every tile
    const int r = quarter * 32 + lane;  // TMEM lane == query row in the tile
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float c = p.scale_log2;
    float* xm = reinterpret_cast<float*>(smem + L::kXchg);
    float* xl = xm + 256;
    bool ok = true;
    int g = 0, ux = 0;  // tiles and work items (with keys) processed
    for (int u = 0; ok; ++u) {
      SeqBase si;
      const int it = ring_get(u, si);
      if (it < 0) break;
      const Item x = item_of(p, it);
      const Seq sq = seq_derive(p, si, x.qtile);
      const int qi = sq.row0 + r;
      const int64_t row = (int64_t)sq.q0 + qi;
      const bool row_valid = r < sq.rows;
      uint16_t* orow = p.out + (row * p.num_heads + x.head) * D;
      if (sq.n_kv == 0) {
        // rows that see no key: zeros and lse = -inf
        if (row_valid) {
          for (int cc = half * (D / 16); cc < (half + 1) * (D / 16); ++cc)
            reinterpret_cast<uint4*>(orow)[cc] = make_uint4(0, 0, 0, 0);
          if (half == 0 && p.lse) p.lse[(int64_t)x.head * p.total_q + row] = -INFINITY;
        }
        continue;
      }
      const int lim = qi + sq.diag;  // last visible key of this row
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < sq.n_kv; ++j) {
        const int gg = g + j, sb = gg & 1;
        if (!mbar_wait(bar(kSFull0 + sb), (gg >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[64];
        PKV_TMEM_LD32(tS(sb) + lane_off + 64 * half, (sr + 0));
        PKV_TMEM_LD32(tS(sb) + lane_off + 64 * half + 32, (sr + 32));
        tmem_wait_ld();

        const int key0 = j * kBN + 64 * half;
        const bool need_mask = (key0 + 63 > sq.row0 + sq.diag) || (key0 + 64 > sq.Lk);
        if (need_mask) {
          const int vis = min(lim, sq.Lk - 1) - key0;  // columns 0..vis are visible
#pragma unroll
          for (int k = 0; k < 64; ++k) sr[k] = (k <= vis) ? sr[k] : __float_as_uint(-INFINITY);
        }
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int k = 0; k < 64; k += 2)
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
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 64; k += 2) {
          float x0, x1;
          f32x2_unpack(ffma2(f32x2_pack(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), c2, nm2), x0, x1);
          const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          sum2[(k >> 1) & 1] = fadd2(sum2[(k >> 1) & 1], f32x2_pack(p0, p1));
          pk[k >> 1] = pack_bf16x2(p0, p1);
        }
        float s00, s01, s10, s11;
        f32x2_unpack(sum2[0], s00, s01);
        f32x2_unpack(sum2[1], s10, s11);
        l = l * alpha + ((s00 + s01) + (s10 + s11));
        m = m_use;

        // rescale O_half when this row's reference max moved (warp-collective TMEM access);
        // the previous tile's PV must have landed first
        if (j > 0 && __any_sync(0xffffffffu, moved && alpha != 1.f)) {
          const int tp = gg - 1;  // previous tile
          if (!mbar_wait(bar(kPvDone0 + (tp & 1)), (tp >> 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t o[32];
            PKV_TMEM_LD32(tO(half) + lane_off + ch * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            PKV_TMEM_ST32(tO(half) + lane_off + ch * 32, o);
          }
        }
        // P_half (bf16 pairs) over the first 32 of this half's S columns
        PKV_TMEM_ST32(tS(sb) + lane_off + 64 * half, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kPFull0 + sb));
      }
      if (!ok) break;
      const int glast = g + sq.n_kv - 1;
      if (!mbar_wait(bar(kPvDone0 + (glast & 1)), (glast >> 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // exchange (m, l) between the two halves of each row
      xm[half * 128 + r] = m;
      xl[half * 128 + r] = l;
      mbar_arrive(bar(kXchgA));
      if (!mbar_wait(bar(kXchgA), ux & 1, abort_flag)) { ok = false; break; }
      const float m0 = xm[r], m1 = xm[128 + r];
      const float l0 = xl[r], l1 = xl[128 + r];
      const float ms = fmaxf(m0, m1);
      const float f0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - ms);
      const float f1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - ms);
      const float lt = l0 * f0 + l1 * f1;
      const float inv = lt > 0.f ? p.v_mul / lt : 0.f;
      const float w0 = f0 * inv, w1 = f1 * inv;
      // this half writes head dims [half*D/2, (half+1)*D/2) of every row
      constexpr int kHalfRowBytes = D;           // D/2 bf16
      constexpr int kCh = kHalfRowBytes / 16;    // 16-byte pieces of a half row
      uint4 mine[kCh];
#pragma unroll
      for (int ch = 0; ch < D / 64; ++ch) {
        const int col = half * (D / 2) + ch * 32;
        uint32_t a[32], bb[32];
        PKV_TMEM_LD32(tO(0) + lane_off + col, a);
        PKV_TMEM_LD32(tO(1) + lane_off + col, bb);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; k += 8) {
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(a[k + e]) * w0 + __uint_as_float(bb[k + e]) * w1;
          mine[(ch * 32 + k) / 8] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                               pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
        }
      }
      // Rows of one head are num_heads*D elements apart, so a thread storing
      // its own row would touch a separate line per 16 bytes.  Instead the
      // warp passes 16 rows at a time through its staging rows in shared
      // memory (16-byte pieces XOR-swizzled by row) and stores whole half rows.
      uint8_t* stg = smem + L::kStage + (warp - 2) * 16 * kHalfRowBytes;
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        if ((lane >> 4) == pass) {
          const int sr = lane & 15;
#pragma unroll
          for (int c = 0; c < kCh; ++c)
            *reinterpret_cast<uint4*>(stg + sr * kHalfRowBytes + ((c ^ (sr & (kCh - 1))) * 16)) = mine[c];
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 16 * kCh / 32; ++i) {
          const int idx = i * 32 + lane;
          const int sr = idx / kCh, c = idx % kCh;
          const int rr = quarter * 32 + pass * 16 + sr;  // row within the tile
          if (rr < sq.rows) {
            const uint4 val = *reinterpret_cast<const uint4*>(stg + sr * kHalfRowBytes + ((c ^ (sr & (kCh - 1))) * 16));
            uint16_t* dst = p.out + ((int64_t)(sq.q0 + sq.row0 + rr) * p.num_heads + x.head) * D + half * (D / 2) + c * 8;
            *reinterpret_cast<uint4*>(dst) = val;
          }
        }
        __syncwarp();
      }
      if (half == 0 && row_valid && p.lse != nullptr)
        p.lse[(int64_t)x.head * p.total_q + row] = lt > 0.f ? (ms + log2f(lt)) * kLn2 : -INFINITY;
      // this thread has read O and the exchange slots; the MMA thread waits for all of them
      // before the next item's first PV (so the softmax warps do not wait here)
      tc_fence_before();
      mbar_arrive(bar(kXchgB));
      g += sq.n_kv;
      ++ux;
    }
    if (!ok) fail();
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// Varlen prep: compacts the sequences that have exactly one query (decode rows
// of a mixed batch) into items[0..*count); the prefill kernel skips them and
// the split-KV decode kernels serve them, one CTA per (split, kv head, item).
// It also resets the prefill kernel's work-item counter.
__global__ void __launch_bounds__(1024) varlen_prep_kernel(const int32_t* __restrict__ cu_q,
                                                           const int32_t* __restrict__ cu_k, int batch,
                                                           int32_t* __restrict__ items, int32_t* __restrict__ count,
                                                           int32_t* __restrict__ item_counter, int route_cap,
                                                           int route_max_q,
                                                           int32_t* __restrict__ cu_g, int64_t gather_cap,
                                                           int32_t* err) {
  __shared__ int n;
  __shared__ int64_t carry;
  if (threadIdx.x == 0) {
    n = 0;
    carry = 0;
    *item_counter = 0;
  }
  __syncthreads();
  if (items != nullptr) {
    // every query row of a sequence with 1..kRouteMaxQ queries (item codes
    // b * kRouteCode + qi; the bound route_cap holds them all)
    for (int b = threadIdx.x; b < batch; b += blockDim.x) {
      const int lq = __ldg(cu_q + b + 1) - __ldg(cu_q + b);
      if (lq >= 1 && lq <= route_max_q) {
        const int base = atomicAdd(&n, lq);
        for (int i = 0; i < lq; ++i)
          if (base + i < route_cap) items[base + i] = b * kRouteCode + i;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) *count = n < route_cap ? n : route_cap;
  }
  if (cu_g != nullptr) {
    // Packed offsets of the gathered sequences (those the prefill kernel
    // serves: more than one query, or any query when nothing is routed):
    // cu_g[b] = sum of their key counts before b.  Exclusive scan, one
    // 32-sequence chunk per warp step, carried across passes.
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __shared__ int64_t warp_sum[32];
    for (int base = 0; base < batch; base += blockDim.x) {
      const int b = base + threadIdx.x;
      int64_t v = 0;
      if (b < batch) {
        const int lq = __ldg(cu_q + b + 1) - __ldg(cu_q + b);
        const int lk = __ldg(cu_k + b + 1) - __ldg(cu_k + b);
        const bool gathered = lq > route_max_q;
        v = gathered && lk > 0 ? lk : 0;
      }
      int64_t x = v;  // inclusive warp scan
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) warp_sum[warp] = x;
      __syncthreads();
      int64_t before = carry;
      for (int w = 0; w < warp; ++w) before += warp_sum[w];
      if (b < batch) cu_g[b] = (int32_t)(before + x - v);
      __syncthreads();
      if (threadIdx.x == 0) {
        for (int w = 0; w < nw; ++w) carry += warp_sum[w];
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      cu_g[batch] = (int32_t)carry;
      if (carry > gather_cap) flag_error(err, PKV_DEVERR_LENGTH);  // rows past the buffer are not gathered
    }
  }
}

// Gather (paged -> packed): key j of every gathered sequence b is copied from
// its cache slot to row cu_g[b] + j of a packed bf16 buffer, for K and V.  An
// FP8 cache is widened exactly (every E4M3 value is a bf16 value; the scales
// are applied by the attention).  Bad block ids are flagged and give zero rows;
// rows at or past `cap` are not written.  CTA (t, b): positions
// [kGatherPos t, kGatherPos (t + 1)), one warp per position at a time; a lane
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
                                                        const int32_t* __restrict__ cu_q,
                                                        const int32_t* __restrict__ cu_k,
                                                        const int32_t* __restrict__ cu_g,
                                                        const int32_t* __restrict__ block_table, int32_t max_blocks,
                                                        int32_t block_size, int32_t num_blocks, int32_t row_elems,
                                                        int route, int64_t cap, uint16_t* __restrict__ k_out,
                                                        uint16_t* __restrict__ v_out, int32_t* err) {
  constexpr int kPer = 4;  // 16-byte output vectors per lane and tensor in one round
  const int b = blockIdx.y;
  const int lq = __ldg(cu_q + b + 1) - __ldg(cu_q + b);
  if (lq <= route) return;  // route: the routed query bound (0: none)
  int lk = __ldg(cu_k + b + 1) - __ldg(cu_k + b);
  if ((int64_t)lk > (int64_t)max_blocks * block_size) {  // more keys than the table holds
    lk = max_blocks * block_size;
    if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(err, PKV_DEVERR_LENGTH);
  }
  const int j0 = blockIdx.x * kGatherPos;
  if (j0 >= lk) return;
  const int64_t g0 = __ldg(cu_g + b);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunks = row_elems >> 3;  // 16-byte bf16 vectors per row
  for (int j = j0 + warp; j < min(lk, j0 + kGatherPos); j += 8) {
    const int64_t row = g0 + j;
    if (row >= cap) break;
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

struct VarlenWs {
  size_t count_off, items_off, decode_off, cu_g_off, gk_off, gv_off, total;
};

// Paged K/V with blocks smaller than this (or FP8) are gathered into a packed
// bf16 buffer first when the caller sizes it (total_k > 0): one small TMA box
// per 16-token page and head-dim half bounds the paged loop, while the gather
// is a plain HBM copy and the packed loop runs at the full tile rate.
constexpr int kGatherBelowBlock = 64;

bool uses_gather(bool paged, int kv_dtype, int block_size, int64_t total_k) {
  return paged && total_k > 0 && (kv_dtype != PKV_BF16 || block_size < kGatherBelowBlock);
}

// [0, 256): the prefill work-item counter and the routed-row count; then the
// routed row list and the decode partials (paged mode), then, when K/V are
// gathered, the packed offsets cu_g[batch+1] and the packed K and V buffers
// of total_k rows each.
// Queries up to which a sequence is routed to the decode kernels: kRouteMaxQ
// when no sequence of the batch has more (then every query row is routed and
// there are total_q items), else 1 (then at most one item per sequence).
int route_max_q(int max_len_q) { return max_len_q <= kRouteMaxQ ? kRouteMaxQ : 1; }
int route_items_bound(int batch, int total_q, int max_len_q) {
  return route_max_q(max_len_q) > 1 ? total_q : (batch < total_q ? batch : total_q);
}

VarlenWs varlen_ws_layout(int batch, int route_items, int num_heads, int num_kv_heads, int head_dim, int max_len_k,
                          bool route, bool gather, int64_t total_k, int kv_dtype) {
  VarlenWs w{0, 0, 0, 0, 0, 0, 256};
  if (batch <= 0) return w;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  if (route && route_items > 0) {
    w.count_off = 4;
    w.items_off = 256;
    w.decode_off = w.items_off + up((size_t)route_items * 4);
    w.total = w.decode_off +
              varlen_decode_workspace(batch, route_items, num_heads, num_kv_heads, head_dim, max_len_k, kv_dtype);
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

template <int D, bool kPaged>
int launch_prefill(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const PrefillParams& p,
                   int batch, cudaStream_t st) {
  auto kern = varlen_prefill_kernel<D, kPaged>;
  const int smem = Smem<D>::kAlloc;
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= 64) dev = 63;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return PKV_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int64_t items = (int64_t)p.n_qtiles * batch * p.num_heads;
  const int grid = (int)(items < device_sm_count() ? items : device_sm_count());
  kern<<<grid, kThreads, smem, st>>>(mq, mk, mv, p);
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
  return pkv::varlen_ws_layout(batch, pkv::route_items_bound(batch, total_q, max_len_q), num_heads, num_kv_heads,
                               head_dim,
                               max_len_k,
                               routes_decode(paged != 0, num_heads, num_kv_heads), gather, total_k, kv_dtype)
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
  using namespace pkv;
  if (batch < 0 || total_q < 0 || total_k < 0 || max_len_q < 0 || max_len_k < 0 || num_heads <= 0 ||
      num_kv_heads <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (head_dim != 128 && head_dim != 64) return PKV_ERR_UNSUPPORTED;
  if (kv_dtype != PKV_BF16 && kv_dtype != PKV_FP8_E4M3 && kv_dtype != PKV_INT8) return PKV_ERR_UNSUPPORTED;
  const bool fp8 = kv_dtype != PKV_BF16;  // one-byte codes (E4M3 or INT8) with per-tensor scales
  // a coded cache is read through the gather (paged mode, total_k > 0)
  if (fp8 && (block_table == nullptr || total_k <= 0)) return PKV_ERR_UNSUPPORTED;
  if (fp8 && (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale)))
    return PKV_ERR_INVALID_ARG;
  if (!causal) return PKV_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  const bool paged = block_table != nullptr;
  if (paged) {
    if (block_size <= 0 || block_size % 16 != 0 || (block_size < 128 && 128 % block_size != 0) ||
        (block_size > 128 && block_size % 128 != 0))
      return PKV_ERR_UNSUPPORTED;
    if (num_blocks <= 0 || max_blocks_per_seq <= 0) return PKV_ERR_INVALID_ARG;
  }
  if (batch == 0 || total_q == 0 || max_len_q == 0) return PKV_OK;
  if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !out) return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return PKV_ERR_INVALID_ARG;

  const bool route = routes_decode(paged, num_heads, num_kv_heads);
  const bool gather = uses_gather(paged, kv_dtype, block_size, total_k);
  const int route_items = route ? route_items_bound(batch, total_q, max_len_q) : 0;
  const int rmq = route ? route_max_q(max_len_q) : 0;  // queries up to which a sequence is routed
  const VarlenWs wl =
      varlen_ws_layout(batch, route_items, num_heads, num_kv_heads, head_dim, max_len_k, route, gather, total_k,
                       kv_dtype);
  if (wl.total > 0 && (workspace == nullptr || workspace_bytes < wl.total ||
                       (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return PKV_ERR_WORKSPACE;
  char* wsb = static_cast<char*>(workspace);

  // Gathered mode runs the packed kernel on the gathered buffers, with the
  // packed offsets cu_g in place of cu_seqlens_k (same lengths for the
  // gathered sequences, zero for the ones the decode kernels take).
  const bool packed_tiles = !paged || gather;
  const void* kt = gather ? static_cast<const void*>(wsb + wl.gk_off) : k;
  const void* vt = gather ? static_cast<const void*>(wsb + wl.gv_off) : v;
  CUtensorMap mq, mk, mv;
  const int64_t kv_rows = !paged ? (int64_t)total_k : gather ? (int64_t)total_k : (int64_t)num_blocks * block_size;
  const int kv_box = packed_tiles ? 128 : (block_size < 128 ? block_size : 128);
  // [rows, heads, dim] bf16, boxes of 64 elements x 1 head x box rows, 128-byte swizzle
  if (!make_tmap_3d(&mq, q, 2, total_q, num_heads, head_dim, 64, 128, 128) ||
      !make_tmap_3d(&mk, kt, 2, kv_rows, num_kv_heads, head_dim, 64, kv_box, 128) ||
      !make_tmap_3d(&mv, vt, 2, kv_rows, num_kv_heads, head_dim, 64, kv_box, 128))
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
  p.n_qtiles = (max_len_q + kBM - 1) / kBM;
  p.batch = batch;
  p.route_decode = rmq;
  // FP8: the gathered codes are exact bf16 values; k_scale joins the logit
  // scale and v_scale the output factor
  p.scale_log2 = scale * kLog2e * (fp8 ? k_scale : 1.f);
  p.v_mul = fp8 ? v_scale : 1.f;
  p.total_q = total_q;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.err = err_flag;
  cudaStream_t st = as_stream(stream);
  int32_t* count = nullptr;
  int32_t* items = nullptr;
  p.item_counter = static_cast<int32_t*>(workspace);
  if (route && route_items > 0) {
    count = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + wl.count_off);
    items = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + wl.items_off);
  }
  int32_t* cu_g = gather ? reinterpret_cast<int32_t*>(wsb + wl.cu_g_off) : nullptr;
  varlen_prep_kernel<<<1, (items != nullptr || gather) ? 1024 : 32, 0, st>>>(
      cu_seqlens_q, cu_seqlens_k, batch, items, count, p.item_counter, route_items, rmq, cu_g, (int64_t)total_k,
      err_flag);
  if (gather) {
    const int gx = (max_len_k + kGatherPos - 1) / kGatherPos;
    const dim3 ggrid((unsigned)(gx > 0 ? gx : 1), (unsigned)batch, 1);
    const int row_elems = num_kv_heads * head_dim;
    uint16_t* gk = reinterpret_cast<uint16_t*>(wsb + wl.gk_off);
    uint16_t* gv = reinterpret_cast<uint16_t*>(wsb + wl.gv_off);
    const auto* kc = static_cast<const uint8_t*>(k);
    const auto* vc = static_cast<const uint8_t*>(v);
    auto gk_kern = kv_dtype == PKV_FP8_E4M3 ? gather_kv_kernel<1>
                   : kv_dtype == PKV_INT8   ? gather_kv_kernel<2>
                                            : gather_kv_kernel<0>;
    gk_kern<<<ggrid, 256, 0, st>>>(kc, vc, cu_seqlens_q, cu_seqlens_k, cu_g, block_table, max_blocks_per_seq,
                                   block_size, num_blocks, row_elems, rmq, total_k, gk, gv, err_flag);
  }
  int rc;
  if (head_dim == 128)
    rc = packed_tiles ? launch_prefill<128, false>(mq, mk, mv, p, batch, st)
                      : launch_prefill<128, true>(mq, mk, mv, p, batch, st);
  else
    rc = packed_tiles ? launch_prefill<64, false>(mq, mk, mv, p, batch, st)
                      : launch_prefill<64, true>(mq, mk, mv, p, batch, st);
  if (rc != PKV_OK || items == nullptr) return rc;
  return launch_varlen_decode(q, k, v, items, count, cu_seqlens_q, cu_seqlens_k, block_table, max_blocks_per_seq,
                              batch, route_items, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                              max_len_k,
                              total_q,
                              scale, kv_dtype, k_scale, v_scale, out, lse, wsb + wl.decode_off,
                              (gather ? wl.cu_g_off : wl.total) - wl.decode_off, err_flag, st);
}
