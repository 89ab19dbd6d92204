// Prefill kernel (K-P): tcgen05 / TMEM / TMA attention, persistent, two
// 128-row query tiles per work tile.
//
// Work unit: one ua_tile of up to 256 packed rows (tokens x the qpk query
// heads of one KV head, the packed GQA tile of
// "vllm_triton_unified_attention_notes"), split into query tiles 0 and 1 of
// 128 rows that share every K/V tile, against their causal key prefix in key
// tiles of 128. The loop is the FA2 forward of the "Fused Attention" notes
// (S = Q K^T, online softmax in base 2, O += P V, O / l at the end); the two
// query tiles are interleaved on the tensor core in the ping-pong manner the
// notes describe for FlashAttention-3, so that one tile's softmax overlaps
// the other tile's matrix products.
// One CTA per SM (at most) takes work tiles from a queue in list order as it
// frees up; the rings and barrier phases run on from one work tile to the
// next, so the next tile's Q and first K/V tiles load while the current one
// finishes, and its output store overlaps the next tile's first products.
//   warp 0      TMA producer of Q (per query tile, refilled once the last S
//               MMA of the previous work tile has read it) and of the K ring;
//   warp 2      TMA producer of the V ring (one box per page, resolved through
//               the block table);
//   warp 1      owns the tensor memory; one thread issues the MMAs in the order
//               S0(j) S1(j) | PV0(j) S0(j+1) | PV1(j) S1(j+1) | ...
//               (S_t into TMEM columns 128t, O_t into 256 + 128t; P_t is read
//               from TMEM where the softmax wrote it over S_t);
//   warp 3      scheduler: one thread claims the next work tile and hands it
//               to the other roles through a shared-memory descriptor;
//   warps 4-7   softmax of query tile 0, one row per thread (TMEM lane);
//   warps 8-11  softmax of query tile 1.
// Softmax: scale, mask by select, running max / sum, P = 2^(x - m) stored as
// bf16 over S; O is rescaled in TMEM only when the row max grew by more than
// 2^8 (exact: P and l use the same stale max); epilogue O / l -> bf16.
// Every mbarrier wait is bounded; a wait that gives up records
// UA_ERR_DEVICE_TIMEOUT, makes the other roles give up, drains the copies and
// MMAs in flight and frees the tensor memory before the CTA exits.
#include <cuda.h>

#include "sm100.cuh"
#include "ua_device.cuh"
#include "ua_kernels.h"

namespace ua {
namespace {

using namespace sm100;

constexpr int kRows = 128;        // query rows per query tile (TMEM lanes, MMA M)
constexpr int kTilesPerCta = 2;   // query tiles per CTA
constexpr int kKeys = 128;        // keys per key tile (MMA N of S, K of PV)
constexpr int kThreads = 384;     // 12 warps: control warpgroup + two softmax warpgroups
// Register split (setmaxnreg): the control warpgroup gives registers back, the
// softmax warpgroups take them. 128 * 56 + 256 * 224 = 64512 = 384 * 168, the
// budget of a launch at 168 registers per thread; the host checks the compiled
// count before every launch so that the increase can always be granted.
constexpr uint32_t kCtrlRegs = 56;
constexpr uint32_t kSoftmaxRegs = 224;
constexpr int kLaunchRegs = 168;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// Work-tile descriptors the scheduler warp keeps ahead: one. A CTA claims its
// next tile only when every role has started the current one, which keeps
// the claims close to the order in which the CTAs run dry.
constexpr int kItemSlots = 1;
constexpr int kItemBytes = 64;  // one descriptor in shared memory
// Arrivals that free a descriptor slot: the two producer threads, the MMA
// thread and the eight softmax warps (one lane each).
constexpr int kItemConsumers = 3 + 8;

// F8: the fp8-products variant (e4m3 Q, K, V and P operands of kind::f8f6f4
// MMAs over an e4m3 cache, head_dim 128): 1-byte elements, so one 128-byte
// swizzled panel holds a whole 128-wide row.
template <int D, bool F8>
struct Smem {
  static_assert(!F8 || D == 128, "fp8 products at head_dim 128");
  static constexpr int kElt = F8 ? 1 : 2;                // operand bytes
  static constexpr int kPanelDims = 128 / kElt;          // head dims per 128-byte panel
  static constexpr int kPanels = D / kPanelDims;
  static constexpr int kKStages = F8 ? 4 : (D == 128 ? 3 : 4);
  static constexpr int kVStages = F8 ? 4 : (D == 128 ? 2 : 4);
  static constexpr int kPanel = kRows * 128;            // one panel of 128 rows: 16 KB
  static constexpr int kTile = kRows * D * kElt;        // 128 x D operands
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTilesPerCta * kTile;
  static constexpr int kV = kK + kKStages * kTile;
  static constexpr int kBar = kV + kVStages * kTile;
  // q_full/q_empty[2], kfull/kempty[KS], vfull/vempty[VS], s_full/p_ready/o_done[2],
  // mma_done, item_full/item_empty[kItemSlots]
  static constexpr int kNumBars = 2 * kTilesPerCta + 2 * kKStages + 2 * kVStages +
                                  3 * kTilesPerCta + 1 + 2 * kItemSlots;
  static constexpr int kMisc = kBar + 8 * kNumBars;
  static constexpr int kItems = kMisc + 64;
  static constexpr int kBytes = kItems + kItemSlots * kItemBytes;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

// The CTA's mbarriers as 32-bit shared-window addresses: one base register
// and constant offsets (8 bytes per barrier).
template <int D, bool F8>
struct Bars {
  static constexpr int KS = Smem<D, F8>::kKStages, VS = Smem<D, F8>::kVStages;
  uint32_t base;
  __device__ __forceinline__ uint32_t at(int i) const { return base + 8u * static_cast<uint32_t>(i); }
  __device__ __forceinline__ uint32_t q_full(int t) const { return at(t); }   // Q of query tile t landed
  __device__ __forceinline__ uint32_t q_empty(int t) const {                  // its last S MMA read it
    return at(kTilesPerCta + t);
  }
  __device__ __forceinline__ uint32_t kfull(int s) const { return at(2 * kTilesPerCta + s); }
  __device__ __forceinline__ uint32_t kempty(int s) const { return at(2 * kTilesPerCta + KS + s); }
  __device__ __forceinline__ uint32_t vfull(int s) const {
    return at(2 * kTilesPerCta + 2 * KS + s);
  }
  __device__ __forceinline__ uint32_t vempty(int s) const {
    return at(2 * kTilesPerCta + 2 * KS + VS + s);
  }
  __device__ __forceinline__ uint32_t s_full(int t) const {
    return at(2 * kTilesPerCta + 2 * KS + 2 * VS + t);
  }
  __device__ __forceinline__ uint32_t p_ready(int t) const {
    return at(3 * kTilesPerCta + 2 * KS + 2 * VS + t);
  }
  __device__ __forceinline__ uint32_t o_done(int t) const {
    return at(4 * kTilesPerCta + 2 * KS + 2 * VS + t);
  }
  __device__ __forceinline__ uint32_t mma_done() const {
    return at(5 * kTilesPerCta + 2 * KS + 2 * VS);
  }
  __device__ __forceinline__ uint32_t item_full(int s) const {   // descriptor s written
    return at(5 * kTilesPerCta + 2 * KS + 2 * VS + 1 + s);
  }
  __device__ __forceinline__ uint32_t item_empty(int s) const {  // every role has read it
    return at(5 * kTilesPerCta + 2 * KS + 2 * VS + 1 + kItemSlots + s);
  }
};

// Geometry of one work tile, computed the same way by every role.
struct Geometry {
  int q_start, ctx, nrows, kv_lo, kv_hi;
  int rows[kTilesPerCta];    // valid rows of each query tile
  int ntiles[kTilesPerCta];  // key tiles each query tile needs
  int nmax;                  // key tiles loaded
};

// One work tile as the scheduler warp hands it to the other roles.
struct Item {
  int seq, kv_head, row0;
  int end;  // 1: no more work tiles for this CTA
  Geometry g;
};
static_assert(sizeof(Item) <= kItemBytes, "work-tile descriptor too large");

// Per-sequence values from the device arrays; ranges are clamped so that
// disagreeing host/device lengths cannot send a read out of bounds.
__device__ __forceinline__ Geometry geometry_of(const PrefillParams& p, const ua_tile& tile) {
  Geometry g;
  g.q_start = p.cu_query_lens[tile.seq];
  const int qlen = p.cu_query_lens[tile.seq + 1] - g.q_start;
  const int kv_len = p.kv_lens[tile.seq];
  g.ctx = kv_len - qlen;
  g.nrows = min(tile.nrows, qlen * p.qpk - tile.row0);
  g.kv_hi = min(min(tile.kv_hi, kv_len), p.max_blocks_per_seq * p.block_size);
  g.kv_lo = tile.kv_lo;
  g.nmax = 0;
#pragma unroll
  for (int t = 0; t < kTilesPerCta; ++t) {
    g.rows[t] = max(0, min(kRows, g.nrows - t * kRows));
    g.ntiles[t] = 0;
    if (g.rows[t] > 0) {
      const int last = tile.row0 + t * kRows + g.rows[t] - 1;
      const int hi = p.causal ? min(g.kv_hi, g.ctx + last / p.qpk + 1) : g.kv_hi;
      g.ntiles[t] = hi > g.kv_lo ? (hi - g.kv_lo + kKeys - 1) / kKeys : 0;
    }
    g.nmax = max(g.nmax, g.ntiles[t]);
  }
  return g;
}

// Give up: record the error once and tell the other roles.
__device__ __forceinline__ void give_up(const PrefillParams& p, volatile int32_t* abort) {
  record_error(p.err, UA_ERR_DEVICE_TIMEOUT);
  *abort = 1;
}

// ------------------------------------------------------------------ scheduler
// One thread of warp 3 claims the CTA's next work tile from the shared queue
// (p.counters[0], a ticket per claim), reads it and the sequence lengths it
// needs from global memory, and publishes it in a shared-memory ring; the
// other roles never wait on a global load between work tiles (those loads
// would queue behind the previous tile's output stores). When the queue is
// empty it publishes an end marker. The last CTA to finish (p.counters[1])
// resets both counters for the next launch; a CTA that gives up still counts
// itself, so the reset happens on the error path too.
template <int D, bool F8>
__device__ __forceinline__ void scheduler_role(const PrefillParams& p, const Bars<D, F8>& bar,
                                               uint8_t* ring, volatile int32_t* abort) {
  for (int k = 0;; ++k) {
    const int s = k % kItemSlots;
    if (k >= kItemSlots &&
        !mbar_wait(bar.item_empty(s), ((k / kItemSlots) - 1) & 1, abort, p.timeout_ns)) {
      give_up(p, abort);
      break;
    }
    Item it = {};
    const int idx = atomicAdd(&p.counters[0], 1);
    it.end = idx >= p.num_tiles ? 1 : 0;
    if (!it.end) {
      const ua_tile tile = p.tiles[idx];
      it.seq = tile.seq;
      it.kv_head = tile.kv_head;
      it.row0 = tile.row0;
      it.g = geometry_of(p, tile);
    }
    *reinterpret_cast<Item*>(ring + s * kItemBytes) = it;
    mbar_arrive(bar.item_full(s));  // release: the descriptor is visible to its readers
    if (it.end) break;
  }
  __threadfence();
  if (atomicAdd(&p.counters[1], 1) == static_cast<int>(gridDim.x) - 1) {
    atomicExch(&p.counters[0], 0);
    atomicExch(&p.counters[1], 0);
  }
}

// Wait for work-tile descriptor k and copy it out of the ring. The caller
// then frees the slot (one arrival per consumer thread or softmax warp).
template <int D, bool F8>
__device__ __forceinline__ bool take_item(const PrefillParams& p, const Bars<D, F8>& bar,
                                          const uint8_t* ring, int k, Item& it,
                                          volatile int32_t* abort) {
  const int s = k % kItemSlots;
  if (!mbar_wait(bar.item_full(s), (k / kItemSlots) & 1, abort, p.timeout_ns)) return false;
  it = *reinterpret_cast<const Item*>(ring + s * kItemBytes);
  return true;
}

// ------------------------------------------------------------------ producers
// Key tile j of a work tile into one ring slot: one TMA box per page (or per
// 128 rows of a larger page) and 64-wide panel. Every page id is read from
// the block table and checked; a missing or out-of-range page is loaded from
// an out-of-range block coordinate, which TMA fills with zeros.
template <int D, bool F8>
__device__ __forceinline__ void load_key_tile(const CUtensorMap* map, const PrefillParams& p,
                                              const Item& tile, const Geometry& g, int j,
                                              uint8_t* dst, uint32_t full) {
  using L = Smem<D, F8>;
  constexpr int kPanels = L::kPanels;
  const int boxes = kKeys / p.rows_per_box;
  const int base = g.kv_lo + j * kKeys;
  mbar_arrive_expect_tx(full, L::kTile);
  if (boxes == 1) {
    // Pages of at least a key tile: one box (and one page-table load).
    int32_t blk = static_cast<int32_t>(p.num_blocks);  // out of range: zero fill
    int32_t slot = 0;
    if (base < g.kv_hi) {
      const int32_t id =
          p.block_tables[static_cast<int64_t>(tile.seq) * p.max_blocks_per_seq + base / p.block_size];
      if (id >= 0 && static_cast<int64_t>(id) < p.num_blocks) {
        blk = id;
        slot = base % p.block_size;
      } else {
        record_error(p.err, UA_ERR_BOUNDS);
      }
    }
#pragma unroll
    for (int pn = 0; pn < kPanels; ++pn)
      tma_load_4d(dst + pn * L::kPanel, map, full, pn * L::kPanelDims, tile.kv_head, slot, blk);
    return;
  }
  for (int b = 0; b < boxes; ++b) {
    const int key0 = base + b * p.rows_per_box;
    int32_t blk = static_cast<int32_t>(p.num_blocks);  // out of range: zero fill
    int32_t slot = 0;
    if (key0 < g.kv_hi) {
      const int32_t id =
          p.block_tables[static_cast<int64_t>(tile.seq) * p.max_blocks_per_seq + key0 / p.block_size];
      if (id >= 0 && static_cast<int64_t>(id) < p.num_blocks) {
        blk = id;
        slot = key0 % p.block_size;
      } else {
        record_error(p.err, UA_ERR_BOUNDS);
      }
    }
    const int row_off = b * p.rows_per_box * 128;
#pragma unroll
    for (int pn = 0; pn < kPanels; ++pn)
      tma_load_4d(dst + pn * L::kPanel + row_off, map, full, pn * L::kPanelDims, tile.kv_head,
                  slot, blk);
  }
}

// One thread of warp 0: per work tile, Q of query tile 0, the K ring, and Q
// of query tile 1 after the first key tile (a Q buffer is refilled once the
// last S MMA of the previous work tile has read it). One thread of warp 2
// (kIsV): the V ring. Ring positions run on across the CTA's work tiles.
template <int D, bool F8, bool kIsV>
__device__ __forceinline__ void producer_role(const CUtensorMap* map_q, const CUtensorMap* map_kv,
                                              const PrefillParams& p, const uint8_t* ring,
                                              uint8_t* sQ, uint8_t* sRing, uint32_t full,
                                              uint32_t empty, const Bars<D, F8>& bar,
                                              volatile int32_t* abort, volatile int32_t* never) {
  using L = Smem<D, F8>;
  constexpr int kPanels = L::kPanels;
  constexpr int kStages = kIsV ? L::kVStages : L::kKStages;
  prefetch_tmap(map_kv);
  if (!kIsV && !F8) prefetch_tmap(map_q);
  const bool idle = (p.debug_flags & kDebugProducerIdle) != 0;
  int last_phase[kStages];
#pragma unroll
  for (int s = 0; s < kStages; ++s) last_phase[s] = -1;
  int q_loads[kTilesPerCta] = {0, 0};
  bool ok = true;
  // Q of query tile t is loaded exactly when the MMA issuer will consume it.
  auto load_q = [&](const Item& tile, const Geometry& g, int t) {
    if (F8 || g.ntiles[t] <= 0) return true;  // F8: the softmax warps write Q
    if (q_loads[t] > 0 &&
        !mbar_wait(bar.q_empty(t), (q_loads[t] - 1) & 1, abort, p.timeout_ns))
      return false;
    mbar_arrive_expect_tx(bar.q_full(t), kRows * D * 2);
#pragma unroll
    for (int pn = 0; pn < kPanels; ++pn)
      tma_load_3d(sQ + t * L::kTile + pn * L::kPanel, map_q, bar.q_full(t), pn * 64,
                  tile.kv_head * p.qpk, g.q_start + (tile.row0 + t * kRows) / p.qpk);
    ++q_loads[t];
    return true;
  };
  if (!idle) {
    int step = 0;  // position in the ring sequence
    for (int k = 0; ok; ++k) {
      Item tile;
      if (!take_item<D, F8>(p, bar, ring, k, tile, abort)) {
        ok = false;
        break;
      }
      mbar_arrive(bar.item_empty(k % kItemSlots));
      if (tile.end) break;
      const Geometry& g = tile.g;
      if (g.nmax <= 0) continue;
      if (!kIsV) ok = load_q(tile, g, 0);
      for (int j = 0; ok && j < g.nmax; ++j, ++step) {
        const int s = step % kStages;
        if (step >= kStages &&
            !mbar_wait(empty + 8u * s, ((step / kStages) - 1) & 1, abort, p.timeout_ns)) {
          ok = false;
          break;
        }
        load_key_tile<D, F8>(map_kv, p, tile, g, j, sRing + s * L::kTile, full + 8u * s);
        last_phase[s] = step / kStages;
        if (!kIsV && j == 0) ok = load_q(tile, g, 1);
      }
    }
    if (!ok) give_up(p, abort);
  }
  // Drain: every load issued completes before the CTA may exit.
#pragma unroll
  for (int s = 0; s < kStages; ++s)
    if (last_phase[s] >= 0 && !mbar_wait(full + 8u * s, last_phase[s] & 1, never, p.timeout_ns))
      give_up(p, abort);
  if (!kIsV) {
#pragma unroll
    for (int t = 0; t < kTilesPerCta; ++t)
      if (q_loads[t] > 0 && !mbar_wait(bar.q_full(t), (q_loads[t] - 1) & 1, never, p.timeout_ns))
        give_up(p, abort);
  }
}

// ------------------------------------------------------------------ MMA issuer
// Per work tile: S0(0) S1(0) | PV0(j) S0(j+1) PV1(j) S1(j+1) | ...; ring
// positions and the per-query-tile barrier phases run on across work tiles.
template <int D, bool F8>
__device__ __forceinline__ void mma_role(const PrefillParams& p, const uint8_t* ring, uint8_t* sQ,
                                         uint8_t* sK, uint8_t* sV, uint32_t tmem,
                                         const Bars<D, F8>& bar, volatile int32_t* abort,
                                         volatile int32_t* never) {
  using L = Smem<D, F8>;
  constexpr int KS = L::kKStages, VS = L::kVStages;
  constexpr uint32_t idesc_s =
      F8 ? idesc_e4m3_f32(kRows, kKeys, 0, 0) : idesc_bf16_f32(kRows, kKeys, 0, 0);
  constexpr uint32_t idesc_o = F8 ? idesc_e4m3_f32(kRows, D, 0, 1) : idesc_bf16_f32(kRows, D, 0, 1);
  // One MMA covers kStep elements of the contraction: 32 bytes of every
  // operand row (16 bf16 or 32 e4m3 values).
  constexpr int kStep = 32 / L::kElt;
  // Each operand descriptor is built once per group of MMAs; the k-th MMA
  // adds its byte offset / 16 to the 14-bit start-address field (shared
  // addresses stay below 256 KB, so the field cannot overflow).
  auto issue_s = [&](int t, int gj) {
    const uint64_t qd = smem_desc_sw128(opaque_u32(smem_u32(sQ)) + t * L::kTile, 16, 1024);
    const uint64_t kd = smem_desc_sw128(smem_u32(sK) + (gj % KS) * L::kTile, 16, 1024);
#pragma unroll
    for (int k = 0; k < D / kStep; ++k) {
      const uint64_t off = static_cast<uint64_t>(((k / 4) * L::kPanel + (k % 4) * 32) >> 4);
      if constexpr (F8) mma_ss_f8(tmem + t * kKeys, qd + off, kd + off, idesc_s, k > 0 ? 1u : 0u);
      else mma_ss(tmem + t * kKeys, qd + off, kd + off, idesc_s, k > 0 ? 1u : 0u);
    }
    mma_commit(bar.s_full(t));
  };
  // P from TMEM (kStep keys = 8 columns per MMA), V's rows kStep * 128 bytes
  // apart per MMA.
  auto issue_pv = [&](int t, int gj, bool acc) {
    const uint64_t vd = smem_desc_sw128(smem_u32(sV) + (gj % VS) * L::kTile, L::kPanel, 1024);
#pragma unroll
    for (int k = 0; k < kKeys / kStep; ++k) {
      const uint64_t off = static_cast<uint64_t>((k * kStep * 128) >> 4);
      if constexpr (F8)
        mma_ts_f8(tmem + 256 + t * 128, tmem + t * kKeys + 8 * k, vd + off, idesc_o,
                  (acc || k > 0) ? 1u : 0u);
      else
        mma_ts(tmem + 256 + t * 128, tmem + t * kKeys + 8 * k, vd + off, idesc_o,
               (acc || k > 0) ? 1u : 0u);
    }
    mma_commit(bar.o_done(t));
  };
  int step = 0;                       // ring position of key tile 0 of the work tile
  int done[kTilesPerCta] = {0, 0};    // key tiles of each query tile so far
  int q_used[kTilesPerCta] = {0, 0};  // Q loads consumed per query tile
  bool ok = true;
  for (int k = 0; ok; ++k) {
    Item it;
    if (!take_item<D, F8>(p, bar, ring, k, it, abort)) {
      ok = false;
      break;
    }
    mbar_arrive(bar.item_empty(k % kItemSlots));
    if (it.end) break;
    const Geometry& g = it.g;
    if (g.nmax <= 0) continue;
    const int n0 = g.ntiles[0], n1 = g.ntiles[1];
    ok = mbar_wait(bar.kfull(step % KS), (step / KS) & 1, abort, p.timeout_ns);
    if (ok && n0 > 0) {
      ok = mbar_wait(bar.q_full(0), q_used[0] & 1, abort, p.timeout_ns);
      if (ok) {
        tc_fence_after();
        issue_s(0, step);
        if (n0 == 1) mma_commit(bar.q_empty(0));
      }
    }
    if (ok && n1 > 0) {
      ok = mbar_wait(bar.q_full(1), q_used[1] & 1, abort, p.timeout_ns);
      if (ok) {
        tc_fence_after();
        issue_s(1, step);
        if (n1 == 1) mma_commit(bar.q_empty(1));
      }
    }
    if (!ok) break;
    mma_commit(bar.kempty(step % KS));
    for (int j = 0; j < g.nmax; ++j) {
      const int gj = step + j;
      if (!mbar_wait(bar.vfull(gj % VS), (gj / VS) & 1, abort, p.timeout_ns)) {
        ok = false;
        break;
      }
      if (j < n0) {
        if (!mbar_wait(bar.p_ready(0), (done[0] + j) & 1, abort, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(0, gj, j > 0);
      }
      const bool more = j + 1 < g.nmax;
      if (more) {
        if (!mbar_wait(bar.kfull((gj + 1) % KS), ((gj + 1) / KS) & 1, abort, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (j + 1 < n0) {
          issue_s(0, gj + 1);
          if (j + 2 == n0) mma_commit(bar.q_empty(0));
        }
      }
      if (j < n1) {
        if (!mbar_wait(bar.p_ready(1), (done[1] + j) & 1, abort, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(1, gj, j > 0);
      }
      mma_commit(bar.vempty(gj % VS));
      if (more) {
        if (j + 1 < n1) {
          issue_s(1, gj + 1);
          if (j + 2 == n1) mma_commit(bar.q_empty(1));
        }
        mma_commit(bar.kempty((gj + 1) % KS));
      }
    }
    step += g.nmax;
    done[0] += n0;
    done[1] += n1;
    q_used[0] += n0 > 0;
    q_used[1] += n1 > 0;
  }
  if (!ok) give_up(p, abort);
  // Drain: every MMA issued has completed before the tensor memory is freed.
  mma_commit(bar.mma_done());
  if (!mbar_wait(bar.mma_done(), 0, never, p.timeout_ns)) give_up(p, abort);
}
// ------------------------------------------------------------------ softmax
// What the softmax of one query tile needs of a work tile, as scalars (a
// runtime index into the descriptor would put it in local memory).
struct SoftmaxTile {
  int kv_head, row0, q_start, ctx, kv_lo, kv_hi, nmax;
  int n_t;     // key tiles of this query tile
  int rows_t;  // valid rows of this query tile
};

// Query tile t of one work tile, one thread per row r (TMEM lane r). A warp may
// only touch TMEM lanes 32 * (warp % 4) .. + 31, which fixes the rows of each
// warp. `done` is the number of key tiles this query tile has already had in
// earlier work tiles (barrier phases), `step` the ring position of key tile 0.
template <int D, bool F8>
__device__ __forceinline__ bool softmax_tile(const PrefillParams& p, const SoftmaxTile& g, int t,
                                             int done, int step, uint8_t* sQ, uint8_t* sV,
                                             uint32_t tmem,
                                             const Bars<D, F8>& bar, volatile int32_t* abort,
                                             int warp, int lane) {
  using L = Smem<D, F8>;
  constexpr int kPanels = L::kPanels;
  constexpr int VS = L::kVStages;
  const int n_t = g.n_t;
  const uint32_t quarter = static_cast<uint32_t>(warp & 3);
  const int r = static_cast<int>(quarter) * 32 + lane;
  const uint32_t lane_addr = (quarter * 32) << 16;
  const uint32_t s_tmem = tmem + lane_addr + t * kKeys;
  const uint32_t o_tmem = tmem + lane_addr + 256 + t * 128;
  const int rr = min(r, g.rows_t - 1);   // rows past the end behave like the last one
  const int row = g.row0 + t * kRows + rr;
  const int pos = g.ctx + row / p.qpk;
  // Scores are used as x = s * c with c >= 0: a negative scale flips the sign
  // of the raw scores once, so that the row max is always a max.
  const bool neg = p.score_scale_log2 < 0.f;
  float c = neg ? -p.score_scale_log2 : p.score_scale_log2;
  if constexpr (F8) {
    // This thread's Q row to e4m3 with its own scale (inv = 448 / max |q|,
    // binary32; 1 for a zero row or a row past the end), written into query
    // tile t's operand tile in the 128-byte swizzled layout TMA would give it
    // (16-byte chunk k of row r at chunk k ^ (r % 8)). The previous work
    // tile's products that read this tile have completed (its last P V did,
    // before this warp's epilogue). The scores then carry 1 / inv.
    static_assert(D == 128, "one 128-byte row per query row");
    uint32_t w[D / 2];
    if (r < g.rows_t) {
      const uint4* src = reinterpret_cast<const uint4*>(
          reinterpret_cast<const uint8_t*>(p.q) +
          (static_cast<int64_t>(g.q_start + row / p.qpk) * p.num_q_heads + g.kv_head * p.qpk +
           row % p.qpk) * D * 2);
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        const uint4 v = src[i];
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < D / 2; ++i) w[i] = 0u;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < D / 2; ++i)
      amax = fmax3(amax, fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i])));
    const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
    uint8_t* qrow = sQ + t * L::kTile + r * 128;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t e[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t a = w[8 * k + 2 * i], b = w[8 * k + 2 * i + 1];
        e[i] = to_e4m3x4(__fmul_rn(bf16_lo(a), inv), __fmul_rn(bf16_hi(a), inv),
                         __fmul_rn(bf16_lo(b), inv), __fmul_rn(bf16_hi(b), inv));
      }
      *reinterpret_cast<uint4*>(qrow + ((k ^ (r & 7)) * 16)) = make_uint4(e[0], e[1], e[2], e[3]);
    }
    fence_proxy_async_smem();
    mbar_arrive(bar.q_full(t));
    c = __fdiv_rn(c, inv);
  }
  float m = -INFINITY, l = 0.f;
  for (int j = 0; j < n_t; ++j) {
    if (!__all_sync(0xffffffffu, mbar_wait(bar.s_full(t), (done + j) & 1, abort, p.timeout_ns)))
      return false;
    tc_fence_after();
    const int base = g.kv_lo + j * kKeys;
    // Raw scores; the scale is folded into one fma per pair below.
    float x[kKeys];
    {
      uint32_t v[kKeys / 32][32];
#pragma unroll
      for (int ch = 0; ch < kKeys / 32; ++ch) tmem_ld32(s_tmem + ch * 32, v[ch]);
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < kKeys / 32; ++ch)
#pragma unroll
        for (int i = 0; i < 32; ++i) x[ch * 32 + i] = __uint_as_float(v[ch][i]);
    }
    if (neg) {
#pragma unroll
      for (int i = 0; i < kKeys; ++i) x[i] = -x[i];
    }
    // Mask by select: keys past the range, past the row's position (causal)
    // or at or below pos - window.
    const int hi_col = min(g.kv_hi, p.causal ? pos + 1 : g.kv_hi) - base;
    const int lo_col = p.window > 0 ? pos - p.window + 1 - base : INT_MIN;
    if (hi_col < kKeys || lo_col > 0) {
#pragma unroll
      for (int i = 0; i < kKeys; ++i)
        if (i >= hi_col || i < lo_col) x[i] = -INFINITY;
    }
    // Row max with independent 3-input partial maxima.
    constexpr int kAcc = 8;
    float mxp[kAcc];
#pragma unroll
    for (int a = 0; a < kAcc; ++a) mxp[a] = x[a];
#pragma unroll
    for (int i = kAcc; i < kKeys; i += 2)
      mxp[(i / 2) % kAcc] = fmax3(mxp[(i / 2) % kAcc], x[i], x[i + 1]);
    const float mx_raw = fmax3(fmax3(mxp[0], mxp[1], mxp[2]), fmax3(mxp[3], mxp[4], mxp[5]),
                               fmaxf(mxp[6], mxp[7]));
    const float m_new = fmaxf(m, mx_raw * c);
    const bool grow = (m == -INFINITY) || (m_new > m + kRescaleThreshold);
    const float m_use = grow ? m_new : m;
    const float alpha = grow ? ((m == -INFINITY) ? 0.f : ex2(m - m_use)) : 1.f;
    const float sub = (m_use == -INFINITY) ? 0.f : m_use;
    // p = 2^(x * c - m): one paired fma per two keys, then ex2; paired sums.
    const uint64_t c2 = f2_pack(c, c), nsub2 = f2_pack(-sub, -sub);
    uint64_t sum2[kAcc / 2];
#pragma unroll
    for (int a = 0; a < kAcc / 2; ++a) sum2[a] = f2_pack(0.f, 0.f);
    // P packed for the P V products: bf16 pairs, or e4m3 quadruples (F8:
    // p <= 2^8 against the lagging reference, inside e4m3's range; l sums the
    // unrounded p).
    constexpr int kPk = F8 ? kKeys / 4 : kKeys / 2;
    uint32_t pk[kPk];
    float q0 = 0.f, q1 = 0.f;
#pragma unroll
    for (int i = 0; i < kKeys / 2; ++i) {
      float e0, e1;
      f2_unpack(f2_fma(f2_pack(x[2 * i], x[2 * i + 1]), c2, nsub2), e0, e1);
      const float p0 = ex2(e0), p1 = ex2(e1);
      sum2[i % (kAcc / 2)] = f2_add(sum2[i % (kAcc / 2)], f2_pack(p0, p1));
      if constexpr (F8) {
        if (i % 2 == 0) {
          q0 = p0;
          q1 = p1;
        } else {
          pk[i / 2] = to_e4m3x4(q0, q1, p0, p1);
        }
      } else {
        pk[i] = pack2<false>(p0, p1);
      }
    }
    sum2[0] = f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3]));
    float sum_lo, sum_hi;
    f2_unpack(sum2[0], sum_lo, sum_hi);
    l = l * alpha + (sum_lo + sum_hi);
    m = m_use;
    // Rescale O in TMEM when some row of this warp moved its max (after the
    // exponentials: the raw scores are dead by then, which keeps the register
    // peak low).
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
      if (!__all_sync(0xffffffffu,
                      mbar_wait(bar.o_done(t), (done + j - 1) & 1, abort, p.timeout_ns)))
        return false;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(o_tmem + ch * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
        tmem_st32(o_tmem + ch * 32, v);
      }
    }
    // P over the first 64 (bf16) or 32 (e4m3) columns of this query tile's
    // score columns.
#pragma unroll
    for (int ch = 0; ch < kPk / 32; ++ch) {
      uint32_t v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = pk[ch * 32 + i];
      tmem_st32(s_tmem + ch * 32, v);
    }
    tmem_wait_st();
    // The last key tile may end inside a page: zero the V rows past the range
    // (they can hold anything, and 0 * NaN would reach O).
    const int valid = g.kv_hi - base;
    if (valid < kKeys && j == g.nmax - 1) {
      const int gj = step + j;
      const int sv = gj % VS;
      if (!__all_sync(0xffffffffu, mbar_wait(bar.vfull(sv), (gj / VS) & 1, abort, p.timeout_ns)))
        return false;
      uint8_t* vt = sV + sv * L::kTile;
      const int dead = kKeys - valid;
      for (int idx = r; idx < dead * kPanels * 8; idx += kRows) {
        const int line = idx / 8, chunk = idx % 8;
        *reinterpret_cast<uint4*>(vt + (line / dead) * L::kPanel + (valid + line % dead) * 128 +
                                  chunk * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
    }
    tc_fence_before();
    mbar_arrive(bar.p_ready(t));
  }
  if (!__all_sync(0xffffffffu, mbar_wait(bar.o_done(t), (done + n_t - 1) & 1, abort, p.timeout_ns)))
    return false;
  tc_fence_after();
  // Epilogue: O / l -> bf16 row of the output. The next work tile's first PV
  // into this O is issued only after this warp's next P is ready, i.e. after
  // these loads have completed.
  const float inv = l > 0.f ? p.out_scale / l : 0.f;
  const bool row_ok = r < g.rows_t;
  const int tok = g.q_start + row / p.qpk;
  const int head = g.kv_head * p.qpk + row % p.qpk;
  uint8_t* dst = reinterpret_cast<uint8_t*>(p.out) +
                 (static_cast<int64_t>(tok) * p.num_q_heads + head) * D * 2;
#pragma unroll
  for (int ch = 0; ch < D / 32; ++ch) {
    uint32_t v[32];
    tmem_ld32(o_tmem + ch * 32, v);
    tmem_wait_ld();
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      o[i] = pack2<false>(__uint_as_float(v[2 * i]) * inv, __uint_as_float(v[2 * i + 1]) * inv);
    if (row_ok) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint4*>(dst + ch * 64 + i * 16) =
            make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    }
  }
  return true;
}

// Softmax warpgroup of query tile t over the CTA's work tiles.
template <int D, bool F8>
__device__ __forceinline__ void softmax_role(const PrefillParams& p, const uint8_t* ring, int t,
                                             uint8_t* sQ, uint8_t* sV, uint32_t tmem,
                                             const Bars<D, F8>& bar,
                                             volatile int32_t* abort, int warp, int lane) {
  int done = 0, step = 0;
  for (int k = 0;; ++k) {
    Item it;
    if (!__all_sync(0xffffffffu, take_item<D, F8>(p, bar, ring, k, it, abort))) {
      give_up(p, abort);
      return;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar.item_empty(k % kItemSlots));
    if (it.end) break;
    SoftmaxTile st;
    st.kv_head = it.kv_head;
    st.row0 = it.row0;
    st.q_start = it.g.q_start;
    st.ctx = it.g.ctx;
    st.kv_lo = it.g.kv_lo;
    st.kv_hi = it.g.kv_hi;
    st.nmax = it.g.nmax;
    st.n_t = t ? it.g.ntiles[1] : it.g.ntiles[0];
    st.rows_t = t ? it.g.rows[1] : it.g.rows[0];
    if (st.n_t > 0) {
      if (!softmax_tile<D, F8>(p, st, t, done, step, sQ, sV, tmem, bar, abort, warp, lane)) {
        give_up(p, abort);
        return;
      }
      done += st.n_t;
    }
    step += st.nmax;
  }
}

template <int D, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, const PrefillParams p) {
  using L = Smem<D, F8>;
  constexpr int KS = L::kKStages, VS = L::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm + L::kQ;
  uint8_t* sK = sm + L::kK;
  uint8_t* sV = sm + L::kV;
  const Bars<D, F8> bar{smem_u32(sm + L::kBar)};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  volatile int32_t* abort = reinterpret_cast<volatile int32_t*>(sm + L::kMisc + 8);
  volatile int32_t* never = reinterpret_cast<volatile int32_t*>(sm + L::kMisc + 12);
  uint8_t* ring = sm + L::kItems;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // A decode grid queued behind this one with programmatic stream
  // serialization may start once every prefill CTA has started: it then
  // takes the SMs these CTAs leave free. It reads nothing this grid writes.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0 && p.span_start != nullptr) atomicMin(p.span_start, globaltimer_ns());

  if (tid == 0) {
    *abort = 0;
    *never = 0;
    for (int t = 0; t < kTilesPerCta; ++t) {
      mbar_init(bar.q_full(t), F8 ? kRows : 1);  // F8: the softmax threads write Q
      mbar_init(bar.q_empty(t), 1);
    }
    for (int s = 0; s < KS; ++s) {
      mbar_init(bar.kfull(s), 1);
      mbar_init(bar.kempty(s), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(bar.vfull(s), 1);
      mbar_init(bar.vempty(s), 1);
    }
    for (int t = 0; t < kTilesPerCta; ++t) {
      mbar_init(bar.s_full(t), 1);
      mbar_init(bar.p_ready(t), kRows);
      mbar_init(bar.o_done(t), 1);
    }
    mbar_init(bar.mma_done(), 1);
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(bar.item_full(s), 1);
      mbar_init(bar.item_empty(s), kItemConsumers);
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    if (warp == 0 && lane == 0) {
      producer_role<D, F8, false>(&map_q, &map_k, p, ring, sQ, sK, bar.kfull(0), bar.kempty(0), bar,
                              abort, never);
    } else if (warp == 2 && lane == 0) {
      producer_role<D, F8, true>(&map_q, &map_v, p, ring, sQ, sV, bar.vfull(0), bar.vempty(0), bar,
                             abort, never);
    } else if (warp == 1 && lane == 0) {
      mma_role<D, F8>(p, ring, sQ, sK, sV, tmem, bar, abort, never);
    } else if (warp == 3 && lane == 0) {
      scheduler_role<D, F8>(p, bar, ring, abort);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    softmax_role<D, F8>(p, ring, (warp - 4) / 4, sQ, sV, tmem, bar, abort, warp, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0 && p.span_end != nullptr) atomicMax(p.span_end, globaltimer_ns());
}

template <int D, bool F8>
cudaError_t launch_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                     const PrefillParams& p, cudaStream_t stream) {
  // The register split above assumes the launch budget; refuse to launch a
  // build whose register count differs (the increase could never be granted).
  static int checked = 0;
  if (!checked) {
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, prefill_kernel<D, F8>);
    if (e != cudaSuccess) return e;
    if (attr.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    checked = 1;
  }
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = set_smem_once(prefill_kernel<D, F8>, Smem<D, F8>::kAlloc, smem_set);
  if (e != cudaSuccess) return e;
  prefill_kernel<D, F8><<<p.num_ctas, kThreads, Smem<D, F8>::kAlloc, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

bool prefill_supported(int head_dim, int kv_dtype, int qpk, int block_size) {
  if (prefill_is_wide(head_dim)) return prefill_wide_supported(kv_dtype, qpk, block_size);
  return (head_dim == 64 || head_dim == 128) && kv_dtype == UA_KV_BF16 && qpk >= 1 &&
         qpk <= kRows && kRows % qpk == 0 && block_size >= 16 &&
         (kKeys % block_size == 0 || block_size % kKeys == 0);
}

cudaError_t launch_prefill(const PrefillParams& p, const void* q, const void* k_cache,
                           const void* v_cache, int64_t total_q, int head_dim, int num_kv_heads,
                           cudaStream_t stream) {
  if (p.num_tiles <= 0 || p.num_ctas <= 0) return cudaSuccess;
  if (p.counters == nullptr) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv;
  {
    // Q as [total_q][Hq][D]: a box of (64 dims, qpk heads, 128/qpk tokens)
    // lands as 128 packed rows (token-major, head-minor) in one panel.
    const uint64_t D = static_cast<uint64_t>(head_dim);
    uint64_t dims[3] = {D, static_cast<uint64_t>(p.num_q_heads), static_cast<uint64_t>(total_q)};
    uint64_t strides[2] = {D * 2, static_cast<uint64_t>(p.num_q_heads) * D * 2};
    uint32_t box[3] = {64, static_cast<uint32_t>(p.qpk), static_cast<uint32_t>(kRows / p.qpk)};
    cudaError_t e = encode_tiled_map(&mq, 2, 3, q, dims, strides, box, true, 128);
    if (e != cudaSuccess) return e;
  }
  // K/V pages: (64 dims, one head, rows_per_box slots, one block) per box.
  cudaError_t e = encode_kv_page_map(&mk, k_cache, 2, head_dim, num_kv_heads, p.block_size,
                                     p.num_blocks, 64, p.rows_per_box, true);
  if (e == cudaSuccess)
    e = encode_kv_page_map(&mv, v_cache, 2, head_dim, num_kv_heads, p.block_size, p.num_blocks,
                           64, p.rows_per_box, true);
  if (e != cudaSuccess) return e;
  return head_dim == 128 ? launch_d<128, false>(mq, mk, mv, p, stream)
                         : launch_d<64, false>(mq, mk, mv, p, stream);
}

bool prefill_fp8_products_supported(int head_dim, int qpk, int block_size) {
  return head_dim == 128 && qpk >= 1 && qpk <= kRows && kRows % qpk == 0 && block_size >= 16 &&
         (kKeys % block_size == 0 || block_size % kKeys == 0);
}

cudaError_t launch_prefill_fp8_products(const PrefillParams& p, const void* k_cache,
                                        const void* v_cache, int num_kv_heads,
                                        cudaStream_t stream) {
  if (p.num_tiles <= 0 || p.num_ctas <= 0) return cudaSuccess;
  if (p.counters == nullptr || p.q == nullptr) return cudaErrorInvalidValue;
  // K/V pages of e4m3 codes: (128 dims = one 128-byte panel, one head,
  // rows_per_box slots, one block) per box. Q is read by the softmax warps;
  // its tensor map argument is not used (the K map stands in for it).
  CUtensorMap mk, mv;
  cudaError_t e = encode_kv_page_map(&mk, k_cache, 1, 128, num_kv_heads, p.block_size,
                                     p.num_blocks, 128, p.rows_per_box, true);
  if (e == cudaSuccess)
    e = encode_kv_page_map(&mv, v_cache, 1, 128, num_kv_heads, p.block_size, p.num_blocks, 128,
                           p.rows_per_box, true);
  if (e != cudaSuccess) return e;
  return launch_d<128, true>(mk, mk, mv, p, stream);
}

}  // namespace ua
