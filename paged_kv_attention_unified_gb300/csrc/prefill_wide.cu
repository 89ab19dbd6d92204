// Prefill kernel for head_dim 192 and 256 (K-P, wide heads): tcgen05 / TMEM /
// TMA attention, persistent, one 128-row query tile at a time.
//
// Same work and loop as the head_dim 64 / 128 prefill kernel -- packed rows
// (tokens x the qpk query heads of one KV head, the packed GQA tile of
// "vllm_triton_unified_attention_notes") against their causal key prefix, S =
// Q K^T, online softmax in base 2, O += P V, O / l at the end (the FA2
// forward of the "Fused Attention" notes) -- laid out for a wide head D, whose
// O alone takes D of the 512 TMEM columns and whose Q tile takes D/4 KB of
// shared memory:
//   - one query tile of 128 rows per item (the scheduler cuts each 256-row
//     work tile of the plan into its two query tiles);
//   - key tiles of 64 keys; S is double-buffered in TMEM (columns 0 and 64),
//     so the MMA for key tile j+1 runs while the softmax works on tile j,
//     and O sits in columns 256 .. 256 + D - 1;
//   - S = Q K^T as tcgen05 SS-MMAs (M 128, N 64, D / 16 steps of K = 16 along
//     the head), O += P V as TS-MMAs (M 128, N D, P read from TMEM where the
//     softmax wrote it over S);
//   - shared memory: Q (D / 4 KB), a 3-stage K ring and a 2-stage V ring of
//     D / 8 KB stages (64 keys x D dims, D / 64 128-byte swizzled panels each).
// Warps: 0 TMA producer of Q and the K ring, 1 TMEM owner and MMA issuer, 2
// TMA producer of the V ring, 3 scheduler, 4-7 softmax (one row per thread).
// The rings, barrier phases and S buffers run on across items. Every
// mbarrier wait is bounded; a wait that gives up records
// UA_ERR_DEVICE_TIMEOUT, makes the other roles give up, drains the copies and
// MMAs in flight and frees the tensor memory before the CTA exits.
#include <cuda.h>

#include "sm100.cuh"
#include "ua_device.cuh"
#include "ua_kernels.h"

namespace ua {
namespace {

using namespace sm100;

namespace wide {

constexpr int kRows = 128;      // query rows per item (TMEM lanes, MMA M)
constexpr int kKeys = 64;       // keys per key tile (MMA N of S, K of P V)
constexpr int kPlanRows = 256;  // rows of one work tile of the plan (two items)
constexpr int kThreads = 256;   // 8 warps
constexpr int KS = 3;           // K ring stages
constexpr int VS = 2;           // V ring stages
constexpr int kPanelQ = kRows * 128;        // one Q panel: 16 KB
constexpr int kPanelKV = kKeys * 128;       // one K / V panel: 8 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;             // O columns 256 .. 256 + D - 1
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr int kItemBytes = 64;
// Arrivals that free the item slot: two producer threads, the MMA thread and
// the four softmax warps (one lane each).
constexpr int kItemConsumers = 3 + 4;

// Shared-memory layout (byte offsets; the ring stages are 1024-byte aligned).
template <int D>
struct Geo {
  static_assert(D == 192 || D == 256, "head_dim of the wide prefill kernel");
  static constexpr int kPanels = D / 64;           // 128-byte swizzled panels per row block
  static constexpr int kQBytes = kRows * D * 2;    // 48 / 64 KB
  static constexpr int kStage = kKeys * D * 2;     // 24 / 32 KB
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBytes;
  static constexpr int kV = kK + KS * kStage;
  static constexpr int kBar = kV + VS * kStage;
// q_full, q_empty, kfull[KS], kempty[KS], vfull[VS], vempty[VS], s_full[2],
// p_ready[2], o_done[2], mma_done, item_full, item_empty. Key tile g uses S
// buffer g % 2 and the barriers of that parity. A parity wait is only sound
// while its barrier is at most one phase away from the awaited one, and with
// double-buffered S the roles run up to two key tiles apart (S(g) is issued
// before P V(g-1), so the softmax may see S(g) while P V(g-1) still runs):
// one barrier per buffer keeps every waiter within one phase.
  static constexpr int kNumBars = 2 + 2 * KS + 2 * VS + 2 + 2 + 2 + 1 + 2;
  static constexpr int kMisc = kBar + 8 * kNumBars;
  static constexpr int kItems = kMisc + 64;
  static constexpr int kBytes = kItems + kItemBytes;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kAlloc <= 232448, "shared memory of the wide prefill kernel");
};

struct Bars {
  uint32_t base;
  __device__ __forceinline__ uint32_t at(int i) const { return base + 8u * static_cast<uint32_t>(i); }
  __device__ __forceinline__ uint32_t q_full() const { return at(0); }
  __device__ __forceinline__ uint32_t q_empty() const { return at(1); }
  __device__ __forceinline__ uint32_t kfull(int s) const { return at(2 + s); }
  __device__ __forceinline__ uint32_t kempty(int s) const { return at(2 + KS + s); }
  __device__ __forceinline__ uint32_t vfull(int s) const { return at(2 + 2 * KS + s); }
  __device__ __forceinline__ uint32_t vempty(int s) const { return at(2 + 2 * KS + VS + s); }
  __device__ __forceinline__ uint32_t s_full(int b) const { return at(2 + 2 * KS + 2 * VS + b); }
  __device__ __forceinline__ uint32_t p_ready(int b) const { return at(4 + 2 * KS + 2 * VS + b); }
  __device__ __forceinline__ uint32_t o_done(int b) const { return at(6 + 2 * KS + 2 * VS + b); }
  __device__ __forceinline__ uint32_t mma_done() const { return at(8 + 2 * KS + 2 * VS); }
  __device__ __forceinline__ uint32_t item_full() const { return at(9 + 2 * KS + 2 * VS); }
  __device__ __forceinline__ uint32_t item_empty() const { return at(10 + 2 * KS + 2 * VS); }
};

// One 128-row query tile as the scheduler hands it to the other roles.
struct Item {
  int seq, kv_head, row0, rows;  // packed rows [row0, row0 + rows) of the KV head
  int q_start, ctx, kv_lo, kv_hi;
  int ntiles;                    // key tiles of 64 from kv_lo
  int end;                       // 1: no more items for this CTA
};
static_assert(sizeof(Item) <= kItemBytes, "item descriptor too large");

__device__ __forceinline__ void give_up(const PrefillParams& p, volatile int32_t* abort) {
  record_error(p.err, UA_ERR_DEVICE_TIMEOUT);
  *abort = 1;
}

// Item k: wait for its descriptor and copy it out (the caller frees the slot).
__device__ __forceinline__ bool take_item(const PrefillParams& p, const Bars& bar,
                                          const uint8_t* slot, int k, Item& it,
                                          volatile int32_t* abort) {
  if (!mbar_wait(bar.item_full(), k & 1, abort, p.timeout_ns)) return false;
  it = *reinterpret_cast<const Item*>(slot);
  return true;
}

// ------------------------------------------------------------------ scheduler
// One thread of warp 3: claims the next work tile of the plan (256 rows) from
// the shared queue, cuts it into its two 128-row query tiles and publishes
// them one at a time (each once every role has taken the previous one). Per
// query tile the key range ends at the last visible key of its last row.
__device__ __forceinline__ void scheduler_role(const PrefillParams& p, const Bars& bar,
                                               uint8_t* slot, volatile int32_t* abort) {
  int k = 0;
  auto publish = [&](const Item& it) {
    if (k > 0 && !mbar_wait(bar.item_empty(), (k - 1) & 1, abort, p.timeout_ns)) return false;
    *reinterpret_cast<Item*>(slot) = it;
    mbar_arrive(bar.item_full());   // release: the descriptor is visible to its readers
    ++k;
    return true;
  };
  bool ok = true;
  while (ok) {
    const int idx = atomicAdd(&p.counters[0], 1);
    if (idx >= p.num_tiles) {
      Item end = {};
      end.end = 1;
      ok = publish(end);
      break;
    }
    const ua_tile tile = p.tiles[idx];
    const int q_start = p.cu_query_lens[tile.seq];
    const int qlen = p.cu_query_lens[tile.seq + 1] - q_start;
    const int kv_len = p.kv_lens[tile.seq];
    const int nrows = min(tile.nrows, qlen * p.qpk - tile.row0);
    const int kv_hi = min(min(tile.kv_hi, kv_len), p.max_blocks_per_seq * p.block_size);
    for (int t = 0; ok && t * kRows < min(nrows, kPlanRows); ++t) {
      Item it = {};
      it.seq = tile.seq;
      it.kv_head = tile.kv_head;
      it.row0 = tile.row0 + t * kRows;
      it.rows = min(kRows, nrows - t * kRows);
      it.q_start = q_start;
      it.ctx = kv_len - qlen;
      it.kv_lo = tile.kv_lo;
      it.kv_hi = kv_hi;
      const int last = it.row0 + it.rows - 1;
      const int hi = p.causal ? min(kv_hi, it.ctx + last / p.qpk + 1) : kv_hi;
      it.ntiles = hi > it.kv_lo ? (hi - it.kv_lo + kKeys - 1) / kKeys : 0;
      if (it.ntiles > 0) ok = publish(it);
    }
  }
  if (!ok) give_up(p, abort);
  __threadfence();
  if (atomicAdd(&p.counters[1], 1) == static_cast<int>(gridDim.x) - 1) {
    atomicExch(&p.counters[0], 0);
    atomicExch(&p.counters[1], 0);
  }
}

// ------------------------------------------------------------------ producers
// Key tile j of an item into one ring stage: one TMA box per page (or per 64
// rows of a larger page) and 64-wide panel. Every page id is read from the
// block table and checked; a missing or out-of-range page is loaded from an
// out-of-range block coordinate, which TMA fills with zeros.
template <int D>
__device__ __forceinline__ void load_key_tile(const CUtensorMap* map, const PrefillParams& p,
                                              const Item& it, int j, uint8_t* dst, uint32_t full) {
  constexpr int kPanels = Geo<D>::kPanels, kStage = Geo<D>::kStage;
  const int boxes = kKeys / p.rows_per_box;
  const int base = it.kv_lo + j * kKeys;
  mbar_arrive_expect_tx(full, kStage);
  if (boxes == 1) {
    // Pages of at least a key tile: one box (and one page-table load).
    int32_t blk = static_cast<int32_t>(p.num_blocks);  // out of range: zero fill
    int32_t slot = 0;
    if (base < it.kv_hi) {
      const int32_t id =
          p.block_tables[static_cast<int64_t>(it.seq) * p.max_blocks_per_seq + base / p.block_size];
      if (id >= 0 && static_cast<int64_t>(id) < p.num_blocks) {
        blk = id;
        slot = base % p.block_size;
      } else {
        record_error(p.err, UA_ERR_BOUNDS);
      }
    }
#pragma unroll
    for (int pn = 0; pn < kPanels; ++pn)
      tma_load_4d(dst + pn * kPanelKV, map, full, pn * 64, it.kv_head, slot, blk);
    return;
  }
  for (int b = 0; b < boxes; ++b) {
    const int key0 = base + b * p.rows_per_box;
    int32_t blk = static_cast<int32_t>(p.num_blocks);  // out of range: zero fill
    int32_t slot = 0;
    if (key0 < it.kv_hi) {
      const int32_t id =
          p.block_tables[static_cast<int64_t>(it.seq) * p.max_blocks_per_seq + key0 / p.block_size];
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
      tma_load_4d(dst + pn * kPanelKV + row_off, map, full, pn * 64, it.kv_head, slot, blk);
  }
}

// One thread of warp 0 (Q and the K ring) or of warp 2 (kIsV: the V ring).
// Ring positions run on across items.
template <int D, bool kIsV>
__device__ __forceinline__ void producer_role(const CUtensorMap* map_q, const CUtensorMap* map_kv,
                                              const PrefillParams& p, const uint8_t* slot,
                                              uint8_t* sQ, uint8_t* sRing, const Bars& bar,
                                              volatile int32_t* abort, volatile int32_t* never) {
  constexpr int kPanels = Geo<D>::kPanels, kQBytes = Geo<D>::kQBytes, kStage = Geo<D>::kStage;
  constexpr int kStages = kIsV ? VS : KS;
  prefetch_tmap(map_kv);
  if (!kIsV) prefetch_tmap(map_q);
  const bool idle = (p.debug_flags & kDebugProducerIdle) != 0;
  int last_phase[kStages];
#pragma unroll
  for (int s = 0; s < kStages; ++s) last_phase[s] = -1;
  int q_loads = 0;
  bool ok = true;
  if (!idle) {
    int step = 0;  // ring position
    for (int k = 0; ok; ++k) {
      Item it;
      if (!take_item(p, bar, slot, k, it, abort)) {
        ok = false;
        break;
      }
      mbar_arrive(bar.item_empty());
      if (it.end) break;
      if (!kIsV) {
        // Q of this item, once the last S MMA of the previous item has read Q
        if (q_loads > 0 && !mbar_wait(bar.q_empty(), (q_loads - 1) & 1, abort, p.timeout_ns)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar.q_full(), kQBytes);
#pragma unroll
        for (int pn = 0; pn < kPanels; ++pn)
          tma_load_3d(sQ + pn * kPanelQ, map_q, bar.q_full(), pn * 64, it.kv_head * p.qpk,
                      it.q_start + it.row0 / p.qpk);
        ++q_loads;
      }
      for (int j = 0; j < it.ntiles; ++j, ++step) {
        const int s = step % kStages;
        const uint32_t empty = kIsV ? bar.vempty(s) : bar.kempty(s);
        if (step >= kStages &&
            !mbar_wait(empty, ((step / kStages) - 1) & 1, abort, p.timeout_ns)) {
          ok = false;
          break;
        }
        load_key_tile<D>(map_kv, p, it, j, sRing + s * kStage, kIsV ? bar.vfull(s) : bar.kfull(s));
        last_phase[s] = step / kStages;
      }
    }
    if (!ok) give_up(p, abort);
  }
  // Drain: every load issued completes before the CTA may exit.
#pragma unroll
  for (int s = 0; s < kStages; ++s) {
    const uint32_t full = kIsV ? bar.vfull(s) : bar.kfull(s);
    if (last_phase[s] >= 0 && !mbar_wait(full, last_phase[s] & 1, never, p.timeout_ns))
      give_up(p, abort);
  }
  if (!kIsV && q_loads > 0 && !mbar_wait(bar.q_full(), (q_loads - 1) & 1, never, p.timeout_ns))
    give_up(p, abort);
}

// ------------------------------------------------------------------ MMA issuer
// Per item: S(0) S(1) | PV(0) S(2) | PV(1) S(3) | ... | PV(n-1); key tile g
// (counted across items) uses S buffer g % 2, K and V ring position g.
template <int D>
__device__ __forceinline__ void mma_role(const PrefillParams& p, const uint8_t* slot, uint8_t* sQ,
                                         uint8_t* sK, uint8_t* sV, uint32_t tmem, const Bars& bar,
                                         volatile int32_t* abort, volatile int32_t* never) {
  constexpr int kStage = Geo<D>::kStage;
  constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, kKeys, 0, 0);
  constexpr uint32_t idesc_o = idesc_bf16_f32(kRows, D, 0, 1);
  // S(g) = Q K(g)^T into S buffer g % 2; the k-th MMA steps 16 head dims,
  // adding its byte offset / 16 to the descriptors' start-address fields.
  auto issue_s = [&](int g) {
    const uint64_t qd = smem_desc_sw128(opaque_u32(smem_u32(sQ)), 16, 1024);
    const uint64_t kd = smem_desc_sw128(smem_u32(sK) + (g % KS) * kStage, 16, 1024);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint64_t qo = static_cast<uint64_t>(((k / 4) * kPanelQ + (k % 4) * 32) >> 4);
      const uint64_t ko = static_cast<uint64_t>(((k / 4) * kPanelKV + (k % 4) * 32) >> 4);
      mma_ss(tmem + (g % 2) * kKeys, qd + qo, kd + ko, idesc_s, k > 0 ? 1u : 0u);
    }
    mma_commit(bar.s_full(g % 2));
    mma_commit(bar.kempty(g % KS));
  };
  // O (+)= P(g) V(g): P from the first 32 columns of S buffer g % 2, the k-th
  // MMA steps 16 keys (8 TMEM columns of bf16 pairs, 2 KB of the V stage).
  auto issue_pv = [&](int g, bool acc) {
    const uint64_t vd = smem_desc_sw128(smem_u32(sV) + (g % VS) * kStage, kPanelKV, 1024);
#pragma unroll
    for (int k = 0; k < kKeys / 16; ++k)
      mma_ts(tmem + kOCol, tmem + (g % 2) * kKeys + 8 * k,
             vd + static_cast<uint64_t>((k * 2048) >> 4), idesc_o, (acc || k > 0) ? 1u : 0u);
    mma_commit(bar.o_done(g % 2));
    mma_commit(bar.vempty(g % VS));
  };
  int g0 = 0;      // key tiles issued before this item
  int q_used = 0;  // Q loads consumed
  bool ok = true;
  for (int k = 0; ok; ++k) {
    Item it;
    if (!take_item(p, bar, slot, k, it, abort)) {
      ok = false;
      break;
    }
    mbar_arrive(bar.item_empty());
    if (it.end) break;
    const int n = it.ntiles;
    ok = mbar_wait(bar.q_full(), q_used & 1, abort, p.timeout_ns);
    for (int j = 0; ok && j < min(n, 2); ++j) {
      const int g = g0 + j;
      ok = mbar_wait(bar.kfull(g % KS), (g / KS) & 1, abort, p.timeout_ns);
      if (!ok) break;
      tc_fence_after();
      issue_s(g);
      if (j == n - 1) mma_commit(bar.q_empty());
    }
    for (int j = 0; ok && j < n; ++j) {
      const int g = g0 + j;
      if (!mbar_wait(bar.vfull(g % VS), (g / VS) & 1, abort, p.timeout_ns) ||
          !mbar_wait(bar.p_ready(g % 2), (g / 2) & 1, abort, p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_pv(g, j > 0);
      if (j + 2 < n) {
        if (!mbar_wait(bar.kfull((g + 2) % KS), ((g + 2) / KS) & 1, abort, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(g + 2);
        if (j + 2 == n - 1) mma_commit(bar.q_empty());
      }
    }
    g0 += n;
    ++q_used;
  }
  if (!ok) give_up(p, abort);
  // Drain: every MMA issued has completed before the tensor memory is freed.
  mma_commit(bar.mma_done());
  if (!mbar_wait(bar.mma_done(), 0, never, p.timeout_ns)) give_up(p, abort);
}

// ------------------------------------------------------------------ softmax
// Warps 4-7, one thread per row r (TMEM lane r; warp w may only touch lanes
// 32 (w % 4) .. + 31). g0: key tiles of earlier items (barrier phases and S
// buffers).
template <int D>
__device__ __forceinline__ bool softmax_item(const PrefillParams& p, const Item& it, int g0,
                                             uint8_t* sV, uint32_t tmem, const Bars& bar,
                                             volatile int32_t* abort, int warp, int lane) {
  constexpr int kPanels = Geo<D>::kPanels, kStage = Geo<D>::kStage;
  const uint32_t quarter = static_cast<uint32_t>(warp & 3);
  const int r = static_cast<int>(quarter) * 32 + lane;
  const uint32_t lane_addr = (quarter * 32) << 16;
  const uint32_t o_tmem = tmem + lane_addr + kOCol;
  const int rr = min(r, it.rows - 1);   // rows past the end behave like the last one
  const int row = it.row0 + rr;
  const int pos = it.ctx + row / p.qpk;
  // Scores are used as x = s * c with c >= 0: a negative scale flips the sign
  // of the raw scores once, so that the row max is always a max.
  const bool neg = p.score_scale_log2 < 0.f;
  const float c = neg ? -p.score_scale_log2 : p.score_scale_log2;
  float m = -INFINITY, l = 0.f;
  const int n = it.ntiles;
  for (int j = 0; j < n; ++j) {
    const int g = g0 + j;
    const uint32_t s_tmem = tmem + lane_addr + (g % 2) * kKeys;
    if (!__all_sync(0xffffffffu, mbar_wait(bar.s_full(g % 2), (g / 2) & 1, abort, p.timeout_ns)))
      return false;
    tc_fence_after();
    const int base = it.kv_lo + j * kKeys;
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
    const int hi_col = min(it.kv_hi, p.causal ? pos + 1 : it.kv_hi) - base;
    const int lo_col = p.window > 0 ? pos - p.window + 1 - base : INT_MIN;
    if (hi_col < kKeys || lo_col > 0) {
#pragma unroll
      for (int i = 0; i < kKeys; ++i)
        if (i >= hi_col || i < lo_col) x[i] = -INFINITY;
    }
    constexpr int kAcc = 8;
    float mxp[kAcc];
#pragma unroll
    for (int a = 0; a < kAcc; ++a) mxp[a] = x[a];
#pragma unroll
    for (int i = kAcc; i < kKeys; i += 2)
      mxp[(i / 2) % kAcc] = fmax3(mxp[(i / 2) % kAcc], x[i], x[i + 1]);
    const float mx_raw = fmax3(fmax3(mxp[0], mxp[1], mxp[2]), fmax3(mxp[3], mxp[4], mxp[5]),
                               fmaxf(mxp[6], mxp[7]));
    // The reference max moves only when the row max grew by more than 2^8:
    // P and l use the same stale reference, so the result is exact up to
    // rounding and O is rescaled only on those steps.
    const float m_new = fmaxf(m, mx_raw * c);
    const bool grow = (m == -INFINITY) || (m_new > m + kRescaleThreshold);
    const float m_use = grow ? m_new : m;
    const float alpha = grow ? ((m == -INFINITY) ? 0.f : ex2(m - m_use)) : 1.f;
    const float sub = (m_use == -INFINITY) ? 0.f : m_use;
    const uint64_t c2 = f2_pack(c, c), nsub2 = f2_pack(-sub, -sub);
    uint64_t sum2[kAcc / 2];
#pragma unroll
    for (int a = 0; a < kAcc / 2; ++a) sum2[a] = f2_pack(0.f, 0.f);
    uint32_t pk[kKeys / 2];
#pragma unroll
    for (int i = 0; i < kKeys / 2; ++i) {
      float e0, e1;
      f2_unpack(f2_fma(f2_pack(x[2 * i], x[2 * i + 1]), c2, nsub2), e0, e1);
      const float p0 = ex2(e0), p1 = ex2(e1);
      sum2[i % (kAcc / 2)] = f2_add(sum2[i % (kAcc / 2)], f2_pack(p0, p1));
      pk[i] = pack2<false>(p0, p1);
    }
    sum2[0] = f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3]));
    float sum_lo, sum_hi;
    f2_unpack(sum2[0], sum_lo, sum_hi);
    l = l * alpha + (sum_lo + sum_hi);
    m = m_use;
    // Rescale O in TMEM when some row of this warp moved its reference (the
    // previous P V must have completed first).
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
      if (!__all_sync(0xffffffffu,
                      mbar_wait(bar.o_done((g - 1) % 2), ((g - 1) / 2) & 1, abort, p.timeout_ns)))
        return false;
      tc_fence_after();
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(o_tmem + ch * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
        tmem_st32(o_tmem + ch * 32, v);
      }
    }
    // P (bf16 pairs) over the first 32 columns of this key tile's S buffer.
    tmem_st32(s_tmem, pk);
    tmem_wait_st();
    // The last key tile may end inside a page: zero the V rows past the range
    // (they can hold anything, and 0 * NaN would reach O).
    const int valid = it.kv_hi - base;
    if (valid < kKeys && j == n - 1) {
      const int sv = g % VS;
      if (!__all_sync(0xffffffffu, mbar_wait(bar.vfull(sv), (g / VS) & 1, abort, p.timeout_ns)))
        return false;
      uint8_t* vt = sV + sv * kStage;
      const int dead = kKeys - valid;
      for (int idx = r; idx < dead * kPanels * 8; idx += kRows) {
        const int line = idx / 8, chunk = idx % 8;
        *reinterpret_cast<uint4*>(vt + (line / dead) * kPanelKV + (valid + line % dead) * 128 +
                                  chunk * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
    }
    tc_fence_before();
    mbar_arrive(bar.p_ready(g % 2));
  }
  // The last P V (key tile g0 + n - 1) and, before it, every earlier one.
  const int gl = g0 + n - 1;
  if (!__all_sync(0xffffffffu,
                  mbar_wait(bar.o_done(gl % 2), (gl / 2) & 1, abort, p.timeout_ns)))
    return false;
  tc_fence_after();
  // Epilogue: O / l -> bf16 row of the output. The next item's first P V into
  // O is issued only after this warp's next P is ready, i.e. after these
  // loads have completed.
  const float inv = l > 0.f ? p.out_scale / l : 0.f;
  const bool row_ok = r < it.rows;
  const int tok = it.q_start + row / p.qpk;
  const int head = it.kv_head * p.qpk + row % p.qpk;
  uint8_t* dst = reinterpret_cast<uint8_t*>(p.out) +
                 (static_cast<int64_t>(tok) * p.num_q_heads + head) * D * 2;
#pragma unroll 1
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

template <int D>
__device__ __forceinline__ void softmax_role(const PrefillParams& p, const uint8_t* slot,
                                             uint8_t* sV, uint32_t tmem, const Bars& bar,
                                             volatile int32_t* abort, int warp, int lane) {
  int g0 = 0;
  for (int k = 0;; ++k) {
    Item it;
    if (!__all_sync(0xffffffffu, take_item(p, bar, slot, k, it, abort))) {
      give_up(p, abort);
      return;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar.item_empty());
    if (it.end) break;
    if (!softmax_item<D>(p, it, g0, sV, tmem, bar, abort, warp, lane)) {
      give_up(p, abort);
      return;
    }
    g0 += it.ntiles;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_wide_kernel(const __grid_constant__ CUtensorMap map_q,
                        const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v, const PrefillParams p) {
  using G = Geo<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm + G::kQ;
  uint8_t* sK = sm + G::kK;
  uint8_t* sV = sm + G::kV;
  const Bars bar{smem_u32(sm + G::kBar)};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + G::kMisc);
  volatile int32_t* abort = reinterpret_cast<volatile int32_t*>(sm + G::kMisc + 8);
  volatile int32_t* never = reinterpret_cast<volatile int32_t*>(sm + G::kMisc + 12);
  uint8_t* slot = sm + G::kItems;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // A decode grid queued behind this one with programmatic stream
  // serialization may start once every CTA here has started; it reads
  // nothing this grid writes.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0 && p.span_start != nullptr) atomicMin(p.span_start, globaltimer_ns());

  if (tid == 0) {
    *abort = 0;
    *never = 0;
    mbar_init(bar.q_full(), 1);
    mbar_init(bar.q_empty(), 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(bar.kfull(s), 1);
      mbar_init(bar.kempty(s), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(bar.vfull(s), 1);
      mbar_init(bar.vempty(s), 1);
    }
    mbar_init(bar.s_full(0), 1);
    mbar_init(bar.s_full(1), 1);
    mbar_init(bar.p_ready(0), kRows);
    mbar_init(bar.p_ready(1), kRows);
    mbar_init(bar.o_done(0), 1);
    mbar_init(bar.o_done(1), 1);
    mbar_init(bar.mma_done(), 1);
    mbar_init(bar.item_full(), 1);
    mbar_init(bar.item_empty(), kItemConsumers);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) producer_role<D, false>(&map_q, &map_k, p, slot, sQ, sK, bar, abort, never);
  } else if (warp == 1) {
    if (lane == 0) mma_role<D>(p, slot, sQ, sK, sV, tmem, bar, abort, never);
  } else if (warp == 2) {
    if (lane == 0) producer_role<D, true>(&map_q, &map_v, p, slot, sQ, sV, bar, abort, never);
  } else if (warp == 3) {
    if (lane == 0) scheduler_role(p, bar, slot, abort);
  } else {
    softmax_role<D>(p, slot, sV, tmem, bar, abort, warp, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0 && p.span_end != nullptr) atomicMax(p.span_end, globaltimer_ns());
}

template <int D>
cudaError_t launch(const PrefillParams& p, const void* q, const void* k_cache,
                   const void* v_cache, int64_t total_q, int num_kv_heads, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  {
    // Q as [total_q][Hq][D]: a box of (64 dims, qpk heads, 128/qpk tokens)
    // lands as 128 packed rows (token-major, head-minor) in one panel.
    uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(p.num_q_heads),
                        static_cast<uint64_t>(total_q)};
    uint64_t strides[2] = {static_cast<uint64_t>(D) * 2,
                           static_cast<uint64_t>(p.num_q_heads) * D * 2};
    uint32_t box[3] = {64, static_cast<uint32_t>(p.qpk), static_cast<uint32_t>(kRows / p.qpk)};
    cudaError_t e = encode_tiled_map(&mq, 2, 3, q, dims, strides, box, true, 128);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = encode_kv_page_map(&mk, k_cache, 2, D, num_kv_heads, p.block_size,
                                     p.num_blocks, 64, p.rows_per_box, true);
  if (e == cudaSuccess)
    e = encode_kv_page_map(&mv, v_cache, 2, D, num_kv_heads, p.block_size, p.num_blocks, 64,
                           p.rows_per_box, true);
  if (e != cudaSuccess) return e;
  static std::atomic<uint64_t> smem_set{0};
  e = set_smem_once(prefill_wide_kernel<D>, Geo<D>::kAlloc, smem_set);
  if (e != cudaSuccess) return e;
  prefill_wide_kernel<D><<<p.num_ctas, kThreads, Geo<D>::kAlloc, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}


}  // namespace wide
}  // namespace

bool prefill_wide_supported(int kv_dtype, int qpk, int block_size) {
  return kv_dtype == UA_KV_BF16 && qpk >= 1 && qpk <= wide::kRows && wide::kRows % qpk == 0 &&
         block_size >= 16 && (wide::kKeys % block_size == 0 || block_size % wide::kKeys == 0);
}

bool prefill_is_wide(int head_dim) { return head_dim == 192 || head_dim == 256; }

int prefill_wide_rows_per_box(int block_size) {
  return block_size < wide::kKeys ? block_size : wide::kKeys;
}

cudaError_t launch_prefill_wide(const PrefillParams& p, const void* q, const void* k_cache,
                                const void* v_cache, int64_t total_q, int head_dim,
                                int num_kv_heads, cudaStream_t stream) {
  if (p.num_tiles <= 0 || p.num_ctas <= 0) return cudaSuccess;
  if (p.counters == nullptr || p.rows_per_box != prefill_wide_rows_per_box(p.block_size))
    return cudaErrorInvalidValue;
  switch (head_dim) {
    case 192: return wide::launch<192>(p, q, k_cache, v_cache, total_q, num_kv_heads, stream);
    case 256: return wide::launch<256>(p, q, k_cache, v_cache, total_q, num_kv_heads, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ua
