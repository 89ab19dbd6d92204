// Prefill kernel (K-P): tcgen05 / TMEM / TMA attention, two 128-row query
// tiles per CTA.
//
// Work unit: one ua_tile of up to 256 packed rows (tokens x the qpk query
// heads of one KV head, the packed GQA tile of
// "vllm_triton_unified_attention_notes"), split into query tiles 0 and 1 of
// 128 rows that share every K/V tile, against their causal key prefix in key
// tiles of 128. The loop is the FA2 forward of the "Fused Attention" notes
// (S = Q K^T, online softmax in base 2, O += P V, O / l at the end); the two
// query tiles are interleaved on the tensor core in the ping-pong manner the
// notes describe for FlashAttention-3, so that one tile's softmax overlaps
// the other tile's matrix products:
//   warp 0      TMA producer of Q (both tiles) and of the K ring, and
//   warp 2      TMA producer of the V ring (one box per page, resolved through
//               the block table);
//   warp 1      owns the tensor memory; one thread issues the MMAs in the order
//               S0(j) S1(j) | PV0(j) S0(j+1) | PV1(j) S1(j+1) | ...
//               (S_t into TMEM columns 128t, O_t into 256 + 128t; P_t is read
//               from TMEM where the softmax wrote it over S_t);
//   warp 3      idle (it completes the control warpgroup);
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

template <int D>
struct Smem {
  static constexpr int kKStages = D == 128 ? 3 : 4;
  static constexpr int kVStages = D == 128 ? 2 : 4;
  static constexpr int kPanel = kRows * 128;           // one 64-wide bf16 panel: 16 KB
  static constexpr int kTile = kRows * D * 2;           // 128 x D bf16
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTilesPerCta * kTile;
  static constexpr int kV = kK + kKStages * kTile;
  static constexpr int kBar = kV + kVStages * kTile;
  // q_full, kfull/kempty[KS], vfull/vempty[VS], s_full/p_ready/o_done[2], mma_done
  static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 3 * kTilesPerCta + 1;
  static constexpr int kMisc = kBar + 8 * kNumBars;
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

struct Bars {
  uint64_t* q_full;
  uint64_t* kfull;
  uint64_t* kempty;
  uint64_t* vfull;
  uint64_t* vempty;
  uint64_t* s_full;   // [2]
  uint64_t* p_ready;  // [2]
  uint64_t* o_done;   // [2]
  uint64_t* mma_done;
};

template <int KS, int VS>
__device__ __forceinline__ Bars bars_at(uint64_t* b) {
  Bars r;
  r.q_full = b;
  r.kfull = b + 1;
  r.kempty = r.kfull + KS;
  r.vfull = r.kempty + KS;
  r.vempty = r.vfull + VS;
  r.s_full = r.vempty + VS;
  r.p_ready = r.s_full + kTilesPerCta;
  r.o_done = r.p_ready + kTilesPerCta;
  r.mma_done = r.o_done + kTilesPerCta;
  return r;
}

// Per-CTA geometry shared by every role.
struct Geometry {
  int q_start, ctx, nrows, kv_lo, kv_hi;
  int rows[kTilesPerCta];    // valid rows of each query tile
  int ntiles[kTilesPerCta];  // key tiles each query tile needs
  int nmax;                  // key tiles loaded
};

// Give up: record the error once and tell the other roles.
__device__ __forceinline__ void give_up(const PrefillParams& p, volatile int32_t* abort) {
  record_error(p.err, UA_ERR_DEVICE_TIMEOUT);
  *abort = 1;
}

// ------------------------------------------------------------------ producer
// One thread of warp 0: Q of both query tiles, then the K ring. One thread of
// warp 2: the V ring.
// Every page id is read from the block table and checked; a missing or
// out-of-range page is loaded from an out-of-range block coordinate, which
// TMA fills with zeros.
template <int D, bool kIsV>
__device__ __forceinline__ void producer_role(const CUtensorMap* map_q, const CUtensorMap* map_kv,
                                              const PrefillParams& p, const ua_tile& tile,
                                              const Geometry& g, uint8_t* sQ, uint8_t* sRing,
                                              uint64_t* full, uint64_t* empty, int stages,
                                              uint64_t* q_full, volatile int32_t* abort,
                                              volatile int32_t* never) {
  using L = Smem<D>;
  constexpr int kPanels = D / 64;
  prefetch_tmap(map_kv);
  const bool idle = (p.debug_flags & kDebugProducerIdle) != 0;
  int last_phase[4] = {-1, -1, -1, -1};
  if (!idle) {
    if (!kIsV) {
      prefetch_tmap(map_q);
      int active = 0;
      for (int t = 0; t < kTilesPerCta; ++t) active += g.rows[t] > 0;
      mbar_arrive_expect_tx(q_full, active * kRows * D * 2);
      for (int t = 0; t < kTilesPerCta; ++t) {
        if (g.rows[t] <= 0) continue;
        for (int pn = 0; pn < kPanels; ++pn)
          tma_load_3d(sQ + t * L::kTile + pn * L::kPanel, map_q, q_full, pn * 64,
                      tile.kv_head * p.qpk, g.q_start + (tile.row0 + t * kRows) / p.qpk);
      }
    }
    const int boxes = kKeys / p.rows_per_box;
    for (int j = 0; j < g.nmax; ++j) {
      const int s = j % stages;
      if (j >= stages &&
          !mbar_wait(&empty[s], ((j / stages) - 1) & 1, abort, p.timeout_ns)) {
        give_up(p, abort);
        break;
      }
      const int base = g.kv_lo + j * kKeys;
      mbar_arrive_expect_tx(&full[s], kKeys * D * 2);
      for (int b = 0; b < boxes; ++b) {
        const int key0 = base + b * p.rows_per_box;
        int32_t blk = static_cast<int32_t>(p.num_blocks);  // out of range: zero fill
        int32_t slot = 0;
        if (key0 < g.kv_hi) {
          const int32_t id = p.block_tables[static_cast<int64_t>(tile.seq) *
                                                p.max_blocks_per_seq + key0 / p.block_size];
          if (id >= 0 && static_cast<int64_t>(id) < p.num_blocks) {
            blk = id;
            slot = key0 % p.block_size;
          } else {
            record_error(p.err, UA_ERR_BOUNDS);
          }
        }
        const int row_off = b * p.rows_per_box * 128;
        for (int pn = 0; pn < kPanels; ++pn)
          tma_load_4d(sRing + s * L::kTile + pn * L::kPanel + row_off, map_kv, &full[s],
                      pn * 64, tile.kv_head, slot, blk);
      }
      last_phase[s] = j / stages;
    }
  }
  // Drain: every load issued completes before the CTA may exit.
  for (int s = 0; s < stages; ++s)
    if (last_phase[s] >= 0 && !mbar_wait(&full[s], last_phase[s] & 1, never, p.timeout_ns))
      give_up(p, abort);
  if (!kIsV && !idle && !mbar_wait(q_full, 0, never, p.timeout_ns)) give_up(p, abort);
}

// ------------------------------------------------------------------ MMA issuer
template <int D>
__device__ __forceinline__ void mma_role(const PrefillParams& p, const Geometry& g, uint8_t* sQ,
                                         uint8_t* sK, uint8_t* sV, uint32_t tmem,
                                         const Bars& bar, volatile int32_t* abort,
                                         volatile int32_t* never) {
  using L = Smem<D>;
  constexpr int KS = L::kKStages, VS = L::kVStages;
  constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, kKeys, 0, 0);
  constexpr uint32_t idesc_o = idesc_bf16_f32(kRows, D, 0, 1);
  auto issue_s = [&](int t, int j) {
    const uint32_t q_addr = smem_u32(sQ + t * L::kTile);
    const uint32_t k_addr = smem_u32(sK + (j % KS) * L::kTile);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k / 4) * L::kPanel + (k % 4) * 32;
      mma_ss(tmem + t * kKeys, smem_desc_sw128(q_addr + off, 16, 1024),
             smem_desc_sw128(k_addr + off, 16, 1024), idesc_s, k > 0 ? 1u : 0u);
    }
    mma_commit(&bar.s_full[t]);
  };
  auto issue_pv = [&](int t, int j) {
    const uint32_t v_addr = smem_u32(sV + (j % VS) * L::kTile);
#pragma unroll
    for (int k = 0; k < kKeys / 16; ++k)
      mma_ts(tmem + 256 + t * 128, tmem + t * kKeys + 8 * k,
             smem_desc_sw128(v_addr + k * 2048, L::kPanel, 1024), idesc_o,
             (j > 0 || k > 0) ? 1u : 0u);
    mma_commit(&bar.o_done[t]);
  };
  const int n0 = g.ntiles[0], n1 = g.ntiles[1];
  bool ok = mbar_wait(bar.q_full, 0, abort, p.timeout_ns) &&
            mbar_wait(&bar.kfull[0], 0, abort, p.timeout_ns);
  if (ok) {
    tc_fence_after();
    if (n0 > 0) issue_s(0, 0);
    if (n1 > 0) issue_s(1, 0);
    mma_commit(&bar.kempty[0]);
  }
  for (int j = 0; ok && j < g.nmax; ++j) {
    if (!mbar_wait(&bar.vfull[j % VS], (j / VS) & 1, abort, p.timeout_ns)) {
      ok = false;
      break;
    }
    if (j < n0) {
      if (!mbar_wait(&bar.p_ready[0], j & 1, abort, p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_pv(0, j);
    }
    const bool more = j + 1 < g.nmax;
    if (more) {
      if (!mbar_wait(&bar.kfull[(j + 1) % KS], ((j + 1) / KS) & 1, abort, p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (j + 1 < n0) issue_s(0, j + 1);
    }
    if (j < n1) {
      if (!mbar_wait(&bar.p_ready[1], j & 1, abort, p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_pv(1, j);
    }
    mma_commit(&bar.vempty[j % VS]);
    if (more) {
      if (j + 1 < n1) issue_s(1, j + 1);
      mma_commit(&bar.kempty[(j + 1) % KS]);
    }
  }
  if (!ok) give_up(p, abort);
  // Drain: every MMA issued has completed before the tensor memory is freed.
  mma_commit(bar.mma_done);
  if (!mbar_wait(bar.mma_done, 0, never, p.timeout_ns)) give_up(p, abort);
}

// ------------------------------------------------------------------ softmax
// Query tile t, one thread per row r (TMEM lane r). A warp may only touch TMEM
// lanes 32 * (warp % 4) .. + 31, which fixes the rows of each warp.
template <int D>
__device__ __forceinline__ void softmax_role(const PrefillParams& p, const ua_tile& tile,
                                             const Geometry& g, int t, uint8_t* sV,
                                             uint32_t tmem, const Bars& bar,
                                             volatile int32_t* abort, int warp, int lane) {
  using L = Smem<D>;
  constexpr int kPanels = D / 64;
  constexpr int VS = L::kVStages;
  const int n_t = g.ntiles[t];
  if (n_t <= 0) return;
  const uint32_t quarter = static_cast<uint32_t>(warp & 3);
  const int r = static_cast<int>(quarter) * 32 + lane;
  const uint32_t lane_addr = (quarter * 32) << 16;
  const uint32_t s_tmem = tmem + lane_addr + t * kKeys;
  const uint32_t o_tmem = tmem + lane_addr + 256 + t * 128;
  const int rr = min(r, g.rows[t] - 1);   // rows past the end behave like the last one
  const int row = tile.row0 + t * kRows + rr;
  const int pos = g.ctx + row / p.qpk;
  // Scores are used as x = s * c with c >= 0: a negative scale flips the sign
  // of the raw scores once, so that the row max is always a max.
  const bool neg = p.score_scale_log2 < 0.f;
  const float c = neg ? -p.score_scale_log2 : p.score_scale_log2;
  float m = -INFINITY, l = 0.f;
  bool ok = true;
  for (int j = 0; j < n_t; ++j) {
    ok = __all_sync(0xffffffffu, mbar_wait(&bar.s_full[t], j & 1, abort, p.timeout_ns));
    if (!ok) break;
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
    const float rowsum = sum_lo + sum_hi;
    l = l * alpha + rowsum;
    m = m_use;
    // Rescale O in TMEM when some row of this warp moved its max.
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bar.o_done[t], (j - 1) & 1, abort, p.timeout_ns));
      if (!ok) break;
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
    // P (bf16) over the first 64 columns of this query tile's score columns.
#pragma unroll
    for (int ch = 0; ch < kKeys / 64; ++ch) {
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
      const int sv = j % VS;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar.vfull[sv], (j / VS) & 1, abort, p.timeout_ns));
      if (!ok) break;
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
    mbar_arrive(&bar.p_ready[t]);
  }
  if (ok)
    ok = __all_sync(0xffffffffu, mbar_wait(&bar.o_done[t], (n_t - 1) & 1, abort, p.timeout_ns));
  if (!ok) {
    give_up(p, abort);
    return;
  }
  tc_fence_after();
  // Epilogue: O / l -> bf16 row of the output.
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const bool row_ok = r < g.rows[t];
  const int tok = g.q_start + row / p.qpk;
  const int head = tile.kv_head * p.qpk + row % p.qpk;
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
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, const PrefillParams p) {
  using L = Smem<D>;
  constexpr int KS = L::kKStages, VS = L::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm + L::kQ;
  uint8_t* sK = sm + L::kK;
  uint8_t* sV = sm + L::kV;
  const Bars bar = bars_at<KS, VS>(reinterpret_cast<uint64_t*>(sm + L::kBar));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  volatile int32_t* abort = reinterpret_cast<volatile int32_t*>(sm + L::kMisc + 8);
  volatile int32_t* never = reinterpret_cast<volatile int32_t*>(sm + L::kMisc + 12);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const ua_tile tile = p.tiles[blockIdx.x];
  // Per-sequence values from the device arrays; ranges are clamped so that
  // disagreeing host/device lengths cannot send a read out of bounds.
  Geometry g;
  g.q_start = p.cu_query_lens[tile.seq];
  const int qlen = p.cu_query_lens[tile.seq + 1] - g.q_start;
  const int kv_len = p.kv_lens[tile.seq];
  g.ctx = kv_len - qlen;
  g.nrows = min(tile.nrows, qlen * p.qpk - tile.row0);
  g.kv_hi = min(min(tile.kv_hi, kv_len), p.max_blocks_per_seq * p.block_size);
  g.kv_lo = tile.kv_lo;
  g.nmax = 0;
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

  if (tid == 0) {
    *abort = 0;
    *never = 0;
    mbar_init(bar.q_full, 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(&bar.kfull[s], 1);
      mbar_init(&bar.kempty[s], 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&bar.vfull[s], 1);
      mbar_init(&bar.vempty[s], 1);
    }
    for (int t = 0; t < kTilesPerCta; ++t) {
      mbar_init(&bar.s_full[t], 1);
      mbar_init(&bar.p_ready[t], kRows);
      mbar_init(&bar.o_done[t], 1);
    }
    mbar_init(bar.mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    if (g.nmax > 0) {
      if (warp == 0 && lane == 0) {
        producer_role<D, false>(&map_q, &map_k, p, tile, g, sQ, sK, bar.kfull, bar.kempty, KS,
                                bar.q_full, abort, never);
      } else if (warp == 2 && lane == 0) {
        producer_role<D, true>(&map_q, &map_v, p, tile, g, sQ, sV, bar.vfull, bar.vempty, VS,
                               bar.q_full, abort, never);
      } else if (warp == 1 && lane == 0) {
        mma_role<D>(p, g, sQ, sK, sV, tmem, bar, abort, never);
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    if (g.nmax > 0) softmax_role<D>(p, tile, g, (warp - 4) / 4, sV, tmem, bar, abort, warp, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                     const PrefillParams& p, cudaStream_t stream) {
  // The register split above assumes the launch budget; refuse to launch a
  // build whose register count differs (the increase could never be granted).
  static int checked = 0;
  if (!checked) {
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, prefill_kernel<D>);
    if (e != cudaSuccess) return e;
    if (attr.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    checked = 1;
  }
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Smem<D>::kAlloc);
  if (e != cudaSuccess) return e;
  prefill_kernel<D><<<p.num_tiles, kThreads, Smem<D>::kAlloc, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

bool prefill_supported(int head_dim, int kv_dtype, int qpk, int block_size) {
  return (head_dim == 64 || head_dim == 128) && kv_dtype == UA_KV_BF16 && qpk >= 1 &&
         qpk <= kRows && kRows % qpk == 0 && block_size >= 16 &&
         (kKeys % block_size == 0 || block_size % kKeys == 0);
}

cudaError_t launch_prefill(const PrefillParams& p, const void* q, const void* k_cache,
                           const void* v_cache, int64_t total_q, int head_dim, int num_kv_heads,
                           cudaStream_t stream) {
  if (p.num_tiles <= 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  {
    // Q as [total_q][Hq][D]: a box of (64 dims, qpk heads, 128/qpk tokens)
    // lands as 128 packed rows (token-major, head-minor) in one panel.
    const uint64_t D = static_cast<uint64_t>(head_dim);
    uint64_t dims[3] = {D, static_cast<uint64_t>(p.num_q_heads), static_cast<uint64_t>(total_q)};
    uint64_t strides[2] = {D * 2, static_cast<uint64_t>(p.num_q_heads) * D * 2};
    uint32_t box[3] = {64, static_cast<uint32_t>(p.qpk), static_cast<uint32_t>(kRows / p.qpk)};
    cudaError_t e = encode_tiled_map(&mq, 2, 3, q, dims, strides, box, true, false);
    if (e != cudaSuccess) return e;
  }
  // K/V pages: (64 dims, one head, rows_per_box slots, one block) per box.
  cudaError_t e = encode_kv_page_map(&mk, k_cache, 2, head_dim, num_kv_heads, p.block_size,
                                     p.num_blocks, 64, p.rows_per_box, true);
  if (e == cudaSuccess)
    e = encode_kv_page_map(&mv, v_cache, 2, head_dim, num_kv_heads, p.block_size, p.num_blocks,
                           64, p.rows_per_box, true);
  if (e != cudaSuccess) return e;
  return head_dim == 128 ? launch_d<128>(mq, mk, mv, p, stream)
                         : launch_d<64>(mq, mk, mv, p, stream);
}

}  // namespace ua
