// Prefill kernel (K-P): tcgen05 / TMEM / TMA attention over 128-row tiles.
//
// Work unit: one ua_tile of 128 packed rows (128/qpk query tokens x the qpk
// query heads of one KV head, the packed GQA tile of
// "vllm_triton_unified_attention_notes") against its causal key prefix, in
// key tiles of 128. The loop is the FA2 forward of the "Fused Attention" notes
// (S = Q K^T, online softmax in base 2, O += P V, O / l at the end) laid out
// the Blackwell way, with the warp specialisation and producer/consumer
// overlap the notes describe for FlashAttention-3:
//   warp 0      TMA producer: Q once, then K and V pages of each key tile
//               (one box per page, resolved through the block table) into a
//               two-stage shared-memory ring;
//   warp 1      owns the tensor memory; one thread issues the MMAs:
//               S_j = Q K_j^T into one of two TMEM score buffers (so S_{j+1}
//               runs while the softmax works on S_j), then O += P_j V_j with
//               P_j read from TMEM;
//   warps 2-5   softmax, one query row per thread (TMEM lane): scale, mask,
//               running max / sum, P_j = 2^(x - m) written back over S_j as
//               bf16, O rescaled in TMEM only when the max grew by more than
//               2^8 (exact: the same stale max is used for P and l), then the
//               epilogue O / l -> bf16.
// Every mbarrier wait is bounded; a wait that gives up records
// UA_ERR_DEVICE_TIMEOUT, makes the other roles give up, drains the copies and
// MMAs in flight and frees the tensor memory before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "sm100.cuh"
#include "ua_device.cuh"
#include "ua_kernels.h"

namespace ua {
namespace {

using namespace sm100;

constexpr int kRows = 128;       // query rows per tile (TMEM lanes, MMA M)
constexpr int kKeys = 128;       // keys per key tile (MMA N of S, K of PV)
constexpr int kThreads = 192;    // 6 warps
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// K/V ring depth: as deep as 227 KB of shared memory allows.
template <int D>
constexpr int stages_for() { return D == 128 ? 3 : 4; }

template <int D>
struct Smem {
  static constexpr int kStages = stages_for<D>();
  static constexpr int kPanel = kRows * 128;           // one 64-wide bf16 panel: 16 KB
  static constexpr int kTile = kRows * D * 2;           // 128 x D bf16
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;
  static constexpr int kV = kK + kStages * kTile;
  static constexpr int kBar = kV + kStages * kTile;
  // barriers: q_full, kfull[S], vfull[S], kv_empty[S], s_full[2], p_ready[2], o_done, mma_done
  static constexpr int kNumBars = 1 + 3 * kStages + 2 + 2 + 2;
  static constexpr int kMisc = kBar + 8 * kNumBars;
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

struct Bars {
  uint64_t* q_full;
  uint64_t* kfull;
  uint64_t* vfull;
  uint64_t* kv_empty;
  uint64_t* s_full;
  uint64_t* p_ready;
  uint64_t* o_done;
  uint64_t* mma_done;
};

template <int kStages>
__device__ __forceinline__ Bars bars_at(uint64_t* b) {
  Bars r;
  r.q_full = b;
  r.kfull = b + 1;
  r.vfull = b + 1 + kStages;
  r.kv_empty = b + 1 + 2 * kStages;
  r.s_full = b + 1 + 3 * kStages;
  r.p_ready = r.s_full + 2;
  r.o_done = r.p_ready + 2;
  r.mma_done = r.o_done + 1;
  return r;
}

// Give up: record the error once and tell the other roles.
__device__ __forceinline__ void give_up(const PrefillParams& p, volatile int32_t* abort) {
  record_error(p.err, UA_ERR_DEVICE_TIMEOUT);
  *abort = 1;
}

// ------------------------------------------------------------------ producer
template <int D>
__device__ __forceinline__ void producer_role(const CUtensorMap* map_q, const CUtensorMap* map_k,
                                              const CUtensorMap* map_v, const PrefillParams& p,
                                              const ua_tile& tile, int q_start, int kv_lo,
                                              int kv_hi, int n_tiles, uint8_t* sQ, uint8_t* sK,
                                              uint8_t* sV, const Bars& bar,
                                              volatile int32_t* abort, volatile int32_t* never) {
  using L = Smem<D>;
  constexpr int kPanels = D / 64;
  constexpr int kStages = L::kStages;
  prefetch_tmap(map_q);
  prefetch_tmap(map_k);
  prefetch_tmap(map_v);
  const bool idle = (p.debug_flags & kDebugProducerIdle) != 0;
  int issued[kStages] = {};
  if (!idle) {
    mbar_arrive_expect_tx(bar.q_full, kRows * D * 2);
    for (int pn = 0; pn < kPanels; ++pn)
      tma_load_3d(sQ + pn * L::kPanel, map_q, bar.q_full, pn * 64, tile.kv_head * p.qpk,
                  q_start + tile.row0 / p.qpk);
    const int boxes = kKeys / p.rows_per_box;
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % kStages;
      if (j >= kStages &&
          !mbar_wait(&bar.kv_empty[s], ((j / kStages) - 1) & 1, abort, p.timeout_ns)) {
        give_up(p, abort);
        break;
      }
      const int base = kv_lo + j * kKeys;
      mbar_arrive_expect_tx(&bar.kfull[s], kKeys * D * 2);
      mbar_arrive_expect_tx(&bar.vfull[s], kKeys * D * 2);
      for (int b = 0; b < boxes; ++b) {
        const int key0 = base + b * p.rows_per_box;
        int32_t blk = static_cast<int32_t>(p.num_blocks);  // out of range: zero fill
        int32_t slot = 0;
        if (key0 < kv_hi) {
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
        for (int pn = 0; pn < kPanels; ++pn) {
          tma_load_4d(sK + s * L::kTile + pn * L::kPanel + row_off, map_k, &bar.kfull[s],
                      pn * 64, tile.kv_head, slot, blk);
          tma_load_4d(sV + s * L::kTile + pn * L::kPanel + row_off, map_v, &bar.vfull[s],
                      pn * 64, tile.kv_head, slot, blk);
        }
      }
      issued[s] = j / kStages + 1;
    }
  }
  // Drain: every load issued completes before the CTA may exit.
  for (int s = 0; s < kStages; ++s) {
    if (issued[s] > 0) {
      const uint32_t par = (issued[s] - 1) & 1;
      if (!mbar_wait(&bar.kfull[s], par, never, p.timeout_ns) ||
          !mbar_wait(&bar.vfull[s], par, never, p.timeout_ns))
        give_up(p, abort);
    }
  }
  if (!idle && !mbar_wait(bar.q_full, 0, never, p.timeout_ns)) give_up(p, abort);
}

// ------------------------------------------------------------------ MMA issuer
template <int D>
__device__ __forceinline__ void mma_role(const PrefillParams& p, int n_tiles, uint8_t* sQ,
                                         uint8_t* sK, uint8_t* sV, uint32_t tmem,
                                         const Bars& bar, volatile int32_t* abort,
                                         volatile int32_t* never) {
  using L = Smem<D>;
  constexpr int kStages = L::kStages;
  constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, kKeys, 0, 0);
  constexpr uint32_t idesc_o = idesc_bf16_f32(kRows, D, 0, 1);
  const uint32_t tmem_o = tmem + 256;
  const uint32_t q_addr = smem_u32(sQ);
  auto issue_s = [&](int j) {
    const int s = j % kStages;
    const uint32_t k_addr = smem_u32(sK + s * L::kTile);
    const uint32_t d_tmem = tmem + (j & 1) * kKeys;
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k / 4) * L::kPanel + (k % 4) * 32;
      mma_ss(d_tmem, smem_desc_sw128(q_addr + off, 16, 1024),
             smem_desc_sw128(k_addr + off, 16, 1024), idesc_s, k > 0 ? 1u : 0u);
    }
    mma_commit(&bar.s_full[j & 1]);
  };
  bool ok = mbar_wait(bar.q_full, 0, abort, p.timeout_ns) &&
            mbar_wait(&bar.kfull[0], 0, abort, p.timeout_ns);
  if (ok) {
    tc_fence_after();
    issue_s(0);
  }
  for (int j = 0; ok && j < n_tiles; ++j) {
    if (j + 1 < n_tiles) {
      const int s1 = (j + 1) % kStages;
      if (!mbar_wait(&bar.kfull[s1], ((j + 1) / kStages) & 1, abort, p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_s(j + 1);
    }
    const int s = j % kStages;
    if (!mbar_wait(&bar.p_ready[j & 1], (j >> 1) & 1, abort, p.timeout_ns) ||
        !mbar_wait(&bar.vfull[s], (j / kStages) & 1, abort, p.timeout_ns)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const uint32_t v_addr = smem_u32(sV + s * L::kTile);
    const uint32_t p_tmem = tmem + (j & 1) * kKeys;
#pragma unroll
    for (int k = 0; k < kKeys / 16; ++k)
      mma_ts(tmem_o, p_tmem + 8 * k, smem_desc_sw128(v_addr + k * 2048, L::kPanel, 1024),
             idesc_o, (j > 0 || k > 0) ? 1u : 0u);
    mma_commit(bar.o_done);
    mma_commit(&bar.kv_empty[s]);
  }
  if (!ok) give_up(p, abort);
  // Drain: every MMA issued has completed before the tensor memory is freed.
  mma_commit(bar.mma_done);
  if (!mbar_wait(bar.mma_done, 0, never, p.timeout_ns)) give_up(p, abort);
}

// ------------------------------------------------------------------ softmax
// One thread per query row r (TMEM lane r); warps 2..5 own lane quarters
// 2, 3, 0, 1 (a warp may only touch TMEM lanes 32 * (warp % 4) .. + 31).
template <int D>
__device__ __forceinline__ void softmax_role(const PrefillParams& p, const ua_tile& tile,
                                             int q_start, int ctx, int nrows, int kv_lo,
                                             int kv_hi, int n_tiles, uint8_t* sV, uint32_t tmem,
                                             const Bars& bar, volatile int32_t* abort, int warp,
                                             int lane) {
  using L = Smem<D>;
  constexpr int kPanels = D / 64;
  constexpr int kStages = L::kStages;
  const uint32_t tmem_o = tmem + 256;
  const int quarter = warp & 3;
  const int r = quarter * 32 + lane;
  const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
  const int rr = min(r, max(nrows - 1, 0));   // rows past the end behave like the last one
  const int pos = ctx + (tile.row0 + rr) / p.qpk;
  const float c = p.score_scale_log2;
  float m = -INFINITY, l = 0.f;
  bool ok = true;
  for (int j = 0; j < n_tiles; ++j) {
    ok = __all_sync(0xffffffffu, mbar_wait(&bar.s_full[j & 1], (j >> 1) & 1, abort, p.timeout_ns));
    if (!ok) break;
    tc_fence_after();
    const int base = kv_lo + j * kKeys;
    const uint32_t s_tmem = tmem + lane_addr + (j & 1) * kKeys;
    float x[kKeys];
    {
      uint32_t v[kKeys / 32][32];
#pragma unroll
      for (int ch = 0; ch < kKeys / 32; ++ch) tmem_ld32(s_tmem + ch * 32, v[ch]);
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < kKeys / 32; ++ch)
#pragma unroll
        for (int i = 0; i < 32; ++i) x[ch * 32 + i] = __uint_as_float(v[ch][i]) * c;
    }
    // Mask by select: keys past the range, past the row's position (causal)
    // or at or below pos - window.
    const int hi_col = min(kv_hi, p.causal ? pos + 1 : kv_hi) - base;
    const int lo_col = p.window > 0 ? pos - p.window + 1 - base : INT_MIN;
    if (hi_col < kKeys || lo_col > 0) {
#pragma unroll
      for (int i = 0; i < kKeys; ++i)
        if (i >= hi_col || i < lo_col) x[i] = -INFINITY;
    }
    // Row max with independent partial maxima (no 128-long dependency chain).
    constexpr int kAcc = 8;
    float mxp[kAcc];
#pragma unroll
    for (int a = 0; a < kAcc; ++a) mxp[a] = x[a];
#pragma unroll
    for (int i = kAcc; i < kKeys; ++i) mxp[i % kAcc] = fmaxf(mxp[i % kAcc], x[i]);
#pragma unroll
    for (int w = kAcc / 2; w > 0; w /= 2)
#pragma unroll
      for (int a = 0; a < w; ++a) mxp[a] = fmaxf(mxp[a], mxp[a + w]);
    const float mx = mxp[0];
    const float m_new = fmaxf(m, mx);
    const bool grow = (m == -INFINITY) || (m_new > m + kRescaleThreshold);
    const float m_use = grow ? m_new : m;
    const float alpha = grow ? ((m == -INFINITY) ? 0.f : ex2(m - m_use)) : 1.f;
    const float sub = (m_use == -INFINITY) ? 0.f : m_use;
    float sump[kAcc];
#pragma unroll
    for (int a = 0; a < kAcc; ++a) sump[a] = 0.f;
    uint32_t pk[kKeys / 2];
#pragma unroll
    for (int i = 0; i < kKeys / 2; ++i) {
      const float p0 = ex2(x[2 * i] - sub), p1 = ex2(x[2 * i + 1] - sub);
      sump[i % kAcc] += p0 + p1;
      pk[i] = pack2<false>(p0, p1);
    }
#pragma unroll
    for (int w = kAcc / 2; w > 0; w /= 2)
#pragma unroll
      for (int a = 0; a < w; ++a) sump[a] += sump[a + w];
    const float rowsum = sump[0];
    l = l * alpha + rowsum;
    m = m_use;
    // Rescale O in TMEM when some row of this warp moved its max.
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar.o_done, (j - 1) & 1, abort, p.timeout_ns));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(tmem_o + lane_addr + ch * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
        tmem_st32(tmem_o + lane_addr + ch * 32, v);
      }
    }
    // P (bf16) over the first 64 columns of this score buffer.
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
    const int valid = kv_hi - base;
    if (valid < kKeys) {
      const int s = j % kStages;
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&bar.vfull[s], (j / kStages) & 1, abort, p.timeout_ns));
      if (!ok) break;
      uint8_t* vt = sV + s * L::kTile;
      const int dead = kKeys - valid;
      for (int idx = r; idx < dead * kPanels * 8; idx += 128) {
        const int line = idx / 8, chunk = idx % 8;
        const int row = valid + line % dead;
        const int pn = line / dead;
        *reinterpret_cast<uint4*>(vt + pn * L::kPanel + row * 128 + chunk * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
    }
    tc_fence_before();
    mbar_arrive(&bar.p_ready[j & 1]);
  }
  if (ok)
    ok = __all_sync(0xffffffffu, mbar_wait(bar.o_done, (n_tiles - 1) & 1, abort, p.timeout_ns));
  if (!ok) {
    give_up(p, abort);
    return;
  }
  tc_fence_after();
  // Epilogue: O / l -> bf16 row of the output.
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const bool row_ok = r < nrows;
  const int tok = q_start + (tile.row0 + rr) / p.qpk;
  const int head = tile.kv_head * p.qpk + (tile.row0 + rr) % p.qpk;
  uint8_t* dst = reinterpret_cast<uint8_t*>(p.out) +
                 (static_cast<int64_t>(tok) * p.num_q_heads + head) * D * 2;
#pragma unroll
  for (int ch = 0; ch < D / 32; ++ch) {
    uint32_t v[32];
    tmem_ld32(tmem_o + lane_addr + ch * 32, v);
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
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm + L::kQ;
  uint8_t* sK = sm + L::kK;
  uint8_t* sV = sm + L::kV;
  constexpr int kStages = L::kStages;
  const Bars bar = bars_at<kStages>(reinterpret_cast<uint64_t*>(sm + L::kBar));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  volatile int32_t* abort = reinterpret_cast<volatile int32_t*>(sm + L::kMisc + 8);
  volatile int32_t* never = reinterpret_cast<volatile int32_t*>(sm + L::kMisc + 12);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const ua_tile tile = p.tiles[blockIdx.x];
  // Per-sequence values from the device arrays; ranges are clamped so that
  // disagreeing host/device lengths cannot send a read out of bounds.
  const int q_start = p.cu_query_lens[tile.seq];
  const int qlen = p.cu_query_lens[tile.seq + 1] - q_start;
  const int kv_len = p.kv_lens[tile.seq];
  const int ctx = kv_len - qlen;
  const int nrows = min(tile.nrows, qlen * p.qpk - tile.row0);
  const int kv_hi = min(min(tile.kv_hi, kv_len), p.max_blocks_per_seq * p.block_size);
  const int kv_lo = tile.kv_lo;
  const int n_tiles = (nrows > 0 && kv_hi > kv_lo) ? (kv_hi - kv_lo + kKeys - 1) / kKeys : 0;

  if (tid == 0) {
    *abort = 0;
    *never = 0;
    mbar_init(bar.q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar.kfull[s], 1);
      mbar_init(&bar.vfull[s], 1);
      mbar_init(&bar.kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar.s_full[b], 1);
      mbar_init(&bar.p_ready[b], 128);
    }
    mbar_init(bar.o_done, 1);
    mbar_init(bar.mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (n_tiles > 0) {
    if (warp == 0) {
      if (lane == 0)
        producer_role<D>(&map_q, &map_k, &map_v, p, tile, q_start, kv_lo, kv_hi, n_tiles, sQ,
                         sK, sV, bar, abort, never);
    } else if (warp == 1) {
      if (lane == 0) mma_role<D>(p, n_tiles, sQ, sK, sV, tmem, bar, abort, never);
    } else {
      softmax_role<D>(p, tile, q_start, ctx, nrows, kv_lo, kv_hi, n_tiles, sV, tmem, bar,
                      abort, warp, lane);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

template <int D>
cudaError_t launch_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                     const PrefillParams& p, cudaStream_t stream) {
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
  auto encode = encode_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t D = static_cast<cuuint64_t>(head_dim);
  CUtensorMap mq, mk, mv;
  {
    // Q as [total_q][Hq][D]: a box of (64 dims, qpk heads, 128/qpk tokens)
    // lands as 128 packed rows (token-major, head-minor) in one panel.
    cuuint64_t dims[3] = {D, static_cast<cuuint64_t>(p.num_q_heads),
                          static_cast<cuuint64_t>(total_q)};
    cuuint64_t strides[2] = {D * 2, static_cast<cuuint64_t>(p.num_q_heads) * D * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(p.qpk),
                         static_cast<cuuint32_t>(kRows / p.qpk)};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // K/V cache as [num_blocks][block_size][Hkv][D]: one box = (64 dims, one
    // head, rows_per_box slots, one block); an out-of-range block coordinate
    // reads zeros.
    cuuint64_t dims[4] = {D, static_cast<cuuint64_t>(num_kv_heads),
                          static_cast<cuuint64_t>(p.block_size),
                          static_cast<cuuint64_t>(p.num_blocks)};
    cuuint64_t strides[3] = {D * 2, static_cast<cuuint64_t>(num_kv_heads) * D * 2,
                             static_cast<cuuint64_t>(p.block_size) * num_kv_heads * D * 2};
    cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(p.rows_per_box), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    for (int which = 0; which < 2; ++which) {
      void* base = const_cast<void*>(which == 0 ? k_cache : v_cache);
      if (encode(which == 0 ? &mk : &mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims,
                 strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
          CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
  }
  return head_dim == 128 ? launch_d<128>(mq, mk, mv, p, stream)
                         : launch_d<64>(mq, mk, mv, p, stream);
}

}  // namespace ua
