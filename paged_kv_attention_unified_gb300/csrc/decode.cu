// Split-KV decode kernel (K-D): a bandwidth-bound pass over the paged cache.
//
// Work unit: one ua_tile = up to 8 packed (token, head) rows of one sequence
// and KV head (all query heads of a GQA group share one K/V stream, as in the
// packed Q tile of "vllm_triton_unified_attention_notes") over one key range
// [kv_lo, kv_hi) -- a whole range, or one split piece whose partial result is
// merged later by the log-sum-exp combine (FlashDecoding, "Fused Attention"
// notes; run_flash_splitkv_fwd in "flashatten takeaways EP2 工程").
//
// Design for sm_103a. Decode is HBM-bound (about 4-16 flop per cache byte).
// Each warp owns a ring of shared-memory stages; one lane issues, per 16-key
// step, one TMA box of K and one of V (the 16 slots of one KV head in one
// page) a few steps ahead of the math, and the warp reads the landed page
// into registers and keeps the math on the tensor pipe with m16n8k16 MMAs in
// a transposed orientation:
//   S^T[key, row]  = K[key, :] . Q[row, :]      (M = 16 keys, N = 8 rows)
//   O^T[d, row]   += V^T[d, key] . P^T[key, row] (M = 16 dims, N = 8 rows)
// Keys on M and the GQA rows on N waste no MMA rows when 8 query heads share
// a KV head. The score fragment becomes the PV operand with one movmatrix
// transpose per 8x8 block. Because the contraction index of both products
// and the M index of the second may be permuted freely, the kernel assigns
// keys and head dimensions to lanes so that the shared-memory fragment reads
// take the minimum number of wavefronts (4 lanes x 16 B of one K row, 8 lanes
// x 16 B of one V row, with the 128-byte swizzle of the staged page).
// Online softmax in base 2 ("Fused Attention" notes, _attn_fwd_inner): running
// max m, running sum l, rescale factor 2^(m_old - m_new). Optionally a unified
// max (FlashDecoding++, "Fused Attention" notes): a preset reference replaces
// the first step's max, with the running max as the fallback.
// Four warps per CTA take interleaved 16-key steps of the tile's range and
// merge their (m, l, O) through shared memory at the end. A split piece
// leaves its normalised partial and base-2 lse in the workspace; with arrival
// counters given, the last piece of a group to finish merges the group in the
// same launch (otherwise the combine kernel does).
#include "sm100.cuh"
#include "ua_device.cuh"
#include "planner.h"
#include "ua_kernels.h"

namespace ua {

namespace {

// Values per shared-memory load: as many as fill 16 bytes, else 8 or 4 bytes,
// dividing the n values a lane reads per row.
constexpr int load_vals(int n, int elt) {
  int v = 16 / elt;
  while (v * elt > 4 && n % v != 0) v /= 2;
  return v;
}

// Head dims: any multiple of 32 up to 256.
template <int D, bool FP8>
struct DecodeCfg {
  static_assert(D % 32 == 0 && D >= 32 && D <= 256, "head_dim");
  static constexpr int ELT = FP8 ? 1 : 2;                       // cache element bytes
  static constexpr int KVALS = D / 4;                           // K values per row per lane
  static constexpr int KE = load_vals(KVALS, ELT);              // K values per load
  static constexpr int KW = KVALS * ELT / 4;                    // ... as 32-bit words
  static constexpr int NKL = KVALS / KE;                        // K loads per row
  static constexpr int VVALS = D / 8;                           // V values per key per lane
  static constexpr int VE = load_vals(VVALS, ELT);              // V values per load
  static constexpr int VW = VVALS * ELT / 4;
  static constexpr int NVL = VVALS / VE;
  static constexpr int VLB = VE * ELT;                          // bytes per V load (16, 8 or 4)
  static constexpr int NC = D / 16;                             // MMA chunks along D
  static constexpr int QW = KVALS / 2;                          // Q words (16-bit pairs)
  static_assert(KVALS % KE == 0 && VVALS % VE == 0 && KE * ELT >= 4 && VLB >= 4, "loads");
};

// A load of B bytes (16, 8 or 4) from shared memory into consecutive words.
template <int B>
__device__ __forceinline__ void lds_words(uint32_t* w, const uint8_t* src, bool ok) {
  if constexpr (B == 16) {
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (ok) x = *reinterpret_cast<const uint4*>(src);
    w[0] = x.x;
    w[1] = x.y;
    w[2] = x.z;
    w[3] = x.w;
  } else if constexpr (B == 8) {
    uint2 x = make_uint2(0u, 0u);
    if (ok) x = *reinterpret_cast<const uint2*>(src);
    w[0] = x.x;
    w[1] = x.y;
  } else {
    w[0] = ok ? *reinterpret_cast<const uint32_t*>(src) : 0u;
  }
}

constexpr int kWarps = kDecodeWarps;
constexpr int kThreads = kWarps * 32;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// How far a unified-max reference may sit above a row's first max (log2
// units): P values down to 2^-64 times the largest are still normal bf16
// numbers, while f16 P (the e4m3 path) has no range to spare beyond what the
// running-max path already uses (largest P in [1, 2^8]).
template <bool FP8>
constexpr float kUnifiedAbove = FP8 ? 0.0f : 64.0f;

// Key slot (0..15) of a step held as MMA row m of S^T. Chosen so that the
// PV contraction slots 2t, 2t+1, 2t+8, 2t+9 of lane t are keys 4t..4t+3.
__device__ __forceinline__ int key_of_row(int m) {
  return (m < 8) ? ((m & 1) ? 2 * m - 1 : 2 * m) : ((m & 1) ? 2 * m - 15 : 2 * m - 14);
}

// Head-dimension index of K/Q value u (0..D/4-1) of lane t.
template <int D, bool FP8>
__device__ __forceinline__ int k_dim(int u, int t) {
  using C = DecodeCfg<D, FP8>;
  return (u / C::KE) * 4 * C::KE + t * C::KE + (u % C::KE);
}

// Head-dimension index of V value v (0..D/8-1) of lane group g.
template <int D, bool FP8>
__device__ __forceinline__ int v_dim(int v, int g) {
  using C = DecodeCfg<D, FP8>;
  return (v / C::VE) * 8 * C::VE + g * C::VE + (v % C::VE);
}

// Shared-memory layout of one 16-key page of K or V as TMA lands it. Rows of
// at least 128 bytes arrive as 128-byte-wide panels (16 rows each) with the
// 128-byte swizzle: the 16-byte chunk c of row r sits at chunk c ^ (r % 8).
// The fragment reads below touch 8 rows at one column (K) or 4 whole rows (V)
// per instruction; with the swizzle both take the minimum of 4 wavefronts
// (unswizzled, the 8 K rows at a 256-byte stride share half of the banks).
// The e4m3 path keeps plain rows: its K reads are half as many and its
// conversion work leaves no issue slots for the swizzled address arithmetic
// (measured: slower with the swizzle). So do bf16 rows that are not a whole
// number of 128-byte panels (head dims 32, 96, 160, 224).
template <int D, bool FP8>
struct PageLayout {
  static constexpr int kRowBytes = D * (FP8 ? 1 : 2);
  static constexpr bool kSwizzle = !FP8 && kRowBytes % 128 == 0;
  static constexpr int kBoxDims = kSwizzle ? 128 / (FP8 ? 1 : 2) : D;  // elements per box row
  static constexpr int kPanels = kSwizzle ? kRowBytes / 128 : 1;
  static constexpr int kPanelBytes = 16 * (kSwizzle ? 128 : kRowBytes);
  // Byte address of row `key`, byte `o` of the row (o a multiple of 8).
  __device__ static __forceinline__ int at(int key, int o) {
    if constexpr (kSwizzle) {
      const int within = o & 127;
      return (o >> 7) * kPanelBytes + key * 128 + ((((within >> 4) ^ (key & 7))) << 4) +
             (within & 15);
    } else {
      return key * kRowBytes + o;
    }
  }
};

template <int D, bool FP8>
struct StepRegs {
  uint32_t k[2][DecodeCfg<D, FP8>::KW];   // K rows key_of_row(g), key_of_row(g+8)
  uint32_t v[4][DecodeCfg<D, FP8>::VW];   // V rows 4t .. 4t+3
};

// Registers of one 16-key step from its shared-memory stage: kp / vp hold the
// step's K and V rows (16 rows of head_dim elements, as the TMA box lands).
// Keys at or beyond kv_hi read as zero (the page may hold anything there).
template <int D, bool FP8>
__device__ __forceinline__ void read_k(StepRegs<D, FP8>& r, const uint8_t* kp, int base,
                                       int kv_hi, int g, int t) {
  using C = DecodeCfg<D, FP8>;
  using PL = PageLayout<D, FP8>;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int key = key_of_row(g + 8 * h);
    const bool ok = base + key < kv_hi;
    constexpr int kB = C::KE * C::ELT;  // bytes per load
#pragma unroll
    for (int l = 0; l < C::NKL; ++l)
      lds_words<kB>(&r.k[h][l * (kB / 4)], kp + PL::at(key, (l * 4 * C::KE + t * C::KE) * C::ELT),
                    ok);
  }
}

template <int D, bool FP8>
__device__ __forceinline__ void read_v(StepRegs<D, FP8>& r, const uint8_t* vp, int base,
                                       int kv_hi, int g, int t) {
  using C = DecodeCfg<D, FP8>;
  using PL = PageLayout<D, FP8>;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int key = 4 * t + j;
    const bool ok = base + key < kv_hi;
#pragma unroll
    for (int l = 0; l < C::NVL; ++l)
      lds_words<C::VLB>(&r.v[j][l * (C::VLB / 4)],
                        vp + PL::at(key, (l * 8 * C::VE + g * C::VE) * C::ELT), ok);
  }
}

// Head dims above 128 read V only after the softmax, so that the K and V
// fragments of a step are never live together (register budget).
template <int D>
constexpr bool kLateV = D > 128;

// Per-warp online-softmax state for the two rows (columns n = 2t, 2t+1) a lane
// holds, plus its O^T accumulator fragments.
template <int D>
struct WarpState {
  float acc[D / 16][4];
  float m[2];
  float l[2];  // lane-partial sums; reduced over the 8 lane groups at the end
};

struct StepMask {
  int kv_hi;       // keys >= kv_hi are outside the range
  int hi_full;     // keys < hi_full are visible to every row (upper side)
  int lo_full;     // keys >= lo_full are visible to every row (lower side)
  int pos[2];      // query position of the lane's two rows
  int causal;
  int window;
  float phi2;      // unified max in log2 units of the scaled score; NaN: off
};

template <int D, bool FP8>
__device__ __forceinline__ void compute_step(WarpState<D>& st, StepRegs<D, FP8>& r,
                                             const uint8_t* vp, int kv_hi,
                                             const uint32_t (&qb)[D / 16][2], const float (&cc)[2],
                                             const StepMask& mk, int base, int g, int t) {
  using C = DecodeCfg<D, FP8>;
  // S^T = K Q^T for the 16 keys of this step, in two independent accumulation
  // chains (even and odd head-dim chunks) that are added at the end: half the
  // dependent MMA latency per step.
  float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int c = 0; c < C::NC; ++c) {
    uint32_t a[4];
    if constexpr (FP8) {
      e4m3x4_to_f16x2x2(r.k[0][c], a[0], a[2]);
      e4m3x4_to_f16x2x2(r.k[1][c], a[1], a[3]);
    } else {
      a[0] = r.k[0][2 * c];
      a[1] = r.k[1][2 * c];
      a[2] = r.k[0][2 * c + 1];
      a[3] = r.k[1][2 * c + 1];
    }
    mma16816<FP8>(s[c & 1], a, qb[c][0], qb[c][1]);
  }
  float x[4];
  x[0] = (s[0][0] + s[1][0]) * cc[0];
  x[1] = (s[0][1] + s[1][1]) * cc[1];
  x[2] = (s[0][2] + s[1][2]) * cc[0];
  x[3] = (s[0][3] + s[1][3]) * cc[1];
  // Masking (a select, so that nothing read from outside the visible set can
  // reach the result) only on steps that straddle a bound.
  if (base < mk.lo_full || base + 16 > mk.hi_full) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = base + key_of_row(g + 8 * (e >> 1));
      const int pos = mk.pos[e & 1];
      bool ok = key < mk.kv_hi;
      if (mk.causal) ok = ok && key <= pos;
      if (mk.window > 0) ok = ok && key > pos - mk.window;
      x[e] = ok ? x[e] : -INFINITY;
    }
  }
  // Row max over the 16 keys: the lane's two keys, then the 8 lane groups.
  float mx[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 4));
    mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 8));
    mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 16));
  }
  // The reference max moves only when the row max grew by more than 2^8
  // (log2 units 8): P and l use the same stale reference, so the result is
  // exact up to rounding, P stays below 2^8, and the O rescale (a multiply of
  // every accumulator) runs only on the rare steps where some row moved.
  // With a unified max phi2, a row's first visible step takes phi2 as its
  // reference when its max lies in [phi2 - kUnifiedAbove, phi2 + 8]; outside
  // that range (overflow or underflow risk) it falls back to its own max, and
  // later steps move the reference up as above.
  float p[4], alpha[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const bool first = st.m[j] == -INFINITY;
    const float m_new = fmaxf(st.m[j], mx[j]);
    const bool grow = first || (m_new > st.m[j] + kRescaleThreshold);
    float m_use = grow ? m_new : st.m[j];
    if (first && mx[j] <= mk.phi2 + kRescaleThreshold && mx[j] >= mk.phi2 - kUnifiedAbove<FP8>)
      m_use = mk.phi2;
    // Rows with nothing visible yet keep m = -inf; subtract 0 instead so that
    // no -inf - -inf appears.
    const float sub = (m_use == -INFINITY) ? 0.f : m_use;
    alpha[j] = grow ? ex2(st.m[j] - sub) : 1.f;
    p[j] = ex2(x[j] - sub);
    p[j + 2] = ex2(x[j + 2] - sub);
    st.l[j] = st.l[j] * alpha[j] + p[j] + p[j + 2];
    st.m[j] = m_use;
  }
  if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
    for (int c = 0; c < C::NC; ++c) {
      st.acc[c][0] *= alpha[0];
      st.acc[c][2] *= alpha[0];
      st.acc[c][1] *= alpha[1];
      st.acc[c][3] *= alpha[1];
    }
  }
  if constexpr (kLateV<D>) read_v<D, FP8>(r, vp, base, kv_hi, g, t);
  // P^T as the B operand of the PV product: transpose the two 8x8 blocks.
  const uint32_t pb0 = movmatrix_trans(pack2<FP8>(p[0], p[1]));
  const uint32_t pb1 = movmatrix_trans(pack2<FP8>(p[2], p[3]));
  // O^T += V^T P^T.
#pragma unroll
  for (int c = 0; c < C::NC; ++c) {
    uint32_t a[4];
    if constexpr (FP8) {
      const uint32_t sel = (c & 1) ? 0x7362u : 0x5140u;
      const uint32_t lo = __byte_perm(r.v[0][c >> 1], r.v[1][c >> 1], sel);
      const uint32_t hi = __byte_perm(r.v[2][c >> 1], r.v[3][c >> 1], sel);
      e4m3x4_to_f16x2x2(lo, a[0], a[1]);
      e4m3x4_to_f16x2x2(hi, a[2], a[3]);
    } else {
      a[0] = __byte_perm(r.v[0][c], r.v[1][c], 0x5410u);
      a[1] = __byte_perm(r.v[0][c], r.v[1][c], 0x7632u);
      a[2] = __byte_perm(r.v[2][c], r.v[3][c], 0x5410u);
      a[3] = __byte_perm(r.v[2][c], r.v[3][c], 0x7632u);
    }
    mma16816<FP8>(st.acc[c], a, pb0, pb1);
  }
}

// Shared memory of one CTA: a ring of R stages per warp, each holding the K
// and V rows (16 x head_dim, in the page layout above) of one 16-key step as
// TMA lands them; then one mbarrier per stage. After the loop the ring is
// reused for the cross-warp merge. The sizes come from the scheduler's copy of
// the decode geometry, which also sizes splits by the CTAs an SM holds.
template <int D, bool FP8>
struct Ring {
  static constexpr int kElt = FP8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElt;
  static constexpr int kStage = decode_stage_bytes(D, kElt);
  static constexpr int kStages = decode_ring_stages(D, kElt);
  static constexpr int kRing = kWarps * kStages * kStage;
  static constexpr int kBars = kRing;
  static constexpr int kMisc = kBars + 8 * kWarps * kStages;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment (swizzle atoms)
  static constexpr int kCtasPerSm = decode_ctas_per_sm(D, kElt);
  static_assert(kAlloc == decode_smem_bytes(D, kElt), "decode shared memory");
  static_assert(kWarps * UA_DECODE_ROWS * (D + 2) * 4 <= kRing, "merge buffers alias the ring");
};

template <int D, bool FP8>
__global__ void __launch_bounds__(kThreads, Ring<D, FP8>::kCtasPerSm)
    decode_kernel(const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const KernelParams p) {
  using C = DecodeCfg<D, FP8>;
  using RC = Ring<D, FP8>;
  constexpr int R = RC::kStages;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(dsm + RC::kBars);
  volatile int32_t* never = reinterpret_cast<volatile int32_t*>(dsm + RC::kMisc);
  // merge buffers (valid only after the loop; they alias the ring)
  float (*red_acc)[UA_DECODE_ROWS][D] = reinterpret_cast<float (*)[UA_DECODE_ROWS][D]>(dsm);
  float (*red_m)[UA_DECODE_ROWS] =
      reinterpret_cast<float (*)[UA_DECODE_ROWS]>(dsm + kWarps * UA_DECODE_ROWS * D * 4);
  float (*red_l)[UA_DECODE_ROWS] = red_m + kWarps;

  const ua_tile tile = p.tiles[blockIdx.x];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  if (threadIdx.x == 0 && p.span_start != nullptr) atomicMin(p.span_start, sm100::globaltimer_ns());
  auto stamp_end = [&]() {
    if (threadIdx.x == 0 && p.span_end != nullptr) atomicMax(p.span_end, sm100::globaltimer_ns());
  };
  if (threadIdx.x == 0) {
    *never = 0;
    for (int i = 0; i < kWarps * R; ++i) sm100::mbar_init(&bars[i], 1);
    sm100::fence_mbar_init();
  }
  __syncthreads();

  // Per-sequence values from the device arrays; every range is clamped so
  // that disagreeing host/device lengths cannot send a read out of bounds.
  const int q_start = p.cu_query_lens[tile.seq];
  const int qlen = p.cu_query_lens[tile.seq + 1] - q_start;
  const int kv_len = p.kv_lens[tile.seq];
  const int ctx = kv_len - qlen;
  const int nrows = min(tile.nrows, qlen * p.qpk - tile.row0);
  const int kv_hi = min(min(tile.kv_hi, kv_len), p.max_blocks_per_seq * p.block_size);
  const int kv_lo = tile.kv_lo;

  // ---- Q fragments (B operand of S^T = K Q^T): row n = g of the tile.
  uint32_t qb[C::NC][2];
  float cc[2];
  {
    uint32_t qw[C::QW];
    const bool row_ok = g < nrows;
    const int r = tile.row0 + (row_ok ? g : 0);
    const int tok = q_start + r / p.qpk;
    const int head = tile.kv_head * p.qpk + r % p.qpk;
    const uint8_t* qrow = reinterpret_cast<const uint8_t*>(p.q) +
                          (static_cast<int64_t>(tok) * p.num_q_heads + head) * D * 2;
#pragma unroll
    for (int l = 0; l < C::NKL; ++l) {
#pragma unroll
      for (int h = 0; h < C::KE / 8; ++h) {
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (row_ok) x = *reinterpret_cast<const uint4*>(qrow + (l * 4 * C::KE + t * C::KE + 8 * h) * 2);
        const int w = l * (C::KE / 2) + 4 * h;
        qw[w + 0] = x.x;
        qw[w + 1] = x.y;
        qw[w + 2] = x.z;
        qw[w + 3] = x.w;
      }
    }
    if constexpr (FP8) {
      // f16 operands for the e4m3 path: scale each Q row by a power of two so
      // that its largest magnitude lies in [2^14, 2^15); exact for every
      // element within 2^-29 of the row maximum. The factor is undone in the
      // per-row score multiplier.
      float amax = 0.f;
#pragma unroll
      for (int w = 0; w < C::QW; ++w) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qw[w]));
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      int e = 0;
      if (amax > 0.f && amax < INFINITY) {
        int E;
        frexpf(amax, &E);
        e = min(max(15 - E, -126), 126);
      }
      const float up = __int_as_float((127 + e) << 23);
      const float down = __int_as_float((127 - e) << 23);
#pragma unroll
      for (int w = 0; w < C::QW; ++w) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qw[w]));
        qw[w] = pack2<true>(f.x * up, f.y * up);
      }
      const float row_mult = p.score_scale_log2 * down;
      cc[0] = __shfl_sync(0xffffffffu, row_mult, 4 * (2 * t));
      cc[1] = __shfl_sync(0xffffffffu, row_mult, 4 * (2 * t + 1));
    } else {
      cc[0] = cc[1] = p.score_scale_log2;
    }
#pragma unroll
    for (int c = 0; c < C::NC; ++c) {
      qb[c][0] = qw[2 * c];
      qb[c][1] = qw[2 * c + 1];
    }
  }

  // ---- Visibility of the lane's two rows (columns n = 2t, 2t+1).
  StepMask mk;
  mk.kv_hi = kv_hi;
  mk.causal = p.causal;
  mk.window = p.window;
  mk.phi2 = p.unified_max_on ? p.unified_max_log2 : __int_as_float(0x7fc00000);
  {
    const int last = max(nrows - 1, 0);
    const int min_pos = ctx + tile.row0 / p.qpk;
    const int max_pos = ctx + (tile.row0 + last) / p.qpk;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int n = 2 * t + j;
      mk.pos[j] = (n < nrows) ? ctx + (tile.row0 + n) / p.qpk : max_pos;
    }
    mk.hi_full = p.causal ? min(kv_hi, min_pos + 1) : kv_hi;
    mk.lo_full = p.window > 0 ? max_pos - p.window + 1 : INT_MIN;
  }

  WarpState<D> st_state;
#pragma unroll
  for (int c = 0; c < C::NC; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) st_state.acc[c][e] = 0.f;
  st_state.m[0] = st_state.m[1] = -INFINITY;
  st_state.l[0] = st_state.l[1] = 0.f;

  // ---- Stream the key range: warp w takes steps w, w+4, w+8, ...; each step
  // is one TMA box of K and one of V (16 keys of one page) into the warp's ring.
  const int nsteps = kv_hi > kv_lo ? (kv_hi - kv_lo + 15) / 16 : 0;
  const int my_n = nsteps > warp ? (nsteps - warp + kWarps - 1) / kWarps : 0;
  auto step_base = [&](int k) { return kv_lo + 16 * (warp + kWarps * k); };
  uint8_t* ring = dsm + warp * R * RC::kStage;
  uint64_t* wbar = bars + warp * R;
  // Page ids, 32 steps at a time: lane l holds the page of step 32c + l.
  int32_t ids = -1;
  auto refill_ids = [&](int c) {
    const int k = 32 * c + lane;
    ids = k < my_n ? p.block_tables[static_cast<int64_t>(tile.seq) * p.max_blocks_per_seq +
                                    step_base(k) / p.block_size]
                   : -1;
  };
  // Whole-warp call: every lane takes part in the shuffle, lane 0 issues.
  auto issue = [&](int k) {
    const int32_t id = __shfl_sync(0xffffffffu, ids, k & 31);
    if (lane == 0) {
      const int base = step_base(k);
      int32_t blk = static_cast<int32_t>(p.num_blocks);  // out of range: TMA fills zeros
      if (id >= 0 && static_cast<int64_t>(id) < p.num_blocks) blk = id;
      else record_error(p.err, UA_ERR_BOUNDS);
      const int st = k % R;
      uint8_t* stage = ring + st * RC::kStage;
      sm100::fence_proxy_async_smem();
      sm100::mbar_arrive_expect_tx(&wbar[st], RC::kStage);
      using PL = PageLayout<D, FP8>;
#pragma unroll
      for (int pn = 0; pn < PL::kPanels; ++pn) {
        sm100::tma_load_4d(stage + pn * PL::kPanelBytes, &map_k, &wbar[st], pn * PL::kBoxDims,
                           tile.kv_head, base % p.block_size, blk);
        sm100::tma_load_4d(stage + 16 * RC::kRowBytes + pn * PL::kPanelBytes, &map_v, &wbar[st],
                           pn * PL::kBoxDims, tile.kv_head, base % p.block_size, blk);
      }
    }
  };
  int issued = 0, done = 0;
  if (my_n > 0) {
    refill_ids(0);
    for (; issued < my_n && issued < R; ++issued) issue(issued);
    StepRegs<D, FP8> r;
    for (; done < my_n; ++done) {
      const int st = done % R;
      const bool ok = __all_sync(0xffffffffu, sm100::mbar_wait(&wbar[st], (done / R) & 1, never,
                                                                p.timeout_ns));
      if (!ok) {
        record_error(p.err, UA_ERR_DEVICE_TIMEOUT);
        break;
      }
      const uint8_t* stage = ring + st * RC::kStage;
      const uint8_t* vstage = stage + 16 * RC::kRowBytes;
      read_k<D, FP8>(r, stage, step_base(done), kv_hi, g, t);
      if constexpr (!kLateV<D>) read_v<D, FP8>(r, vstage, step_base(done), kv_hi, g, t);
      compute_step<D, FP8>(st_state, r, vstage, kv_hi, qb, cc, mk, step_base(done), g, t);
      __syncwarp();  // every lane has consumed the stage: it may be refilled
      if (issued < my_n) {
        if ((issued & 31) == 0) refill_ids(issued >> 5);
        issue(issued);
        ++issued;
      }
    }
    // Copies still in flight (only after a timeout) complete before exit.
    if (lane == 0)
      for (int k = done; k < issued; ++k)
        sm100::mbar_wait(&wbar[k % R], (k / R) & 1, never, p.timeout_ns);
    __syncwarp();
  }
  __syncthreads();  // the ring is reused for the merge below

  // ---- Merge the four warps.
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    st_state.l[j] += __shfl_xor_sync(0xffffffffu, st_state.l[j], 4);
    st_state.l[j] += __shfl_xor_sync(0xffffffffu, st_state.l[j], 8);
    st_state.l[j] += __shfl_xor_sync(0xffffffffu, st_state.l[j], 16);
  }
  if (g == 0) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      red_m[warp][2 * t + j] = st_state.m[j];
      red_l[warp][2 * t + j] = st_state.l[j];
    }
  }
#pragma unroll
  for (int c = 0; c < C::NC; ++c) {
    const int d0 = v_dim<D, FP8>(2 * c, g);
    red_acc[warp][2 * t][d0] = st_state.acc[c][0];
    red_acc[warp][2 * t + 1][d0] = st_state.acc[c][1];
    red_acc[warp][2 * t][d0 + 1] = st_state.acc[c][2];
    red_acc[warp][2 * t + 1][d0 + 1] = st_state.acc[c][3];
  }
  __syncthreads();

  constexpr int kSeg = D / 16;  // dims per thread in the epilogue
  const int n = threadIdx.x / 16;
  const int d0 = (threadIdx.x % 16) * kSeg;
  const bool row_ok = n < nrows;
  float M = -INFINITY, L = 0.f;
  float o[kSeg];
#pragma unroll
  for (int e = 0; e < kSeg; ++e) o[e] = 0.f;
  if (row_ok) {
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w][n]);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = red_m[w][n];
      const float f = (mw == -INFINITY) ? 0.f : ex2(mw - M);
      L += f * red_l[w][n];
#pragma unroll
      for (int e = 0; e < kSeg; ++e) o[e] += f * red_acc[w][n][d0 + e];
    }
  }
  // bf16 output row n of this tile, scaled by `mult`.
  auto store_out = [&](const float* vals, float mult) {
    const int r = tile.row0 + n;
    const int tok = q_start + r / p.qpk;
    const int head = tile.kv_head * p.qpk + r % p.qpk;
    uint32_t packed[kSeg / 2];
#pragma unroll
    for (int e = 0; e < kSeg / 2; ++e)
      packed[e] = pack2<false>(vals[2 * e] * mult, vals[2 * e + 1] * mult);
    uint8_t* dst = reinterpret_cast<uint8_t*>(p.out) +
                   ((static_cast<int64_t>(tok) * p.num_q_heads + head) * D + d0) * 2;
    if constexpr (kSeg % 8 == 0) {
#pragma unroll
      for (int i = 0; i < kSeg / 8; ++i)
        *reinterpret_cast<uint4*>(dst + 16 * i) =
            make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
    } else if constexpr (kSeg % 4 == 0) {
#pragma unroll
      for (int i = 0; i < kSeg / 4; ++i)
        *reinterpret_cast<uint2*>(dst + 8 * i) = make_uint2(packed[2 * i], packed[2 * i + 1]);
    } else {
#pragma unroll
      for (int i = 0; i < kSeg / 2; ++i) *reinterpret_cast<uint32_t*>(dst + 4 * i) = packed[i];
    }
  };
  const float inv = L > 0.f ? p.v_scale / L : 0.f;
  if (tile.slot < 0) {
    if (row_ok) store_out(o, inv);
    stamp_end();
    return;
  }
  // Split piece: normalised partial row and its base-2 log-sum-exp.
  if (row_ok) {
    float* wo = p.ws_o + (static_cast<int64_t>(tile.slot) * UA_DECODE_ROWS + n) * D + d0;
    if constexpr (kSeg % 4 == 0) {
#pragma unroll
      for (int e = 0; e < kSeg; e += 4)
        *reinterpret_cast<float4*>(wo + e) =
            make_float4(o[e] * inv, o[e + 1] * inv, o[e + 2] * inv, o[e + 3] * inv);
    } else {
#pragma unroll
      for (int e = 0; e < kSeg; e += 2)
        *reinterpret_cast<float2*>(wo + e) = make_float2(o[e] * inv, o[e + 1] * inv);
    }
    if (threadIdx.x % 16 == 0)
      p.ws_lse[static_cast<int64_t>(tile.slot) * UA_DECODE_ROWS + n] =
          L > 0.f ? M + log2f(L) : -INFINITY;
  }
  if (p.split_counters == nullptr) {  // a separate combine kernel merges the pieces
    stamp_end();
    return;
  }
  // Fused combine: the last piece of a group to finish merges all of them
  // (weights 2^(lse_s - lse*)), then re-arms the group's counter for the next call.
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int ns = p.groups[tile.group].nsplits;
    s_last = atomicAdd(&p.split_counters[tile.group], 1) == ns - 1;
  }
  __syncthreads();
  if (!s_last) {
    stamp_end();
    return;
  }
  __threadfence();
  const ua_combine_group grp = p.groups[tile.group];
  if (row_ok) {
    const float* lse = p.ws_lse + static_cast<int64_t>(grp.slot0) * UA_DECODE_ROWS + n;
    float Mx = -INFINITY;
    for (int sp = 0; sp < grp.nsplits; ++sp) Mx = fmaxf(Mx, __ldcg(lse + sp * UA_DECODE_ROWS));
    float W = 0.f;
    float acc[kSeg];
#pragma unroll
    for (int e = 0; e < kSeg; ++e) acc[e] = 0.f;
    for (int sp = 0; sp < grp.nsplits; ++sp) {
      const float l = __ldcg(lse + sp * UA_DECODE_ROWS);
      if (l == -INFINITY) continue;
      const float w = ex2(l - Mx);
      W += w;
      const float* src =
          p.ws_o + ((static_cast<int64_t>(grp.slot0) + sp) * UA_DECODE_ROWS + n) * D + d0;
      if constexpr (kSeg % 4 == 0) {
#pragma unroll
        for (int e = 0; e < kSeg; e += 4) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(src + e));
          acc[e] += w * v.x;
          acc[e + 1] += w * v.y;
          acc[e + 2] += w * v.z;
          acc[e + 3] += w * v.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < kSeg; e += 2) {
          const float2 v = __ldcg(reinterpret_cast<const float2*>(src + e));
          acc[e] += w * v.x;
          acc[e + 1] += w * v.y;
        }
      }
    }
    store_out(acc, W > 0.f ? 1.f / W : 0.f);
  }
  if (threadIdx.x == 0) p.split_counters[tile.group] = 0;
  stamp_end();
}

template <int D, bool FP8>
cudaError_t launch_decode_d(const KernelParams& p, cudaStream_t stream, bool after_prefill) {
  CUtensorMap mk, mv;
  const int elt = FP8 ? 1 : 2;
  using PL = PageLayout<D, FP8>;
  // one box = the 16 key rows of one KV head in one page, one 128-byte panel
  // of head dims (swizzled) or the whole row
  cudaError_t e = encode_kv_page_map(&mk, p.k_cache, elt, D, p.num_kv_heads, p.block_size,
                                     p.num_blocks, PL::kBoxDims, 16, PL::kSwizzle);
  if (e == cudaSuccess)
    e = encode_kv_page_map(&mv, p.v_cache, elt, D, p.num_kv_heads, p.block_size, p.num_blocks,
                           PL::kBoxDims, 16, PL::kSwizzle);
  if (e != cudaSuccess) return e;
  static std::atomic<uint64_t> smem_set{0};
  e = set_smem_once(decode_kernel<D, FP8>, Ring<D, FP8>::kAlloc, smem_set);
  if (e != cudaSuccess) return e;
  if (!after_prefill) {
    decode_kernel<D, FP8><<<p.num_tiles, kThreads, Ring<D, FP8>::kAlloc, stream>>>(mk, mv, p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.num_tiles));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Ring<D, FP8>::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<D, FP8>, mk, mv, p);
}

}  // namespace

cudaError_t launch_decode(const KernelParams& p, int head_dim, int kv_dtype, cudaStream_t stream,
                          bool after_prefill) {
  if (p.num_tiles <= 0) return cudaSuccess;
  const bool a = after_prefill;
  const bool f8 = kv_dtype != UA_KV_BF16;
  switch (head_dim) {
    case 32: return f8 ? launch_decode_d<32, true>(p, stream, a) : launch_decode_d<32, false>(p, stream, a);
    case 64: return f8 ? launch_decode_d<64, true>(p, stream, a) : launch_decode_d<64, false>(p, stream, a);
    case 96: return f8 ? launch_decode_d<96, true>(p, stream, a) : launch_decode_d<96, false>(p, stream, a);
    case 128: return f8 ? launch_decode_d<128, true>(p, stream, a) : launch_decode_d<128, false>(p, stream, a);
    case 160: return f8 ? launch_decode_d<160, true>(p, stream, a) : launch_decode_d<160, false>(p, stream, a);
    case 192: return f8 ? launch_decode_d<192, true>(p, stream, a) : launch_decode_d<192, false>(p, stream, a);
    case 224: return f8 ? launch_decode_d<224, true>(p, stream, a) : launch_decode_d<224, false>(p, stream, a);
    case 256: return f8 ? launch_decode_d<256, true>(p, stream, a) : launch_decode_d<256, false>(p, stream, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ua
