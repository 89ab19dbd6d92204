// Device-side helpers shared by the unified paged-KV attention kernels.
#pragma once

#include <climits>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "../../include/ua.h"

namespace ua {

// log2(e): softmax is evaluated as 2^(x*log2e - m) ("Fused Attention" notes,
// _attn_fwd: qk_scale = sm_scale * 1/log(2)).
constexpr float kLog2e = 1.4426950408889634f;

struct KernelParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  void* out;
  const int32_t* cu_query_lens;
  const int32_t* kv_lens;
  const int32_t* block_tables;
  const ua_tile* tiles;
  int32_t num_tiles;
  float* ws_o;       // [slots][UA_DECODE_ROWS][head_dim]
  float* ws_lse;     // [slots][UA_DECODE_ROWS], base-2 log-sum-exp
  int32_t* err;      // device error word
  int64_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t block_size;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t qpk;
  int32_t causal;
  int32_t window;
  float score_scale_log2;  // scale * log2(e) (* k_scale for fp8)
  float v_scale;           // 1 for bf16
  // Fused split combine: per-group arrival counters (zero between calls) and
  // the groups; null counters leave the merge to the combine kernel.
  int32_t* split_counters;
  const ua_combine_group* groups;
  uint64_t timeout_ns;  // bound of every device-side wait
  // Unified max (FlashDecoding++): when on, the preset reference of every
  // decode row, in log2 units of the scaled score (phi * log2(e)).
  int32_t unified_max_on;
  float unified_max_log2;
  // Kernel timing (null: off): first CTA start (atomicMin) and last CTA end
  // (atomicMax) on the device global timer, in ns.
  unsigned long long* span_start;
  unsigned long long* span_end;
};

struct CombineParams {
  const ua_combine_group* groups;
  int32_t num_groups;
  const float* ws_o;
  const float* ws_lse;
  const int32_t* cu_query_lens;
  void* out;
  int32_t num_q_heads;
  int32_t qpk;
};

// ----------------------------------------------------------------------------
// Small PTX wrappers
// ----------------------------------------------------------------------------

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Streaming 16-byte / 8-byte loads of cache data: read-only, not kept in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(r.x), "=r"(r.y)
               : "l"(p));
  return r;
}

// D(16x8, f32) += A(16x16, row) * B(16x8, col), bf16 or f16 inputs.
template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (F16) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// Transpose an 8x8 matrix of 16-bit elements held one row-pair per thread.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (F16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// Four binary32 values -> four e4m3 codes (x0 in the lowest byte), rounded
// to nearest even and saturating.
__device__ __forceinline__ uint32_t to_e4m3x4(float x0, float x1, float x2, float x3) {
  uint16_t lo, hi;
  // the first source operand lands in the upper byte of the pair
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// The two bf16 values of a 32-bit word as binary32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two e4m3 codes in the low 16 bits -> f16x2 (low byte -> low half). Exact:
// every e4m3 value is an f16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
      static_cast<__nv_fp8x2_storage_t>(two_codes & 0xFFFFu), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

// Four e4m3 codes in one word -> two f16x2 words (bytes 0,1 -> lo; bytes 2,3
// -> hi; low byte -> low half). Two conversions, no repacking.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t codes, uint32_t& lo, uint32_t& hi) {
  asm("{\n"
      ".reg .b16 l16, h16;\n"
      "mov.b32 {l16, h16}, %2;\n"
      "cvt.rn.f16x2.e4m3x2 %0, l16;\n"
      "cvt.rn.f16x2.e4m3x2 %1, h16;\n"
      "}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(codes));
}

__device__ __forceinline__ void record_error(int32_t* err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

// Physical page of logical key position t of sequence seq, or -1 when the
// page id read from the block table lies outside [0, num_blocks) (recorded
// as UA_ERR_BOUNDS; the caller then reads nothing from that page).
__device__ __forceinline__ int64_t page_of(const KernelParams& p, int seq, int t) {
  const int32_t id =
      p.block_tables[static_cast<int64_t>(seq) * p.max_blocks_per_seq + t / p.block_size];
  if (id < 0 || static_cast<int64_t>(id) >= p.num_blocks) {
    record_error(p.err, UA_ERR_BOUNDS);
    return -1;
  }
  return id;
}

// Element offset of K/V[page, slot, kv_head, 0] in the paged cache.
__device__ __forceinline__ int64_t kv_row_offset(const KernelParams& p, int64_t page, int slot,
                                                 int kv_head, int head_dim) {
  return ((page * p.block_size + slot) * p.num_kv_heads + kv_head) *
         static_cast<int64_t>(head_dim);
}

}  // namespace ua
