// Staging kernel for prefill over an fp8 (e4m3) cache: widens the keys and
// values the prefill tiles will read from the paged e4m3 cache into a bf16
// staging cache of 128-slot pages, so that the tcgen05 prefill kernel (bf16
// operands) runs on it unchanged.
//
// The widening is exact and scale-free: an e4m3 code has 4 significant bits
// and an exponent within [-9, 8], so its value is a bf16 value; k_scale is
// folded into the score scale and v_scale into the output scale of the
// prefill launch, as for the oracle's dequantised values (code * scale).
// Conversion chain: e4m3x2 -> f16x2 (hardware, exact) -> f32 -> bf16x2
// (exact: no rounding happens for such values). NaN codes stay NaN.
//
// One CTA per staging page (the plan's stage tiles): 8 warps, one key row
// (all KV heads, contiguous in both caches) per warp at a time, 16-byte loads
// (four in flight per lane and cache) before the stores; source pages
// through the block table; rows past the sequence's length are not written
// (the prefill kernel masks those keys and zeroes those value rows).
// HBM-bound: per staged key Hkv * d bytes read per cache, twice that written.
#include <cstdint>
#include <cuda_fp16.h>

#include "planner.h"
#include "ua_device.cuh"
#include "ua_kernels.h"

namespace ua {

namespace {

constexpr int kStageWarps = 8;

// f16x2 -> bf16x2 (exact for widened e4m3 values), element order kept.
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h2) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
  uint32_t b2;
  // the first source operand lands in the upper half
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(b2) : "f"(f.y), "f"(f.x));
  return b2;
}

// Sixteen codes (16 bytes, lowest first) -> sixteen bf16 values (2 x 16 bytes).
__device__ __forceinline__ void widen16(uint4 c, uint4& lo, uint4& hi) {
  uint32_t h[8];
  e4m3x4_to_f16x2x2(c.x, h[0], h[1]);
  e4m3x4_to_f16x2x2(c.y, h[2], h[3]);
  e4m3x4_to_f16x2x2(c.z, h[4], h[5]);
  e4m3x4_to_f16x2x2(c.w, h[6], h[7]);
  lo = make_uint4(f16x2_to_bf16x2(h[0]), f16x2_to_bf16x2(h[1]), f16x2_to_bf16x2(h[2]),
                  f16x2_to_bf16x2(h[3]));
  hi = make_uint4(f16x2_to_bf16x2(h[4]), f16x2_to_bf16x2(h[5]), f16x2_to_bf16x2(h[6]),
                  f16x2_to_bf16x2(h[7]));
}

constexpr int kUnroll = 4;  // 16-byte loads per lane in flight per cache

__global__ void __launch_bounds__(kStageWarps * 32) stage_kernel(const StageParams p) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const ua_tile tile = p.tiles[blockIdx.x];
  const int chunks = p.row_elems / 16;  // 16 codes per load
  const int32_t* table = p.block_tables + static_cast<int64_t>(tile.seq) * p.max_blocks_per_seq;
  for (int t = tile.kv_lo + w; t < tile.kv_hi; t += kStageWarps) {
    if (t / p.block_size >= p.max_blocks_per_seq) break;
    const int32_t blk = table[t / p.block_size];
    if (blk < 0 || static_cast<int64_t>(blk) >= p.num_blocks) {
      if (lane == 0) record_error(p.err, UA_ERR_BOUNDS);
      continue;
    }
    const int64_t src_row = static_cast<int64_t>(blk) * p.block_size + t % p.block_size;
    const int64_t dst_row = static_cast<int64_t>(tile.row0) * kStagePage + (t - tile.kv_lo);
    const uint4* ks = reinterpret_cast<const uint4*>(p.k_src) + src_row * chunks;
    const uint4* vs = reinterpret_cast<const uint4*>(p.v_src) + src_row * chunks;
    uint4* kd = reinterpret_cast<uint4*>(p.k_dst) + dst_row * 2 * chunks;
    uint4* vd = reinterpret_cast<uint4*>(p.v_dst) + dst_row * 2 * chunks;
    for (int c0 = 0; c0 < chunks; c0 += 32 * kUnroll) {
      uint4 kc[kUnroll], vc[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < chunks) {
          kc[u] = ld_stream_v4(ks + c);
          vc[u] = ld_stream_v4(vs + c);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c >= chunks) continue;
        uint4 lo, hi;
        widen16(kc[u], lo, hi);
        kd[2 * c] = lo;
        kd[2 * c + 1] = hi;
        widen16(vc[u], lo, hi);
        vd[2 * c] = lo;
        vd[2 * c + 1] = hi;
      }
    }
  }
}

}  // namespace

cudaError_t launch_stage(const StageParams& p, cudaStream_t stream) {
  if (p.num_tiles <= 0) return cudaSuccess;
  if (p.row_elems % 16 != 0 || p.tiles == nullptr) return cudaErrorInvalidValue;
  stage_kernel<<<p.num_tiles, kStageWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ua
