// Append-KV kernel: writes a step's new keys and values into the paged cache
// before attention reads it (the Append_KV path of the split-KV launcher in
// "flashatten takeaways EP2 工程"; the paged layout and the quantisation path
// of "vllm_triton_unified_attention_notes").
//
// For sequence s and new token i < q_len_s (row cu_query_lens[s] + i of
// k_new / v_new), logical position pos = kv_len_s - q_len_s + i goes to block
// block_tables[s][pos / block_size], slot pos % block_size. One (block, slot)
// holds all KV heads of a token contiguously, and so does one row of k_new, so
// a token is one contiguous copy of num_kv_heads * head_dim elements.
// The host plan cuts every sequence's new tokens into tiles of up to 8 (its
// sequence, first row and first position precomputed, so no search over the
// query offsets runs on the device): one CTA per tile, one warp per token;
// a warp issues all of its row's 16-byte loads before its stores.
// fp8 cache: code = e4m3(x / scale) with the quotient in binary32 (IEEE
// division, round to nearest) and the hardware conversion rounding to nearest
// even with saturation at +-448.
// HBM-bound: per token 2 * Hkv * d * 2 bytes read, 2 * Hkv * d * elt written.
#include <cstdint>

#include "planner.h"
#include "ua_device.cuh"
#include "ua_kernels.h"

namespace ua {

namespace {

constexpr int kWarpsPerCta = 8;   // tokens per append tile (one warp each)
constexpr int kUnroll = 4;        // 16-byte chunks per lane in flight (rows up to 4 KB of bf16)
static_assert(kWarpsPerCta == kAppendTokens, "one warp per token of an append tile");

// Eight bf16 values (one 16-byte chunk) / scale -> eight e4m3 codes.
__device__ __forceinline__ uint2 quantize8(uint4 w, float scale) {
  const float a0 = __fdiv_rn(bf16_lo(w.x), scale), a1 = __fdiv_rn(bf16_hi(w.x), scale);
  const float a2 = __fdiv_rn(bf16_lo(w.y), scale), a3 = __fdiv_rn(bf16_hi(w.y), scale);
  const float a4 = __fdiv_rn(bf16_lo(w.z), scale), a5 = __fdiv_rn(bf16_hi(w.z), scale);
  const float a6 = __fdiv_rn(bf16_lo(w.w), scale), a7 = __fdiv_rn(bf16_hi(w.w), scale);
  return make_uint2(to_e4m3x4(a0, a1, a2, a3), to_e4m3x4(a4, a5, a6, a7));
}

template <bool FP8>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    append_kernel(const AppendParams p) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const ua_tile tile = p.tiles[blockIdx.x];
  if (w >= tile.nrows) return;
  const int j = tile.row0 + w;    // row of k_new / v_new
  const int pos = tile.kv_lo + w; // logical position in the sequence's cache
  int32_t blk = -1;
  if (pos >= 0 && pos / p.block_size < p.max_blocks_per_seq)
    blk = p.block_tables[static_cast<int64_t>(tile.seq) * p.max_blocks_per_seq +
                         pos / p.block_size];
  if (blk < 0 || static_cast<int64_t>(blk) >= p.num_blocks) {
    if (lane == 0) record_error(p.err, UA_ERR_BOUNDS);
    return;
  }
  const int64_t dst_row = static_cast<int64_t>(blk) * p.block_size + pos % p.block_size;
  const int chunks = p.row_elems / 8;  // 16-byte chunks of the bf16 source row
  const uint4* ks = reinterpret_cast<const uint4*>(p.k_new) + static_cast<int64_t>(j) * chunks;
  const uint4* vs = reinterpret_cast<const uint4*>(p.v_new) + static_cast<int64_t>(j) * chunks;
  for (int c0 = 0; c0 < chunks; c0 += 32 * kUnroll) {
    uint4 kx[kUnroll], vx[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int c = c0 + u * 32 + lane;
      if (c < chunks) {
        kx[u] = ld_stream_v4(ks + c);
        vx[u] = ld_stream_v4(vs + c);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int c = c0 + u * 32 + lane;
      if (c >= chunks) continue;
      if constexpr (!FP8) {
        reinterpret_cast<uint4*>(p.k_cache)[dst_row * chunks + c] = kx[u];
        reinterpret_cast<uint4*>(p.v_cache)[dst_row * chunks + c] = vx[u];
      } else {
        reinterpret_cast<uint2*>(p.k_cache)[dst_row * chunks + c] = quantize8(kx[u], p.k_scale);
        reinterpret_cast<uint2*>(p.v_cache)[dst_row * chunks + c] = quantize8(vx[u], p.v_scale);
      }
    }
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  if (p.num_tiles <= 0) return cudaSuccess;
  if (p.row_elems % 8 != 0 || p.tiles == nullptr) return cudaErrorInvalidValue;
  if (p.fp8)
    append_kernel<true><<<p.num_tiles, kWarpsPerCta * 32, 0, stream>>>(p);
  else
    append_kernel<false><<<p.num_tiles, kWarpsPerCta * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ua
