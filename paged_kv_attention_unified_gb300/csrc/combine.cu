// Log-sum-exp combine of split-KV partials (K-C), and the index-check gather.
//
// The combine is the global reduction step of FlashDecoding ("Fused
// Attention" notes, FlashDecoding section) and of the split-KV launcher's
// second kernel ("flashatten takeaways EP2 工程", run_flash_splitkv_fwd):
// each split s of a row left O_s = (sum of p v) / l_s and lse_s = m_s + log2 l_s
// (base 2); the row's output is
//     O = sum_s 2^(lse_s - lse*) O_s,   lse* = log2 sum_s 2^(lse_s).
// A split that saw no visible key has lse_s = -inf and weight 0.
//
// One CTA per combine group (one decode tile cut into pieces): warp n owns
// packed row n, every lane a contiguous run of head_dim/32 dimensions, so the
// partial rows are read with coalesced 16-, 8- or 4-byte loads.
#include "ua_device.cuh"
#include "ua_kernels.h"

namespace ua {

namespace {

template <int D>
__global__ void __launch_bounds__(32 * UA_DECODE_ROWS) combine_kernel(const CombineParams c) {
  __shared__ float wts[UA_DECODE_ROWS][UA_MAX_SPLITS];
  const ua_combine_group grp = c.groups[blockIdx.x];
  const int n = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (n >= grp.nrows) return;
  const int S = min(grp.nsplits, UA_MAX_SPLITS);
  const float* lse = c.ws_lse + static_cast<int64_t>(grp.slot0) * UA_DECODE_ROWS + n;
  float M = -INFINITY;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, lse[s * UA_DECODE_ROWS]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float W = 0.f;
  for (int s = lane; s < S; s += 32) {
    const float l = lse[s * UA_DECODE_ROWS];
    const float w = (l == -INFINITY) ? 0.f : ex2(l - M);
    wts[n][s] = w;
    W += w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
  __syncwarp();
  const float inv = W > 0.f ? 1.f / W : 0.f;

  constexpr int kPer = D / 32;
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  const float* base = c.ws_o + (static_cast<int64_t>(grp.slot0) * UA_DECODE_ROWS + n) * D +
                      lane * kPer;
  for (int s = 0; s < S; ++s) {
    const float w = wts[n][s];
    if (w == 0.f) continue;
    const float* src = base + static_cast<int64_t>(s) * UA_DECODE_ROWS * D;
    if constexpr (kPer % 4 == 0) {
#pragma unroll
      for (int e = 0; e < kPer; e += 4) {
        const float4 v = *reinterpret_cast<const float4*>(src + e);
        acc[e] += w * v.x;
        acc[e + 1] += w * v.y;
        acc[e + 2] += w * v.z;
        acc[e + 3] += w * v.w;
      }
    } else if constexpr (kPer % 2 == 0) {
#pragma unroll
      for (int e = 0; e < kPer; e += 2) {
        const float2 v = *reinterpret_cast<const float2*>(src + e);
        acc[e] += w * v.x;
        acc[e + 1] += w * v.y;
      }
    } else {
#pragma unroll
      for (int e = 0; e < kPer; ++e) acc[e] += w * src[e];
    }
  }
  const int r = grp.row0 + n;
  const int tok = c.cu_query_lens[grp.seq] + r / c.qpk;
  const int head = grp.kv_head * c.qpk + r % c.qpk;
  uint8_t* dst = reinterpret_cast<uint8_t*>(c.out) +
                 ((static_cast<int64_t>(tok) * c.num_q_heads + head) * D + lane * kPer) * 2;
  if constexpr (kPer % 4 == 0) {
#pragma unroll
    for (int e = 0; e < kPer; e += 4)
      *reinterpret_cast<uint2*>(dst + 2 * e) =
          make_uint2(pack2<false>(acc[e] * inv, acc[e + 1] * inv),
                     pack2<false>(acc[e + 2] * inv, acc[e + 3] * inv));
  } else if constexpr (kPer % 2 == 0) {
#pragma unroll
    for (int e = 0; e < kPer; e += 2)
      *reinterpret_cast<uint32_t*>(dst + 2 * e) = pack2<false>(acc[e] * inv, acc[e + 1] * inv);
  } else {
#pragma unroll
    for (int e = 0; e < kPer; ++e)
      *reinterpret_cast<__nv_bfloat16*>(dst + 2 * e) = __float2bfloat16_rn(acc[e] * inv);
  }
}

// One CTA per decode tile: copy the raw K and V rows of its key range.
__global__ void gather_debug_kernel(const KernelParams p, const int64_t* row_offsets,
                                    int row_bytes, uint8_t* k_out, uint8_t* v_out) {
  const ua_tile tile = p.tiles[blockIdx.x];
  const int kv_len = p.kv_lens[tile.seq];
  const int hi = min(min(tile.kv_hi, kv_len), p.max_blocks_per_seq * p.block_size);
  const int n = max(hi - tile.kv_lo, 0);
  const int chunks = row_bytes / 16;
  const int head_dim_elems = row_bytes;  // offsets below are in bytes
  for (int idx = threadIdx.x; idx < n * chunks; idx += blockDim.x) {
    const int key = tile.kv_lo + idx / chunks;
    const int ch = idx % chunks;
    const int64_t page = page_of(p, tile.seq, key);
    const int64_t dst = (row_offsets[blockIdx.x] + (key - tile.kv_lo)) * row_bytes + ch * 16;
    uint4 kx = make_uint4(0u, 0u, 0u, 0u), vx = kx;
    if (page >= 0) {
      const int64_t src =
          kv_row_offset(p, page, key % p.block_size, tile.kv_head, 1) * head_dim_elems + ch * 16;
      kx = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.k_cache) + src);
      vx = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.v_cache) + src);
    }
    *reinterpret_cast<uint4*>(k_out + dst) = kx;
    *reinterpret_cast<uint4*>(v_out + dst) = vx;
  }
}

}  // namespace

cudaError_t launch_combine(const CombineParams& c, int head_dim, cudaStream_t stream) {
  if (c.num_groups <= 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(c.num_groups)), block(32 * UA_DECODE_ROWS);
  switch (head_dim) {
    case 32: combine_kernel<32><<<grid, block, 0, stream>>>(c); break;
    case 64: combine_kernel<64><<<grid, block, 0, stream>>>(c); break;
    case 96: combine_kernel<96><<<grid, block, 0, stream>>>(c); break;
    case 128: combine_kernel<128><<<grid, block, 0, stream>>>(c); break;
    case 160: combine_kernel<160><<<grid, block, 0, stream>>>(c); break;
    case 192: combine_kernel<192><<<grid, block, 0, stream>>>(c); break;
    case 224: combine_kernel<224><<<grid, block, 0, stream>>>(c); break;
    case 256: combine_kernel<256><<<grid, block, 0, stream>>>(c); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_gather_debug(const KernelParams& p, const int64_t* row_offsets, int head_dim,
                                int elt_bytes, void* k_out, void* v_out, cudaStream_t stream) {
  if (p.num_tiles <= 0) return cudaSuccess;
  gather_debug_kernel<<<p.num_tiles, 256, 0, stream>>>(p, row_offsets, head_dim * elt_bytes,
                                                       static_cast<uint8_t*>(k_out),
                                                       static_cast<uint8_t*>(v_out));
  return cudaGetLastError();
}

}  // namespace ua
