// Launch entry points of the device kernels (host side of each .cu file).
#pragma once

#include <atomic>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "ua_device.cuh"

namespace ua {

// Sets a kernel's dynamic shared-memory limit once per device (the driver
// keeps it for the life of the context). `done` is a per-kernel bitmask of
// devices; devices beyond 63 are set on every call.
template <typename Kernel>
cudaError_t set_smem_once(Kernel kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

struct PrefillParams {
  const ua_tile* tiles;       // taken in list order by the persistent CTAs
  int32_t num_tiles;
  const void* q;              // bf16 queries (read directly by the fp8-products kernel)
  int32_t* counters;          // [2] next tile, finished CTAs; zero between launches
  int32_t num_ctas;           // persistent CTAs (at most one per SM)
  const int32_t* cu_query_lens;
  const int32_t* kv_lens;
  const int32_t* block_tables;
  void* out;
  int32_t* err;
  int64_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t block_size;
  int32_t num_q_heads;
  int32_t qpk;
  int32_t causal;
  int32_t window;
  float score_scale_log2;   // scale * log2(e) (* k_scale for a staged fp8 cache)
  float out_scale;          // multiplies O / l (v_scale for a staged fp8 cache, else 1)
  int32_t rows_per_box;     // keys per TMA box: min(block_size, 128)
  uint64_t timeout_ns;      // bound of every mbarrier wait
  int32_t debug_flags;      // bit 0: the producer issues nothing (timeout test)
  // Kernel timing (null: off): the first CTA's start (atomicMin) and the last
  // CTA's end (atomicMax) on the device global timer, in ns.
  unsigned long long* span_start;
  unsigned long long* span_end;
};

// Bit 0 of PrefillParams::debug_flags: the TMA producer skips every load, so
// that the consumers' bounded waits run out (tests the timeout path).
constexpr int32_t kDebugProducerIdle = 1;

// Whether the prefill kernel can take a problem with these parameters
// (host-only check, no CUDA call).
bool prefill_supported(int head_dim, int kv_dtype, int qpk, int block_size);

// Persistent prefill kernel: p.num_ctas CTAs take p.tiles in order as they
// free up (the host encodes the tensor maps from the pointers). Every CTA
// allows a grid queued behind it with programmatic stream serialization to
// start once all of them have started.
cudaError_t launch_prefill(const PrefillParams& p, const void* q, const void* k_cache,
                           const void* v_cache, int64_t total_q, int head_dim,
                           int num_kv_heads, cudaStream_t stream);

// Prefill kernel with fp8 tensor-core products over an e4m3 cache (head_dim
// 128): Q rows quantised to e4m3 per row inside the kernel, S = Q K^T and
// O += P V as kind::f8f6f4 MMAs with P rounded to e4m3. rows_per_box as for
// launch_prefill; score_scale_log2 = scale * log2(e) * k_scale, out_scale =
// v_scale.
bool prefill_fp8_products_supported(int head_dim, int qpk, int block_size);
cudaError_t launch_prefill_fp8_products(const PrefillParams& p, const void* k_cache,
                                        const void* v_cache, int num_kv_heads,
                                        cudaStream_t stream);

// head_dim 192 / 256 prefill kernel (one 128-row query tile at a time,
// 64-key tiles): whether it takes the problem, the keys per TMA box it needs
// (PrefillParams::rows_per_box), and its launch (same parameters as
// launch_prefill).
bool prefill_wide_supported(int kv_dtype, int qpk, int block_size);
int prefill_wide_rows_per_box(int block_size);
bool prefill_is_wide(int head_dim);
cudaError_t launch_prefill_wide(const PrefillParams& p, const void* q, const void* k_cache,
                                const void* v_cache, int64_t total_q, int head_dim,
                                int num_kv_heads, cudaStream_t stream);

// Tensor map of a row-major tensor (dims innermost first, strides in bytes of
// dims 1..rank-1) for bf16 (elt_bytes 2) or byte (elt_bytes 1) elements;
// l2_promotion: L2 fetch width in bytes (64, 128 or 256).
cudaError_t encode_tiled_map(CUtensorMap* map, int elt_bytes, int rank, const void* base,
                             const uint64_t* dims, const uint64_t* strides_bytes,
                             const uint32_t* box, bool swizzle_128b, int l2_promotion);

// Tensor map over a paged cache [num_blocks][block_size][Hkv][head_dim] whose
// box is (box_dims dims, one head, box_rows slots, one block); an out-of-range
// block coordinate reads zeros. L2 fetches are at most one head row wide.
cudaError_t encode_kv_page_map(CUtensorMap* map, const void* cache, int elt_bytes, int head_dim,
                               int num_kv_heads, int block_size, int64_t num_blocks,
                               int box_dims, int box_rows, bool swizzle_128b);

// Split-KV decode kernel over p.tiles[0 .. p.num_tiles). after_prefill: the
// launch directly follows a prefill launch on `stream` and may start as soon
// as every prefill CTA has started (programmatic stream serialization; the
// two grids touch disjoint outputs and share only read-only inputs).
cudaError_t launch_decode(const KernelParams& p, int head_dim, int kv_dtype, cudaStream_t stream,
                          bool after_prefill = false);

// Log-sum-exp combine of split partials into bf16 output rows.
cudaError_t launch_combine(const CombineParams& c, int head_dim, cudaStream_t stream);

// Append-KV: new keys / values of a step into the paged cache.
struct AppendParams {
  const void* k_new;            // [total_tokens][Hkv][d] bf16
  const void* v_new;
  void* k_cache;                // [num_blocks][block_size][Hkv][d] bf16 or e4m3
  void* v_cache;
  const ua_tile* tiles;          // append tiles of the plan (one CTA each)
  int32_t num_tiles;
  const int32_t* block_tables;   // device [num_seqs][max_blocks_per_seq]
  int32_t* err;                  // error word (UA_ERR_BOUNDS)
  int64_t num_blocks;
  int32_t row_elems;             // Hkv * d, a multiple of 8
  int32_t max_blocks_per_seq;
  int32_t block_size;
  int32_t fp8;                   // 1: e4m3 cache
  float k_scale;                 // e4m3 cache: code = e4m3(x / scale)
  float v_scale;
};

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);

// fp8 prefill staging: e4m3 pages of the prefill sequences -> bf16 staging
// pages of 128 slots (exact, scale-free).
struct StageParams {
  const void* k_src;             // e4m3 caches [num_blocks][block_size][Hkv][d]
  const void* v_src;
  void* k_dst;                   // bf16 staging [pages][128][Hkv][d]
  void* v_dst;
  const ua_tile* tiles;          // stage tiles of the plan (one CTA each)
  int32_t num_tiles;
  const int32_t* block_tables;   // device [num_seqs][max_blocks_per_seq]
  int32_t max_blocks_per_seq;
  int32_t block_size;
  int64_t num_blocks;
  int32_t row_elems;             // Hkv * d, a multiple of 8
  int32_t* err;                  // error word (UA_ERR_BOUNDS)
};

cudaError_t launch_stage(const StageParams& p, cudaStream_t stream);

// Test aid: copy the raw K/V rows each tile reads into dense buffers.
cudaError_t launch_gather_debug(const KernelParams& p, const int64_t* row_offsets, int head_dim,
                                int elt_bytes, void* k_out, void* v_out, cudaStream_t stream);

}  // namespace ua
