// ua_forward_static_scratch: the split-KV decode path with its scratch memory
// (tile list, combine groups, split partials, error word) held in one
// file-scope device array, so that a call allocates nothing.
//
// Who needs this: callers that must not allocate device memory themselves --
// for example code embedded in another runtime that owns every device
// allocation through its own pool, plugins loaded into such a host, or
// latency-critical loops in which cudaMalloc (which can synchronise the whole
// device) is not acceptable. They pass inputs and outputs; everything else
// lives in g_scratch below.
//
// The tile list is built on the device from the device copies of the lengths,
// one tile per (sequence, KV head, block of 8 packed rows, split), so no
// host-side scheduling, staging buffer or upload is needed either. The tiles
// are then run by the same decode and combine kernels as ua_forward.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "ua_kernels.h"

namespace ua {
namespace {

// Scratch capacity in bytes; the whole array is resident on every device that
// loads this library, for the life of the process.
constexpr size_t kScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

// The scratch itself. Host code must not use this name as a device address:
// on the host it is only a stand-in for the symbol, so the address a kernel
// gets is looked up per device with cudaGetSymbolAddress (scratch_on_device).
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Layout of the scratch for one call (byte offsets, 256-byte aligned).
struct ScratchLayout {
  size_t tiles, groups, err, ws_o, ws_lse, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

ScratchLayout layout_for(int64_t num_tiles, int64_t num_groups, int64_t num_slots, int head_dim) {
  ScratchLayout l;
  l.tiles = 0;
  l.groups = align256(l.tiles + num_tiles * sizeof(ua_tile));
  l.err = align256(l.groups + num_groups * sizeof(ua_combine_group));
  l.ws_o = align256(l.err + sizeof(int32_t));
  l.ws_lse = align256(l.ws_o + num_slots * UA_DECODE_ROWS * head_dim * sizeof(float));
  l.total = align256(l.ws_lse + num_slots * UA_DECODE_ROWS * sizeof(float));
  return l;
}

// Device address of g_scratch on the current device: looked up once per device
// (with that device current) and remembered.
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

cudaError_t scratch_on_device(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_scratch_addr[dev]);
  return cudaSuccess;
}

// One thread per tile: tile n = ((s * Hkv + g) * row_tiles + rt) * splits + j.
// Same key-range rule as the host scheduler: rows [8 rt, 8 rt + 8) of sequence
// s see keys up to ctx + last token (causal) and above the window; the range,
// starting on a multiple of 16, is cut into `splits` equal pieces of a
// multiple of 16 keys. Rows or pieces that do not exist become empty tiles.
// The grid covers max_q tokens per sequence; one thread per sequence records
// UA_ERR_INVALID_ARG in the error word when the device lengths break the
// call's bounds (more packed rows than the grid holds, kv_len < q_len, or a
// kv_len past the page table), since those rows would otherwise be left
// unwritten or silently masked.
__global__ void build_tiles_kernel(const int32_t* cu_query_lens, const int32_t* kv_lens,
                                   int num_seqs, int num_kv_heads, int qpk, int row_tiles,
                                   int splits, int causal, int window, int64_t max_keys,
                                   ua_tile* tiles, ua_combine_group* groups, int32_t* err) {
  const int64_t n = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = static_cast<int64_t>(num_seqs) * num_kv_heads * row_tiles * splits;
  if (n >= total) return;
  const int j = static_cast<int>(n % splits);
  const int64_t grp = n / splits;
  const int rt = static_cast<int>(grp % row_tiles);
  const int g = static_cast<int>((grp / row_tiles) % num_kv_heads);
  const int s = static_cast<int>(grp / (static_cast<int64_t>(row_tiles) * num_kv_heads));
  const int qlen = cu_query_lens[s + 1] - cu_query_lens[s];
  const int kv = kv_lens[s];
  const int rows = qlen * qpk;
  const int row0 = rt * UA_DECODE_ROWS;
  if (g == 0 && rt == 0 && j == 0 &&
      (qlen < 0 || kv < qlen || static_cast<int64_t>(qlen) * qpk >
                                    static_cast<int64_t>(row_tiles) * UA_DECODE_ROWS ||
       kv > max_keys))
    record_error(err, UA_ERR_INVALID_ARG);
  const int nrows = max(0, min(UA_DECODE_ROWS, rows - row0));
  int lo = 0, hi = 0;
  if (nrows > 0) {
    const int ctx = kv - qlen;
    const int min_pos = ctx + row0 / qpk;
    const int max_pos = ctx + (row0 + nrows - 1) / qpk;
    hi = causal ? min(kv, max_pos + 1) : kv;
    lo = window > 0 ? max(0, min_pos - window + 1) : 0;
    lo = (lo / 16) * 16;
    hi = max(hi, lo);
  }
  const int len = hi - lo;
  const int size = ((len + splits - 1) / splits + 15) / 16 * 16;
  const int p0 = min(hi, lo + j * size);
  const int p1 = min(hi, lo + (j + 1) * size);
  ua_tile t;
  t.seq = s;
  t.kv_head = g;
  t.row0 = row0;
  t.nrows = nrows;
  t.kv_lo = p0;
  t.kv_hi = p1;
  t.slot = splits > 1 ? static_cast<int32_t>(n) : -1;
  t.group = splits > 1 ? static_cast<int32_t>(grp) : -1;
  tiles[n] = t;
  if (splits > 1 && j == 0) {
    ua_combine_group c;
    c.seq = s;
    c.kv_head = g;
    c.row0 = row0;
    c.nrows = nrows;
    c.slot0 = static_cast<int32_t>(n);
    c.nsplits = splits;
    c.pad0 = c.pad1 = 0;
    groups[grp] = c;
  }
}

}  // namespace
}  // namespace ua

extern "C" ua_status ua_forward_static_scratch(
    const void* q, const void* k_cache, const void* v_cache, void* out,
    const int32_t* cu_query_lens, const int32_t* kv_lens, const int32_t* block_tables,
    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int32_t max_blocks_per_seq, int64_t num_blocks, int32_t kv_dtype,
    int32_t max_q, int32_t max_kv, float scale, int32_t causal, int32_t window, float k_scale,
    float v_scale, int32_t num_splits, int32_t* device_error, ua_stream_t stream) {
  using namespace ua;
  // ---- host-side checks (nothing is launched on failure)
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || block_size <= 0 ||
      max_blocks_per_seq < 0 || max_q < 0 || max_kv < 0 || num_splits < 0 ||
      num_splits > UA_MAX_SPLITS || (causal != 0 && causal != 1))
    return UA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return UA_ERR_INVALID_ARG;
  if (kv_dtype != UA_KV_BF16 && kv_dtype != UA_KV_FP8_E4M3) return UA_ERR_INVALID_ARG;
  if (head_dim < 32 || head_dim > 256 || head_dim % 32 != 0) return UA_ERR_UNSUPPORTED;
  if (block_size % 16 != 0) return UA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size < max_kv) return UA_ERR_INVALID_ARG;
  if (num_seqs == 0 || max_q == 0) return UA_OK;
  if (!q || !k_cache || !v_cache || !out || !cu_query_lens || !kv_lens || !block_tables ||
      num_blocks <= 0 || num_blocks >= INT32_MAX)
    return UA_ERR_INVALID_ARG;
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (misaligned(q) || misaligned(k_cache) || misaligned(v_cache) || misaligned(out))
    return UA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return UA_ERR_INVALID_ARG;
  if (kv_dtype == UA_KV_FP8_E4M3 && (!std::isfinite(k_scale) || !std::isfinite(v_scale) ||
                                     k_scale == 0.f || v_scale == 0.f))
    return UA_ERR_INVALID_ARG;

  const int qpk = num_q_heads / num_kv_heads;
  const int64_t row_tiles = (static_cast<int64_t>(max_q) * qpk + UA_DECODE_ROWS - 1) / UA_DECODE_ROWS;
  // splits: as requested, else enough 1024-key pieces for the longest sequence
  int splits = num_splits > 0 ? num_splits : (max_kv + 1023) / 1024;
  splits = splits < 1 ? 1 : (splits > UA_MAX_SPLITS ? UA_MAX_SPLITS : splits);
  const int64_t groups = static_cast<int64_t>(num_seqs) * num_kv_heads * row_tiles;
  auto fits = [&](int sp) {
    const int64_t t = groups * sp;
    return t <= INT32_MAX &&
           layout_for(t, sp > 1 ? groups : 0, sp > 1 ? t : 0, head_dim).total <= kScratchBytes;
  };
  // automatic splits shrink until the call fits; requested splits must fit as given
  while (num_splits == 0 && splits > 1 && !fits(splits)) splits = (splits + 1) / 2;
  if (!fits(splits)) return UA_ERR_WORKSPACE;  // larger than the static scratch
  const int64_t tiles = groups * splits;
  const ScratchLayout lay = layout_for(tiles, splits > 1 ? groups : 0, splits > 1 ? tiles : 0,
                                       head_dim);

  // ---- set-up (first call on this device) and launches
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return UA_ERR_CUDA;
  unsigned char* base = nullptr;
  if (scratch_on_device(dev, &base) != cudaSuccess) return UA_ERR_CUDA;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  ua_tile* d_tiles = reinterpret_cast<ua_tile*>(base + lay.tiles);
  ua_combine_group* d_groups = reinterpret_cast<ua_combine_group*>(base + lay.groups);
  int32_t* d_err = reinterpret_cast<int32_t*>(base + lay.err);
  // the error word is the only scratch that must start at zero
  if (cudaMemsetAsync(d_err, 0, sizeof(int32_t), cs) != cudaSuccess) return UA_ERR_CUDA;
  const int threads = 256;
  build_tiles_kernel<<<static_cast<unsigned>((tiles + threads - 1) / threads), threads, 0, cs>>>(
      cu_query_lens, kv_lens, num_seqs, num_kv_heads, qpk, static_cast<int>(row_tiles), splits,
      causal, window, static_cast<int64_t>(max_blocks_per_seq) * block_size, d_tiles, d_groups,
      d_err);
  if (cudaGetLastError() != cudaSuccess) return UA_ERR_CUDA;

  KernelParams kp{};
  kp.q = q;
  kp.k_cache = k_cache;
  kp.v_cache = v_cache;
  kp.out = out;
  kp.cu_query_lens = cu_query_lens;
  kp.kv_lens = kv_lens;
  kp.block_tables = block_tables;
  kp.tiles = d_tiles;
  kp.num_tiles = static_cast<int32_t>(tiles);
  kp.ws_o = splits > 1 ? reinterpret_cast<float*>(base + lay.ws_o) : nullptr;
  kp.ws_lse = splits > 1 ? reinterpret_cast<float*>(base + lay.ws_lse) : nullptr;
  kp.err = d_err;
  kp.num_blocks = num_blocks;
  kp.max_blocks_per_seq = max_blocks_per_seq;
  kp.block_size = block_size;
  kp.num_q_heads = num_q_heads;
  kp.num_kv_heads = num_kv_heads;
  kp.qpk = qpk;
  kp.causal = causal;
  kp.window = window;
  const bool fp8 = kv_dtype == UA_KV_FP8_E4M3;
  kp.score_scale_log2 = scale * kLog2e * (fp8 ? k_scale : 1.f);
  kp.v_scale = fp8 ? v_scale : 1.f;
  kp.timeout_ns = 2000000000ull;
  if (launch_decode(kp, head_dim, kv_dtype, cs) != cudaSuccess) return UA_ERR_CUDA;
  if (splits > 1) {
    CombineParams cp;
    cp.groups = d_groups;
    cp.num_groups = static_cast<int32_t>(groups);
    cp.ws_o = kp.ws_o;
    cp.ws_lse = kp.ws_lse;
    cp.cu_query_lens = cu_query_lens;
    cp.out = out;
    cp.num_q_heads = num_q_heads;
    cp.qpk = qpk;
    if (launch_combine(cp, head_dim, cs) != cudaSuccess) return UA_ERR_CUDA;
  }
  if (device_error != nullptr &&
      cudaMemcpyAsync(device_error, d_err, sizeof(int32_t), cudaMemcpyDeviceToDevice, cs) !=
          cudaSuccess)
    return UA_ERR_CUDA;
  return UA_OK;
}
