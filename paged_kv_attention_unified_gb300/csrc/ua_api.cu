// C ABI of the unified paged-KV attention forward (declared in include/ua.h):
// plan creation around the CPU scheduler, argument validation, and the kernel
// launches of one forward call.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "planner.h"
#include "ua_kernels.h"

struct ua_plan {
  int device = 0;
  ua::Problem prob;
  ua::Schedule sched;
  ua_plan_info info{};
  // device memory owned by the plan
  void* d_meta = nullptr;          // [tiles | groups | error word | counters | ... | split workspace]
  ua_tile* d_prefill = nullptr;
  ua_tile* d_decode = nullptr;
  ua_combine_group* d_groups = nullptr;
  int32_t* d_err = nullptr;
  int32_t* d_counters = nullptr;   // per combine group, zero between calls
  int32_t* d_prefill_counters = nullptr;  // [2] persistent prefill tile queue, zero between calls
  ua_tile* d_append = nullptr;            // append-KV tiles
  int32_t* d_staged_table = nullptr;      // fp8 prefill: staging page table
  ua_tile* d_stage = nullptr;             // fp8 prefill: stage tiles
  void* d_staged_k = nullptr;             // fp8 prefill: bf16 staging caches
  void* d_staged_v = nullptr;
  // split workspace (inside d_meta): partial rows then lse values
  float* d_ws_o = nullptr;
  float* d_ws_lse = nullptr;
  cudaStream_t last_stream = nullptr;
  int64_t total_q = 0;             // query tokens of the batch (host lengths)
  int32_t debug_flags = 0;         // ua_plan_set_debug
  bool unified_max_on = false;     // ua_plan_set_unified_max
  float unified_max = 0.f;
  uint64_t wait_timeout_ns = 2000000000ull;
  int32_t prefill_ctas_override = 0;  // ua_plan_set_prefill_ctas (0: the scheduler's count)
  bool fp8_products = false;          // ua_plan_set_fp8_products
  // kernel timing (ua_plan_set_profiling)
  struct EventPair {
    cudaEvent_t start = nullptr, stop = nullptr;
    int kind = 0;
  };
  bool profiling = false;
  std::vector<EventPair> ev_pending, ev_free;
  // The prefill and decode kernels time themselves (first CTA start, last CTA
  // end on the device global timer) into slot i of these arrays: an event
  // recorded between the two launches of a mixed batch would stop the decode
  // grid from starting while the prefill grid runs.
  unsigned long long* d_span = nullptr;  // [kSpanSlots] starts, then [kSpanSlots] ends
  std::vector<std::pair<int, int>> span_pending;  // (kind, slot)
};

namespace {

ua_status from_cuda(cudaError_t e) { return e == cudaSuccess ? UA_OK : UA_ERR_CUDA; }

// Plan memory comes from a stream-ordered pool the library owns (one per
// device), which keeps up to kPoolKeepBytes of freed blocks for the next
// plan: a serving loop that builds and drops a plan every step then never
// calls the driver allocator, and destroying a plan does not wait for its
// stream. The pool's own release threshold is a setting of this process only.
constexpr uint64_t kPoolKeepBytes = 1ull << 30;
constexpr int kMaxDevices = 64;

cudaMemPool_t plan_pool(int device) {
  static std::mutex mu;
  static cudaMemPool_t pools[kMaxDevices] = {};
  if (device < 0 || device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (pools[device] == nullptr) {
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = device;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
    uint64_t keep = kPoolKeepBytes;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    pools[device] = pool;
  }
  return pools[device];
}

cudaError_t plan_alloc(void** ptr, size_t bytes, int device, cudaStream_t stream) {
  cudaMemPool_t pool = plan_pool(device);
  if (pool == nullptr) return cudaErrorMemoryAllocation;
  return cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
}

// Pinned host blocks for the plan's tile-list upload. A copy from pageable
// memory first waits for everything queued on its stream (for a step that
// has just queued the H2D copy of its inputs, that is the whole copy); from
// pinned memory it is queued like a kernel, so scheduling the next plan
// overlaps the input copy. A block is reused once the event recorded after
// its copy has completed; blocks are kept for the life of the process.
struct PinnedBlock {
  void* ptr = nullptr;
  size_t bytes = 0;
  cudaEvent_t done = nullptr;
};

std::mutex g_pinned_mu;
std::vector<PinnedBlock> g_pinned_free;

bool pinned_take(size_t bytes, PinnedBlock* out) {
  std::lock_guard<std::mutex> lock(g_pinned_mu);
  for (size_t i = 0; i < g_pinned_free.size(); ++i) {
    PinnedBlock& b = g_pinned_free[i];
    if (b.bytes >= bytes && cudaEventQuery(b.done) == cudaSuccess) {
      *out = b;
      g_pinned_free.erase(g_pinned_free.begin() + static_cast<std::ptrdiff_t>(i));
      return true;
    }
  }
  PinnedBlock b;
  b.bytes = bytes < (64u << 10) ? (64u << 10) : bytes;
  if (cudaMallocHost(&b.ptr, b.bytes) != cudaSuccess) return false;
  if (cudaEventCreateWithFlags(&b.done, cudaEventDisableTiming) != cudaSuccess) {
    cudaFreeHost(b.ptr);
    return false;
  }
  *out = b;
  return true;
}

void pinned_give_back(const PinnedBlock& b) {
  std::lock_guard<std::mutex> lock(g_pinned_mu);
  g_pinned_free.push_back(b);
}

constexpr int kSpanSlots = 1024;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

void free_plan_memory(ua_plan* p) {
  for (auto* v : {&p->ev_pending, &p->ev_free})
    for (auto& e : *v) {
      if (e.start) cudaEventDestroy(e.start);
      if (e.stop) cudaEventDestroy(e.stop);
    }
  p->ev_pending.clear();
  p->ev_free.clear();
  // stream-ordered: the memory returns to the pool once the plan's last
  // stream has finished with it
  if (p->d_span) cudaFreeAsync(p->d_span, p->last_stream);
  p->d_span = nullptr;
  if (p->d_meta) cudaFreeAsync(p->d_meta, p->last_stream);
  if (p->d_staged_k) cudaFreeAsync(p->d_staged_k, p->last_stream);
  if (p->d_staged_v) cudaFreeAsync(p->d_staged_v, p->last_stream);
  p->d_meta = nullptr;
  p->d_staged_k = nullptr;
  p->d_staged_v = nullptr;
}

ua::Problem make_problem(const int32_t* cu, const int32_t* kv, int32_t num_seqs, int32_t hq,
                         int32_t hkv, int32_t d, int32_t bs, int32_t max_blocks, int32_t dtype,
                         int32_t causal, int32_t window, int32_t num_splits, int32_t num_sms,
                         int32_t decode_rows_max) {
  ua::Problem p;
  p.cu_query_lens = cu;
  p.kv_lens = kv;
  p.num_seqs = num_seqs;
  p.num_q_heads = hq;
  p.num_kv_heads = hkv;
  p.head_dim = d;
  p.block_size = bs;
  p.max_blocks_per_seq = max_blocks;
  p.kv_dtype = dtype;
  p.causal = causal;
  p.window = window;
  p.num_splits = num_splits;
  p.num_sms = num_sms;
  p.decode_rows_max = decode_rows_max;
  // An fp8 cache's prefill runs on a bf16 staging copy of 128-slot pages.
  const bool fp8 = dtype == UA_KV_FP8_E4M3;
  p.prefill_ok = hkv > 0 && hq % hkv == 0 &&
                 ua::prefill_supported(d, fp8 ? UA_KV_BF16 : dtype, hq / hkv,
                                       fp8 ? ua::kStagePage : bs);
  p.prefill_staged = fp8 && p.prefill_ok;
  return p;
}

void fill_info(const ua::Schedule& s, int head_dim, int num_sms, ua_plan_info* info) {
  info->num_prefill_tiles = static_cast<int64_t>(s.prefill.size());
  info->num_decode_tiles = static_cast<int64_t>(s.decode.size());
  info->num_combine_groups = static_cast<int64_t>(s.groups.size());
  info->num_slots = s.num_slots;
  info->workspace_bytes = ua::workspace_bytes(s, head_dim);
  info->split_tokens = s.split_tokens;
  info->num_sms = num_sms;
  info->num_prefill_ctas = s.prefill_ctas;
  info->reserved = 0;
}

ua::KernelParams base_params(const ua_plan* plan, const void* q, const void* k, const void* v,
                             void* out, const int32_t* cu, const int32_t* kvl, const int32_t* bt,
                             int64_t num_blocks, float scale, float k_scale, float v_scale) {
  const ua::Problem& pr = plan->prob;
  ua::KernelParams kp;
  std::memset(&kp, 0, sizeof(kp));
  kp.q = q;
  kp.k_cache = k;
  kp.v_cache = v;
  kp.out = out;
  kp.cu_query_lens = cu;
  kp.kv_lens = kvl;
  kp.block_tables = bt;
  kp.ws_o = plan->d_ws_o;
  kp.ws_lse = plan->d_ws_lse;
  kp.err = plan->d_err;
  kp.num_blocks = num_blocks;
  kp.max_blocks_per_seq = pr.max_blocks_per_seq;
  kp.block_size = pr.block_size;
  kp.num_q_heads = pr.num_q_heads;
  kp.num_kv_heads = pr.num_kv_heads;
  kp.qpk = pr.num_q_heads / pr.num_kv_heads;
  kp.causal = pr.causal;
  kp.window = pr.window;
  const bool fp8 = pr.kv_dtype == UA_KV_FP8_E4M3;
  kp.score_scale_log2 = scale * ua::kLog2e * (fp8 ? k_scale : 1.f);
  kp.v_scale = fp8 ? v_scale : 1.f;
  kp.timeout_ns = plan->wait_timeout_ns;
  kp.unified_max_on = plan->unified_max_on ? 1 : 0;
  kp.unified_max_log2 = plan->unified_max * ua::kLog2e;
  return kp;
}

// Record the start event of a timed launch (no-op unless profiling).
ua_plan::EventPair* timing_begin(ua_plan* p, int kind, cudaStream_t cs) {
  if (!p->profiling) return nullptr;
  ua_plan::EventPair e;
  if (!p->ev_free.empty()) {
    e = p->ev_free.back();
    p->ev_free.pop_back();
  } else if (cudaEventCreate(&e.start) != cudaSuccess || cudaEventCreate(&e.stop) != cudaSuccess) {
    return nullptr;
  }
  e.kind = kind;
  cudaEventRecord(e.start, cs);
  p->ev_pending.push_back(e);
  return &p->ev_pending.back();
}

void timing_end(ua_plan::EventPair* e, cudaStream_t cs) {
  if (e) cudaEventRecord(e->stop, cs);
}

// Span slot for a self-timed launch of `kind` (prefill 0, decode 1): the
// kernel's start / end words, or nulls when not profiling or out of slots.
void span_begin(ua_plan* p, int kind, unsigned long long** start, unsigned long long** end) {
  *start = *end = nullptr;
  if (!p->profiling || p->d_span == nullptr) return;
  const int slot = static_cast<int>(p->span_pending.size());
  if (slot >= kSpanSlots) return;
  p->span_pending.emplace_back(kind, slot);
  *start = p->d_span + slot;
  *end = p->d_span + kSpanSlots + slot;
}

// Span words back to "empty": starts at the largest value, ends at zero.
cudaError_t span_reset(ua_plan* p, int slots, cudaStream_t cs) {
  if (slots <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(p->d_span, 0xFF, slots * sizeof(unsigned long long), cs);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(p->d_span + kSpanSlots, 0, slots * sizeof(unsigned long long), cs);
  return e;
}

}  // namespace

extern "C" {

const char* ua_status_string(int32_t status) {
  switch (status) {
    case UA_OK: return "UA_OK";
    case UA_ERR_INVALID_ARG: return "UA_ERR_INVALID_ARG: invalid argument";
    case UA_ERR_UNSUPPORTED: return "UA_ERR_UNSUPPORTED: head_dim, dtype or block_size not built";
    case UA_ERR_CUDA: return "UA_ERR_CUDA: a CUDA call failed";
    case UA_ERR_WORKSPACE: return "UA_ERR_WORKSPACE: workspace missing or too small";
    case UA_ERR_DEVICE_TIMEOUT: return "UA_ERR_DEVICE_TIMEOUT: a device-side wait gave up";
    case UA_ERR_BOUNDS: return "UA_ERR_BOUNDS: page id outside [0, num_blocks)";
    default: return "unknown ua_status";
  }
}

ua_status ua_schedule(const int32_t* cu_query_lens_host, const int32_t* kv_lens_host,
                      int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq,
                      int32_t kv_dtype, int32_t causal, int32_t window, int32_t num_splits,
                      int32_t num_sms, int32_t decode_rows_max, ua_plan_info* info,
                      ua_tile* prefill_tiles, int64_t prefill_cap, ua_tile* decode_tiles,
                      int64_t decode_cap, ua_combine_group* groups, int64_t groups_cap) {
  if (info == nullptr) return UA_ERR_INVALID_ARG;
  const int sms = num_sms > 0 ? num_sms : 152;
  ua::Problem pr = make_problem(cu_query_lens_host, kv_lens_host, num_seqs, num_q_heads,
                                num_kv_heads, head_dim, block_size, max_blocks_per_seq, kv_dtype,
                                causal, window, num_splits, sms, decode_rows_max);
  ua::Schedule s;
  try {
    ua_status st = ua::build_schedule(pr, &s);
    if (st != UA_OK) return st;
  } catch (const std::bad_alloc&) {
    return UA_ERR_INVALID_ARG;
  }
  fill_info(s, head_dim, sms, info);
  if (prefill_tiles) {
    if (prefill_cap < static_cast<int64_t>(s.prefill.size())) return UA_ERR_INVALID_ARG;
    std::memcpy(prefill_tiles, s.prefill.data(), s.prefill.size() * sizeof(ua_tile));
  }
  if (decode_tiles) {
    if (decode_cap < static_cast<int64_t>(s.decode.size())) return UA_ERR_INVALID_ARG;
    std::memcpy(decode_tiles, s.decode.data(), s.decode.size() * sizeof(ua_tile));
  }
  if (groups) {
    if (groups_cap < static_cast<int64_t>(s.groups.size())) return UA_ERR_INVALID_ARG;
    std::memcpy(groups, s.groups.data(), s.groups.size() * sizeof(ua_combine_group));
  }
  return UA_OK;
}

}  // extern "C"

namespace {

// Plan creation. `extra` (if any): host byte ranges appended, 16-byte
// aligned, to the plan's one tile-list upload; *extra_dev receives the device
// address of each (they live as long as the plan).
struct HostRange {
  const void* ptr;
  size_t bytes;
};

ua_status create_plan(ua_plan** out, const int32_t* cu_query_lens_host,
                      const int32_t* kv_lens_host, int32_t num_seqs, int32_t num_q_heads,
                      int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                      int32_t max_blocks_per_seq, int32_t kv_dtype, int32_t causal,
                      int32_t window, int32_t num_splits, int32_t decode_rows_max,
                      ua_stream_t stream, const HostRange* extra, int n_extra,
                      void** extra_dev) {
  if (out == nullptr) return UA_ERR_INVALID_ARG;
  *out = nullptr;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return UA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return UA_ERR_CUDA;
  ua_plan* plan = new (std::nothrow) ua_plan();
  if (plan == nullptr) return UA_ERR_INVALID_ARG;
  plan->device = dev;
  plan->prob = make_problem(cu_query_lens_host, kv_lens_host, num_seqs, num_q_heads,
                            num_kv_heads, head_dim, block_size, max_blocks_per_seq, kv_dtype,
                            causal, window, num_splits, sms, decode_rows_max);
  ua_status st;
  try {
    st = ua::build_schedule(plan->prob, &plan->sched);
  } catch (const std::bad_alloc&) {
    st = UA_ERR_INVALID_ARG;
  }
  if (st != UA_OK) {
    delete plan;
    return st;
  }
  plan->total_q = num_seqs > 0 ? cu_query_lens_host[num_seqs] : 0;
  // The plan keeps no pointer to the caller's host arrays.
  plan->prob.cu_query_lens = nullptr;
  plan->prob.kv_lens = nullptr;
  fill_info(plan->sched, head_dim, sms, &plan->info);

  const ua::Schedule& s = plan->sched;
  const size_t n_pre = s.prefill.size(), n_dec = s.decode.size(), n_grp = s.groups.size();
  const size_t bytes_tiles = (n_pre + n_dec) * sizeof(ua_tile);
  const size_t bytes_groups = n_grp * sizeof(ua_combine_group);
  const size_t off_pc = bytes_tiles + bytes_groups + 16 + n_grp * sizeof(int32_t);
  const size_t n_app = s.append.size();
  const size_t off_app = (off_pc + 2 * sizeof(int32_t) + 15) & ~static_cast<size_t>(15);
  const size_t n_stage = s.stage.size(), n_st = s.staged_table.size();
  const size_t off_stage = off_app + n_app * sizeof(ua_tile);
  const size_t off_st = off_stage + n_stage * sizeof(ua_tile);
  size_t bytes_meta = off_st + n_st * sizeof(int32_t);
  std::vector<size_t> off_extra(static_cast<size_t>(n_extra > 0 ? n_extra : 0));
  for (int i = 0; i < n_extra; ++i) {
    bytes_meta = (bytes_meta + 15) & ~static_cast<size_t>(15);
    off_extra[i] = bytes_meta;
    bytes_meta += extra[i].bytes;
  }
  PinnedBlock staging;
  if (!pinned_take(bytes_meta, &staging)) {
    delete plan;
    return UA_ERR_CUDA;
  }
  uint8_t* host = static_cast<uint8_t*>(staging.ptr);
  // Every list below is copied whole; only the error word, the combine
  // counters and the prefill queue counters (and the padding up to the
  // append tiles) start at zero.
  std::memset(host + bytes_tiles + bytes_groups, 0, off_app - (bytes_tiles + bytes_groups));
  if (n_pre) std::memcpy(host, s.prefill.data(), n_pre * sizeof(ua_tile));
  if (n_dec) std::memcpy(host + n_pre * sizeof(ua_tile), s.decode.data(),
                         n_dec * sizeof(ua_tile));
  if (n_grp) std::memcpy(host + bytes_tiles, s.groups.data(), bytes_groups);
  if (n_app) std::memcpy(host + off_app, s.append.data(), n_app * sizeof(ua_tile));
  if (n_stage) std::memcpy(host + off_stage, s.stage.data(), n_stage * sizeof(ua_tile));
  if (n_st) std::memcpy(host + off_st, s.staged_table.data(), n_st * sizeof(int32_t));
  for (int i = 0; i < n_extra; ++i)
    if (extra[i].bytes) std::memcpy(host + off_extra[i], extra[i].ptr, extra[i].bytes);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  plan->last_stream = cs;
  // The split workspace follows the uploaded part in the same allocation
  // (not copied: every slot is written before it is read).
  const size_t off_ws = (bytes_meta + 255) & ~static_cast<size_t>(255);
  const size_t bytes_alloc = off_ws + static_cast<size_t>(plan->info.workspace_bytes);
  if (plan_alloc(&plan->d_meta, bytes_alloc, plan->device, cs) != cudaSuccess) {
    plan->d_meta = nullptr;
    pinned_give_back(staging);
    free_plan_memory(plan);
    delete plan;
    return UA_ERR_CUDA;
  }
  uint8_t* base = static_cast<uint8_t*>(plan->d_meta);
  plan->d_prefill = reinterpret_cast<ua_tile*>(base);
  plan->d_decode = reinterpret_cast<ua_tile*>(base + n_pre * sizeof(ua_tile));
  plan->d_groups = reinterpret_cast<ua_combine_group*>(base + bytes_tiles);
  plan->d_err = reinterpret_cast<int32_t*>(base + bytes_tiles + bytes_groups);
  plan->d_counters = reinterpret_cast<int32_t*>(base + bytes_tiles + bytes_groups + 16);
  plan->d_prefill_counters = reinterpret_cast<int32_t*>(base + off_pc);
  plan->d_append = reinterpret_cast<ua_tile*>(base + off_app);
  plan->d_stage = reinterpret_cast<ua_tile*>(base + off_stage);
  plan->d_staged_table = reinterpret_cast<int32_t*>(base + off_st);
  for (int i = 0; i < n_extra; ++i) extra_dev[i] = base + off_extra[i];
  if (s.staged_pages > 0) {
    const size_t bytes = static_cast<size_t>(s.staged_pages) * ua::kStagePage *
                         plan->prob.num_kv_heads * head_dim * 2;
    if (plan_alloc(&plan->d_staged_k, bytes, plan->device, cs) != cudaSuccess ||
        plan_alloc(&plan->d_staged_v, bytes, plan->device, cs) != cudaSuccess) {
      pinned_give_back(staging);
      free_plan_memory(plan);
      delete plan;
      return UA_ERR_CUDA;
    }
  }
  if (plan->info.workspace_bytes > 0) {
    plan->d_ws_o = reinterpret_cast<float*>(base + off_ws);
    plan->d_ws_lse = plan->d_ws_o + s.num_slots * UA_DECODE_ROWS * static_cast<int64_t>(head_dim);
  }
  const bool copied =
      cudaMemcpyAsync(plan->d_meta, host, bytes_meta, cudaMemcpyHostToDevice, cs) == cudaSuccess;
  // the block returns to the pool; it is reused only after this event
  cudaEventRecord(staging.done, cs);
  pinned_give_back(staging);
  if (!copied) {
    free_plan_memory(plan);
    delete plan;
    return UA_ERR_CUDA;
  }
  plan->last_stream = cs;
  *out = plan;
  return UA_OK;
}

// ua_forward_host for batches whose query and output copies take about as
// long as the forward itself: the query tokens are cut into runs of about
// kHostRunBytes of q each (2 to kHostMaxRuns runs), each with its own plan,
// and the copies overlap the compute. Run c goes on `stream` (even c) or a
// second compute stream (odd c): the copy of its q, its plan upload and its
// forward, in that order on one stream, so that the next run's q copy
// overlaps this run's forward and the next run's CTAs fill the SMs this
// run's last CTAs leave idle. Its output comes back on a copy stream while
// later runs compute (the host link carries both directions at once). (A q
// copy on a stream of its own, waited for through an event, held back the
// forwards until every q had landed.)
// A cut falls on the first sequence boundary at or after its target, unless
// the sequence holding the target is at least a run long (one long prefill
// would otherwise be a single run): then, when the mask allows it, the cut
// falls inside it. With a causal mask, query rows [a, b) of a sequence with
// context ctx see exactly what a sequence of b - a new tokens and ctx + b
// keys sees; without a mask or window, what one with all kv_len keys sees.
// Such cuts fall on whole prefill tiles and leave both parts too long for
// the decode kernel, so every prefill row takes the same arithmetic as in
// one plan. (More, shorter runs measured slower: eight runs of half
// sequences took 1.29 ms per dense-prefill call, four whole ones 1.18 ms.)
constexpr size_t kHostPipelineMinBytes = size_t{32} << 20;
constexpr size_t kHostRunBytes = size_t{16} << 20;
constexpr int kHostMaxRuns = 4;

// The internal streams of a device (a compute stream and the output copy
// stream), created on first use and kept.
bool host_pipeline_streams(int dev, cudaStream_t (&out)[2]) {
  static std::mutex mu;
  static cudaStream_t streams[kMaxDevices][2] = {};
  if (dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(mu);
  cudaStream_t* st = streams[dev];
  for (int i = 0; i < 2; ++i) {
    if (st[i] == nullptr && cudaStreamCreateWithFlags(&st[i], cudaStreamNonBlocking) != cudaSuccess) {
      st[i] = nullptr;
      return false;
    }
    out[i] = st[i];
  }
  return true;
}

ua_status forward_host_chunked(const void* q_host, void* out_host,
                               const int32_t* cu_query_lens_host, const int32_t* kv_lens_host,
                               const int32_t* block_tables_host, const void* k_cache,
                               const void* v_cache, int32_t num_seqs, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t max_blocks_per_seq, int64_t num_blocks, int32_t kv_dtype,
                               float scale, int32_t causal, int32_t window, float k_scale,
                               float v_scale, int32_t num_splits, int32_t* error_word,
                               ua_stream_t stream) {
  const int32_t* cu = cu_query_lens_host;
  const int64_t total_q = cu[num_seqs];
  const size_t row_bytes = static_cast<size_t>(num_q_heads) * head_dim * 2;
  const size_t q_bytes = static_cast<size_t>(total_q) * row_bytes;
  // Run boundaries in query tokens: tok[c] .. tok[c + 1].
  const int want = static_cast<int>(
      std::min<size_t>(kHostMaxRuns, std::max<size_t>(2, q_bytes / kHostRunBytes)));
  const bool cut_inside = causal != 0 || window <= 0;
  const int64_t qpk = num_q_heads / num_kv_heads;
  const int64_t align = std::max<int64_t>(1, UA_PREFILL_ROWS / qpk);  // tokens per prefill tile
  std::vector<int64_t> tok{0};
  for (int k = 1; k < want; ++k) {
    const int64_t target = total_q * k / want;
    // the sequence holding token `target`
    const int32_t sq = static_cast<int32_t>(std::upper_bound(cu, cu + num_seqs + 1, target) - cu) - 1;
    const int64_t ql = cu[sq + 1] - cu[sq];
    const int64_t boundary = cu[sq] == target ? cu[sq] : cu[sq + 1];
    const int64_t inside = (target - cu[sq]) / align * align;
    const bool inside_ok = cut_inside && ql * want >= total_q && inside > 0 &&
                           inside * qpk > ua::kDefaultDecodeRowsMax &&
                           (ql - inside) * qpk > ua::kDefaultDecodeRowsMax;
    const int64_t cut = inside_ok ? cu[sq] + inside : boundary;
    if (cut > tok.back() && cut < total_q) tok.push_back(cut);
  }
  tok.push_back(total_q);
  const int runs = static_cast<int>(tok.size()) - 1;

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0;
  cudaStream_t lanes[2];
  if (cudaGetDevice(&dev) != cudaSuccess || !host_pipeline_streams(dev, lanes))
    return UA_ERR_CUDA;
  const cudaStream_t compute[2] = {cs, lanes[0]};
  const cudaStream_t s_out = lanes[1];
  // events: [0] buffers allocated, [1 + c] forward of run c done, [1 + runs],
  // [2 + runs] the side streams drained
  std::vector<cudaEvent_t> ev(3 + static_cast<size_t>(runs), nullptr);
  for (cudaEvent_t& e : ev)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
      for (cudaEvent_t x : ev)
        if (x) cudaEventDestroy(x);
      return UA_ERR_CUDA;
    }
  void* dq = nullptr;
  ua_status st = UA_OK;
  if (plan_alloc(&dq, 2 * q_bytes, dev, cs) != cudaSuccess) {
    dq = nullptr;
    st = UA_ERR_CUDA;
  }
  uint8_t* const d_q = static_cast<uint8_t*>(dq);
  uint8_t* const d_out = d_q + q_bytes;
  if (st == UA_OK) {
    st = from_cuda(cudaEventRecord(ev[0], cs));
    for (cudaStream_t x : {compute[1], s_out})
      if (st == UA_OK) st = from_cuda(cudaStreamWaitEvent(x, ev[0], 0));
  }
  std::vector<ua_plan*> plans(static_cast<size_t>(runs), nullptr);
  std::vector<int32_t> cu_run, kv_run;
  for (int c = 0; c < runs && st == UA_OK; ++c) {
    const int64_t t0 = tok[c], t1 = tok[c + 1];
    // sequences s0 .. s0 + n - 1 hold the run's tokens (empty ones between
    // them included, so that their page-table rows stay consecutive)
    const int32_t s0 = static_cast<int32_t>(std::upper_bound(cu, cu + num_seqs + 1, t0) - cu) - 1;
    const int32_t s_last =
        static_cast<int32_t>(std::upper_bound(cu, cu + num_seqs + 1, t1 - 1) - cu) - 1;
    const int32_t n = s_last - s0 + 1;
    const size_t off = static_cast<size_t>(t0) * row_bytes;
    const size_t bytes = static_cast<size_t>(t1 - t0) * row_bytes;
    const cudaStream_t run_stream = compute[c % 2];
    st = from_cuda(cudaMemcpyAsync(d_q + off, static_cast<const uint8_t*>(q_host) + off, bytes,
                                   cudaMemcpyHostToDevice, run_stream));
    if (st != UA_OK) break;
    cu_run.assign(1, 0);
    kv_run.clear();
    for (int32_t i = s0; i <= s_last; ++i) {
      const int64_t a = std::max<int64_t>(t0, cu[i]), b = std::min<int64_t>(t1, cu[i + 1]);
      const int64_t ql = std::max<int64_t>(0, b - a);
      cu_run.push_back(cu_run.back() + static_cast<int32_t>(ql));
      // causal: the keys up to the run's last row of this sequence
      kv_run.push_back(causal != 0 ? static_cast<int32_t>(kv_lens_host[i] - (cu[i + 1] - b))
                                   : kv_lens_host[i]);
    }
    const int32_t* bt = block_tables_host + static_cast<size_t>(s0) * max_blocks_per_seq;
    const HostRange extra[3] = {
        {cu_run.data(), (static_cast<size_t>(n) + 1) * sizeof(int32_t)},
        {kv_run.data(), static_cast<size_t>(n) * sizeof(int32_t)},
        {bt, static_cast<size_t>(n) * static_cast<size_t>(max_blocks_per_seq) * sizeof(int32_t)}};
    void* dev_extra[3] = {nullptr, nullptr, nullptr};
    st = create_plan(&plans[c], cu_run.data(), kv_run.data(), n, num_q_heads, num_kv_heads,
                     head_dim, block_size, max_blocks_per_seq, kv_dtype, causal, window,
                     num_splits, -1, reinterpret_cast<ua_stream_t>(run_stream), extra, 3,
                     dev_extra);
    if (st != UA_OK) break;
    st = ua_forward(plans[c], d_q + off, k_cache, v_cache, d_out + off,
                    static_cast<const int32_t*>(dev_extra[0]),
                    static_cast<const int32_t*>(dev_extra[1]),
                    static_cast<const int32_t*>(dev_extra[2]), num_blocks, plans[c]->sched.max_q,
                    plans[c]->sched.max_kv, scale, k_scale, v_scale,
                    reinterpret_cast<ua_stream_t>(run_stream));
    if (st == UA_OK) st = from_cuda(cudaEventRecord(ev[1 + c], run_stream));
    if (st == UA_OK) st = from_cuda(cudaStreamWaitEvent(s_out, ev[1 + c], 0));
    if (st == UA_OK)
      st = from_cuda(cudaMemcpyAsync(static_cast<uint8_t*>(out_host) + off, d_out + off, bytes,
                                     cudaMemcpyDeviceToHost, s_out));
  }
  // Drain the side streams into `stream` (also after a failure), then free.
  cudaEventRecord(ev[1 + runs], s_out);
  cudaStreamWaitEvent(cs, ev[1 + runs], 0);
  cudaEventRecord(ev[2 + runs], compute[1]);
  cudaStreamWaitEvent(cs, ev[2 + runs], 0);
  if (dq) cudaFreeAsync(dq, cs);
  if (cudaStreamSynchronize(cs) != cudaSuccess && st == UA_OK) st = UA_ERR_CUDA;
  int32_t code = UA_OK;
  for (ua_plan* pl : plans) {
    if (pl == nullptr) continue;
    int32_t v = UA_OK;
    if (st == UA_OK && code == UA_OK &&
        cudaMemcpy(&v, pl->d_err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
      st = UA_ERR_CUDA;
    if (code == UA_OK) code = v;
    ua_plan_destroy(pl);
  }
  if (error_word != nullptr && st == UA_OK) *error_word = code;
  for (cudaEvent_t e : ev) cudaEventDestroy(e);
  return st;
}

}  // namespace

extern "C" {

ua_status ua_plan_create_ex(ua_plan** out, const int32_t* cu_query_lens_host,
                            const int32_t* kv_lens_host, int32_t num_seqs, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int32_t max_blocks_per_seq, int32_t kv_dtype, int32_t causal,
                            int32_t window, int32_t num_splits, int32_t decode_rows_max,
                            ua_stream_t stream) {
  return create_plan(out, cu_query_lens_host, kv_lens_host, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, block_size, max_blocks_per_seq, kv_dtype, causal, window,
                     num_splits, decode_rows_max, stream, nullptr, 0, nullptr);
}

ua_status ua_plan_create(ua_plan** out, const int32_t* cu_query_lens_host,
                         const int32_t* kv_lens_host, int32_t num_seqs, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         int32_t max_blocks_per_seq, int32_t kv_dtype, int32_t causal,
                         int32_t window, int32_t num_splits, ua_stream_t stream) {
  return ua_plan_create_ex(out, cu_query_lens_host, kv_lens_host, num_seqs, num_q_heads,
                           num_kv_heads, head_dim, block_size, max_blocks_per_seq, kv_dtype,
                           causal, window, num_splits, -1, stream);
}

ua_status ua_plan_get_info(const ua_plan* plan, ua_plan_info* info) {
  if (plan == nullptr || info == nullptr) return UA_ERR_INVALID_ARG;
  *info = plan->info;
  return UA_OK;
}

ua_status ua_plan_destroy(ua_plan* plan) {
  if (plan == nullptr) return UA_OK;
  int cur = 0;
  cudaGetDevice(&cur);
  if (cur != plan->device) cudaSetDevice(plan->device);
  free_plan_memory(plan);
  if (cur != plan->device) cudaSetDevice(cur);
  delete plan;
  return UA_OK;
}

ua_status ua_forward(const ua_plan* plan, const void* q, const void* k_cache,
                     const void* v_cache, void* out, const int32_t* cu_query_lens,
                     const int32_t* kv_lens, const int32_t* block_tables, int64_t num_blocks,
                     int32_t max_q, int32_t max_kv, float scale, float k_scale, float v_scale,
                     ua_stream_t stream) {
  if (plan == nullptr) return UA_ERR_INVALID_ARG;
  const ua::Schedule& s = plan->sched;
  const bool any = !s.prefill.empty() || !s.decode.empty();
  if (!any) return UA_OK;
  if (!q || !k_cache || !v_cache || !out || !cu_query_lens || !kv_lens || !block_tables)
    return UA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return UA_ERR_INVALID_ARG;
  if (num_blocks <= 0 || max_q < s.max_q || max_kv < s.max_kv) return UA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return UA_ERR_INVALID_ARG;
  if (plan->prob.kv_dtype == UA_KV_FP8_E4M3 && (!std::isfinite(k_scale) || !std::isfinite(v_scale)))
    return UA_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return UA_ERR_CUDA;
  if (dev != plan->device) return UA_ERR_INVALID_ARG;
  if (num_blocks >= INT32_MAX) return UA_ERR_INVALID_ARG;  // TMA block coordinates are int32

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  ua_plan* mp = const_cast<ua_plan*>(plan);
  mp->last_stream = cs;
  ua::KernelParams kp = base_params(plan, q, k_cache, v_cache, out, cu_query_lens, kv_lens,
                                    block_tables, num_blocks, scale, k_scale, v_scale);
  const bool mixed = !s.prefill.empty() && !s.decode.empty();
  auto run_prefill = [&](cudaStream_t cs) -> ua_status {
    // fp8 cache: either the prefill kernel reads a bf16 staging copy, or (fp8
    // products on) the fp8-products kernel reads the e4m3 cache itself
    const bool f8p = plan->prob.prefill_staged && plan->fp8_products;
    const bool staged = plan->prob.prefill_staged && !f8p;
    const void* pk = k_cache;
    const void* pv = v_cache;
    if (staged) {
      // fp8 cache: widen the prefill sequences' pages into the staging cache
      ua::StageParams sp;
      std::memset(&sp, 0, sizeof(sp));
      sp.k_src = k_cache;
      sp.v_src = v_cache;
      sp.k_dst = plan->d_staged_k;
      sp.v_dst = plan->d_staged_v;
      sp.tiles = plan->d_stage;
      sp.num_tiles = static_cast<int32_t>(s.stage.size());
      sp.block_tables = block_tables;
      sp.max_blocks_per_seq = plan->prob.max_blocks_per_seq;
      sp.block_size = plan->prob.block_size;
      sp.num_blocks = num_blocks;
      sp.row_elems = plan->prob.num_kv_heads * plan->prob.head_dim;
      sp.err = plan->d_err;
      auto* sev = timing_begin(mp, 4, cs);
      if (ua::launch_stage(sp, cs) != cudaSuccess) return UA_ERR_CUDA;
      timing_end(sev, cs);
      pk = plan->d_staged_k;
      pv = plan->d_staged_v;
    }
    ua::PrefillParams pp;
    std::memset(&pp, 0, sizeof(pp));
    pp.tiles = plan->d_prefill;
    pp.num_tiles = static_cast<int32_t>(s.prefill.size());
    pp.q = q;
    pp.counters = plan->d_prefill_counters;
    pp.num_ctas = plan->prefill_ctas_override > 0
                      ? std::min<int32_t>(plan->prefill_ctas_override,
                                          std::min<int32_t>(plan->info.num_sms,
                                                            static_cast<int32_t>(s.prefill.size())))
                      : plan->info.num_prefill_ctas;
    pp.cu_query_lens = cu_query_lens;
    pp.kv_lens = kv_lens;
    pp.block_tables = staged ? plan->d_staged_table : block_tables;
    pp.out = out;
    pp.err = plan->d_err;
    pp.num_blocks = staged ? s.staged_pages : num_blocks;
    pp.max_blocks_per_seq = staged ? s.staged_max_blocks : plan->prob.max_blocks_per_seq;
    pp.block_size = staged ? ua::kStagePage : plan->prob.block_size;
    pp.num_q_heads = plan->prob.num_q_heads;
    pp.qpk = kp.qpk;
    pp.causal = plan->prob.causal;
    pp.window = plan->prob.window;
    pp.score_scale_log2 = kp.score_scale_log2;
    pp.out_scale = kp.v_scale;
    const bool wide = ua::prefill_is_wide(plan->prob.head_dim);
    pp.rows_per_box = wide ? ua::prefill_wide_rows_per_box(pp.block_size)
                           : (pp.block_size < 128 ? pp.block_size : 128);
    pp.timeout_ns = plan->wait_timeout_ns;
    pp.debug_flags = plan->debug_flags;
    // Timing: CUDA events around a kernel that runs alone; in a mixed batch
    // the kernels time themselves (an event between the two launches would
    // hold the decode grid back until the prefill grid ends).
    ua_plan::EventPair* ev = nullptr;
    if (mixed) span_begin(mp, 0, &pp.span_start, &pp.span_end);
    else ev = timing_begin(mp, 0, cs);
    const cudaError_t le =
        f8p  ? ua::launch_prefill_fp8_products(pp, k_cache, v_cache, plan->prob.num_kv_heads, cs)
        : wide ? ua::launch_prefill_wide(pp, q, pk, pv, plan->total_q, plan->prob.head_dim,
                                         plan->prob.num_kv_heads, cs)
               : ua::launch_prefill(pp, q, pk, pv, plan->total_q, plan->prob.head_dim,
                                    plan->prob.num_kv_heads, cs);
    if (le != cudaSuccess) return UA_ERR_CUDA;
    timing_end(ev, cs);
    return UA_OK;
  };
  auto run_decode = [&](cudaStream_t cs, bool after_prefill) -> ua_status {
    kp.tiles = plan->d_decode;
    kp.num_tiles = static_cast<int32_t>(s.decode.size());
    // split pieces are merged inside the decode launch (last piece per group)
    kp.split_counters = s.groups.empty() ? nullptr : plan->d_counters;
    kp.groups = plan->d_groups;
    ua_plan::EventPair* ev = nullptr;
    if (mixed) span_begin(mp, 1, &kp.span_start, &kp.span_end);
    else ev = timing_begin(mp, 1, cs);
    if (ua::launch_decode(kp, plan->prob.head_dim, plan->prob.kv_dtype, cs, after_prefill) !=
        cudaSuccess)
      return UA_ERR_CUDA;
    timing_end(ev, cs);
    return UA_OK;
  };
  if (mixed) {
    // Mixed batch, one stream: every prefill CTA signals at its start that a
    // grid queued behind it with programmatic serialization may launch, so
    // the decode grid starts while the prefill runs -- its CTAs take the SMs
    // the num_prefill_ctas prefill CTAs leave, then the prefill SMs as those
    // CTAs finish. The two grids write disjoint outputs and share only
    // read-only inputs; work queued on `stream` afterwards waits for both.
    const ua_status st_pre = run_prefill(cs);
    if (st_pre != UA_OK) return st_pre;
    return run_decode(cs, true);
  }
  if (!s.prefill.empty()) return run_prefill(cs);
  if (!s.decode.empty()) return run_decode(cs, false);
  return UA_OK;
}

ua_status ua_append_kv(const ua_plan* plan, const void* k_new, const void* v_new, void* k_cache,
                       void* v_cache, const int32_t* block_tables, int64_t num_blocks,
                       float k_scale, float v_scale, ua_stream_t stream) {
  if (plan == nullptr) return UA_ERR_INVALID_ARG;
  if (plan->sched.append.empty()) return UA_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !block_tables) return UA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return UA_ERR_INVALID_ARG;
  if (num_blocks <= 0 || num_blocks >= INT32_MAX) return UA_ERR_INVALID_ARG;
  const bool fp8 = plan->prob.kv_dtype == UA_KV_FP8_E4M3;
  if (fp8 && (!std::isfinite(k_scale) || !std::isfinite(v_scale) || k_scale == 0.f ||
              v_scale == 0.f))
    return UA_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return UA_ERR_CUDA;
  if (dev != plan->device) return UA_ERR_INVALID_ARG;
  ua::AppendParams ap;
  std::memset(&ap, 0, sizeof(ap));
  ap.k_new = k_new;
  ap.v_new = v_new;
  ap.k_cache = k_cache;
  ap.v_cache = v_cache;
  ap.tiles = plan->d_append;
  ap.num_tiles = static_cast<int32_t>(plan->sched.append.size());
  ap.block_tables = block_tables;
  ap.err = plan->d_err;
  ap.num_blocks = num_blocks;
  ap.row_elems = plan->prob.num_kv_heads * plan->prob.head_dim;
  ap.max_blocks_per_seq = plan->prob.max_blocks_per_seq;
  ap.block_size = plan->prob.block_size;
  ap.fp8 = fp8 ? 1 : 0;
  ap.k_scale = k_scale;
  ap.v_scale = v_scale;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  ua_plan* mp = const_cast<ua_plan*>(plan);
  mp->last_stream = cs;
  auto* ev = timing_begin(mp, 3, cs);
  if (ua::launch_append(ap, cs) != cudaSuccess) return UA_ERR_CUDA;
  timing_end(ev, cs);
  return UA_OK;
}

ua_status ua_forward_oneshot(const void* q, const void* k_cache, const void* v_cache, void* out,
                             const int32_t* cu_query_lens_host, const int32_t* kv_lens_host,
                             const int32_t* cu_query_lens, const int32_t* kv_lens,
                             const int32_t* block_tables, int32_t num_seqs,
                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int32_t max_blocks_per_seq,
                             int64_t num_blocks, int32_t kv_dtype, int32_t max_q,
                             int32_t max_kv, float scale, int32_t causal, int32_t window,
                             float k_scale, float v_scale, int32_t num_splits,
                             ua_stream_t stream) {
  ua_plan* plan = nullptr;
  ua_status st = ua_plan_create(&plan, cu_query_lens_host, kv_lens_host, num_seqs, num_q_heads,
                                num_kv_heads, head_dim, block_size, max_blocks_per_seq, kv_dtype,
                                causal, window, num_splits, stream);
  if (st != UA_OK) return st;
  st = ua_forward(plan, q, k_cache, v_cache, out, cu_query_lens, kv_lens, block_tables,
                  num_blocks, max_q, max_kv, scale, k_scale, v_scale, stream);
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess &&
      st == UA_OK)
    st = UA_ERR_CUDA;
  ua_plan_destroy(plan);
  return st;
}

ua_status ua_forward_host(const void* q_host, void* out_host, const int32_t* cu_query_lens_host,
                          const int32_t* kv_lens_host, const int32_t* block_tables_host,
                          const void* k_cache, const void* v_cache, int32_t num_seqs,
                          int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, int32_t max_blocks_per_seq, int64_t num_blocks,
                          int32_t kv_dtype, float scale, int32_t causal, int32_t window,
                          float k_scale, float v_scale, int32_t num_splits,
                          int32_t* error_word, ua_stream_t stream) {
  if (num_seqs < 0 || max_blocks_per_seq < 0 || num_q_heads <= 0 || head_dim <= 0)
    return UA_ERR_INVALID_ARG;
  if (num_seqs > 0 && (!cu_query_lens_host || !kv_lens_host || !block_tables_host))
    return UA_ERR_INVALID_ARG;
  // The query count sizes the q / output buffers, which go first so that
  // the copy of q runs while the host schedules the batch.
  int64_t total_q = 0;
  if (num_seqs > 0) {
    if (cu_query_lens_host[0] != 0) return UA_ERR_INVALID_ARG;
    for (int32_t i = 0; i < num_seqs; ++i)
      if (cu_query_lens_host[i + 1] < cu_query_lens_host[i]) return UA_ERR_INVALID_ARG;
    total_q = cu_query_lens_host[num_seqs];
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const size_t q_bytes =
      static_cast<size_t>(total_q) * static_cast<size_t>(num_q_heads) * head_dim * 2;
  if (q_bytes > 0 && (!q_host || !out_host)) return UA_ERR_INVALID_ARG;
  if (q_bytes >= kHostPipelineMinBytes) {
    // the scheduler validates the rest per run; check the whole batch first
    // so that a bad sequence fails the call before any run starts
    ua::Problem whole = make_problem(cu_query_lens_host, kv_lens_host, num_seqs, num_q_heads,
                                     num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                     kv_dtype, causal, window, num_splits, 152, -1);
    const ua_status vs = ua::validate(whole);
    if (vs != UA_OK) return vs;
    return forward_host_chunked(q_host, out_host, cu_query_lens_host, kv_lens_host,
                                block_tables_host, k_cache, v_cache, num_seqs, num_q_heads,
                                num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                num_blocks, kv_dtype, scale, causal, window, k_scale, v_scale,
                                num_splits, error_word, stream);
  }
  void* dq = nullptr;
  int dev = 0;
  if (q_bytes > 0) {
    if (cudaGetDevice(&dev) != cudaSuccess) return UA_ERR_CUDA;
    if (plan_alloc(&dq, 2 * q_bytes, dev, cs) != cudaSuccess) return UA_ERR_CUDA;
    if (cudaMemcpyAsync(dq, q_host, q_bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess) {
      cudaFreeAsync(dq, cs);
      return UA_ERR_CUDA;
    }
  }
  const HostRange extra[3] = {
      {cu_query_lens_host, (static_cast<size_t>(num_seqs) + 1) * sizeof(int32_t)},
      {kv_lens_host, static_cast<size_t>(num_seqs) * sizeof(int32_t)},
      {block_tables_host,
       static_cast<size_t>(num_seqs) * static_cast<size_t>(max_blocks_per_seq) * sizeof(int32_t)}};
  void* dev_extra[3] = {nullptr, nullptr, nullptr};
  ua_plan* plan = nullptr;
  ua_status st = create_plan(&plan, cu_query_lens_host, kv_lens_host, num_seqs, num_q_heads,
                             num_kv_heads, head_dim, block_size, max_blocks_per_seq, kv_dtype,
                             causal, window, num_splits, -1, stream,
                             num_seqs > 0 ? extra : nullptr, num_seqs > 0 ? 3 : 0, dev_extra);
  if (st != UA_OK) {
    if (dq) cudaFreeAsync(dq, cs);
    return st;
  }
  PinnedBlock word;
  bool have_word = false;
  if (q_bytes > 0) {
    void* dout = static_cast<uint8_t*>(dq) + q_bytes;
    st = ua_forward(plan, dq, k_cache, v_cache, dout, static_cast<const int32_t*>(dev_extra[0]),
                    static_cast<const int32_t*>(dev_extra[1]),
                    static_cast<const int32_t*>(dev_extra[2]), num_blocks, plan->sched.max_q,
                    plan->sched.max_kv, scale, k_scale, v_scale, stream);
    if (st == UA_OK &&
        cudaMemcpyAsync(out_host, dout, q_bytes, cudaMemcpyDeviceToHost, cs) != cudaSuccess)
      st = UA_ERR_CUDA;
    // The error word comes back through a pinned block: a copy into the
    // caller's (usually pageable) word would stage through the driver and
    // hold the host until the forward is done.
    if (st == UA_OK && error_word != nullptr) {
      have_word = pinned_take(sizeof(int32_t), &word);
      if (cudaMemcpyAsync(have_word ? word.ptr : error_word, plan->d_err, sizeof(int32_t),
                          cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        st = UA_ERR_CUDA;
    }
    cudaFreeAsync(dq, cs);
  } else if (error_word != nullptr) {
    *error_word = UA_OK;
  }
  if (cudaStreamSynchronize(cs) != cudaSuccess && st == UA_OK) st = UA_ERR_CUDA;
  if (have_word) {
    if (st == UA_OK) *error_word = *static_cast<const int32_t*>(word.ptr);
    cudaEventRecord(word.done, cs);
    pinned_give_back(word);
  }
  ua_plan_destroy(plan);
  return st;
}

ua_status ua_last_device_error(ua_plan* plan, int32_t* code) {
  if (plan == nullptr || code == nullptr) return UA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(plan->last_stream) != cudaSuccess) return UA_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, plan->d_err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return UA_ERR_CUDA;
  const int32_t zero = 0;
  if (cudaMemcpy(plan->d_err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return UA_ERR_CUDA;
  *code = v;
  return UA_OK;
}

ua_status ua_gather_kv_debug(const ua_plan* plan, const void* k_cache, const void* v_cache,
                             const int32_t* kv_lens, const int32_t* block_tables,
                             int64_t num_blocks, void* k_out, void* v_out, int64_t rows_cap,
                             ua_stream_t stream) {
  if (plan == nullptr || !k_cache || !v_cache || !kv_lens || !block_tables || !k_out || !v_out)
    return UA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_out) || !aligned16(v_out) ||
      num_blocks <= 0)
    return UA_ERR_INVALID_ARG;
  const ua::Schedule& s = plan->sched;
  // Row offsets from the host ranges; the kernel clamps by the device kv_lens,
  // which the caller guarantees equal the plan's.
  std::vector<int64_t> offs(s.decode.size() + 1, 0);
  for (size_t i = 0; i < s.decode.size(); ++i)
    offs[i + 1] = offs[i] + (s.decode[i].kv_hi - s.decode[i].kv_lo);
  if (offs.back() > rows_cap) return UA_ERR_INVALID_ARG;
  if (s.decode.empty()) return UA_OK;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  int64_t* d_offs = nullptr;
  if (cudaMalloc(&d_offs, offs.size() * sizeof(int64_t)) != cudaSuccess) return UA_ERR_CUDA;
  ua_status st = from_cuda(cudaMemcpyAsync(d_offs, offs.data(), offs.size() * sizeof(int64_t),
                                           cudaMemcpyHostToDevice, cs));
  if (st == UA_OK) {
    ua::KernelParams kp = base_params(plan, nullptr, k_cache, v_cache, nullptr, nullptr, kv_lens,
                                      block_tables, num_blocks, 1.f, 1.f, 1.f);
    kp.tiles = plan->d_decode;
    kp.num_tiles = static_cast<int32_t>(s.decode.size());
    const int elt = plan->prob.kv_dtype == UA_KV_FP8_E4M3 ? 1 : 2;
    st = from_cuda(ua::launch_gather_debug(kp, d_offs, plan->prob.head_dim, elt, k_out, v_out, cs));
  }
  if (cudaStreamSynchronize(cs) != cudaSuccess && st == UA_OK) st = UA_ERR_CUDA;
  cudaFree(d_offs);
  return st;
}

ua_status ua_plan_set_profiling(ua_plan* plan, int32_t enable) {
  if (plan == nullptr) return UA_ERR_INVALID_ARG;
  if (enable && plan->d_span == nullptr) {
    void* ptr = nullptr;
    if (plan_alloc(&ptr, 2 * kSpanSlots * sizeof(unsigned long long), plan->device,
                   plan->last_stream) != cudaSuccess)
      return UA_ERR_CUDA;
    plan->d_span = static_cast<unsigned long long*>(ptr);
    if (span_reset(plan, kSpanSlots, plan->last_stream) != cudaSuccess) return UA_ERR_CUDA;
  }
  plan->profiling = enable != 0;
  return UA_OK;
}

ua_status ua_plan_kernel_times(ua_plan* plan, float* ms, int64_t* launches) {
  if (plan == nullptr || ms == nullptr || launches == nullptr) return UA_ERR_INVALID_ARG;
  for (int k = 0; k < UA_KERNEL_KINDS; ++k) {
    ms[k] = 0.f;
    launches[k] = 0;
  }
  if (cudaStreamSynchronize(plan->last_stream) != cudaSuccess) return UA_ERR_CUDA;
  ua_status st = UA_OK;
  for (auto& e : plan->ev_pending) {
    float t = 0.f;
    if (cudaEventElapsedTime(&t, e.start, e.stop) != cudaSuccess) st = UA_ERR_CUDA;
    ms[e.kind] += t;
    launches[e.kind] += 1;
    plan->ev_free.push_back(e);
  }
  plan->ev_pending.clear();
  const int used = static_cast<int>(plan->span_pending.size());
  if (used > 0) {
    std::vector<unsigned long long> t(2 * kSpanSlots);
    if (cudaMemcpy(t.data(), plan->d_span, 2 * kSpanSlots * sizeof(unsigned long long),
                   cudaMemcpyDeviceToHost) != cudaSuccess)
      return UA_ERR_CUDA;
    for (const auto& ks : plan->span_pending) {
      const unsigned long long t0 = t[ks.second], t1 = t[kSpanSlots + ks.second];
      if (t1 >= t0) ms[ks.first] += static_cast<float>(static_cast<double>(t1 - t0) * 1e-6);
      launches[ks.first] += 1;
    }
    plan->span_pending.clear();
    if (span_reset(plan, used, plan->last_stream) != cudaSuccess ||
        cudaStreamSynchronize(plan->last_stream) != cudaSuccess)
      st = UA_ERR_CUDA;
  }
  return st;
}

ua_status ua_plan_set_debug(ua_plan* plan, int32_t flags, int64_t wait_timeout_ns) {
  if (plan == nullptr || flags < 0 || wait_timeout_ns < 0) return UA_ERR_INVALID_ARG;
  plan->debug_flags = flags;
  plan->wait_timeout_ns = wait_timeout_ns > 0 ? static_cast<uint64_t>(wait_timeout_ns)
                                              : 2000000000ull;
  return UA_OK;
}

ua_status ua_plan_set_prefill_ctas(ua_plan* plan, int32_t num_ctas) {
  if (plan == nullptr || num_ctas < 0) return UA_ERR_INVALID_ARG;
  plan->prefill_ctas_override = num_ctas;
  return UA_OK;
}

ua_status ua_plan_set_fp8_products(ua_plan* plan, int32_t enable) {
  if (plan == nullptr || (enable != 0 && enable != 1)) return UA_ERR_INVALID_ARG;
  if (enable) {
    const ua::Problem& pr = plan->prob;
    if (pr.kv_dtype != UA_KV_FP8_E4M3 || !pr.prefill_staged ||
        !ua::prefill_fp8_products_supported(pr.head_dim, pr.num_q_heads / pr.num_kv_heads,
                                            pr.block_size))
      return UA_ERR_UNSUPPORTED;
  }
  plan->fp8_products = enable != 0;
  return UA_OK;
}

ua_status ua_plan_set_unified_max(ua_plan* plan, int32_t enable, float phi) {
  if (plan == nullptr || (enable != 0 && enable != 1)) return UA_ERR_INVALID_ARG;
  if (enable && !(std::fabs(phi) <= 1e30f)) return UA_ERR_INVALID_ARG;  // NaN, inf, huge
  plan->unified_max_on = enable != 0;
  plan->unified_max = enable ? phi : 0.f;
  return UA_OK;
}

}  // extern "C"
