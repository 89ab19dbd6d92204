/*
 * ua.h -- C ABI of the unified paged-KV attention forward for GB300 (sm_103a).
 *
 * What it computes. For every sequence s of a batch, every query token i of s
 * and every query head h, the attention output
 *
 *     out[cu[s]+i, h, :] = softmax_t(scale * <q[cu[s]+i, h, :], k_t>) v_t
 *
 * over the keys t visible to that query, where k_t / v_t are read from a
 * block-paged cache through the sequence's page table. This is the boxed
 * O_{t+1} equation of "flashatten takeaways EP2 工程" (kv cache section) with
 * the tensor layout, page table, GQA grouping and context length of
 * "vllm_triton_unified_attention_notes" (test_triton_unified_attn,
 * unified_attention and kernel_unified_attention_2d sections):
 *
 *   q            [total_q, num_q_heads, head_dim]                 bf16
 *   k/v cache    [num_blocks, block_size, num_kv_heads, head_dim] bf16 or fp8 e4m3
 *                (strides block_size*Hkv*d, Hkv*d, d, 1: all KV heads of one
 *                 (block, slot) are contiguous)
 *   out          [total_q, num_q_heads, head_dim]                 bf16
 *   cu_query_lens[num_seqs+1]  int32, cu[0] = 0, cu[s+1] = cu[s] + q_len(s)
 *   kv_lens      [num_seqs]    int32, kv_len(s) >= q_len(s); it counts the
 *                              new query tokens, whose K/V are already cached
 *   block_tables [num_seqs, max_blocks_per_seq] int32; logical block j of s
 *                lives in physical block block_tables[s*max_blocks_per_seq+j]
 *
 * Visibility: query head h uses KV head h / (Hq/Hkv) (contiguous groups).
 * Query i of s sits at position pos = kv_len(s) - q_len(s) + i; key t is
 * visible iff t < kv_len(s), and (causal == 0 or t <= pos), and
 * (window <= 0 or t > pos - window).
 *
 * fp8 e4m3 caches hold per-tensor scaled values: the key is code * k_scale,
 * the value code * v_scale ("vllm_triton_unified_attention_notes", the load
 * and quantisation branch). k_scale / v_scale are ignored for bf16 caches.
 *
 * Work split. A plan (ua_plan_create) is built on the host from host copies of
 * the lengths: a CPU scheduler turns (sequence, KV head, row block) programs
 * into a flat tile list, cutting long key ranges into split-KV pieces whose
 * partial results are merged by a log-sum-exp combine ("flashatten takeaways
 * EP2 工程", run_flash_splitkv_fwd and its combine kernel; FlashDecoding in
 * the "Fused Attention" notes). It replaces the per-program binary search over
 * the query prefix sums that the vLLM kernel performs at run time.
 *
 * Supported: every head_dim that is a multiple of 32 from 32 to 256 in the
 * decode kernel, which also runs any prefill no prefill kernel takes; a
 * tcgen05 prefill kernel at head_dim 64 and 128 (256-row tiles, 128-key
 * tiles) and one at head_dim 192 and 256 (one 128-row query tile and 64-key
 * tiles at a time, block sizes that 64 divides or that divide 64);
 * block_size a multiple of 16; any GQA ratio (the prefill kernels take ratios
 * dividing 128; sequences they cannot take run in the decode kernel).
 *
 * Conventions.
 *  - The caller owns every tensor argument; the plan owns its device tile list,
 *    per-plan error word, split workspace and, for an fp8 cache with prefill
 *    work, a bf16 staging copy of the pages that work reads (all allocated
 *    stream-ordered from a pool the library keeps per device), and frees them
 *    in ua_plan_destroy.
 *  - Device pointers must be 16-byte aligned and tensors contiguous.
 *  - All device work is ordered on the stream argument (in a mixed batch the
 *    decode grid is launched behind the prefill grid on that stream with
 *    programmatic stream serialization, so that it starts on the SMs the
 *    prefill grid leaves free);
 *    nothing synchronises the host except ua_last_device_error,
 *    ua_plan_kernel_times, ua_forward_oneshot and ua_forward_host.
 *  - No entry point calls exit, abort or a device trap. Invalid arguments are
 *    rejected with a negative status before anything is launched.
 */
#ifndef UA_H
#define UA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-identical to cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* ua_stream_t;

typedef enum {
  UA_OK = 0,
  UA_ERR_INVALID_ARG = -1,   /* bad size, length, pointer or alignment */
  UA_ERR_UNSUPPORTED = -2,   /* valid but not built: head_dim, dtype, block_size */
  UA_ERR_CUDA = -3,          /* a CUDA runtime/driver call failed */
  UA_ERR_WORKSPACE = -4,     /* workspace missing or too small */
  UA_ERR_DEVICE_TIMEOUT = -5,/* a bounded device-side wait gave up (error word) */
  UA_ERR_BOUNDS = -6         /* a page id outside [0, num_blocks) was met (error word) */
} ua_status;

typedef enum { UA_KV_BF16 = 0, UA_KV_FP8_E4M3 = 1 } ua_kv_dtype;

/* One unit of scheduled work, 8 x int32 (32 bytes), shared by the prefill
 * and decode lists. Rows are the packed (token, head) pairs of one KV head:
 * row r of sequence s and KV head g is query token r / qpk and query head
 * g * qpk + r % qpk, qpk = Hq / Hkv (the packed GQA tile of the vLLM kernel). */
typedef struct {
  int32_t seq;      /* sequence index */
  int32_t kv_head;  /* KV head g */
  int32_t row0;     /* first packed row of this tile */
  int32_t nrows;    /* rows in this tile (<= 8 decode, <= 256 prefill) */
  int32_t kv_lo;    /* first key position this tile reads */
  int32_t kv_hi;    /* one past the last key position this tile reads */
  int32_t slot;     /* split workspace slot, or -1: write the output directly */
  int32_t group;    /* combine group of the split, or -1 */
} ua_tile;

/* A combine group: the consecutive workspace slots holding the split partials
 * of one (sequence, KV head, row block). */
typedef struct {
  int32_t seq, kv_head, row0, nrows;
  int32_t slot0;    /* first slot */
  int32_t nsplits;  /* number of consecutive slots, 2..UA_MAX_SPLITS */
  int32_t pad0, pad1;
} ua_combine_group;

#define UA_MAX_SPLITS 128
#define UA_DECODE_ROWS 8     /* rows of one decode tile */
#define UA_PREFILL_ROWS 256  /* rows of one prefill tile: two tcgen05 M=128 query tiles */

typedef struct {
  int64_t num_prefill_tiles;
  int64_t num_decode_tiles;    /* includes every split piece */
  int64_t num_combine_groups;
  int64_t num_slots;           /* split workspace slots */
  int64_t workspace_bytes;     /* bytes of split workspace the plan owns */
  int32_t split_tokens;        /* key tokens per split piece (0: no splits) */
  int32_t num_sms;             /* SM count the schedule was sized for */
  int32_t num_prefill_ctas;    /* CTAs of the persistent prefill launch, one per SM; they take
                                  the prefill tiles in list order. min(num_sms, prefill tiles)
                                  without decode tiles; with decode tiles too, the count that
                                  balances the two kernels (the decode kernel takes the other
                                  SMs while the prefill runs) */
  int32_t reserved;            /* zero */
} ua_plan_info;

typedef struct ua_plan ua_plan;

/*
 * ua_schedule -- the CPU scheduler alone: host memory only, no CUDA call.
 * Validates the problem and writes the tile lists the plan would upload.
 * Call once with NULL arrays to read the counts into *info, then again with
 * arrays of at least those lengths (the *_cap arguments give their lengths in
 * elements; too small a capacity returns UA_ERR_INVALID_ARG).
 * num_splits: 0 = automatic, n > 0 = cut every decode tile's key range into
 * min(n, ceil(len/16)) pieces; at most UA_MAX_SPLITS. Automatic: pieces of
 * about one CTA slot's average load (tiles of nearly one length: unsplit
 * when a bf16 batch of 256 or more tiles fills one wave of slots, else the
 * cut that fills whole waves); a batch left unsplit that overfills one wave
 * by at most half a wave cuts the tiles that start last into pieces of at
 * least 256 keys (tail pieces), so that they fill the slots the first wave
 * frees. num_sms <= 0 means 152.
 * decode_rows_max: sequences with q_len * qpk <= this value go to the decode
 * kernel, the others to a prefill kernel (when one takes the problem:
 * head_dim 64, 128, 192 or 256, 128 % qpk == 0, and a bf16 cache whose
 * block_size and the key tile (128 keys at head dim 64 / 128, 64 at head dim
 * 192 / 256) divide one another, or any fp8 cache); < 0 means the built-in
 * default (32).
 * The prefill list is in the order the persistent prefill CTAs take it
 * (grouped by sequence and KV head, the shortest tiles last); the decode list
 * is longest first.
 */
ua_status ua_schedule(const int32_t* cu_query_lens_host, const int32_t* kv_lens_host,
                      int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq,
                      int32_t kv_dtype, int32_t causal, int32_t window, int32_t num_splits,
                      int32_t num_sms, int32_t decode_rows_max, ua_plan_info* info,
                      ua_tile* prefill_tiles, int64_t prefill_cap,
                      ua_tile* decode_tiles, int64_t decode_cap,
                      ua_combine_group* groups, int64_t groups_cap);

/*
 * ua_plan_create -- the CPU work scheduler of the forward. It replaces the
 * run-time search for each program's sequence over the query prefix sums
 * (find_seq_idx) and the grid sizing of the host wrapper in
 * "vllm_triton_unified_attention_notes" (unified_attention section), and
 * picks the split-KV piece count that run_flash_splitkv_fwd chooses per
 * launch in "flashatten takeaways EP2 工程" (split-KV launcher section).
 * Runs the scheduler for the current CUDA device and uploads
 * the tile lists with one stream-ordered copy (from a pinned block the
 * library recycles, so the host does not wait for earlier work on `stream`);
 * allocates the plan's device memory (tile lists, error word, split
 * workspace, fp8 prefill staging) stream-ordered from the library's pool.
 * Arguments as ua_schedule; num_sms is queried from the device.
 * Returns UA_ERR_INVALID_ARG / UA_ERR_UNSUPPORTED for a rejected problem,
 * UA_ERR_CUDA when an allocation or copy fails (nothing is leaked).
 */
ua_status ua_plan_create(ua_plan** out, const int32_t* cu_query_lens_host,
                         const int32_t* kv_lens_host, int32_t num_seqs, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         int32_t max_blocks_per_seq, int32_t kv_dtype, int32_t causal,
                         int32_t window, int32_t num_splits, ua_stream_t stream);

/* Same with an explicit decode/prefill row threshold (see ua_schedule). */
ua_status ua_plan_create_ex(ua_plan** out, const int32_t* cu_query_lens_host,
                            const int32_t* kv_lens_host, int32_t num_seqs, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int32_t max_blocks_per_seq, int32_t kv_dtype, int32_t causal,
                            int32_t window, int32_t num_splits, int32_t decode_rows_max,
                            ua_stream_t stream);

/*
 * ua_forward -- attention for the batch the plan was built for: the boxed
 * O_{t+1} = softmax(q K^T) V equation of "flashatten takeaways EP2 工程" (kv
 * cache section) over the paged cache, evaluated tile by tile as
 * kernel_unified_attention_2d does in "vllm_triton_unified_attention_notes"
 * (Q tile load, paged K/V load through the block table, causal mask against
 * the context length, online softmax with running max and sum), with the
 * online-softmax recurrence of _attn_fwd_inner ("Fused Attention" notes) and
 * the split-KV log-sum-exp combine (FlashDecoding, same notes).
 * q, k_cache, v_cache, out: device tensors in the layouts above.
 * cu_query_lens, kv_lens, block_tables: device copies. cu_query_lens and
 * kv_lens must hold the values given to the plan; the kernels read them for
 * each tile's query offset and masking and clamp every key range by
 * kv_lens[seq], and the page index by max_blocks_per_seq.
 * num_blocks: physical blocks in each cache; a page id outside
 * [0, num_blocks) is never dereferenced: the page is treated as masked and
 * UA_ERR_BOUNDS is recorded in the plan's error word.
 * max_q / max_kv: the largest q_len / kv_len (checked against the plan).
 * scale: multiplies q.k as given (not assumed to be 1/sqrt(d)).
 * Launches the prefill kernel (after the staging kernel for an fp8 cache)
 * and the decode kernel (which merges split pieces itself) in the order of
 * `stream`: when the batch has both, the decode grid follows the prefill grid
 * on `stream` as a programmatic dependent launch that may start once every
 * prefill CTA has begun (so after everything queued on `stream` before the
 * call): the prefill CTAs hold num_prefill_ctas SMs and the decode CTAs
 * stream the cache on the others, then on the prefill SMs as they free up.
 * Work queued on `stream` afterwards sees the whole result. Not thread-safe per plan:
 * calls that share a plan must be ordered (they share its split workspace).
 */
ua_status ua_forward(const ua_plan* plan, const void* q, const void* k_cache,
                     const void* v_cache, void* out, const int32_t* cu_query_lens,
                     const int32_t* kv_lens, const int32_t* block_tables, int64_t num_blocks,
                     int32_t max_q, int32_t max_kv, float scale, float k_scale, float v_scale,
                     ua_stream_t stream);

/*
 * ua_forward_oneshot -- the whole call in one: host copies of the lengths
 * (for the scheduler) plus the device tensors; builds a transient plan,
 * runs ua_forward, and frees the plan after the stream has drained it.
 * Synchronises `stream` before returning.
 */
ua_status ua_forward_oneshot(const void* q, const void* k_cache, const void* v_cache, void* out,
                             const int32_t* cu_query_lens_host, const int32_t* kv_lens_host,
                             const int32_t* cu_query_lens, const int32_t* kv_lens,
                             const int32_t* block_tables, int32_t num_seqs,
                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int32_t max_blocks_per_seq,
                             int64_t num_blocks, int32_t kv_dtype, int32_t max_q,
                             int32_t max_kv, float scale, int32_t causal, int32_t window,
                             float k_scale, float v_scale, int32_t num_splits,
                             ua_stream_t stream);

/*
 * ua_forward_host -- one serving step from host buffers: the whole of
 * ua_forward_oneshot, with the queries, output, lengths and page tables in
 * host memory and the paged K/V cache resident on the device. Schedules the
 * batch, uploads the tile list together with the lengths and page tables in
 * one copy, copies q to the device, runs the forward, copies the output
 * back, and synchronises `stream` before returning.
 * From 32 MiB of q the copies would take about as long
 * as the forward, so the query tokens are cut into runs of about 16 MiB of
 * q (2 to 4 runs), each scheduled on its own. A cut falls on the first
 * sequence boundary at or after its target; but inside a sequence at least
 * a run long, with a causal mask or with neither mask nor window (on a
 * whole prefill tile, both parts still prefill-sized): rows [a, b) of a
 * sequence with context ctx run as a sequence of b - a tokens with ctx + b
 * keys (causal) or all kv_len keys (no mask). The runs alternate between `stream` and an internal compute
 * stream (each run: copy of its q, plan upload, forward), so that one run's
 * q copy overlaps the previous run's forward, and each output comes back on
 * an internal copy stream while later runs compute. Prefill rows are
 * bit-identical either way; decode rows may differ in rounding, since their
 * split-KV pieces are chosen per run. The whole batch is validated before
 * the first run starts.
 * q_host, out_host: [total_q, num_q_heads, head_dim] bf16 in host memory
 *   (page-locked memory, e.g. cudaHostAlloc, gives asynchronous copies;
 *   pageable memory works, its copies synchronise).
 * cu_query_lens_host [num_seqs+1], kv_lens_host [num_seqs],
 * block_tables_host [num_seqs, max_blocks_per_seq]: host int32, as for
 *   ua_forward.
 * k_cache, v_cache: device caches, as for ua_forward.
 * error_word: optional host int32 that receives the call's device error
 *   word (UA_OK, UA_ERR_BOUNDS or UA_ERR_DEVICE_TIMEOUT); may be NULL.
 * Device memory for the plan, q and the output comes from the library's
 * stream-ordered pool and is returned to it before the call returns.
 * Returns as ua_plan_create and ua_forward.
 */
ua_status ua_forward_host(const void* q_host, void* out_host, const int32_t* cu_query_lens_host,
                          const int32_t* kv_lens_host, const int32_t* block_tables_host,
                          const void* k_cache, const void* v_cache, int32_t num_seqs,
                          int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, int32_t max_blocks_per_seq, int64_t num_blocks,
                          int32_t kv_dtype, float scale, int32_t causal, int32_t window,
                          float k_scale, float v_scale, int32_t num_splits,
                          int32_t* error_word, ua_stream_t stream);

/*
 * ua_append_kv -- write a step's new keys and values into the paged cache
 * (the Append_KV path of the split-KV launcher in "flashatten takeaways EP2
 * 工程"), before ua_forward reads them. For sequence s of the plan and new
 * token i < q_len_s (row cu_query_lens[s] + i of k_new / v_new), logical
 * position pos = kv_len_s - q_len_s + i is written at block
 * block_tables[s][pos / block_size], slot pos % block_size, all KV heads.
 * The positions come from the lengths the plan was built with (one tile of
 * up to 8 new tokens per CTA, listed by the plan).
 * k_new, v_new: device [total_q, num_kv_heads, head_dim] bf16 (the plan's
 *   total_q = cu_query_lens_host[num_seqs]), contiguous, 16-byte aligned.
 * k_cache, v_cache: the caches of ua_forward (written in place).
 * block_tables: the device page table (as for ua_forward).
 * fp8 (e4m3) cache: code = e4m3(x / k_scale) (v_scale for V), the quotient
 *   in binary32, rounded to nearest even, saturating at +-448, NaN stays NaN;
 *   the scales must be finite and non-zero. bf16 cache: a copy (scales
 *   ignored).
 * A page id outside [0, num_blocks) (or a position past the page table) is
 * not written; UA_ERR_BOUNDS is recorded in the plan's error word.
 * Stream-ordered on `stream`; issue it before ua_forward on the same stream.
 * Returns UA_ERR_INVALID_ARG for null or misaligned pointers, a bad
 * num_blocks or scale, or a stream on another device than the plan's.
 */
ua_status ua_append_kv(const ua_plan* plan, const void* k_new, const void* v_new, void* k_cache,
                       void* v_cache, const int32_t* block_tables, int64_t num_blocks,
                       float k_scale, float v_scale, ua_stream_t stream);

/* Counts and sizes of a plan (host memory only). */
ua_status ua_plan_get_info(const ua_plan* plan, ua_plan_info* info);

/* Kernel timing for measurement tools. While enabled, ua_forward and
 * ua_append_kv record a CUDA event pair on their stream around each kernel
 * launch (a few microseconds per launch). The exception is a batch with both
 * prefill and decode tiles, whose two kernels overlap: there each of the two
 * records its own span instead (first CTA start to last CTA end, device
 * global timer), so that no event sits between the launches.
 * ua_plan_kernel_times synchronises, sums the elapsed milliseconds and launch
 * counts per kernel kind since the last read -- index 0 prefill, 1 decode,
 * 2 combine, 3 append, 4 fp8 prefill staging -- into ms[0..UA_KERNEL_KINDS-1]
 * / launches[0..UA_KERNEL_KINDS-1], and clears them. Up to 1024 self-timed
 * launches are kept between reads; later ones are not counted. */
#define UA_KERNEL_KINDS 5
ua_status ua_plan_set_profiling(ua_plan* plan, int32_t enable);
ua_status ua_plan_kernel_times(ua_plan* plan, float* ms, int64_t* launches);

/* Test aid for the device-side failure path. flags bit 0 makes the prefill
 * kernel's TMA producer issue nothing, so its consumers' bounded waits run
 * out: the kernel records UA_ERR_DEVICE_TIMEOUT in the error word, drains
 * and frees what it holds, and exits (the output of the affected tiles is
 * undefined). wait_timeout_ns bounds every device-side wait (0: 2 s default).
 * Both apply to later ua_forward calls on this plan. */
ua_status ua_plan_set_debug(ua_plan* plan, int32_t flags, int64_t wait_timeout_ns);

/* Unified max for decode work (FlashDecoding++, "Fused Attention" notes:
 * a preset value stands in for each row's maximum, with a fallback when the
 * scores leave its range). With enable = 1, every row the decode kernel
 * processes starts from phi -- in units of the scaled score scale * q.k
 * (times k_scale for an e4m3 cache), the argument of softmax's exp -- as the
 * value subtracted before exponentiation, instead of the maximum of its first
 * keys. Fallback: when the first visible keys' maximum m lies outside
 * [phi - 64 / log2(e), phi + 8 / log2(e)] (bf16 cache) or
 * [phi, phi + 8 / log2(e)] (e4m3 cache, whose P operand is f16), or later
 * keys exceed the reference by more than 8 / log2(e), the row uses its
 * running maximum, as with enable = 0. The result is the same softmax up to
 * rounding either way; phi only moves where the rescales happen. Prefill
 * tiles keep the running maximum. enable = 0 restores the default.
 * phi must be finite (|phi| <= 1e30); applies to later ua_forward calls. */
ua_status ua_plan_set_unified_max(ua_plan* plan, int32_t enable, float phi);

/* Tuning aid: run the prefill kernel of later ua_forward calls on this plan
 * with num_ctas persistent CTAs (capped at the SM count and the prefill tile
 * count) instead of the scheduler's num_prefill_ctas; 0 restores it. Results
 * do not depend on it. */
ua_status ua_plan_set_prefill_ctas(ua_plan* plan, int32_t num_ctas);

/* fp8 tensor-core products for the prefill tiles of an fp8 (e4m3) cache:
 * the low-precision path of the "Fused Attention" notes (Q.K^T on fp8
 * operands, P cast to fp8 ahead of P.V; the block-quantised FP8 path of
 * their FlashAttention-3 summary). With enable = 1, later ua_forward calls
 * run the prefill tiles in a kernel that reads the e4m3 cache directly (no
 * bf16 staging copy): each query row is quantised to e4m3 with its own scale
 * (448 / max |q|, binary32), S = Q K^T and O += P V are kind::f8f6f4 MMAs,
 * and P (exp relative to the row's running max, <= 1) is rounded to e4m3,
 * while l sums the unrounded P. Accuracy is that of the fp8 operands
 * (about 2^-4 relative per element) rather than of the exact dequantised
 * cache; decode tiles keep their f16 products. enable = 0 restores the
 * staged path. Returns UA_ERR_UNSUPPORTED unless the plan has an e4m3 cache,
 * head_dim 128, 128 % qpk == 0 and a block size that divides or is divided
 * by 128 (and at least 16); UA_ERR_INVALID_ARG for a null plan or an enable
 * other than 0 / 1. */
ua_status ua_plan_set_fp8_products(ua_plan* plan, int32_t enable);

/* Synchronises the plan's last stream, reads the device error word
 * (UA_OK, UA_ERR_BOUNDS or UA_ERR_DEVICE_TIMEOUT) into *code and clears it. */
ua_status ua_last_device_error(ua_plan* plan, int32_t* code);

/* Frees the plan. Its device memory is released stream-ordered on the last
 * stream the plan was used on (no host synchronisation): work already queued
 * there may still use it, later work must not. */
ua_status ua_plan_destroy(ua_plan* plan);

/* Static string for a status code (never NULL). */
const char* ua_status_string(int32_t status);

/*
 * ua_gather_kv_debug -- test aid for bit-exact index checks. For every decode
 * tile of the plan, in order, copies the raw K and V rows of its key range
 * [kv_lo, kv_hi) (clamped by kv_lens[seq]) for its KV head into k_out/v_out,
 * packed tile after tile, rows of head_dim elements of the cache's element
 * size. The row offset of tile n is the sum of the clamped range lengths of
 * tiles 0..n-1. Page ids are resolved exactly as in ua_forward. The outputs
 * must hold `rows_cap` rows.
 */
ua_status ua_gather_kv_debug(const ua_plan* plan, const void* k_cache, const void* v_cache,
                             const int32_t* kv_lens, const int32_t* block_tables,
                             int64_t num_blocks, void* k_out, void* v_out, int64_t rows_cap,
                             ua_stream_t stream);

/*
 * ua_forward_static_scratch -- the same attention for callers that cannot
 * allocate device memory. The pages describe no such entry point; it exists
 * for code that runs inside another runtime owning every device allocation
 * (its own memory pool, a plugin host), or in loops where cudaMalloc, which
 * can synchronise the whole device, is not acceptable.
 *
 * It allocates nothing: the tile list, combine groups, split partials and
 * error word live in one static device array of 16 MiB inside libua.so,
 * which every GPU that loads the library keeps until the process exits. The
 * tile list is built on the device from the device copies of the lengths
 * (one tile per sequence, KV head, block of 8 packed rows and split), and every
 * sequence runs through the split-KV decode kernel and the combine kernel.
 *
 * Meant for decode-shaped batches (small max_q): the tile grid gives every
 * sequence ceil(max_q * Hq / Hkv / 8) row blocks, so one long query in the
 * batch makes every sequence launch that many (mostly empty) decode CTAs;
 * mixed batches with long prefills belong on ua_forward.
 *
 * Arguments as ua_forward_oneshot, without host lengths: max_q / max_kv must
 * bound every q_len / kv_len (max_q sizes the tile grid); num_splits 0 picks
 * ceil(max_kv / 1024) pieces (at most UA_MAX_SPLITS, fewer if needed to fit),
 * n > 0 uses exactly n. scale must be finite; for an e4m3 cache k_scale and
 * v_scale must be finite and non-zero (else UA_ERR_INVALID_ARG, nothing
 * launched). device_error: optional device int32 that receives the call's
 * error word; may be NULL. The word is UA_OK, or UA_ERR_BOUNDS (a page id
 * outside [0, num_blocks)), UA_ERR_DEVICE_TIMEOUT (a bounded wait of the
 * decode kernel gave up) or UA_ERR_INVALID_ARG (the device lengths break the
 * call's bounds: q_len above max_q, kv_len below q_len, or kv_len beyond
 * max_blocks_per_seq * block_size); the output of the affected rows is then
 * undefined.
 * Returns UA_ERR_WORKSPACE when the call's scratch (32 B per tile and per
 * group, plus 8 * (head_dim + 1) * 4 B per tile when split) exceeds 16 MiB;
 * nothing is launched then.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. Every call shares the one array and leaves its
 * contents behind: calls whose work overlaps on the GPU (different streams,
 * or different host threads) race on it and must be ordered by the caller.
 */
ua_status ua_forward_static_scratch(const void* q, const void* k_cache, const void* v_cache,
                                    void* out, const int32_t* cu_query_lens,
                                    const int32_t* kv_lens, const int32_t* block_tables,
                                    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t block_size,
                                    int32_t max_blocks_per_seq, int64_t num_blocks,
                                    int32_t kv_dtype, int32_t max_q, int32_t max_kv, float scale,
                                    int32_t causal, int32_t window, float k_scale, float v_scale,
                                    int32_t num_splits, int32_t* device_error,
                                    ua_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* UA_H */
