// Host-side work scheduler for the unified paged-KV attention forward.
//
// Replaces the per-program binary search over the query prefix sums and the
// "2D or 3D kernel" choice of the vLLM Triton kernel
// ("vllm_triton_unified_attention_notes", find_seq_idx and the unified_attention
// host wrapper) with a precomputed, flat tile list built once per batch on the
// CPU from host copies of the lengths.
#pragma once

#include <cstdint>
#include <climits>
#include <vector>

#include "../../include/ua.h"

namespace ua {

struct Problem {
  const int32_t* cu_query_lens = nullptr;  // host [num_seqs + 1]
  const int32_t* kv_lens = nullptr;        // host [num_seqs]
  int32_t num_seqs = 0;
  int32_t num_q_heads = 0;
  int32_t num_kv_heads = 0;
  int32_t head_dim = 0;
  int32_t block_size = 0;
  int32_t max_blocks_per_seq = 0;
  int32_t kv_dtype = UA_KV_BF16;
  int32_t causal = 1;
  int32_t window = 0;
  int32_t num_splits = 0;       // 0: automatic
  int32_t num_sms = 152;
  int32_t decode_rows_max = -1; // < 0: default
  bool prefill_ok = false;      // the prefill kernel can take this problem
  bool prefill_staged = false;  // fp8 cache: the prefill kernel reads a bf16 staging copy
};

struct Schedule {
  // Prefill tiles in the order the persistent prefill CTAs take them.
  std::vector<ua_tile> prefill;
  // Persistent prefill CTAs (one per SM). Without decode work: min(SMs,
  // prefill tiles). With decode work too, fewer, so that the decode kernel
  // streams the cache on the other SMs while the prefill runs (see
  // mixed_prefill_ctas).
  int32_t prefill_ctas = 0;
  int64_t prefill_blocks = 0;   // prefill work in 128 x 128 (query row, key) blocks
  int64_t decode_bytes = 0;     // K/V bytes the decode tiles read
  std::vector<ua_tile> decode;
  // fp8 caches: the keys and values the prefill tiles read are first widened
  // to bf16 into a staging cache of kStagePage-slot pages (a sequence's pages
  // consecutive), which the prefill kernel reads through staged_table
  // [num_seqs][staged_max_blocks] (-1: no page). One stage tile per page:
  // seq, row0 = staging page, nrows = logical page index, [kv_lo, kv_hi) =
  // the keys it holds.
  std::vector<int32_t> staged_table;
  std::vector<ua_tile> stage;
  int32_t staged_max_blocks = 0;
  int64_t staged_pages = 0;
  // Append-KV tiles: up to kAppendTokens consecutive new tokens of one
  // sequence: seq, row0 = first token (row of k_new), nrows = tokens,
  // kv_lo = logical cache position of the first token, kv_hi = kv_lo + nrows.
  std::vector<ua_tile> append;
  std::vector<ua_combine_group> groups;
  int64_t num_slots = 0;
  int32_t split_tokens = 0;
  int32_t max_q = 0;
  int32_t max_kv = 0;
};

// Granularity of key ranges: one decode step reads 16 tokens, so split pieces
// and decode ranges start on multiples of 16.
constexpr int kKeyStep = 16;
// Decode kernel geometry, shared by the kernel and the scheduler. Each of
// the four warps of a CTA owns a ring of TMA stages, one stage holding the K
// and V rows of one 16-key step: 16 KB of ring per warp where that gives 2 to
// 8 stages, two stages at the widest heads.
constexpr int kDecodeWarps = 4;
constexpr int decode_stage_bytes(int head_dim, int elt_bytes) {
  return 2 * kKeyStep * head_dim * elt_bytes;
}
constexpr int decode_ring_stages(int head_dim, int elt_bytes) {
  return 16384 / decode_stage_bytes(head_dim, elt_bytes) < 2
             ? 2
             : (16384 / decode_stage_bytes(head_dim, elt_bytes) > 8
                    ? 8
                    : 16384 / decode_stage_bytes(head_dim, elt_bytes));
}
// Dynamic shared memory of one CTA: the rings, one mbarrier per stage, 16
// bytes of flags and 1 KB of slack for the 1024-byte alignment of the
// swizzle atoms.
constexpr int decode_smem_bytes(int head_dim, int elt_bytes) {
  return kDecodeWarps * decode_ring_stages(head_dim, elt_bytes) *
             (decode_stage_bytes(head_dim, elt_bytes) + 8) +
         16 + 1024;
}
// Resident decode CTAs per SM: as many as the 228 KB of shared memory of an
// SM hold (1 KB of it reserved per CTA), at most three (the register budget
// of 128-thread CTAs up to head_dim 128) and at most two above head_dim 128.
// The kernel is compiled for this many CTAs per SM; the scheduler sizes
// automatic splits with it (pieces of about the average load of one CTA slot
// in a single wave, so that long sequences are cut and short ones not).
constexpr int decode_ctas_per_sm(int head_dim, int elt_bytes = 2) {
  return (233472 / (decode_smem_bytes(head_dim, elt_bytes) + 1024)) < (head_dim > 128 ? 2 : 3)
             ? 233472 / (decode_smem_bytes(head_dim, elt_bytes) + 1024)
             : (head_dim > 128 ? 2 : 3);
}
static_assert(decode_ctas_per_sm(128) == 3 && decode_ctas_per_sm(256) == 1 &&
                  decode_ctas_per_sm(256, 1) == 2 && decode_ctas_per_sm(192) == 2 &&
                  decode_ctas_per_sm(224) == 1 && decode_ctas_per_sm(32) == 3,
              "decode residency");
// Cost of one split piece beyond its keys (CTA start, ring fill, merge and
// store), in key tokens: used when automatic splits are fitted to whole waves.
constexpr int kPieceOverheadTokens = 128;
// bf16 decode CTAs (head_dim >= 128) that keep HBM busy by themselves: each
// keeps 64 KB or more of K/V in flight, and 256 unsplit tiles of 8192 keys
// (one per CTA, 1.7 per SM) stream at 0.99 of the copy peak, while cutting
// them into waves of 456 pieces loses 10 % to the extra pieces and the wave
// tails. Uniform batches with at least this many tiles in one wave stay
// unsplit.
constexpr int kDecodeSaturatingCtas = 256;
// Smallest automatic split piece, in key tokens.
constexpr int kMinSplitTokens = 256;
// Default: sequences with q_len * qpk above this go to the prefill kernel
// (when it can take the problem; otherwise every sequence is decode work).
constexpr int kDefaultDecodeRowsMax = 32;
// Key tile of the prefill kernel: its key ranges start on multiples of this.
constexpr int kPrefillKeyTile = 128;
// Rows of one tcgen05 query tile of the prefill kernel (two per prefill tile).
constexpr int kPrefillQueryTile = 128;
// Slots per page of the bf16 staging cache of fp8 prefills.
constexpr int kStagePage = 128;
// New tokens per append tile (one warp each in the append kernel).
constexpr int kAppendTokens = 8;
// Share of the prefill work (in 128 x 128 query-key blocks) kept for the end
// of the prefill list: the shortest tiles, so that the CTAs finish together.
constexpr double kPrefillTailShare = 1.0 / 16.0;

// Mixed batches: the prefill kernel takes one whole SM per CTA (its shared
// memory excludes decode CTAs there), the decode kernel the SMs it leaves.
// With P prefill CTAs the prefill part takes about blocks * t_block / P, the
// decode part streams at min(HBM, (SMs - P) * per-SM rate) meanwhile and at
// the full HBM rate once the prefill SMs free up; P minimises the modelled
// step time. Constants measured on GB300 (bf16, head_dim 128): one 128 x 128
// block of one query tile costs about 1.3 us of one SM; decode streams about
// 6.5 bytes/ns from HBM in all and at most kDecodeSmBytesPerNs per SM.
constexpr double kPrefillBlockNs = 1300.0;
constexpr double kDecodeHbmBytesPerNs = 6500.0;
constexpr double kDecodeSmBytesPerNs = 90.0;
int32_t mixed_prefill_ctas(int64_t prefill_blocks, int64_t decode_bytes, int64_t prefill_tiles,
                           int num_sms, int head_dim);

// Validate the problem (host arrays included).
ua_status validate(const Problem& p);

// Validate and build the schedule.
ua_status build_schedule(const Problem& p, Schedule* out);

// Workspace bytes for a schedule: per slot, UA_DECODE_ROWS rows of head_dim
// fp32 partial outputs plus UA_DECODE_ROWS fp32 log-sum-exp values.
int64_t workspace_bytes(const Schedule& s, int head_dim);

}  // namespace ua
