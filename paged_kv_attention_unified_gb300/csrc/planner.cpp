// Host-side work scheduler (see planner.h).
#include "planner.h"

#include <algorithm>
#include <climits>
#include <functional>

namespace ua {

namespace {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
inline int64_t round_down(int64_t a, int64_t b) { return (a / b) * b; }

// Key range [lo, hi) read by the packed rows [row0, row0 + nrows) of one
// sequence. Query token i = row / qpk sits at pos = ctx + i; with a causal
// mask it sees keys up to pos, with a window only keys above pos - window.
// lo is rounded down to the 16-token step; the kernels mask what lies below
// the true bound.
void key_range(const Problem& p, int32_t ctx, int32_t kv_len, int32_t row0, int32_t nrows,
               int32_t* lo, int32_t* hi) {
  const int qpk = p.num_q_heads / p.num_kv_heads;
  const int64_t min_pos = ctx + row0 / qpk;
  const int64_t max_pos = ctx + (row0 + nrows - 1) / qpk;
  int64_t h = p.causal ? std::min<int64_t>(kv_len, max_pos + 1) : kv_len;
  int64_t l = 0;
  if (p.window > 0) l = std::max<int64_t>(0, min_pos - p.window + 1);
  l = round_down(l, kKeyStep);
  if (h < l) h = l;
  *lo = static_cast<int32_t>(l);
  *hi = static_cast<int32_t>(h);
}

// Piece length for decode tiles of (nearly) one key length L: with pieces of
// about the average slot load, T tiles cut into k pieces each would leave a
// short last wave (T * k just above a multiple of the CTA slots: e.g. 64
// tiles of 131072 keys in 8 pieces are 512 CTAs on 456 slots, the last 56
// holding only 12 % of a tile). Equal pieces run in waves, so the step takes
// about ceil(T * k / slots) * (L / k + overhead); the k that minimises this
// (the fewest pieces on a tie) sets the length.
int64_t wave_fit_chunk(int64_t tiles, int64_t len, int64_t slots) {
  const int64_t k_max = std::min<int64_t>(UA_MAX_SPLITS, std::max<int64_t>(1, len / kMinSplitTokens));
  int64_t best_size = len, best_cost = INT64_MAX;
  for (int64_t k = 1; k <= k_max; ++k) {
    const int64_t size = round_up(ceil_div(len, k), kKeyStep);
    const int64_t pieces = ceil_div(len, size);
    const int64_t cost = ceil_div(tiles * pieces, slots) * (size + kPieceOverheadTokens);
    if (cost < best_cost) {
      best_cost = cost;
      best_size = size;
    }
  }
  return best_size;
}

// Work of a tile: keys read x packed rows.
inline int64_t work_of(const ua_tile& t) {
  return static_cast<int64_t>(t.kv_hi - t.kv_lo) * t.nrows;
}

// Indices 0..n-1 ordered by the keys (a, b, c) ascending, ties by index: a
// stable sort on precomputed keys (the lists are generated in (sequence, KV
// head, row, key) order, so the index is the documented final tie-break).
struct SortKey {
  int64_t a, b, c;
  int32_t idx;
};

std::vector<int32_t> order_by(std::vector<SortKey>& keys) {
  std::sort(keys.begin(), keys.end(), [](const SortKey& x, const SortKey& y) {
    if (x.a != y.a) return x.a < y.a;
    if (x.b != y.b) return x.b < y.b;
    if (x.c != y.c) return x.c < y.c;
    return x.idx < y.idx;
  });
  std::vector<int32_t> order(keys.size());
  for (size_t i = 0; i < keys.size(); ++i) order[i] = keys[i].idx;
  return order;
}

template <typename T>
void permute(std::vector<T>& v, const std::vector<int32_t>& order) {
  std::vector<T> out;
  out.reserve(v.size());
  for (int32_t i : order) out.push_back(v[static_cast<size_t>(i)]);
  v.swap(out);
}

}  // namespace

ua_status validate(const Problem& p) {
  if (p.num_seqs < 0 || p.num_q_heads <= 0 || p.num_kv_heads <= 0 || p.head_dim <= 0 ||
      p.block_size <= 0 || p.max_blocks_per_seq < 0)
    return UA_ERR_INVALID_ARG;
  if (p.num_q_heads % p.num_kv_heads != 0) return UA_ERR_INVALID_ARG;
  if (p.kv_dtype != UA_KV_BF16 && p.kv_dtype != UA_KV_FP8_E4M3) return UA_ERR_INVALID_ARG;
  if (p.num_splits < 0 || p.num_splits > UA_MAX_SPLITS) return UA_ERR_INVALID_ARG;
  if (p.causal != 0 && p.causal != 1) return UA_ERR_INVALID_ARG;
  if (p.num_seqs > 0 && (p.cu_query_lens == nullptr || p.kv_lens == nullptr))
    return UA_ERR_INVALID_ARG;
  if (p.head_dim < 32 || p.head_dim > 256 || p.head_dim % 32 != 0) return UA_ERR_UNSUPPORTED;
  if (p.block_size % kKeyStep != 0) return UA_ERR_UNSUPPORTED;
  if (p.num_seqs == 0) return UA_OK;
  if (p.cu_query_lens[0] != 0) return UA_ERR_INVALID_ARG;
  const int64_t qpk = p.num_q_heads / p.num_kv_heads;
  for (int s = 0; s < p.num_seqs; ++s) {
    const int64_t q0 = p.cu_query_lens[s], q1 = p.cu_query_lens[s + 1];
    const int64_t ql = q1 - q0, kv = p.kv_lens[s];
    if (ql < 0 || kv < 0 || kv < ql) return UA_ERR_INVALID_ARG;
    if (ceil_div(kv, p.block_size) > p.max_blocks_per_seq) return UA_ERR_INVALID_ARG;
    if (ql * qpk > INT32_MAX) return UA_ERR_INVALID_ARG;
  }
  // key positions must fit the page table in int32 arithmetic
  if (static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size > INT32_MAX)
    return UA_ERR_INVALID_ARG;
  return UA_OK;
}

ua_status build_schedule(const Problem& p, Schedule* out) {
  ua_status st = validate(p);
  if (st != UA_OK) return st;
  Schedule s;
  const int qpk = p.num_q_heads / p.num_kv_heads;
  const int64_t rows_max = !p.prefill_ok ? INT64_MAX
                           : (p.decode_rows_max < 0 ? kDefaultDecodeRowsMax : p.decode_rows_max);
  const int num_sms = p.num_sms > 0 ? p.num_sms : 152;

  // 1. Prefill tiles, and the decode row blocks: a decode sequence's packed
  // rows in runs of UA_DECODE_ROWS with their key ranges, which are the same
  // for each of its KV heads (its tiles are (KV head, row block) in that
  // order).
  struct DecodeBlock {
    int32_t seq, row0, nrows, kv_lo, kv_hi;
  };
  std::vector<DecodeBlock> blocks;
  std::vector<int32_t> span_end;  // per decode sequence: end of its blocks
  {
    int64_t n_blk = 0, n_pre = 0, n_app = 0, n_dseq = 0;
    for (int32_t q = 0; q < p.num_seqs; ++q) {
      const int64_t ql = p.cu_query_lens[q + 1] - p.cu_query_lens[q];
      const int64_t rows = ql * qpk;
      if (rows <= rows_max) {
        n_blk += ceil_div(rows, UA_DECODE_ROWS);
        ++n_dseq;
      } else {
        n_pre += ceil_div(rows, UA_PREFILL_ROWS) * p.num_kv_heads;
      }
      n_app += ceil_div(ql, kAppendTokens);
    }
    blocks.reserve(static_cast<size_t>(n_blk));
    span_end.reserve(static_cast<size_t>(n_dseq));
    s.prefill.reserve(static_cast<size_t>(n_pre));
    s.append.reserve(static_cast<size_t>(n_app));
  }
  for (int32_t q = 0; q < p.num_seqs; ++q) {
    const int32_t ql = p.cu_query_lens[q + 1] - p.cu_query_lens[q];
    const int32_t kv = p.kv_lens[q];
    s.max_q = std::max(s.max_q, ql);
    s.max_kv = std::max(s.max_kv, kv);
    if (ql == 0) continue;
    const int32_t ctx = kv - ql;
    const int64_t rows = static_cast<int64_t>(ql) * qpk;
    if (rows <= rows_max) {
      for (int64_t r0 = 0; r0 < rows; r0 += UA_DECODE_ROWS) {
        DecodeBlock b;
        b.seq = q;
        b.row0 = static_cast<int32_t>(r0);
        b.nrows = static_cast<int32_t>(std::min<int64_t>(UA_DECODE_ROWS, rows - r0));
        key_range(p, ctx, kv, b.row0, b.nrows, &b.kv_lo, &b.kv_hi);
        blocks.push_back(b);
      }
      span_end.push_back(static_cast<int32_t>(blocks.size()));
      continue;
    }
    const size_t first = s.prefill.size();
    for (int64_t r0 = 0; r0 < rows; r0 += UA_PREFILL_ROWS) {
      ua_tile t;
      t.seq = q;
      t.kv_head = 0;
      t.row0 = static_cast<int32_t>(r0);
      t.nrows = static_cast<int32_t>(std::min<int64_t>(UA_PREFILL_ROWS, rows - r0));
      key_range(p, ctx, kv, t.row0, t.nrows, &t.kv_lo, &t.kv_hi);
      t.kv_lo = static_cast<int32_t>(round_down(t.kv_lo, kPrefillKeyTile));
      t.slot = -1;
      t.group = -1;
      s.prefill.push_back(t);
    }
    const size_t per_head = s.prefill.size() - first;
    for (int32_t g = 1; g < p.num_kv_heads; ++g) {
      for (size_t i = 0; i < per_head; ++i) {
        ua_tile t = s.prefill[first + i];
        t.kv_head = g;
        s.prefill.push_back(t);
      }
    }
  }

  // Append tiles: each sequence's new tokens in runs of kAppendTokens.
  for (int32_t q = 0; q < p.num_seqs; ++q) {
    const int32_t q0 = p.cu_query_lens[q];
    const int32_t ql = p.cu_query_lens[q + 1] - q0;
    const int32_t ctx = p.kv_lens[q] - ql;
    for (int32_t j = 0; j < ql; j += kAppendTokens) {
      ua_tile t;
      t.seq = q;
      t.kv_head = 0;
      t.row0 = q0 + j;
      t.nrows = std::min(kAppendTokens, ql - j);
      t.kv_lo = ctx + j;
      t.kv_hi = t.kv_lo + t.nrows;
      t.slot = -1;
      t.group = -1;
      s.append.push_back(t);
    }
  }

  // 2. Split-KV for decode tiles (FlashDecoding): one chunk length C for the
  // whole batch, so that pieces are equal-sized and load-balance well.
  const int64_t heads = p.num_kv_heads;
  const int64_t n_tiles = static_cast<int64_t>(blocks.size()) * heads;
  int64_t total = 0, longest = 0, shortest = INT64_MAX;
  for (const DecodeBlock& b : blocks) {
    total += (b.kv_hi - b.kv_lo) * heads;
    longest = std::max<int64_t>(longest, b.kv_hi - b.kv_lo);
    shortest = std::min<int64_t>(shortest, b.kv_hi - b.kv_lo);
  }
  int64_t chunk = 0;  // 0: do not split
  const int64_t slots = static_cast<int64_t>(num_sms) * decode_ctas_per_sm(p.head_dim, p.kv_dtype == UA_KV_BF16 ? 2 : 1);
  if (p.num_splits == 0 && n_tiles > 0 && total > 0) {
    chunk = round_up(std::max<int64_t>(kMinSplitTokens, ceil_div(total, slots)), kKeyStep);
    chunk = std::max<int64_t>(chunk, round_up(ceil_div(longest, UA_MAX_SPLITS), kKeyStep));
    if (chunk < longest && shortest * 16 >= longest * 15) {
      // Tiles of (nearly) one length: unsplit when they alone fill HBM in
      // one wave (bf16, rows of at least 256 bytes), else whole waves.
      const bool saturating = p.kv_dtype == UA_KV_BF16 && p.head_dim >= 128 &&
                              n_tiles >= kDecodeSaturatingCtas && n_tiles <= slots;
      chunk = saturating ? longest : wave_fit_chunk(n_tiles, longest, slots);
    }
    if (chunk >= longest) chunk = 0;
  }
  s.split_tokens = static_cast<int32_t>(chunk);
  // Tail pieces. Unsplit tiles that overfill one wave of CTA slots by at most
  // half a wave leave a second wave of `late` whole tiles behind the first:
  // the step takes two tile times for little more than one tile time of work.
  // The `late` tiles that start last in the longest-first order below are cut
  // into k = slots / late pieces (each of at least kMinSplitTokens keys), so
  // they fill the slots the first wave frees and end a fraction of a tile
  // after it.
  int64_t tail_k = 0;
  if (p.num_splits == 0 && chunk == 0 && n_tiles > slots) {
    const int64_t k = std::min<int64_t>(UA_MAX_SPLITS, slots / (n_tiles - slots));
    if (k >= 2) tail_k = k;
  }

  // Per block: the pieces of its tiles (size, count) in the batch rule and,
  // with tail pieces, for a late tile.
  struct Cut {
    int64_t size, pieces;
  };
  auto cut = [](int64_t len, int64_t pieces) {
    const int64_t size = round_up(ceil_div(len, pieces), kKeyStep);
    return Cut{size, std::max<int64_t>(1, ceil_div(len, size))};
  };
  const size_t nb = blocks.size();
  std::vector<Cut> plan(nb), late_plan(tail_k > 0 ? nb : 0);
  for (size_t i = 0; i < nb; ++i) {
    const int64_t len = blocks[i].kv_hi - blocks[i].kv_lo;
    if (p.num_splits > 0)
      plan[i] = cut(len, std::max<int64_t>(1, std::min<int64_t>(p.num_splits, ceil_div(len, kKeyStep))));
    else if (chunk > 0 && len > chunk)
      plan[i] = Cut{chunk, ceil_div(len, chunk)};
    else
      plan[i] = Cut{len, 1};
    if (tail_k > 0) {
      const int64_t n = std::min<int64_t>(tail_k, len / kMinSplitTokens);
      late_plan[i] = n >= 2 ? cut(len, n) : Cut{len, 1};
    }
  }

  // 3. Longest work (keys x rows) first, so the tail of the grid holds the
  // short pieces; equal work in (sequence, KV head, row, key) order, the
  // generation order. The distinct works are few (at most four per block:
  // whole and last piece, in each plan): pieces are counted per work, then
  // written in generation order straight to their place.
  // work of a full piece and of the last piece of a tile of block b cut by c
  auto whole_work = [](const DecodeBlock& b, const Cut& c) { return c.size * b.nrows; };
  auto last_work = [](const DecodeBlock& b, const Cut& c) {
    return (b.kv_hi - b.kv_lo - (c.pieces - 1) * c.size) * b.nrows;
  };
  std::vector<int64_t> works;
  works.reserve(4 * nb);
  for (size_t i = 0; i < nb; ++i) {
    works.push_back(whole_work(blocks[i], plan[i]));
    works.push_back(last_work(blocks[i], plan[i]));
    if (tail_k > 0) {
      works.push_back(whole_work(blocks[i], late_plan[i]));
      works.push_back(last_work(blocks[i], late_plan[i]));
    }
  }
  std::sort(works.begin(), works.end(), std::greater<int64_t>());
  works.erase(std::unique(works.begin(), works.end()), works.end());
  auto rank_of = [&](int64_t w) {
    return static_cast<int32_t>(std::lower_bound(works.begin(), works.end(), w,
                                                 std::greater<int64_t>()) - works.begin());
  };
  struct Ranks {
    int32_t whole, last;
  };
  std::vector<Ranks> rank(nb), late_rank(tail_k > 0 ? nb : 0);
  for (size_t i = 0; i < nb; ++i) {
    rank[i] = Ranks{rank_of(whole_work(blocks[i], plan[i])), rank_of(last_work(blocks[i], plan[i]))};
    if (tail_k > 0)
      late_rank[i] = Ranks{rank_of(whole_work(blocks[i], late_plan[i])),
                           rank_of(last_work(blocks[i], late_plan[i]))};
  }
  // Late tiles: with tail pieces every tile is whole in the batch rule, so a
  // tile's place in the longest-first order of whole tiles is the number of
  // tiles of larger work plus those of its work generated before it.
  std::vector<int64_t> late_from;  // per work rank: first late index among its tiles
  if (tail_k > 0) {
    std::vector<int64_t> count(works.size(), 0);
    for (size_t i = 0; i < nb; ++i) count[static_cast<size_t>(rank[i].last)] += heads;
    late_from.resize(works.size());
    int64_t before = 0;
    for (size_t r = 0; r < works.size(); ++r) {
      late_from[r] = std::max<int64_t>(0, slots - before);
      before += count[r];
    }
  }
  // Tiles run in generation order (sequence, KV head, row block). late(i):
  // whether the next tile of block i is late (`seen` counts the whole tiles
  // of each work so far).
  std::vector<int64_t> seen(tail_k > 0 ? works.size() : 0, 0);
  auto late = [&](size_t i) {
    if (tail_k == 0) return false;
    const size_t r = static_cast<size_t>(rank[i].last);
    return seen[r]++ >= late_from[r];
  };
  // Pieces per work, then each piece written to its place.
  std::vector<int64_t> place(works.size() + 1, 0);
  int64_t n_pieces = 0, n_groups = 0;
  auto count = [&](const Cut& c, const Ranks& r, int64_t tiles) {
    place[static_cast<size_t>(r.whole) + 1] += (c.pieces - 1) * tiles;
    place[static_cast<size_t>(r.last) + 1] += tiles;
    n_pieces += c.pieces * tiles;
    n_groups += c.pieces > 1 ? tiles : 0;
  };
  if (tail_k == 0) {
    for (size_t i = 0; i < nb; ++i) count(plan[i], rank[i], heads);
  } else {
    size_t b0 = 0;
    for (int32_t e : span_end) {
      for (int32_t g = 0; g < p.num_kv_heads; ++g)
        for (size_t i = b0; i < static_cast<size_t>(e); ++i)
          if (late(i)) count(late_plan[i], late_rank[i], 1);
          else count(plan[i], rank[i], 1);
      b0 = static_cast<size_t>(e);
    }
    std::fill(seen.begin(), seen.end(), 0);
  }
  for (size_t r = 0; r < works.size(); ++r) place[r + 1] += place[r];
  s.decode.resize(static_cast<size_t>(n_pieces));
  s.groups.resize(static_cast<size_t>(n_groups));
  ua_tile* const out_tiles = s.decode.data();
  ua_combine_group* const out_groups = s.groups.data();
  int64_t* const at = place.data();
  int32_t slot = 0, gid = 0;
  size_t b0 = 0;
  for (int32_t e : span_end) {
    for (int32_t g = 0; g < p.num_kv_heads; ++g) {
      for (size_t i = b0; i < static_cast<size_t>(e); ++i) {
        const bool is_late = late(i);
        const DecodeBlock& b = blocks[i];
        const Cut& c = is_late ? late_plan[i] : plan[i];
        const Ranks& r = is_late ? late_rank[i] : rank[i];
        ua_tile t;
        t.seq = b.seq;
        t.kv_head = g;
        t.row0 = b.row0;
        t.nrows = b.nrows;
        t.kv_lo = b.kv_lo;
        t.kv_hi = b.kv_hi;
        t.slot = -1;
        t.group = -1;
        if (c.pieces == 1) {
          out_tiles[at[r.last]++] = t;
          continue;
        }
        ua_combine_group& grp = out_groups[gid];
        grp.seq = b.seq;
        grp.kv_head = g;
        grp.row0 = b.row0;
        grp.nrows = b.nrows;
        grp.slot0 = slot;
        grp.nsplits = static_cast<int32_t>(c.pieces);
        grp.pad0 = grp.pad1 = 0;
        t.group = gid++;
        const int32_t size = static_cast<int32_t>(c.size);
        for (int64_t k = 0; k + 1 < c.pieces; ++k) {
          t.kv_hi = t.kv_lo + size;
          t.slot = slot++;
          out_tiles[at[r.whole]++] = t;
          t.kv_lo = t.kv_hi;
        }
        t.kv_hi = b.kv_hi;
        t.slot = slot++;
        out_tiles[at[r.last]++] = t;
      }
    }
    b0 = static_cast<size_t>(e);
  }
  s.num_slots = slot;

  // Prefill tiles stay grouped by (sequence, KV head), longest group first and
  // longest tile first inside a group: CTAs running at the same time then read
  // the same K/V rows, which stay in L2 (a head's K/V is a few MB; all heads
  // at once would not fit).
  if (!s.prefill.empty()) {
    std::vector<int64_t> group_work(static_cast<size_t>(p.num_seqs) * p.num_kv_heads, 0);
    auto gi = [&](const ua_tile& t) {
      return static_cast<size_t>(t.seq) * p.num_kv_heads + t.kv_head;
    };
    for (const ua_tile& t : s.prefill) group_work[gi(t)] += work_of(t);
    std::vector<SortKey> keys(s.prefill.size());
    for (size_t i = 0; i < s.prefill.size(); ++i) {
      const ua_tile& t = s.prefill[i];
      keys[i] = {-group_work[gi(t)], static_cast<int64_t>(gi(t)), -work_of(t),
                 static_cast<int32_t>(i)};
    }
    permute(s.prefill, order_by(keys));
  }
  // Staging pages for an fp8 cache: per sequence with prefill tiles, the
  // logical pages of kStagePage keys from the lowest key any of its tiles
  // reads to its last key.
  if (p.prefill_staged && !s.prefill.empty()) {
    std::vector<int64_t> lo(p.num_seqs, INT64_MAX);
    for (const ua_tile& t : s.prefill) lo[t.seq] = std::min<int64_t>(lo[t.seq], t.kv_lo);
    int32_t max_pages = 0;
    for (int32_t q = 0; q < p.num_seqs; ++q)
      if (lo[q] != INT64_MAX)
        max_pages = std::max<int32_t>(max_pages,
                                      static_cast<int32_t>(ceil_div(p.kv_lens[q], kStagePage)));
    s.staged_max_blocks = max_pages;
    s.staged_table.assign(static_cast<size_t>(p.num_seqs) * max_pages, -1);
    int64_t next = 0;
    for (int32_t q = 0; q < p.num_seqs; ++q) {
      if (lo[q] == INT64_MAX) continue;
      const int64_t pages = ceil_div(p.kv_lens[q], kStagePage);
      for (int64_t i = lo[q] / kStagePage; i < pages; ++i) {
        s.staged_table[static_cast<size_t>(q) * max_pages + i] = static_cast<int32_t>(next);
        ua_tile t;
        t.seq = q;
        t.kv_head = 0;
        t.row0 = static_cast<int32_t>(next);
        t.nrows = static_cast<int32_t>(i);
        t.kv_lo = static_cast<int32_t>(i * kStagePage);
        t.kv_hi = static_cast<int32_t>(std::min<int64_t>(p.kv_lens[q], (i + 1) * kStagePage));
        t.slot = -1;
        t.group = -1;
        s.stage.push_back(t);
        ++next;
      }
    }
    s.staged_pages = next;
  }

  // 4. The persistent prefill CTAs take tiles in list order as they free up.
  // The bulk keeps the order above; the shortest tiles, up to
  // kPrefillTailShare of the work, move to the end, longest first, so that no
  // CTA starts a long tile while the others run dry.
  if (!s.prefill.empty()) {
    const size_t n = s.prefill.size();
    std::vector<int64_t> cost(n, 0);
    int64_t total_cost = 0;
    for (size_t i = 0; i < n; ++i) {
      const ua_tile& t = s.prefill[i];
      const int32_t ql = p.cu_query_lens[t.seq + 1] - p.cu_query_lens[t.seq];
      for (int32_t r0 = t.row0; r0 < t.row0 + t.nrows; r0 += kPrefillQueryTile) {
        int32_t lo = 0, hi = 0;
        const int32_t rows = std::min(kPrefillQueryTile, t.row0 + t.nrows - r0);
        key_range(p, p.kv_lens[t.seq] - ql, p.kv_lens[t.seq], r0, rows, &lo, &hi);
        cost[i] += ceil_div(std::max<int64_t>(0, hi - t.kv_lo), kPrefillKeyTile);
      }
      total_cost += cost[i];
    }
    std::vector<SortKey> keys(n);
    for (size_t i = 0; i < n; ++i) keys[i] = {cost[i], 0, 0, static_cast<int32_t>(i)};
    const std::vector<int32_t> by_cost = order_by(keys);
    std::vector<char> in_tail(n, 0);
    int64_t tail_cost = 0;
    for (size_t k = 0; k < n; ++k) {
      const size_t i = static_cast<size_t>(by_cost[k]);
      if (static_cast<double>(tail_cost + cost[i]) > kPrefillTailShare * total_cost) break;
      tail_cost += cost[i];
      in_tail[i] = 1;
    }
    // bulk in list order, then the tail longest first (ties in list order)
    std::vector<SortKey> tkeys;
    std::vector<int32_t> order;
    order.reserve(n);
    for (size_t i = 0; i < n; ++i)
      if (in_tail[i]) tkeys.push_back({-cost[i], 0, 0, static_cast<int32_t>(i)});
      else order.push_back(static_cast<int32_t>(i));
    for (int32_t i : order_by(tkeys)) order.push_back(i);
    permute(s.prefill, order);
    s.prefill_blocks = total_cost;
    s.prefill_ctas = static_cast<int32_t>(std::min<int64_t>(num_sms, static_cast<int64_t>(n)));
  }
  {
    // the pieces of a tile cover its keys once: `total` keys in all
    const int elt = p.kv_dtype == UA_KV_FP8_E4M3 ? 1 : 2;
    s.decode_bytes = total * 2 * static_cast<int64_t>(p.head_dim) * elt;
  }
  if (!s.prefill.empty() && !s.decode.empty())
    s.prefill_ctas = mixed_prefill_ctas(s.prefill_blocks, s.decode_bytes,
                                        static_cast<int64_t>(s.prefill.size()), num_sms,
                                        p.head_dim);
  *out = std::move(s);
  return UA_OK;
}

int32_t mixed_prefill_ctas(int64_t prefill_blocks, int64_t decode_bytes, int64_t prefill_tiles,
                           int num_sms, int head_dim) {
  const int64_t cap = std::min<int64_t>(num_sms, prefill_tiles);
  if (cap <= 1 || decode_bytes <= 0) return static_cast<int32_t>(std::max<int64_t>(cap, 1));
  const double work_ns = static_cast<double>(prefill_blocks) * kPrefillBlockNs * head_dim / 128.0;
  double best_t = 0.0;
  int64_t best_p = cap;
  for (int64_t P = 1; P <= cap; ++P) {
    const double tp = work_ns / static_cast<double>(P);
    const double bw =
        std::min(kDecodeHbmBytesPerNs, static_cast<double>(num_sms - P) * kDecodeSmBytesPerNs);
    const double left = static_cast<double>(decode_bytes) - bw * tp;
    const double t = left > 0.0 ? tp + left / kDecodeHbmBytesPerNs : tp;
    if (P == 1 || t < best_t) {
      best_t = t;
      best_p = P;
    }
  }
  return static_cast<int32_t>(best_p);
}

int64_t workspace_bytes(const Schedule& s, int head_dim) {
  return s.num_slots * UA_DECODE_ROWS * (static_cast<int64_t>(head_dim) + 1) *
         static_cast<int64_t>(sizeof(float));
}

}  // namespace ua
