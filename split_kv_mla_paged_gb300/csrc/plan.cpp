// Host split planner and workspace sizing for paged MLA decode.
//
// Two planners:
//  * target_ctas > 0 reproduces the per-request plan printed in TensorRT-LLM
//    issue #20510 ("Repro 2": H12 q8 splits 94/49/25/12/6 at 128K and
//    100/50/25/12/6 at 1M for B = 1..16, split cap raised to 128):
//    t = max(1, target / B) splits per request, chunk = roundup128(ceil(L / t)),
//    splits = ceil(L / chunk).
//  * target_ctas <= 0 is the GB300 planner.  One CTA of the split kernel fills
//    an SM (its shared memory holds two or three 72 KB KV stages), so it
//    balances whole waves of sm_count CTAs, with up to MLA_MAX_SPLITS splits
//    per request (a single long request fills every SM): one chunk for the
//    whole batch (the skewed-batch finding in the same issue's follow-up: a
//    common split size plus early exit of empty split slots beats one wave
//    per request), a minimum of one 128-token tile per split (the short-KV
//    finding there), at most two waves of CTAs (the 2 x SMs grid CTA budget
//    of PR #20380, "Description"; only a batch whose requests alone exceed it
//    gets one split each), and an estimate of each CTA's fixed cost (prologue
//    plus the partial it writes and the merge reads) to choose between one
//    and two waves.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <string>

#include "mla_internal.h"

namespace mla {

static thread_local std::string g_last_error;

void set_error(const std::string& msg) { g_last_error = msg; }

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
static int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// The GB300 planner's CTA budget, in waves of sm_count CTAs.
constexpr int kMaxWaves = 2;
// SMs assumed by the merge's KvSplit budget when the caller passes none (the
// pages' planner mode): a GB300.
constexpr int kDefaultSms = 152;

// CTAs the split kernel launches with a common chunk (empty slots excluded).
static int64_t ctas_for_chunk(const int32_t* lens, int batch, int64_t chunk, int groups) {
  int64_t n = 0;
  for (int b = 0; b < batch; ++b) n += ceil_div(lens[b], chunk);
  return n * groups;
}

}  // namespace mla

using namespace mla;

extern "C" const char* mla_last_error(void) { return g_last_error.c_str(); }

extern "C" size_t mla_decode_workspace_size(int32_t batch, int32_t q_len, int32_t num_heads,
                                            int32_t max_splits) {
  if (batch < 1 || q_len < 1 || num_heads < 1 || max_splits < 1) return 0;
  const int64_t rows = static_cast<int64_t>(batch) * q_len * num_heads;
  return ws_total(rows, max_splits);
}

extern "C" int mla_decode_plan(const int32_t* kv_lens, int32_t batch, int32_t num_heads,
                               int32_t q_len, int32_t sm_count, int32_t target_ctas,
                               int32_t* splits_out, int32_t* chunk_out, int32_t* kv_split_out,
                               size_t* workspace_bytes_out) {
  if (!kv_lens || !splits_out || !chunk_out || !kv_split_out || !workspace_bytes_out) {
    set_error("mla_decode_plan: null pointer argument");
    return MLA_ERR_INVALID_ARG;
  }
  if (batch < 1 || num_heads < 1 || q_len < 1) {
    set_error("mla_decode_plan: batch, num_heads and q_len must be >= 1");
    return MLA_ERR_INVALID_ARG;
  }
  if (static_cast<int64_t>(num_heads) * q_len > MLA_MAX_ROWS) {
    set_error("mla_decode_plan: num_heads * q_len exceeds MLA_MAX_ROWS");
    return MLA_ERR_UNSUPPORTED;
  }
  int64_t lmax = 0;
  for (int b = 0; b < batch; ++b) {
    if (kv_lens[b] < q_len || kv_lens[b] < 1) {
      set_error("mla_decode_plan: kv_lens[" + std::to_string(b) + "] = " +
                std::to_string(kv_lens[b]) + " is below q_len (" + std::to_string(q_len) + ")");
      return MLA_ERR_INVALID_ARG;
    }
    if (kv_lens[b] > INT32_MAX - MLA_TILE_TOKENS) {
      set_error("mla_decode_plan: kv length too large");
      return MLA_ERR_INVALID_ARG;
    }
    lmax = std::max<int64_t>(lmax, kv_lens[b]);
  }
  const RowGroups rg = row_groups_fp8(num_heads * q_len);
  const int64_t T = MLA_TILE_TOKENS;

  if (target_ctas > 0) {
    // The pages' formula counts splits per request; row groups (CTAs that
    // share a split's KV range) come on top of the target.
    const int64_t t = std::max<int64_t>(1, target_ctas / static_cast<int64_t>(batch));
    for (int b = 0; b < batch; ++b) {
      int64_t chunk = round_up(ceil_div(kv_lens[b], t), T);
      if (ceil_div(kv_lens[b], chunk) > MLA_PAGES_SPLIT_CAP)
        chunk = round_up(ceil_div(kv_lens[b], MLA_PAGES_SPLIT_CAP), T);
      chunk_out[b] = static_cast<int32_t>(chunk);
      splits_out[b] = static_cast<int32_t>(ceil_div(kv_lens[b], chunk));
    }
  } else {
    if (sm_count < 1) {
      set_error("mla_decode_plan: sm_count must be >= 1 when target_ctas <= 0");
      return MLA_ERR_INVALID_ARG;
    }
    // Fixed cost of one CTA in token-equivalents of KV streaming: ~2.5 us of
    // prologue/epilogue at ~76 tokens/us per SM, plus writing and re-reading
    // its partials (rows x 2 KB each way) at 576 B per token.
    const int64_t c0 = 200 + static_cast<int64_t>(rg.rows) * 2 * 2048 / MLA_HEAD_DIM;
    const int64_t cmin = std::max<int64_t>(T, round_up(ceil_div(lmax, MLA_MAX_SPLITS), T));
    const int64_t cmax = std::max<int64_t>(cmin, round_up(lmax, T));
    int64_t best_chunk = cmax;
    double best_cost = -1.0;
    for (int w = 1; w <= kMaxWaves; ++w) {
      const int64_t slots = static_cast<int64_t>(w) * sm_count;
      if (ctas_for_chunk(kv_lens, batch, cmax, rg.groups) > slots) continue;
      int64_t lo = cmin / T, hi = cmax / T;  // smallest chunk/T that fits `slots`
      while (lo < hi) {
        const int64_t mid = (lo + hi) / 2;
        if (ctas_for_chunk(kv_lens, batch, mid * T, rg.groups) <= slots)
          hi = mid;
        else
          lo = mid + 1;
      }
      const int64_t chunk = lo * T;
      const int64_t n = ctas_for_chunk(kv_lens, batch, chunk, rg.groups);
      const double cost = static_cast<double>(ceil_div(n, sm_count)) * static_cast<double>(chunk + c0);
      if (best_cost < 0.0 || cost < best_cost) {
        best_cost = cost;
        best_chunk = chunk;
      }
    }
    for (int b = 0; b < batch; ++b) {
      chunk_out[b] = static_cast<int32_t>(best_chunk);
      splits_out[b] = static_cast<int32_t>(ceil_div(kv_lens[b], best_chunk));
    }
  }
  int32_t max_splits = 1;
  for (int b = 0; b < batch; ++b) max_splits = std::max(max_splits, splits_out[b]);
  // Merge thread groups (KvSplit): PR #20380 "Description" takes the largest
  // power of two up to the cap that still gives every group whole work and
  // keeps the grid within its CTA budget.  Here: the largest power of two up
  // to 16 with at least two partials per group and merged rows x groups <= 6 x SMs
  // (the merge runs rows x 4 CTAs of 32 threads per group, so this keeps it
  // near a third of the GPU's thread slots; past that, more groups add
  // threads but no parallel loads).  Fitted to the
  // merge-only sweep on GB300 (rows 12-768, 6-152 splits, every KvSplit):
  // within 5 % of the best KvSplit per point in total, against 14 % for
  // "about four partials per group".
  // Only the rows of requests with more than one split are merged (the
  // others are written by the split kernel and their merge CTAs exit at once).
  int64_t rows = 0;
  for (int b = 0; b < batch; ++b)
    if (splits_out[b] > 1) rows += static_cast<int64_t>(num_heads) * q_len;
  const int64_t budget = 6 * static_cast<int64_t>(sm_count > 0 ? sm_count : kDefaultSms);
  int32_t g = 16;
  while (g > 1 && (g * 2 > max_splits || rows * g > budget)) g >>= 1;
  *kv_split_out = g;
  *workspace_bytes_out = mla_decode_workspace_size(batch, q_len, num_heads, max_splits);
  return MLA_OK;
}

// The item list of a plan for row groups `rg` (shared by the FP8 and BF16
// builders, whose kernels group rows differently).
static int plan_items(const char* who_c, const int32_t* splits, int32_t batch, int32_t num_heads,
                      int32_t q_len, bool bf16, int32_t* items_out, int32_t capacity,
                      int32_t* n_items_out) {
  const std::string who(who_c);
  if (!splits || !n_items_out) {
    set_error(who + ": null pointer argument");
    return MLA_ERR_INVALID_ARG;
  }
  if (batch < 1 || num_heads < 1 || q_len < 1 || batch > MLA_ITEM_MAX_BATCH) {
    set_error(who + ": batch in [1, MLA_ITEM_MAX_BATCH], num_heads, q_len >= 1");
    return MLA_ERR_INVALID_ARG;
  }
  if (static_cast<int64_t>(num_heads) * q_len > MLA_MAX_ROWS) {
    set_error(who + ": num_heads * q_len exceeds MLA_MAX_ROWS");
    return MLA_ERR_UNSUPPORTED;
  }
  const RowGroups rg = bf16 ? row_groups(num_heads * q_len) : row_groups_fp8(num_heads * q_len);
  int32_t max_splits = 0;
  int64_t total = 0;
  for (int b = 0; b < batch; ++b) {
    if (splits[b] < 1 || splits[b] > MLA_MAX_SPLITS) {
      set_error(who + ": splits[" + std::to_string(b) + "] out of range");
      return MLA_ERR_INVALID_ARG;
    }
    max_splits = std::max(max_splits, splits[b]);
    total += static_cast<int64_t>(splits[b]) * rg.groups;
  }
  *n_items_out = static_cast<int32_t>(total);
  if (!items_out) return MLA_OK;  // size query
  if (capacity < total) {
    set_error(who + ": capacity " + std::to_string(capacity) + " below the " +
              std::to_string(total) + " items");
    return MLA_ERR_INVALID_ARG;
  }
  // Split-major: every request's split s before anyone's split s + 1; the row
  // groups of one split are adjacent.
  int64_t k = 0;
  for (int32_t s = 0; s < max_splits; ++s)
    for (int b = 0; b < batch; ++b)
      if (s < splits[b])
        for (int g = 0; g < rg.groups; ++g)
          items_out[k++] = (b << MLA_ITEM_B_SHIFT) | (s << MLA_ITEM_S_SHIFT) | g;
  return MLA_OK;
}

extern "C" int mla_decode_plan_items(const int32_t* splits, int32_t batch, int32_t num_heads,
                                     int32_t q_len, int32_t* items_out, int32_t capacity,
                                     int32_t* n_items_out) {
  return plan_items("mla_decode_plan_items", splits, batch, num_heads, q_len, false, items_out,
                    capacity, n_items_out);
}

extern "C" int mla_decode_plan_items_bf16(const int32_t* splits, int32_t batch, int32_t num_heads,
                                          int32_t q_len, int32_t* items_out, int32_t capacity,
                                          int32_t* n_items_out) {
  return plan_items("mla_decode_plan_items_bf16", splits, batch, num_heads, q_len, true,
                    items_out, capacity, n_items_out);
}
