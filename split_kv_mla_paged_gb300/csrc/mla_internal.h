// Host-side helpers shared by the planner and the launchers.
#pragma once
#include <cstddef>
#include <cstdint>
#include <string>

#include "../../include/mla_decode.h"

namespace mla {

// Rows (heads x query tokens) one CTA of the split-KV kernel handles, in
// multiples of 16 (the MMA N step).  BF16 kernels: at most 48 (TMEM holds two
// S^T buffers and O^T for 48 rows; shared memory two P^T buffers next to two
// KV stages).  FP8 kernels: 16, 32 or 48 rows as for BF16, and one 96-row
// configuration for larger groups (one S^T buffer, both E4M3 terms of P
// accumulated into one O^T, one P^T buffer), so that an H12 q8 request (96
// rows) reads each KV tile once.  More rows use more CTAs (row groups).
constexpr int kMaxRowsPerCta = 48;
constexpr int kMaxRowsPerCtaFp8 = 96;

struct RowGroups {
  int groups;   // CTAs per (request, split) along the row dimension
  int rows;     // real rows per group (the last group may hold fewer)
  int nr;       // rows rounded up to a CTA configuration (MMA N)
};

inline RowGroups row_groups(int total_rows, int max_rows = kMaxRowsPerCta) {
  RowGroups g;
  g.groups = (total_rows + max_rows - 1) / max_rows;
  if (g.groups < 1) g.groups = 1;
  g.rows = (total_rows + g.groups - 1) / g.groups;
  g.nr = (g.rows + 15) / 16 * 16;
  return g;
}

// FP8 grouping: up to 48 rows in one CTA of 16, 32 or 48 rows; above that,
// groups of at most 96 rows, each in a 96-row CTA.
inline RowGroups row_groups_fp8(int total_rows) {
  if (total_rows <= kMaxRowsPerCta) return row_groups(total_rows);
  RowGroups g = row_groups(total_rows, kMaxRowsPerCtaFp8);
  g.nr = kMaxRowsPerCtaFp8;
  return g;
}

// Workspace layout: [status header 256 B][ml: rows*S*2 fp32][o: rows*S*512 fp32]
constexpr size_t kStatusBytes = 256;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline size_t ws_ml_offset() { return kStatusBytes; }
inline size_t ws_o_offset(int64_t rows, int64_t max_splits) {
  return kStatusBytes + align_up(static_cast<size_t>(rows * max_splits) * 2 * sizeof(float), 256);
}
inline size_t ws_total(int64_t rows, int64_t max_splits) {
  return ws_o_offset(rows, max_splits) +
         static_cast<size_t>(rows * max_splits) * MLA_LATENT_DIM * sizeof(float);
}

void set_error(const std::string& msg);

}  // namespace mla
