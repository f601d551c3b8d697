// Host-side helpers shared by the planner and the launchers.
#pragma once
#include <cstddef>
#include <cstdint>
#include <string>

#include "../../include/mla_decode.h"

namespace mla {

// Rows (heads x query tokens) one CTA of the split-KV kernel handles, in
// multiples of 16 (the MMA N step).  At most 48: TMEM then holds two S^T
// buffers (2 x NR columns) and O^T for both E4M3 terms of P
// (4 blocks x 2 x NR columns) in 512 columns, and shared memory holds two
// P^T buffers next to two KV stages.  More rows use more CTAs (row groups).
constexpr int kMaxRowsPerCta = 48;

struct RowGroups {
  int groups;   // CTAs per (request, split) along the row dimension
  int rows;     // real rows per group (the last group may hold fewer)
  int nr;       // rows rounded up to a multiple of 16 (MMA N)
};

inline RowGroups row_groups(int total_rows) {
  RowGroups g;
  g.groups = (total_rows + kMaxRowsPerCta - 1) / kMaxRowsPerCta;
  if (g.groups < 1) g.groups = 1;
  g.rows = (total_rows + g.groups - 1) / g.groups;
  g.nr = (g.rows + 15) / 16 * 16;
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
