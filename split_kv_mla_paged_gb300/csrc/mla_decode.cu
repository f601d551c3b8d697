// Paged FP8 MLA decode for GB300 (sm_103a): split-KV kernel (TMA + tcgen05 +
// TMEM) and the C-ABI launchers of the decode (the online-softmax merge
// kernel is in mla_merge.cu).
//
// Problem statement: TensorRT-LLM issue #20510 "CuTe DSL FP8 MLA decode
// regression" (sections "Setup", "Repro 1", "Repro 2", "Analysis"): E4M3 Q
// and paged E4M3 KV, 512 latent + 64 rope per row, page size 32, K = the whole
// row, V = its first 512 values, BF16 output and fp32 softmax stats, the KV
// range split across CTAs with per-split partials merged afterwards.
//
// Split-KV kernel design (one CTA per (request, split, row group), one CTA per
// SM):
//  * The MMA is "swapped": tokens are the M = 128 dimension and a row group of
//    the request's query rows (heads x query tokens, padded: NR = 16, 32, 48
//    or 96 per CTA) is N.  S^T[128 tok x NR] = K[128 x 576] Q^T and
//    O^T[512 x 2NR] += V^T[512 x 128 tok] [P_hi | P_lo]^T, as four M = 128
//    MMAs over the latent dims.  With H*q = 12 this does 16 columns of work
//    instead of padding 12 rows to 128, and S^T plus O^T fit TMEM
//    (2*NR + 4*2NR <= 512).  The 96-row configuration (H12 q8 in one CTA, so
//    each KV tile is read from shared memory once for all 96 rows) keeps one
//    S^T buffer and accumulates P_hi and P_lo into the same O^T with two MMAs
//    (96 + 4*96 columns), with one P^T buffer and per-thread row sums.
//  * One TMA-staged copy of each KV tile (4 pages x 576 B x 32 tokens, 128 B
//    swizzle for the latent blocks, 64 B for the rope block) serves as the K
//    operand (K-major) and as the V operand (MN-major over the same bytes), so
//    each KV byte is read from HBM once.
//  * Online softmax in log2 units with integer reference maxima: per row the
//    reference k is ceil(running max) and p = 2^(t - k + 8) is computed as
//    ex2(t - rint(t)) * 2^(rint(t) - k + 8).  Every rescale is then an exact
//    power of two, so the E4M3-quantised P fed to the PV MMA, and every
//    partial, is the same for any split plan up to exact scaling.
//  * Warp roles: warp 0 issues TMA, warp 1 issues the QK tcgen05.mma (and
//    owns TMEM), warp 2 the PV ones, and the next four warps (eight from 32
//    rows up; for 96 rows an idle warp 3, then twelve; TMEM lane quadrant =
//    warp % 4) run the softmax, the rare O correction and the epilogue.
//  * The 96-row configuration fills and releases its two KV stages block by
//    block (rope, then the four latent blocks), so a tile's load overlaps the
//    previous tile's PV.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>

#include "mla_device.cuh"

namespace mla {

constexpr int kTileTokens = 128;
constexpr uint32_t kTileBytes = kTileTokens * MLA_HEAD_DIM;  // 73728
constexpr uint32_t kLatBlockBytes = kTileTokens * 128;       // 16384: one 128-dim block
constexpr uint32_t kRopeOffset = 4 * kLatBlockBytes;         // 65536
constexpr uint32_t kPageLatBytes = MLA_PAGE_SIZE * 128;      // 4096
constexpr uint32_t kPageRopeBytes = MLA_PAGE_SIZE * 64;      // 2048
constexpr uint32_t kPageBytes = MLA_PAGE_SIZE * MLA_HEAD_DIM;


template <int NR>
struct Cfg {
  static_assert(NR == 16 || NR == 32 || NR == 48 || NR == kMaxRowsPerCtaFp8, "NR");
  // kWide: the 96-row configuration.  TMEM holds one S^T buffer and O^T for
  // 96 rows; the two E4M3 terms of P^T go through two PV MMAs into the same
  // O^T, and each softmax thread keeps its own row sums across tiles (so the
  // shared-memory reduction buffers fit next to two KV stages, Q and P^T).
  static constexpr bool kWide = NR > kMaxRowsPerCta;
  // P^T = hi + lo.  Up to 48 rows both terms go through one PV MMA with
  // N = 2*NR (O^T holds the hi and lo products side by side and the epilogue
  // adds them), so V is read from shared memory once per tile.
  static constexpr int OW = kWide ? NR : 2 * NR;  // O^T columns per latent block
  static constexpr int NS = kWide ? 1 : 2;        // S^T buffers in TMEM
  static constexpr uint32_t kTmemUsed = NS * NR + 4 * OW;
  static_assert(kTmemUsed <= 512, "TMEM");
  // Softmax warpgroups: two (each owning half the rows) from 32 rows up,
  // three (32 rows each) for the 96-row configuration.
  static constexpr int SWG = kWide ? 3 : NR >= 32 ? 2 : 1;
  static constexpr int NRH = NR / SWG;
  static_assert(NRH % 8 == 0, "rows per softmax warpgroup");
  // Warp 0 TMA, warp 1 QK issuer (and TMEM owner), warp 2 PV issuer, then
  // the softmax warpgroups.  Each issuer blocks on its own barriers; for the
  // 96-row CTA this measured 2 % faster on H96 q8 B1 1M (and 1 % slower on
  // MTP q8 B16 128K) than one warp polling both, and the polling loop lost
  // 4 % to any extra work in it.
  static constexpr int kMmaWarps = 2;
  // 96 rows: an idle fourth warp makes warps 0-3 one warpgroup, so that
  // setmaxnreg can move registers from it to the three softmax warpgroups:
  // launched with 128 per thread (512 threads), warpgroup 0 drops to 56 and
  // the softmax warpgroups rise to 152 (56 x 128 + 152 x 384 = 128 x 512).
  // Measured against two softmax warpgroups of 48 rows at 168 registers
  // (which spilled): MTP q8 B16 128K 371.6 -> 361.2 us, B1 45.1 -> 41.4 us,
  // H96 q8 B1 1M 1332.7 -> 1305.7 us.
  static constexpr int kIdleWarps = kWide ? 1 : 0;
  static constexpr int kSoftmaxWarp0 = 1 + kMmaWarps + kIdleWarps;
  static constexpr int kRegsLaunch = 128, kRegsLow = 56, kRegsHigh = 152;
  static_assert(!kWide || (kRegsLow * 128 + kRegsHigh * 128 * SWG <= kRegsLaunch * 512 &&
                           32 * kSoftmaxWarp0 + 128 * SWG == 512),
                "register split");
  static constexpr int kThreads = 32 * kSoftmaxWarp0 + 128 * SWG;
  static constexpr uint32_t kTmemCols =
      kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64 : kTmemUsed <= 128 ? 128
      : kTmemUsed <= 256 ? 256 : 512;
  static constexpr uint32_t kOCol = NS * NR;
  // Shared memory, offsets from a 1024-byte aligned base.
  static constexpr uint32_t kPHalf = NR * kTileTokens;  // one E4M3 term of P^T
  static constexpr uint32_t kPBytes = 2 * kPHalf;       // hi + lo
  // Reductions: tile maxima 16 NR B, row sums 32 NR B (double-buffered by
  // tile parity; with per-thread sums, 96 rows, the once-per-item reduction
  // shares the tile maxima's buffer), references 4 NR B.
  static constexpr uint32_t kRedSumBytes = kWide ? 0 : 32 * NR;
  // 96 rows: the KV stages are filled and released per block (rope, then the
  // four 128-dim latent blocks), each with its own full and empty barrier.
  static constexpr bool kBlockStages = kWide;
  static constexpr uint32_t kBlkBarBytes = kBlockStages ? 2 * 2 * 5 * 8 : 0;
  static constexpr uint32_t kAuxBytes =
      192 + 20 * NR + kRedSumBytes + (kWide ? 4 * NR : 0) + kBlkBarBytes;
  static constexpr uint32_t kQBytes = NR * MLA_HEAD_DIM;
  // Three KV stages fit when P^T can live in the rope block of its own stage
  // (QK has consumed that block before P is written): NR = 16.  Otherwise two
  // stages and separate P^T buffers (two when they fit, else one).
  static constexpr bool kPInStage =
      kPBytes <= kTileTokens * 64 &&
      3 * kTileBytes + kQBytes + kAuxBytes + 1024 <= 232448u;
  static constexpr int NST = kPInStage ? 3 : 2;
  static constexpr uint32_t kKV = 0;
  static constexpr uint32_t kQ = NST * kTileBytes;
  static constexpr uint32_t kP = kQ + kQBytes;
  static constexpr int NPB = kPInStage ? 0
                             : (kP + 2 * kPBytes + kAuxBytes + 1024 <= 232448u) ? 2 : 1;
  static_assert(NPB != 1 || kWide, "P^T needs two buffers or a slot in each KV stage");
  static constexpr uint32_t kAux = kP + NPB * kPBytes;
  // PV completions alternate between two barriers by tile parity; the second
  // takes a slot this configuration does not use (the second P^T-free
  // barrier when P^T lives in the stages, else the third stage's full one).
  static constexpr int kBarOdone1 = kPInStage ? BAR_PFREE1 : BAR_FULL0 + 2;
  static_assert(kPInStage || NST == 2, "the third stage's barrier must be free");
  // aux: mbarriers, tmem slot, flags, reductions
  static constexpr uint32_t kBars = kAux;               // 19 x 8 B
  static constexpr uint32_t kTmemSlot = kAux + 152;     // 4 B
  static constexpr uint32_t kFlags = kAux + 160;        // 3 x 4 B
  static constexpr uint32_t kStageInfo = kAux + 176;    // NST x 4 B: rows loaded per page
  static constexpr uint32_t kRedMax = kAux + 192;       // 4 x NR floats
  // Row owner r reads red_max[.][r] before writing alpha[r]: alpha reuses
  // red_max's first row.
  static constexpr uint32_t kAlpha = kRedMax;           // NR floats
  // (2 x) 4 x NR floats; 96 rows: the tile maxima's buffer.  Each warpgroup
  // writes its own rows' slots of either, so one warpgroup's sums and
  // another's tile maxima never meet.
  static constexpr uint32_t kRedSum = kWide ? kRedMax : kRedMax + 16 * NR;
  static constexpr uint32_t kKref = kRedMax + 16 * NR + kRedSumBytes;  // NR floats
  // 96 rows: kref holds each row's vote threshold k + 0.75, and kKci its
  // integer exponent offset for softmax_weight_kc (NR ints).
  static constexpr uint32_t kKci = kKref + 4 * NR;
  // Block barriers: full (stage s, block b) at 8 (5 s + b), empty at 8 (10 + 5 s + b).
  static constexpr uint32_t kBlkBars = kKci + (kWide ? 4 * NR : 0);
  static_assert(kBlkBars % 8 == 0, "mbarrier alignment");
  static constexpr uint32_t kEnd = kBlkBars + kBlkBarBytes;
  static_assert(kEnd - kAux <= kAuxBytes, "aux layout");
  static_assert(NR != 16 || NST == 3, "16-row CTAs must keep three KV stages");
  static constexpr uint32_t kSmemBytes = kEnd + 1024;   // + alignment slack
  static_assert(kSmemBytes <= 232448u, "shared memory");
};


// Rows of a staged tile that hold no loaded key: pages that were not loaded
// (past the split's end, outside a window or an unused selection slot) and
// the tail of a request's last page.  The warp zeroes them (all 576 bytes of
// a row: four 128-byte latent blocks and the 64-byte rope block) so V holds
// no stale or NaN bytes (0 * NaN would poison the PV sum).  kGather: `info`
// holds the rows loaded per page, one byte each; otherwise the first `valid`
// rows of the tile are keys of the split.
template <bool kGather>
__device__ __forceinline__ void zero_unloaded_rows(uint8_t* kvp, int lane, uint32_t info,
                                                   int valid) {
  const uint4 z = make_uint4(0, 0, 0, 0);
  auto zero_rows = [&](int r0, int nrow) {
    for (int idx = lane; idx < nrow * 36; idx += 32) {
      const int r = r0 + idx / 36;
      const int c = idx % 36;
      uint4* dst;
      if (c < 32)
        dst = reinterpret_cast<uint4*>(kvp + (c / 8) * kLatBlockBytes + r * 128 + (c % 8) * 16);
      else
        dst = reinterpret_cast<uint4*>(kvp + kRopeOffset + r * 64 + (c - 32) * 16);
      *dst = z;
    }
  };
  if constexpr (kGather) {
    if (info != 0x20202020u) {
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        const int nv = static_cast<int>((info >> (8 * q)) & 0xFFu);
        if (nv < MLA_PAGE_SIZE) zero_rows(q * MLA_PAGE_SIZE + nv, MLA_PAGE_SIZE - nv);
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
  } else {
    if (valid < kTileTokens) {
      zero_rows(valid, kTileTokens - valid);
      fence_proxy_async_smem();
      __syncwarp();
    }
  }
}

// One work item of the split kernel: split `split` of request b, row group
// grp, with the key range, scales and row counts every role derives the
// same way.
struct ItemInfo {
  int b, split, grp, L, nsplit, q_b, tok_end, t0, win_lo, win_hi, row0, rows_here, rows_valid,
      n_tiles;
  bool sparse;
  float c_log2, kv_scale;
};

// Item (b, split, grp): the plan checks (a bad plan is reported as
// MLA_ERR_INVALID_ARG and gives false), then the split's token range in the
// planned space (positions, or the compact range of a page selection), the
// key window, the first tile (whole tiles below a dense window are skipped;
// tiles stay aligned to the split start, so pages stay whole), the scales and
// the row counts.
template <bool kGather>
__device__ __forceinline__ bool item_info(const DecodeParams& p, int b, int split, int grp,
                                          ItemInfo& it) {
  it.b = b;
  it.split = split;
  it.grp = grp;
  it.L = p.kv_lens[b];
  it.nsplit = p.splits[b];
  const int chunk = p.chunks[b];
  // With selected pages the split plan covers the compact range of the
  // selection (32 * topk tokens); otherwise the key positions [0, L).
  it.sparse = kGather && p.block_idx != nullptr;
  const int Lspace = it.sparse ? p.topk * MLA_PAGE_SIZE : it.L;
  it.q_b = p.query_lens ? p.query_lens[b] : p.q_len;  // this request's query tokens
  const bool bad = it.L < 1 || it.q_b < 1 || it.q_b > p.q_len || (p.causal && it.L < it.q_b) ||
                   it.nsplit > p.max_splits || chunk < kTileTokens ||
                   (chunk % kTileTokens) != 0 ||
                   static_cast<int64_t>(it.nsplit) * chunk < Lspace ||
                   static_cast<int64_t>(it.nsplit - 1) * chunk >= Lspace ||
                   static_cast<int64_t>(it.L) > static_cast<int64_t>(p.max_pages) * MLA_PAGE_SIZE;
  if (bad) {
    if (threadIdx.x == 0) report(p.status, MLA_ERR_INVALID_ARG);
    return false;
  }
  const int tok_begin = split * chunk;
  it.tok_end = min(Lspace, tok_begin + chunk);
  // Key window in positions ([0, L) without one).
  it.win_lo = 0;
  it.win_hi = it.L;
  if (kGather && p.kv_bounds) {
    it.win_lo = max(0, p.kv_bounds[2 * b]);
    it.win_hi = min(it.L, p.kv_bounds[2 * b + 1]);
  }
  it.t0 = tok_begin;
  if (kGather && !it.sparse) {
    it.tok_end = min(it.tok_end, it.win_hi);
    if (it.win_lo >= it.tok_end)
      it.t0 = it.tok_end;  // nothing of the window in this split
    else if (it.win_lo > tok_begin)
      it.t0 = tok_begin + (it.win_lo - tok_begin) / kTileTokens * kTileTokens;
  }
  it.c_log2 = p.c_log2;
  it.kv_scale = p.kv_scale;
  if (p.q_scale_dev || p.kv_scale_dev || p.sm_scale_dev) {
    const float qs = p.q_scale_dev ? *p.q_scale_dev : p.q_scale_h;
    it.kv_scale = p.kv_scale_dev ? *p.kv_scale_dev : p.kv_scale;
    const float ss = p.sm_scale_dev ? *p.sm_scale_dev : p.sm_scale_h;
    it.c_log2 = ss * qs * it.kv_scale * 1.4426950408889634f;
  }
  it.row0 = grp * p.rows_per_group;  // first row of this group
  it.rows_here = min(p.rows_per_group, p.rows_per_req - it.row0);
  // Rows of real query tokens (the others are padding slots of a shorter
  // query block: no key is visible to them).
  it.rows_valid = max(0, min(it.rows_here, it.q_b * p.num_heads - it.row0));
  it.n_tiles = (it.rows_valid > 0 && it.tok_end > it.t0)
                   ? (it.tok_end - it.t0 + kTileTokens - 1) / kTileTokens
                   : 0;
  return true;
}

// Decodes a CTA item-list entry; false (reported) for an item outside the
// batch or the row groups.
__device__ __forceinline__ bool decode_item(const DecodeParams& p, int it, int ngroups, int& b,
                                            int& split, int& grp) {
  b = it >> MLA_ITEM_B_SHIFT;
  split = (it >> MLA_ITEM_S_SHIFT) & ((1 << (MLA_ITEM_B_SHIFT - MLA_ITEM_S_SHIFT)) - 1);
  grp = it & ((1 << MLA_ITEM_S_SHIFT) - 1);
  if (it < 0 || b >= p.batch || grp >= ngroups) {
    if (threadIdx.x == 0) report(p.status, MLA_ERR_INVALID_ARG);
    return false;
  }
  return true;
}

// kGather: the variant for restricted key sets (key windows, selected pages):
// tiles may have pages that are not loaded, and every score is masked by its
// key position.  The plain variant (kGather = false) covers full key ranges,
// with or without ragged query counts.  kMode: 0 the (request, split x row
// group) grid, 1 the CTA item list (one item per CTA), 2 persistent CTAs
// that each loop over items blockIdx.x, blockIdx.x + gridDim.x, ... of the
// list, carrying every barrier phase from one item to the next so that the
// next item's Q and first tiles load while the current one finishes.
template <int NR, bool kGather, int kMode>
__global__ void __launch_bounds__(Cfg<NR>::kThreads, 1)
    mla_split_kv_kernel(const __grid_constant__ CUtensorMap tm_kv_lat,
                        const __grid_constant__ CUtensorMap tm_kv_rope,
                        const __grid_constant__ CUtensorMap tm_q_lat,
                        const __grid_constant__ CUtensorMap tm_q_rope, const DecodeParams p) {
  using C = Cfg<NR>;
  constexpr bool kPersist = kMode == 2;
  // Grid (request, split x row group), dispatched split-major: every
  // request's first splits go out before anyone's later ones, so the empty
  // slots of short requests (split >= splits[b], exiting at once) do not hold
  // back real work in a skewed batch; the row groups of one split are
  // `batch` CTAs apart and run in the same wave, so L2 serves their repeated
  // reads of the same KV tiles.  The item list holds exactly the CTAs that
  // have work, in the same order.
  const int ngroups = (p.rows_per_req + p.rows_per_group - 1) / p.rows_per_group;
  ItemInfo first{};
  if constexpr (!kPersist) {
    int b, split, grp;
    if constexpr (kMode == 1) {
      if (!decode_item(p, p.cta_items[blockIdx.x], ngroups, b, split, grp)) return;
    } else {
      split = blockIdx.y / ngroups;
      grp = blockIdx.y - split * ngroups;
      b = blockIdx.x;
    }
    if (split >= p.splits[b]) return;  // empty split slot of a shorter request
    if (!item_info<kGather>(p, b, split, grp, first)) return;
  }
  // The n-th item of this CTA: 2 = `it` holds it, 1 = skip it (reported),
  // 0 = no more.  Every role walks the same sequence.
  auto next_item = [&](int n, ItemInfo& it) -> int {
    if constexpr (!kPersist) {
      if (n > 0) return 0;
      it = first;
      return 2;
    } else {
      const int64_t idx = blockIdx.x + static_cast<int64_t>(n) * gridDim.x;
      if (idx >= p.num_items) return 0;
      int b, split, grp;
      if (!decode_item(p, p.cta_items[idx], ngroups, b, split, grp)) return 1;
      if (split >= p.splits[b]) return 1;
      return item_info<kGather>(p, b, split, grp, it) ? 2 : 1;
    }
  };
  // Binds an item's values to the names the role bodies use.
#define MLA_ITEM_NAMES(it)                                                                    \
  const int b = it.b, split = it.split, L = it.L, nsplit = it.nsplit, q_b = it.q_b;          \
  const int tok_end = it.tok_end, t0 = it.t0, win_lo = it.win_lo, win_hi = it.win_hi;        \
  const int row0 = it.row0, rows_here = it.rows_here, rows_valid = it.rows_valid;            \
  const int n_tiles = it.n_tiles;                                                            \
  const bool sparse = it.sparse;                                                             \
  const float c_log2 = it.c_log2, kv_scale = it.kv_scale;                                    \
  (void)b; (void)split; (void)L; (void)nsplit; (void)q_b; (void)tok_end; (void)t0;           \
  (void)win_lo; (void)win_hi; (void)row0; (void)rows_here; (void)rows_valid; (void)n_tiles;   \
  (void)sparse; (void)c_log2; (void)kv_scale

  // One item per CTA with contiguous pages: the producer's first page-id
  // window is read before the set-up below, so that its latency overlaps it.
  int pre_window = 0;
  if constexpr (!kPersist && !kGather) {
    if ((threadIdx.x >> 5) == 0) {
      const int pi = first.t0 / MLA_PAGE_SIZE + static_cast<int>(threadIdx.x & 31);
      if (pi < (first.tok_end + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE)
        pre_window = p.page_table[static_cast<int64_t>(first.b) * p.max_pages + pi];
    }
  }
  (void)pre_window;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(base);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kBars + 8u * i; };
  // Block barriers (kBlockStages): block b of stage s, b = 0..3 the latent
  // blocks, 4 the rope block.
  auto full_blk = [&](int st, int b) -> uint32_t { return sbase + C::kBlkBars + 8u * (5 * st + b); };
  auto empty_blk = [&](int st, int b) -> uint32_t {
    return sbase + C::kBlkBars + 8u * (10 + 5 * st + b);
  };
  (void)full_blk;
  (void)empty_blk;
  volatile int* flags = reinterpret_cast<volatile int*>(base + C::kFlags);
  volatile int* abort_flag = flags + 2;
  float* red_max = reinterpret_cast<float*>(base + C::kRedMax);
  float* red_sum = reinterpret_cast<float*>(base + C::kRedSum);
  float* kref = reinterpret_cast<float*>(base + C::kKref);
  float* alpha_s = reinterpret_cast<float*>(base + C::kAlpha);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int k = 0; k < C::NST; ++k) {
      mbar_init(bar(BAR_FULL0 + k), 1);
      mbar_init(bar(BAR_EMPTY0 + k), 1);
    }
    if constexpr (C::kBlockStages) {
      for (int k = 0; k < C::NST; ++k)
        for (int b = 0; b < 5; ++b) {
          mbar_init(full_blk(k, b), 1);
          mbar_init(empty_blk(k, b), 1);
        }
    }
    mbar_init(bar(BAR_QFULL), 1);
    mbar_init(bar(BAR_SFULL0), 1);
    mbar_init(bar(BAR_SFULL1), 1);
    mbar_init(bar(BAR_SFREE0), 128 * C::SWG);
    mbar_init(bar(BAR_SFREE1), 128 * C::SWG);
    mbar_init(bar(BAR_PFULL0), 128 * C::SWG);
    mbar_init(bar(BAR_PFULL1), 128 * C::SWG);
    mbar_init(bar(BAR_PFREE0), 1);
    mbar_init(bar(BAR_PFREE1), 1);
    mbar_init(bar(BAR_ODONE), 1);
    mbar_init(bar(C::kBarOdone1), 1);
    // Per item: the PV warp's commit after its last PV (every QK result has
    // been consumed by then); Q free again after the QK warp's last QK; O^T
    // read by the softmax warpgroups.
    mbar_init(bar(BAR_FINAL), 1);
    mbar_init(bar(BAR_QFREE), 1);
    mbar_init(bar(BAR_OFREE), 128 * C::SWG);
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    fence_mbar_init();
  }
  // Rows start with no reference (every thread takes a few, next to thread
  // 0's barrier set-up).
  for (int r = threadIdx.x; r < NR; r += C::kThreads) {
    kref[r] = -INFINITY;
    if constexpr (C::kWide) reinterpret_cast<int*>(base + C::kKci)[r] = kKcNone;
  }
  if (warp == 1) {
    tmem_alloc(sbase + C::kTmemSlot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base + C::kTmemSlot);

  if (warp < C::kSoftmaxWarp0) {
    // Producer, MMA issuers (and the 96-row configuration's idle warp): one
    // warpgroup, whose registers go to the softmax warpgroups.
    if constexpr (C::kWide) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegsLow));
    if (warp == 0) {
      // ================= TMA producer =================
      if (lane == 0) {
        tma_prefetch_desc(&tm_kv_lat);
        tma_prefetch_desc(&tm_kv_rope);
        tma_prefetch_desc(&tm_q_lat);
        tma_prefetch_desc(&tm_q_rope);
      }
      const uint64_t pol = l2_policy_evict_first();
      volatile uint32_t* stage_info = reinterpret_cast<volatile uint32_t*>(base + C::kStageInfo);
      int issued = 0;  // tiles issued, all items
      int armed_part = 0;  // block stages: blocks out of a tile cut short by a failed wait
      int st = 0, round = 0;
      int nq = 0;      // items whose Q was loaded
      bool ok = true;
      for (int n = 0; ok && (kPersist || n == 0); ++n) {
        ItemInfo item;
        const int r = next_item(n, item);
        if (r == 0) break;
        if (r == 1) continue;
        MLA_ITEM_NAMES(item);
        // Q of this item, once the previous item's QKs are done with the buffer.
        if (nq > 0) {
          bool q_ok = mbar_wait_abort(bar(BAR_QFREE), (nq - 1) & 1, p.wait_cycles, abort_flag);
          q_ok = __all_sync(0xffffffffu, q_ok && !*abort_flag);
          if (!q_ok) {
            if (lane == 0) {
              report(p.status, MLA_ERR_TIMEOUT);
              *abort_flag = 1;
            }
            ok = false;
            break;
          }
        }
        if (lane == 0) {
          const int qrow = b * p.rows_per_req + row0;
          mbar_arrive_expect_tx(bar(BAR_QFULL), C::kQBytes);
#pragma unroll
          for (int d = 0; d < 4; ++d)
            tma_load_2d(sbase + C::kQ + d * NR * 128, &tm_q_lat, d * 128, qrow, bar(BAR_QFULL));
          tma_load_2d(sbase + C::kQ + 4 * NR * 128, &tm_q_rope, MLA_LATENT_DIM, qrow,
                      bar(BAR_QFULL));
        }
        ++nq;
        const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.max_pages;
        const int page0 = t0 / MLA_PAGE_SIZE;
        const int page_end = (tok_end + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE;  // exclusive
        // Page ids of 8 tiles (32 pages) per window, one per lane; the next
        // window is fetched a window ahead so its latency is hidden.  kGather
        // also keeps, per page, the number of its rows to load (0: not loaded):
        // compact page cp maps to logical page lp (cp itself, or the selection's
        // entry), which is loaded when it holds keys inside the window and before
        // the end of the split (dense) or of the request (selection).
        int last_lp = -1;  // selection: the entry before this window (order check)
        auto load_window = [&](int w, int& nv_out) -> int {
          const int pi = page0 + w * 32 + lane;
          int pg = 0;
          nv_out = 0;
          if constexpr (!kGather) {
            if (pi < page_end) {
              pg = (!kPersist && w == 0) ? pre_window : pt[pi];
              if (pg < 0 || pg >= p.num_pages) {
                report(p.status, MLA_ERR_INVALID_ARG);
                pg = 0;
              }
            }
          } else {
            int lp = -1;
            if (pi < page_end) {
              lp = pi;
              if (sparse) lp = (pi < p.topk) ? p.block_idx[static_cast<int64_t>(b) * p.topk + pi] : -1;
            }
            if (sparse) {
              // Selected pages must be listed in increasing order, each once.
              int prev = __shfl_up_sync(0xffffffffu, lp, 1);
              if (lane == 0) prev = last_lp;
              if (lp >= 0 && prev >= 0 && lp <= prev) report(p.status, MLA_ERR_INVALID_ARG);
              last_lp = __shfl_sync(0xffffffffu, lp, 31);
            }
            const int64_t end_pos = sparse ? win_hi : tok_end;
            const int64_t first = static_cast<int64_t>(lp) * MLA_PAGE_SIZE;
            if (lp >= 0 && first < end_pos && first + MLA_PAGE_SIZE > win_lo) {
              pg = pt[lp];
              if (pg < 0 || pg >= p.num_pages) {
                report(p.status, MLA_ERR_INVALID_ARG);
                pg = 0;
              }
              nv_out = static_cast<int>(end_pos - first < MLA_PAGE_SIZE ? end_pos - first : MLA_PAGE_SIZE);
            }
          }
          return pg;
        };
        int window_nv, window_next_nv;
        int window = load_window(0, window_nv);
        int window_next = load_window(1, window_next_nv);
        for (int i = 0; i < n_tiles; ++i) {
          if (i > 0 && (i & 7) == 0) {
            window = window_next;
            window_nv = window_next_nv;
            window_next = load_window((i >> 3) + 1, window_next_nv);
          }
          ok = !expired_here(p, WAIT_STAGE_FREE, i);
          if (ok && round > 0 && !C::kBlockStages)
            ok = mbar_wait_abort(bar(BAR_EMPTY0 + st), (round - 1) & 1, p.wait_cycles, abort_flag);
          ok = __all_sync(0xffffffffu, ok && !*abort_flag);
          if (!ok) {
            if (lane == 0) {
              report(p.status, MLA_ERR_TIMEOUT);
              *abort_flag = 1;
            }
            break;
          }
          // Lane q (< 4) takes the id of the tile's page q.
          const int src = (i & 7) * 4 + (lane & 3);
          const int my_page = __shfl_sync(0xffffffffu, window, src);
          const int tp0 = page0 + i * 4;
          bool my_load;
          uint32_t info = 0;
          if constexpr (kGather) {
            // Rows to load of pages 0-3, one byte each, for the QK warp (which
            // zeroes the rest); published by the arrive below.
            const int my_nv = __shfl_sync(0xffffffffu, window_nv, src);
            my_load = my_nv > 0;
            const int n1 = __shfl_sync(0xffffffffu, my_nv, 1);
            const int n2 = __shfl_sync(0xffffffffu, my_nv, 2);
            const int n3 = __shfl_sync(0xffffffffu, my_nv, 3);
            info = static_cast<uint32_t>(my_nv) | (static_cast<uint32_t>(n1) << 8) |
                   (static_cast<uint32_t>(n2) << 16) | (static_cast<uint32_t>(n3) << 24);
          } else {
            my_load = tp0 + (lane & 3) < page_end;
          }
          const int nload = __popc(__ballot_sync(0xffffffffu, lane < 4 && my_load));
          const uint32_t kv = sbase + C::kKV + st * kTileBytes;
          const int row = my_page * MLA_PAGE_SIZE;
          if constexpr (C::kBlockStages) {
            // Block by block as the previous tile of this stage releases them:
            // the rope block after its QK, latent block d after its PV block d.
            // The rows-loaded word goes out with the first block's barrier.
            int armed = 0;  // blocks of this tile whose copies are out
#pragma unroll 1
            for (int bi = 0; bi < 5; ++bi) {
              const int blk = (bi == 0) ? 4 : bi - 1;
              if (round > 0) {
                ok = mbar_wait_abort(empty_blk(st, blk), (round - 1) & 1, p.wait_cycles,
                                     abort_flag);
                ok = __all_sync(0xffffffffu, ok && !*abort_flag);
                if (!ok) break;
              }
              const uint32_t fb = full_blk(st, blk);
              if (lane == 0) {
                if (kGather && bi == 0) stage_info[st] = info;
                mbar_arrive_expect_tx(fb, nload * (blk == 4 ? kPageRopeBytes : kPageLatBytes));
              }
              __syncwarp();
              if (lane < 4 && my_load) {
                if (blk == 4)
                  tma_load_2d_hint(kv + kRopeOffset + lane * kPageRopeBytes, &tm_kv_rope,
                                   MLA_LATENT_DIM, row, fb, pol);
                else
                  tma_load_2d_hint(kv + blk * kLatBlockBytes + lane * kPageLatBytes, &tm_kv_lat,
                                   blk * 128, row, fb, pol);
              }
              __syncwarp();
              ++armed;
            }
            if (!ok) {
              if (lane == 0) {
                report(p.status, MLA_ERR_TIMEOUT);
                *abort_flag = 1;
              }
              armed_part = armed;  // drained below
              break;
            }
          } else {
            const uint32_t fb = bar(BAR_FULL0 + st);
            if (lane == 0) {
              if constexpr (kGather) stage_info[st] = info;
              mbar_arrive_expect_tx(fb, nload * kPageBytes);
            }
            __syncwarp();
            // Lanes 0-3 issue one page each (5 boxes: 4 latent blocks + rope).
            if (lane < 4 && my_load) {
#pragma unroll
              for (int d = 0; d < 4; ++d)
                tma_load_2d_hint(kv + d * kLatBlockBytes + lane * kPageLatBytes, &tm_kv_lat,
                                 d * 128, row, fb, pol);
              tma_load_2d_hint(kv + kRopeOffset + lane * kPageRopeBytes, &tm_kv_rope,
                               MLA_LATENT_DIM, row, fb, pol);
            }
            __syncwarp();
          }
          ++issued;
          if (++st == C::NST) {
            st = 0;
            ++round;
          }
        }
      }
      // Before the CTA can exit, the copies this warp issued must have landed
      // (they have, unless a wait elsewhere ran out).  The full barrier of a
      // stage is at most one phase behind the producer, so these waits are exact.
      if (lane == 0) {
        for (int k = max(0, issued - C::NST); k < issued; ++k) {
          if constexpr (C::kBlockStages) {
            // Blocks of the stage re-armed for a tile cut short have landed
            // for tile k (their release needed it); that tile's own blocks
            // are one phase ahead, waited for after this loop.
            const int skip = (k + C::NST == issued) ? armed_part : 0;
            for (int bi = skip; bi < 5; ++bi)
              mbar_wait(full_blk(k % C::NST, bi == 0 ? 4 : bi - 1), (k / C::NST) & 1,
                        kWaitLimitCycles);
          } else {
            mbar_wait(bar(BAR_FULL0 + k % C::NST), (k / C::NST) & 1, kWaitLimitCycles);
          }
        }
        for (int bi = 0; bi < armed_part; ++bi)
          mbar_wait(full_blk(st, bi == 0 ? 4 : bi - 1), round & 1, kWaitLimitCycles);
        if (nq > 0) mbar_wait(bar(BAR_QFULL), (nq - 1) & 1, kWaitLimitCycles);
      }
      __syncwarp();
    } else if (warp == 1 || warp == 2) {
      // ================= MMA issuers: warp 1 QK, warp 2 PV =================
      // Two issuing warps keep the tensor pipe fed with QK(i + 1) while PV(i)
      // goes out: one warp issuing both left ~30 % of the pipe's rate unused
      // at these N (measured with a probe of the issue rate).
      constexpr uint32_t kIdQK = idesc_e4m3(128, NR, 0, 0);
      constexpr uint32_t kIdPV = idesc_e4m3(128, C::OW, 1, 1);
      bool ok = true;
      auto fail = [&]() {
        if (lane == 0) {
          report(p.status, MLA_ERR_TIMEOUT);
          *abort_flag = 1;
        }
      };
      // PV of tile j of an item (tile g of the CTA, KV in stage jst, P^T in
      // buffer pb); lane 0 issues.
      auto issue_pv = [&](int j, int g, int jst, int pb) {
        tc_fence_after();
        const uint32_t kv = sbase + C::kKV + jst * kTileBytes;
        const uint32_t pbuf = C::kPInStage ? kv + kRopeOffset : sbase + C::kP + pb * C::kPBytes;
#pragma unroll
        for (int d = 0; d < 4; ++d) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t a = smem_desc(kv + d * kLatBlockBytes + ks * 4096, 16384, 1024,
                                         kLayoutSW128);
            const uint32_t acc = (j > 0 || ks > 0) ? 1u : 0u;
            // B = P^T, MN-major: 16-row groups 2048 B apart (hi groups, then lo
            // groups), 8-token groups 128 B apart.
            const uint64_t bd = smem_desc(pbuf + ks * 512, 128, 2048, kLayoutNone);
            umma_f8(tmem + C::kOCol + d * C::OW, a, bd, kIdPV, acc);
            if constexpr (C::kWide) {
              // The lo term: a second MMA into the same O^T columns.
              const uint64_t bl = smem_desc(pbuf + C::kPHalf + ks * 512, 128, 2048, kLayoutNone);
              umma_f8(tmem + C::kOCol + d * C::OW, a, bl, kIdPV, 1u);
            }
          }
          // Latent block d of the stage is free once these MMAs complete.
          if constexpr (C::kBlockStages) umma_commit(empty_blk(jst, d));
        }
        if constexpr (!C::kBlockStages) umma_commit(bar(BAR_EMPTY0 + jst));
        if (!C::kPInStage) umma_commit(bar(BAR_PFREE0 + pb));
        umma_commit(bar((g & 1) ? C::kBarOdone1 : BAR_ODONE));
      };
      // One 32-dim K step of QK (KV in stage ist, S^T buffer sb): steps 0-15
      // the latent blocks, 16-17 the rope block.
      auto qk_step = [&](int ist, int sb, int kk, bool acc) {
        const uint32_t kv = sbase + C::kKV + ist * kTileBytes;
        uint64_t a, bd;
        if (kk < 16) {
          const int d = kk >> 2, sub = kk & 3;
          a = smem_desc(kv + d * kLatBlockBytes + sub * 32, 16, 1024, kLayoutSW128);
          bd = smem_desc(sbase + C::kQ + d * NR * 128 + sub * 32, 16, 1024, kLayoutSW128);
        } else {
          const int sub = kk - 16;
          a = smem_desc(kv + kRopeOffset + sub * 32, 16, 512, kLayoutSW64);
          bd = smem_desc(sbase + C::kQ + 4 * NR * 128 + sub * 32, 16, 512, kLayoutSW64);
        }
        umma_f8(tmem + sb * NR, a, bd, kIdQK, acc ? 1u : 0u);
      };
      // QK of tile i (KV in stage ist) into S buffer sb; lane 0 issues.
      auto issue_qk = [&](int ist, int sb) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 18; ++kk) qk_step(ist, sb, kk, kk > 0);
        umma_commit(bar(BAR_SFULL0 + sb));
      };
      if (warp == 1) {
        // QK(j) once its tile has landed, its S^T buffer is free and PV(j - 2)
        // has completed (so the softmax's wait for PV(j - 1) stays within one
        // phase of its barrier; QK(j) still overlaps PV(j - 1)).  Tile indices
        // for buffers and phases count across the CTA's items (g).
        int st = 0, round = 0, g = 0;
        int nq = 0;  // items started
        for (int n = 0; ok && (kPersist || n == 0); ++n) {
          ItemInfo item;
          const int r = next_item(n, item);
          if (r == 0) break;
          if (r == 1) continue;
          MLA_ITEM_NAMES(item);
          ++nq;
          bool w = mbar_wait_abort(bar(BAR_QFULL), (nq - 1) & 1, p.wait_cycles, abort_flag);
          ok = __all_sync(0xffffffffu, w && !*abort_flag);
          for (int j = 0; ok && j < n_tiles; ++j, ++g) {
            const int sb = (C::NS == 2) ? (g & 1) : 0;
            const int use = (C::NS == 2) ? (g >> 1) : g;
            // Block stages: the rope block arrives first.
            w = !expired_here(p, WAIT_TILE_FULL, j) &&
                mbar_wait_abort(C::kBlockStages ? full_blk(st, 4) : bar(BAR_FULL0 + st), round & 1,
                                p.wait_cycles, abort_flag);
            if (w && use >= 1)
              w = mbar_wait_abort(bar(BAR_SFREE0 + sb), (use - 1) & 1, p.wait_cycles, abort_flag);
            // The 96-row CTA needs no PV(g - 2) wait: its softmax waited for
            // PV(g - 2) (the P^T buffer) before writing P(g - 1), which keeps its
            // wait for PV(g - 1) within one phase; the tile's stage implies
            // PV(g - 2) anyway.
            if (w && g >= 2 && !C::kWide)
              w = mbar_wait_abort(bar(((g - 2) & 1) ? C::kBarOdone1 : BAR_ODONE),
                                  ((g - 2) >> 1) & 1, p.wait_cycles, abort_flag);
            w = __all_sync(0xffffffffu, w && !*abort_flag);
            if (!w) {
              ok = false;
              break;
            }
            // Rows loaded per page, as the producer published them with the
            // stage's full barrier (observed above).
            const uint32_t info =
                kGather ? *reinterpret_cast<volatile uint32_t*>(base + C::kStageInfo + 4 * st) : 0u;
            const int valid = tok_end - (t0 + j * kTileTokens);
            if constexpr (C::kBlockStages) {
              // Rope steps first, then each latent block's four steps as it
              // lands.  A tile with rows to zero (which span every block)
              // waits for all of it first.
              const bool partial = kGather ? (info != 0x20202020u) : (valid < kTileTokens);
              if (partial) {
                for (int blk = 0; w && blk < 4; ++blk)
                  w = mbar_wait_abort(full_blk(st, blk), round & 1, p.wait_cycles, abort_flag);
                w = __all_sync(0xffffffffu, w && !*abort_flag);
                if (!w) {
                  ok = false;
                  break;
                }
                zero_unloaded_rows<kGather>(base + C::kKV + st * kTileBytes, lane, info, valid);
              }
              if (lane == 0) {
                tc_fence_after();
                qk_step(st, sb, 16, false);
                qk_step(st, sb, 17, true);
              }
              __syncwarp();
              for (int blk = 0; blk < 4; ++blk) {
                if (!partial) {
                  w = mbar_wait_abort(full_blk(st, blk), round & 1, p.wait_cycles, abort_flag);
                  w = __all_sync(0xffffffffu, w && !*abort_flag);
                  if (!w) break;
                }
                if (lane == 0) {
                  tc_fence_after();
#pragma unroll
                  for (int sub = 0; sub < 4; ++sub) qk_step(st, sb, blk * 4 + sub, true);
                }
                __syncwarp();
              }
              if (!w) {
                ok = false;
                break;
              }
              // S^T is complete, and the rope block free, once these MMAs are.
              if (lane == 0) {
                umma_commit(bar(BAR_SFULL0 + sb));
                umma_commit(empty_blk(st, 4));
              }
              __syncwarp();
            } else {
              zero_unloaded_rows<kGather>(base + C::kKV + st * kTileBytes, lane, info, valid);
              if (lane == 0) issue_qk(st, sb);
              __syncwarp();
            }
            if (++st == C::NST) {
              st = 0;
              ++round;
            }
          }
          // Q is free for the next item once these QKs complete (also on the
          // way out: the drain below waits for it).
          if (lane == 0) umma_commit(bar(BAR_QFREE));
          __syncwarp();
        }
        if (!ok) fail();
        // This warp's MMAs complete before the CTA releases TMEM.
        if (nq > 0) mbar_wait(bar(BAR_QFREE), (nq - 1) & 1, kWaitLimitCycles);
      } else {
        // PV(i) as soon as its P^T is ready; the first PV of an item overwrites
        // O^T, so it waits until the softmax has read the previous item's.
        int st = 0, g = 0;
        int nq = 0;  // items started
        for (int n = 0; ok && (kPersist || n == 0); ++n) {
          ItemInfo item;
          const int r = next_item(n, item);
          if (r == 0) break;
          if (r == 1) continue;
          MLA_ITEM_NAMES(item);
          ++nq;
          if (nq > 1) {
            const bool w =
                mbar_wait_abort(bar(BAR_OFREE), (nq - 2) & 1, p.wait_cycles, abort_flag);
            ok = __all_sync(0xffffffffu, w && !*abort_flag);
          }
          for (int i = 0; ok && i < n_tiles; ++i, ++g) {
            const int pb = (C::NPB == 1) ? 0 : (g & 1);
            const int use = (C::NPB == 1) ? g : (g >> 1);
            bool w = !expired_here(p, WAIT_P_FULL, i) &&
                     mbar_wait_abort(bar(BAR_PFULL0 + pb), use & 1, p.wait_cycles, abort_flag);
            w = __all_sync(0xffffffffu, w && !*abort_flag);
            if (!w) {
              ok = false;
              break;
            }
            if (lane == 0) issue_pv(i, g, st, pb);
            __syncwarp();
            if (++st == C::NST) st = 0;
          }
          // One commit after the item's last PV: the epilogue reads O^T after
          // it (every QK result has been consumed by then).
          if (lane == 0) umma_commit(bar(BAR_FINAL));
          __syncwarp();
        }
        if (!ok) fail();
        // This warp's MMAs complete before the CTA releases TMEM.
        if (nq > 0) mbar_wait(bar(BAR_FINAL), (nq - 1) & 1, kWaitLimitCycles);
      }
    }
  } else {
    if constexpr (C::kWide) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegsHigh));
    // ===== softmax warpgroups (warps kSoftmaxWarp0 .. kSoftmaxWarp0 + 4*SWG - 1) =====
    // SWG warpgroups share each tile: warpgroup g owns rows [g*NRH, (g+1)*NRH)
    // of every token (two warps per SM sub-partition when SWG = 2, so one
    // warp's latency hides behind the other's).  TMEM lane quadrant = warp % 4.
    // Every warp passes the same sequence of named barriers whether or not a
    // wait ran out (a failed wait only turns `ok` off and skips the work), so a
    // timeout can never leave the group split across barriers.
    constexpr int NRH = C::NRH;
    constexpr int NT = 128 * C::SWG;
    const int quad = warp & 3;
    const int rbase = ((warp - C::kSoftmaxWarp0) >> 2) * NRH;  // first row of this warpgroup
    const int tok_lane = quad * 32 + lane;  // TMEM lane == token index within the tile
    const int sid = threadIdx.x - 32 * C::kSoftmaxWarp0;  // 0..NT-1
    // Owner of a row's state (reference, sum): thread `sid` of row `sid` up to
    // 48 rows; with 96 rows the first 32 threads of each warpgroup own its
    // rows, so that a warpgroup's vote and reference update synchronise only
    // its own 128 threads (named barriers per warpgroup).
    const int wgi = (warp - C::kSoftmaxWarp0) >> 2;
    const int own = C::kWide ? (((sid & 127) < NRH) ? rbase + (sid & 127) : -1)
                             : (sid < NR ? sid : -1);
    const uint32_t vote_bar = C::kWide ? kVoteBarrierWg0 + wgi : kVoteBarrier;
    const uint32_t smx_bar = C::kWide ? kSoftmaxBarrierWg0 + wgi : kSoftmaxBarrier;
    (void)vote_bar;
    (void)smx_bar;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    int g = 0;   // tiles of the CTA's earlier items (S^T / P^T buffer phases)
    int nq = 0;  // items started
    bool ok = true;
    for (int n = 0; kPersist || n == 0; ++n) {
      ItemInfo item;
      const int r = next_item(n, item);
      if (r == 0) break;
      if (r == 1) continue;
      MLA_ITEM_NAMES(item);
      ++nq;
      float k_row = -INFINITY;  // owner state: reference (integer, log2 units)
      float l_row = 0.0f;       // owner state: sum of weights relative to k_row - 8
      // This thread's copy of its rows' references; the 96-row configuration
      // reads its rows' thresholds and exponent offsets from shared memory
      // instead (owners write them only between B1 and B2, when every thread
      // has passed the tile's vote and none has reached its weights), which
      // keeps the 32-row thread within its registers.
      float kreg[C::kWide ? 1 : NRH];
#pragma unroll
      for (int k = 0; k < (C::kWide ? 1 : NRH); ++k) kreg[k] = -INFINITY;
      // 96 rows: this thread's sums of its token's weights per row, relative to
      // the row's current reference (reduced once, after the last tile).
      float lsum[C::kWide ? NRH : 1];
#pragma unroll
      for (int k = 0; k < (C::kWide ? NRH : 1); ++k) lsum[k] = 0.0f;
      const float c = c_log2;
      // Smallest visibility limit over this group's rows (MTP verify: the first
      // query token of the block sees the fewest keys).
      const int qi_first = row0 / p.num_heads;
      const int lim_min = p.causal ? min(tok_end, L - q_b + qi_first + 1) : tok_end;
      const int my_row0 = row0 + rbase;  // first request row of this warpgroup
      const int my_rows = max(0, min(NRH, rows_valid - rbase));
      // Selection: logical page ids of 8 tiles' compact pages, one per lane
      // (this warp's token page is page `quad` of its tile).
      auto sel_window = [&](int w) -> int {
        const int cp = t0 / MLA_PAGE_SIZE + w * 32 + lane;
        return (cp < p.topk) ? p.block_idx[static_cast<int64_t>(b) * p.topk + cp] : -1;
      };
      int sel_cur = -1, sel_next = -1;
      if (sparse) {
        sel_cur = sel_window(0);
        sel_next = sel_window(1);
      }
      // Scale the scores of tile i by c and mask them (-inf): rows past the real
      // query rows, tokens past the split, and (MTP verify) tokens after the
      // row's query position; with restricted key sets the key position decides.
      auto scale_mask = [&](float (&t)[NRH], int i) {
        const int tile_tok0 = t0 + i * kTileTokens;
        const int j = tile_tok0 + tok_lane;
        if constexpr (kGather) {
          // Restricted key sets: the token's key position decides.
          int64_t pos = j;
          bool tok_ok = j < tok_end;
          if (sparse) {
            if (i > 0 && (i & 7) == 0) {
              sel_cur = sel_next;
              sel_next = sel_window((i >> 3) + 1);
            }
            const int lp = __shfl_sync(0xffffffffu, sel_cur, (i & 7) * 4 + quad);
            pos = static_cast<int64_t>(lp) * MLA_PAGE_SIZE + lane;
            tok_ok = tok_ok && lp >= 0;
          }
          tok_ok = tok_ok && pos >= win_lo && pos < win_hi;
          int qi = my_row0 / p.num_heads;
          int h = my_row0 - qi * p.num_heads;
#pragma unroll
          for (int k = 0; k < NRH; ++k) {
            const bool vis = tok_ok && k < my_rows && (!p.causal || pos < L - q_b + qi + 1);
            t[k] = vis ? t[k] * c : -INFINITY;
            if (++h == p.num_heads) {
              h = 0;
              ++qi;
            }
          }
        } else if (tile_tok0 + kTileTokens <= lim_min) {
#pragma unroll
          for (int k = 0; k < NRH; ++k) t[k] = (k < my_rows) ? t[k] * c : -INFINITY;
        } else {
          int qi = my_row0 / p.num_heads;
          int h = my_row0 - qi * p.num_heads;
#pragma unroll
          for (int k = 0; k < NRH; ++k) {
            const int lim = p.causal ? min(tok_end, L - q_b + qi + 1) : tok_end;
            t[k] = (k < my_rows && j < lim) ? t[k] * c : -INFINITY;
            if (++h == p.num_heads) {
              h = 0;
              ++qi;
            }
          }
        }
      };
      if constexpr (C::kWide) {
        // 96 rows: each thread holds 32 rows of one token.  Per tile: load S^T
        // and free it, scale and mask, vote on the rows' thresholds (k + 0.75,
        // from shared memory), then weights from the rows' integer exponent
        // offsets (softmax_weight_kc), the row sums of this thread, and P^T as
        // hi and lo E4M3 terms through packed halves.
        float* thr = kref;                                  // k + 0.75 per row
        int* kci = reinterpret_cast<int*>(base + C::kKci);  // exponent offset per row
        for (int i = 0; i < n_tiles; ++i) {
          if (ok)
            ok = !expired_here(p, WAIT_S_FULL, i) &&
                 mbar_wait_abort(bar(BAR_SFULL0), (g + i) & 1, p.wait_cycles, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok && lane == 0) *abort_flag = 1;  // the other roles stop waiting
          float t[NRH];
          if (ok) {
            tc_fence_after();
            uint32_t r[NRH];
#pragma unroll
            for (int cc = 0; cc < NRH / 16; ++cc)
              tmem_ld16(tmem + lane_addr + rbase + cc * 16,
                        *reinterpret_cast<uint32_t(*)[16]>(&r[cc * 16]));
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < NRH; ++k) t[k] = __uint_as_float(r[k]);
            tc_fence_before();
            mbar_arrive(bar(BAR_SFREE0));
          } else {
#pragma unroll
            for (int k = 0; k < NRH; ++k) t[k] = 0.0f;
          }
          if (!kGather && my_rows == NRH && t0 + i * kTileTokens + kTileTokens <= lim_min) {
#pragma unroll
            for (int k = 0; k < NRH; ++k) t[k] *= c;
          } else {
            scale_mask(t, i);
          }
          // Vote: does some score exceed its row's threshold?
          bool over = false;
#pragma unroll
          for (int k4 = 0; k4 < NRH / 4; ++k4) {
            const float4 th = *reinterpret_cast<const float4*>(thr + rbase + 4 * k4);
            over |= (t[4 * k4] > th.x) | (t[4 * k4 + 1] > th.y) | (t[4 * k4 + 2] > th.z) |
                    (t[4 * k4 + 3] > th.w);
          }
          const bool any_over = bar_sync_or(vote_bar, 128, over);
          if (any_over) {
            {
              float tm[NRH];
#pragma unroll
              for (int k = 0; k < NRH; ++k) tm[k] = t[k];
              warp_reduce_rows<NRH, true>(tm, lane, red_max + quad * NR + rbase);
            }
            named_bar_sync(smx_bar, 128);  // B1: tile maxima ready
            if (own >= 0) {
              const float mt = fmaxf(fmaxf(red_max[own], red_max[NR + own]),
                                     fmaxf(red_max[2 * NR + own], red_max[3 * NR + own]));
              float k_new = k_row;
              if (mt > k_row + 0.75f) k_new = ceilf(mt);
              float alpha = 1.0f;
              if (k_new != k_row && k_row != -INFINITY) {
                const int e = static_cast<int>(k_row - k_new);
                alpha = (e < -126) ? 0.0f : pow2i(e);
              }
              k_row = k_new;
              thr[own] = k_new + 0.75f;
              kci[own] = (k_new == -INFINITY) ? kKcNone
                                              : 135 - 0x4B400000 - static_cast<int>(k_new);
              alpha_s[own] = alpha;
            }
            named_bar_sync(smx_bar, 128);  // B2: references ready
            // This thread's sums follow their rows' references; a row whose
            // reference moved needs its O^T columns rescaled (the same answer
            // for every thread of the warpgroup).
            bool corr = false;
#pragma unroll
            for (int k = 0; k < NRH; ++k) {
              const float al = alpha_s[rbase + k];
              lsum[k] *= al;
              corr |= al != 1.0f;
            }
            if (ok && corr && i > 0) {
              // Rescale the O^T columns of rows whose reference moved (rare),
              // once PV(i - 1) is done (its completion barrier is within one
              // phase of the awaited one, as in the other configurations).
              ok = mbar_wait_abort(bar(((g + i - 1) & 1) ? C::kBarOdone1 : BAR_ODONE),
                                   ((g + i - 1) >> 1) & 1, p.wait_cycles, abort_flag);
              ok = __all_sync(0xffffffffu, ok);
              if (ok) {
                tc_fence_after();
#pragma unroll 1
                for (int d = 0; d < 4; ++d) {
#pragma unroll
                  for (int cc = 0; cc < NRH / 8; ++cc) {
                    uint32_t r[8];
                    const uint32_t addr = tmem + lane_addr + C::kOCol + d * C::OW + rbase + cc * 8;
                    tmem_ld8(addr, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                      r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha_s[rbase + cc * 8 + k]);
                    tmem_st8(addr, r);
                  }
                }
                tmem_st_wait();
              }
            }
          }
          // Weights 2^(t - k + 8) and this thread's row sums.
#pragma unroll
          for (int k4 = 0; k4 < NRH / 4; ++k4) {
            const int4 kc = *reinterpret_cast<const int4*>(kci + rbase + 4 * k4);
            t[4 * k4] = softmax_weight_kc(t[4 * k4], kc.x);
            t[4 * k4 + 1] = softmax_weight_kc(t[4 * k4 + 1], kc.y);
            t[4 * k4 + 2] = softmax_weight_kc(t[4 * k4 + 2], kc.z);
            t[4 * k4 + 3] = softmax_weight_kc(t[4 * k4 + 3], kc.w);
          }
#pragma unroll
          for (int k = 0; k < NRH; ++k) lsum[k] += t[k];
          // P^T (one buffer): wait until PV(i - 1) has read it.
          if (ok && expired_here(p, WAIT_P_FREE, i)) ok = false;
          if (ok && g + i >= 1)
            ok = mbar_wait_abort(bar(BAR_PFREE0), (g + i - 1) & 1, p.wait_cycles, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok && lane == 0) *abort_flag = 1;
          if (ok) {
            // MN-major [term][NR/16 row groups][128 tokens][16 rows]: one
            // 16-byte store per term and 16-row group.
            uint8_t* pbuf = base + C::kP;
#pragma unroll
            for (int g = 0; g < NRH / 16; ++g) {
              uint32_t h[8], l[8];
#pragma unroll
              for (int m = 0; m < 8; ++m)
                split_e4m3x2_h(t[g * 16 + 2 * m], t[g * 16 + 2 * m + 1], h[m], l[m]);
              const uint4 vh = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16),
                                          h[4] | (h[5] << 16), h[6] | (h[7] << 16));
              const uint4 vl = make_uint4(l[0] | (l[1] << 16), l[2] | (l[3] << 16),
                                          l[4] | (l[5] << 16), l[6] | (l[7] << 16));
              const uint32_t off = ((rbase >> 4) + g) * 2048 + tok_lane * 16;
              *reinterpret_cast<uint4*>(pbuf + off) = vh;
              *reinterpret_cast<uint4*>(pbuf + C::kPHalf + off) = vl;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(BAR_PFULL0));
          }
        }
      } else {
        for (int i = 0; i < n_tiles; ++i) {
          const int sb = (C::NS == 2) ? ((g + i) & 1) : 0;
          const int use = (C::NS == 2) ? ((g + i) >> 1) : (g + i);
          if (ok)
            ok = !expired_here(p, WAIT_S_FULL, i) &&
                 mbar_wait_abort(bar(BAR_SFULL0 + sb), use & 1, p.wait_cycles, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok && lane == 0) *abort_flag = 1;  // the other roles stop waiting
          float t[NRH];
          if (ok) {
            tc_fence_after();
            uint32_t r[NRH];
#pragma unroll
            for (int cc = 0; cc < NRH / 8; ++cc)
              tmem_ld8(tmem + lane_addr + sb * NR + rbase + cc * 8,
                       *reinterpret_cast<uint32_t(*)[8]>(&r[cc * 8]));
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < NRH; ++k) t[k] = __uint_as_float(r[k]);
            tc_fence_before();
            mbar_arrive(bar(BAR_SFREE0 + sb));
          } else {
#pragma unroll
            for (int k = 0; k < NRH; ++k) t[k] = 0.0f;
          }
          scale_mask(t, i);
          // Reference check.  A row's reference k only has to bound its scores:
          // with p = 2^(t - k + 8), E4M3 holds p up to 448 = 2^8.8, so any k with
          // t <= k + 0.75 works.  One vote finds whether some score of the tile
          // exceeds its row's reference; only then (always on the first tile)
          // are the tile maxima reduced and references raised to ceil(max).
          bool over = false;
#pragma unroll
          for (int k = 0; k < NRH; ++k) over |= t[k] > kreg[k] + 0.75f;
          const bool any_over = bar_sync_or(kVoteBarrier, NT, over);
          // Owners fold the previous tile's row sums (relative to its reference).
          if (sid < NR && i > 0) {
            const float* rs = red_sum + ((i - 1) & 1) * 4 * NR;
            l_row += (rs[sid] + rs[NR + sid]) + (rs[2 * NR + sid] + rs[3 * NR + sid]);
          }
          if (any_over) {
            {
              float tm[NRH];
#pragma unroll
              for (int k = 0; k < NRH; ++k) tm[k] = t[k];
              warp_reduce_rows<NRH, true>(tm, lane, red_max + quad * NR + rbase);
            }
            // The correction flag: cleared before B1 (every read of its last
            // value happened before this tile's vote), set by owners after B1,
            // read by all after B2.
            if (sid == 0) flags[0] = 0;
            named_bar_sync(kSoftmaxBarrier, NT);  // B1: tile maxima ready
            if (sid < NR) {
              const float mt = fmaxf(fmaxf(red_max[sid], red_max[NR + sid]),
                                     fmaxf(red_max[2 * NR + sid], red_max[3 * NR + sid]));
              float k_new = k_row;
              if (mt > k_row + 0.75f) k_new = ceilf(mt);
              float alpha = 1.0f;
              if (k_new != k_row && k_row != -INFINITY) {
                const int e = static_cast<int>(k_row - k_new);
                alpha = (e < -126) ? 0.0f : pow2i(e);
                flags[0] = 1;
              }
              l_row *= alpha;
              k_row = k_new;
              kref[sid] = k_new;
              alpha_s[sid] = alpha;
            }
            named_bar_sync(kSoftmaxBarrier, NT);  // B2: references ready
#pragma unroll
            for (int k = 0; k < NRH; ++k) kreg[k] = kref[rbase + k];
            const bool corr = flags[0] != 0;
            if (ok && corr && i > 0) {
              // Rescale the O^T columns (hi and lo) of rows whose reference moved
              // (rare), once PV(i-1) is done.  PV completions alternate between
              // two barriers, and the one of PV(i-1)'s parity is within one phase
              // of the awaited one: s_full(i) implies PV(i-2) completed (QK(i)
              // waits for it) and PV(i+1) needs a later tile's P^T.
              ok = mbar_wait_abort(bar(((g + i - 1) & 1) ? C::kBarOdone1 : BAR_ODONE),
                                   ((g + i - 1) >> 1) & 1, p.wait_cycles, abort_flag);
              ok = __all_sync(0xffffffffu, ok);
              if (ok) {
                tc_fence_after();
#pragma unroll 1
                for (int d = 0; d < 4; ++d) {
#pragma unroll
                  for (int half = 0; half < 2; ++half) {
#pragma unroll
                    for (int cc = 0; cc < NRH / 8; ++cc) {
                      uint32_t r[8];
                      const uint32_t addr =
                          tmem + lane_addr + C::kOCol + d * C::OW + half * NR + rbase + cc * 8;
                      tmem_ld8(addr, r);
                      tmem_ld_wait();
#pragma unroll
                      for (int k = 0; k < 8; ++k)
                        r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha_s[rbase + cc * 8 + k]);
                      tmem_st8(addr, r);
                    }
                  }
                }
                tmem_st_wait();
              }
            }
          }
          // Weights 2^(t - k + 8), exact power-of-two scaling.
#pragma unroll
          for (int k = 0; k < NRH; ++k) t[k] = softmax_weight<(C::SWG > 1)>(t[k], kreg[k]);
          // P^T as two E4M3 terms into shared memory, MN-major:
          // [term][NR/16 row groups][128 tokens][16 rows]; this thread writes its
          // token's bytes for rows rbase .. rbase + NRH, 16 (or 8) rows per store.
          // P barriers (and buffers) alternate by tile parity; the PV issuer
          // uses the same rule.
          const int pb = (g + i) & 1;
          const int puse = (g + i) >> 1;
          if (ok && !C::kPInStage && expired_here(p, WAIT_P_FREE, i)) ok = false;
          if (ok && !C::kPInStage && puse >= 1)
            ok = mbar_wait_abort(bar(BAR_PFREE0 + pb), (puse - 1) & 1, p.wait_cycles, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok && lane == 0) *abort_flag = 1;
          if (ok) {
            // P^T of tile i goes to the rope block of its KV stage (consumed by
            // QK(i), which s_full(i) reports complete) or to a P buffer.
            uint8_t* pbuf = C::kPInStage
                                ? base + C::kKV + ((g + i) % C::NST) * kTileBytes + kRopeOffset
                                : base + C::kP + pb * C::kPBytes;
            if constexpr (NRH % 16 == 0) {
              // Whole 16-row groups: one 16-byte store per term and group, the
              // warp's 32 tokens covering 512 contiguous bytes (no bank conflict).
#pragma unroll
              for (int g = 0; g < NRH / 16; ++g) {
                const int row = rbase + g * 16;
                uint4 vh, vl;
                split_e4m3x4(&t[g * 16 + 0], vh.x, vl.x);
                split_e4m3x4(&t[g * 16 + 4], vh.y, vl.y);
                split_e4m3x4(&t[g * 16 + 8], vh.z, vl.z);
                split_e4m3x4(&t[g * 16 + 12], vh.w, vl.w);
                const uint32_t off = (row >> 4) * 2048 + tok_lane * 16;
                *reinterpret_cast<uint4*>(pbuf + off) = vh;
                *reinterpret_cast<uint4*>(pbuf + C::kPHalf + off) = vl;
              }
            } else {
#pragma unroll
              for (int g = 0; g < NRH / 8; ++g) {
                const int row = rbase + g * 8;
                uint2 vh, vl;
                split_e4m3x4(&t[g * 8 + 0], vh.x, vl.x);
                split_e4m3x4(&t[g * 8 + 4], vh.y, vl.y);
                const uint32_t off = (row >> 4) * 2048 + tok_lane * 16 + (row & 15);
                *reinterpret_cast<uint2*>(pbuf + off) = vh;
                *reinterpret_cast<uint2*>(pbuf + C::kPHalf + off) = vl;
              }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(BAR_PFULL0 + pb));
          }
          // Row sums of the unquantised weights, reduced per tile and folded in
          // by the owners after the next tile's vote (double-buffered by tile
          // parity).
          warp_reduce_rows<NRH, false>(t, lane, red_sum + (i & 1) * 4 * NR + quad * NR + rbase);
        }
      }
      if (!ok && lane == 0) {
        report(p.status, MLA_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // ---- epilogue ----
      if constexpr (C::kWide) {
        // The per-thread sums, reduced over the 32 tokens of each warp; the
        // owners add the four lane quadrants below.
        warp_reduce_rows<NRH, false>(lsum, lane, red_sum + quad * NR + rbase);
      }
      named_bar_sync(kSoftmaxBarrier, NT);
      const bool single = (nsplit == 1);
      float* scale_s = alpha_s;
      if (own >= 0) {
        if (n_tiles > 0) {
          const float* rs = red_sum + (C::kWide ? 0 : ((n_tiles - 1) & 1) * 4 * NR);
          l_row += (rs[own] + rs[NR + own]) + (rs[2 * NR + own] + rs[3 * NR + own]);
        }
        const float m_s = (k_row == -INFINITY) ? -INFINITY : k_row - 8.0f;
        const int64_t grow = static_cast<int64_t>(b) * p.rows_per_req + row0 + own;
        float sc = 0.0f;
        if (own < rows_here) {
          if (single) {
            // A sink is one more (zero-valued) key: it joins the denominator.
            const float sink2 = p.sinks
                                    ? p.sinks[(row0 + own) % p.num_heads] * 1.4426950408889634f
                                    : -INFINITY;
            const float mm = fmaxf(l_row > 0.0f ? m_s : -INFINITY, sink2);
            const float a = (l_row > 0.0f) ? exp2f(m_s - mm) : 0.0f;
            const float den = l_row * a + (sink2 == -INFINITY ? 0.0f : exp2f(sink2 - mm));
            const float ls = (den > 0.0f) ? 0.6931471805599453f * (mm + log2f(den)) : -INFINITY;
            if (p.lse) p.lse[grow] = ls;
            sc = (den > 0.0f) ? kv_scale * p.output_scale * a / den : 0.0f;
          } else {
            float* ml = p.ws_ml + (grow * p.max_splits + split) * 2;
            ml[0] = m_s;
            ml[1] = l_row;
            sc = kv_scale;
          }
        }
        scale_s[own] = sc;
        // The 96-row configuration's thresholds and exponent offsets start the
        // next item with no reference (every thread is past its last read).
        if constexpr (C::kWide) {
          kref[own] = -INFINITY;
          reinterpret_cast<int*>(base + C::kKci)[own] = kKcNone;
        }
      }
      named_bar_sync(kSoftmaxBarrier, NT);
      // The PV warp commits BAR_FINAL once per item, after its last PV.
      bool fin = !expired_here(p, WAIT_FINAL, 0) &&
                 mbar_wait(bar(BAR_FINAL), (nq - 1) & 1, p.wait_cycles);
      fin = __all_sync(0xffffffffu, fin);
      if (!fin && lane == 0) report(p.status, MLA_ERR_TIMEOUT);
      if (ok && fin && n_tiles > 0) {
        tc_fence_after();
        // Per latent block: every column of this warpgroup's rows (and their
        // lo products up to 48 rows) in one batch of TMEM loads and one wait,
        // then the stores.  Row k of the warpgroup goes to base + k * stride.
        const int64_t grow0 = static_cast<int64_t>(b) * p.rows_per_req + row0 + rbase;
        const int64_t stride = single ? MLA_LATENT_DIM
                                      : static_cast<int64_t>(p.max_splits) * MLA_LATENT_DIM;
        float* const obase = single ? nullptr
                                    : p.ws_o + (grow0 * p.max_splits + split) * MLA_LATENT_DIM;
        const int nrow = min(NRH, rows_here - rbase);  // rows of this warpgroup to store
        // With a P^T buffer to spare (free after the item's last PV), each
        // warp turns its 32 dims x 8 rows at a time around through 1 KB of it,
        // so that a lane stores 4 contiguous dims of a row (16 B of a partial,
        // 8 B of BF16 output) instead of one dim of each of four rows.
        float* const scr = reinterpret_cast<float*>(base + C::kP) +
                           (warp - C::kSoftmaxWarp0) * 256;
        constexpr bool transpose = !C::kPInStage;
        // The rows' scales in registers: read from shared memory inside the
        // store loops, each would wait behind the previous row's stores (the
        // compiler cannot tell the two shared-memory pointers apart).
        float sc_r[NRH];
#pragma unroll
        for (int k = 0; k < NRH; ++k) sc_r[k] = scale_s[rbase + k];
#pragma unroll 1
        for (int d = 0; d < 4; ++d) {
          const int dim = d * 128 + tok_lane;
          uint32_t r[NRH], r2[C::kWide ? 1 : NRH];
          const uint32_t addr = tmem + lane_addr + C::kOCol + d * C::OW + rbase;
#pragma unroll
          for (int cc = 0; cc < NRH / 8; ++cc) {
            tmem_ld8(addr + cc * 8, *reinterpret_cast<uint32_t(*)[8]>(&r[cc * 8]));
            if constexpr (!C::kWide)  // the lo term's product
              tmem_ld8(addr + NR + cc * 8, *reinterpret_cast<uint32_t(*)[8]>(&r2[cc * 8]));
          }
          tmem_ld_wait();
          if constexpr (transpose) {
            const int dim4 = d * 128 + quad * 32 + (lane & 7) * 4;  // this lane's 4 dims
#pragma unroll
            for (int c8 = 0; c8 < NRH / 8; ++c8) {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const int k = c8 * 8 + kk;
                const float o = C::kWide ? __uint_as_float(r[k])
                                         : __uint_as_float(r[k]) + __uint_as_float(r2[k]);
                scr[kk * 32 + lane] = o * sc_r[k];
              }
              __syncwarp();
#pragma unroll
              for (int m = 0; m < 2; ++m) {
                const int kk = m * 4 + (lane >> 3);
                const float4 v4 = *reinterpret_cast<const float4*>(scr + kk * 32 + (lane & 7) * 4);
                const int k = c8 * 8 + kk;
                if (k < nrow) {
                  if (single) {
                    const int64_t off = (grow0 + k) * MLA_LATENT_DIM + dim4;
                    __nv_bfloat162 lo2 = __floats2bfloat162_rn(v4.x, v4.y);
                    __nv_bfloat162 hi2 = __floats2bfloat162_rn(v4.z, v4.w);
                    uint2 packed;
                    packed.x = *reinterpret_cast<uint32_t*>(&lo2);
                    packed.y = *reinterpret_cast<uint32_t*>(&hi2);
                    *reinterpret_cast<uint2*>(p.out + off) = packed;
                    if (p.out_f32) *reinterpret_cast<float4*>(p.out_f32 + off) = v4;
                  } else {
                    *reinterpret_cast<float4*>(obase + k * stride + dim4) = v4;
                  }
                }
              }
              __syncwarp();
            }
          } else {
#pragma unroll
            for (int k = 0; k < NRH; ++k) {
              if (k < nrow) {
                const float o = C::kWide ? __uint_as_float(r[k])
                                         : __uint_as_float(r[k]) + __uint_as_float(r2[k]);
                const float v = o * sc_r[k];
                if (single) {
                  const int64_t off = (grow0 + k) * MLA_LATENT_DIM + dim;
                  p.out[off] = __float2bfloat16_rn(v);
                  if (p.out_f32) p.out_f32[off] = v;
                } else {
                  obase[k * stride + dim] = v;
                }
              }
            }
          }
        }
      } else if (ok && fin && n_tiles == 0 && single) {
        // No key of this split is visible to any row here (padding query slots,
        // an empty window or selection): O = 0.  Partials need only (-inf, 0),
        // written above; the merge gives such slots weight 0 without reading O.
#pragma unroll 1
        for (int d = 0; d < 4; ++d) {
          const int dim = d * 128 + tok_lane;
          for (int row = rbase; row < min(rows_here, rbase + NRH); ++row) {
            const int64_t grow = static_cast<int64_t>(b) * p.rows_per_req + row0 + row;
            p.out[grow * MLA_LATENT_DIM + dim] = __float2bfloat16_rn(0.0f);
            if (p.out_f32) p.out_f32[grow * MLA_LATENT_DIM + dim] = 0.0f;
          }
        }
      }
      // Persistent CTAs: every warp is done with its P^T scratch before any
      // writes the next item's P^T.
      if (kPersist && !C::kPInStage) named_bar_sync(kSoftmaxBarrier, NT);
      // O^T has been read: the next item's first PV may overwrite it.
      tc_fence_before();
      mbar_arrive(bar(BAR_OFREE));
      g += n_tiles;
      if (!ok) break;  // after a wait ran out the remaining items are not run
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  // This CTA's partials are written: the merge may start once every CTA is here.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#undef MLA_ITEM_NAMES



// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D uint8 view [rows, 576] with a (box_x, box_y) box.
static bool make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint32_t box_x,
                     uint32_t box_y, CUtensorMapSwizzle sw) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {MLA_HEAD_DIM, rows};
  cuuint64_t strides[1] = {MLA_HEAD_DIM};
  cuuint32_t box[2] = {box_x, box_y};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NR, bool kGather, int kMode>
static cudaError_t launch_split_t(const void* q, const void* kv, int64_t num_pages, int batch,
                                int groups, int num_ctas, const DecodeParams& prm,
                                cudaStream_t stream) {
  using C = Cfg<NR>;
  static std::atomic<uint64_t> attr_done{0};
  {
    const cudaError_t e = ensure_smem_attr(mla_split_kv_kernel<NR, kGather, kMode>,
                                           static_cast<int>(C::kSmemBytes), attr_done);
    if (e != cudaSuccess) return e;
  }
  if constexpr (C::kWide) {
    // setmaxnreg.inc waits until the registers exist: launch only if the
    // kernel's register count covers the split.
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, mla_split_kv_kernel<NR, kGather, kMode>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * C::kThreads < C::kRegsLow * 128 + C::kRegsHigh * 128 * C::SWG)
      return cudaErrorInvalidConfiguration;
  }
  CUtensorMap kv_lat, kv_rope, q_lat, q_rope;
  const uint64_t kv_rows = static_cast<uint64_t>(num_pages) * MLA_PAGE_SIZE;
  const uint64_t q_rows = static_cast<uint64_t>(batch) * prm.rows_per_req;
  if (!make_map(&kv_lat, kv, kv_rows, 128, MLA_PAGE_SIZE, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&kv_rope, kv, kv_rows, 64, MLA_PAGE_SIZE, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&q_lat, q, q_rows, 128, NR, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&q_rope, q, q_rows, 64, NR, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  // Persistent: num_ctas CTAs loop over the prm.num_items items of the list.
  const dim3 grid = kMode != 0 ? dim3(num_ctas) : dim3(batch, prm.max_splits * groups);
  mla_split_kv_kernel<NR, kGather, kMode>
      <<<grid, C::kThreads, C::kSmemBytes, stream>>>(kv_lat, kv_rope, q_lat, q_rope, prm);
  return cudaGetLastError();
}

template <int NR, bool kGather>
static cudaError_t launch_split(const void* q, const void* kv, int64_t num_pages, int batch,
                                int groups, int num_ctas, const DecodeParams& prm,
                                cudaStream_t stream) {
  // The item-list mapping and the persistent loop are their own
  // instantiations, so the grid variant's code is what it is without them.
  if (!prm.cta_items)
    return launch_split_t<NR, kGather, 0>(q, kv, num_pages, batch, groups, num_ctas, prm, stream);
  if (num_ctas < prm.num_items)
    return launch_split_t<NR, kGather, 2>(q, kv, num_pages, batch, groups, num_ctas, prm, stream);
  return launch_split_t<NR, kGather, 1>(q, kv, num_pages, batch, groups, num_ctas, prm, stream);
}

std::atomic<long long> g_wait_cycles{0};
std::atomic<int> g_debug_expire{-1};

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

int cuda_fail(const char* what, cudaError_t e) {
  set_error(std::string(what) + ": " + cudaGetErrorString(e));
  return MLA_ERR_CUDA;
}

}  // namespace mla

using namespace mla;

namespace mla {

// Validated launch state shared by mla_decode, mla_decode_splitkv and
// mla_decode_merge.
struct DecodeLaunch {
  DecodeParams prm;
  MergeParams mp;
  RowGroups rg;
  int batch;
  int kv_split;
  int max_splits;
  int num_ctas;  // length of prm.cta_items (0 without an item list)
  int phases = MLA_PHASE_ALL;
};

static int prepare_decode(const void* q_fp8, const void* kv_pages_fp8, int64_t num_pages,
                          const int32_t* page_table, int32_t max_pages_per_req,
                          const int32_t* kv_lens, const int32_t* splits, const int32_t* chunks,
                          int32_t max_splits, int32_t kv_split, int32_t batch, int32_t q_len,
                          int32_t num_heads, int32_t causal, float q_scale, float kv_scale,
                          float softmax_scale, void* workspace, size_t workspace_bytes,
                          void* out_bf16, float* lse_f32, float* out_f32_debug,
                          const char* who, DecodeLaunch* dl) {
  const std::string w(who);
  if (!q_fp8 || !kv_pages_fp8 || !page_table || !kv_lens || !splits || !chunks || !workspace ||
      !out_bf16) {
    set_error(w + ": null pointer argument");
    return MLA_ERR_INVALID_ARG;
  }
  if (batch < 1 || q_len < 1 || num_heads < 1 || max_pages_per_req < 1 || num_pages < 1) {
    set_error(w + ": batch, q_len, num_heads, max_pages_per_req and num_pages must be >= 1");
    return MLA_ERR_INVALID_ARG;
  }
  if (static_cast<int64_t>(num_heads) * q_len > MLA_MAX_ROWS) {
    set_error(w + ": num_heads * q_len exceeds MLA_MAX_ROWS");
    return MLA_ERR_UNSUPPORTED;
  }
  if (batch > 65535) {
    set_error(w + ": batch exceeds 65535");
    return MLA_ERR_UNSUPPORTED;
  }
  if (num_pages * MLA_PAGE_SIZE > INT32_MAX) {
    set_error(w + ": page pool too large for 32-bit TMA row coordinates");
    return MLA_ERR_UNSUPPORTED;
  }
  if (max_splits < 1 || max_splits > MLA_MAX_SPLITS) {
    set_error(w + ": max_splits must be in [1, MLA_MAX_SPLITS]");
    return MLA_ERR_INVALID_ARG;
  }
  if (kv_split != 1 && kv_split != 2 && kv_split != 4 && kv_split != 8 && kv_split != 16) {
    set_error(w + ": kv_split must be 1, 2, 4, 8 or 16");
    return MLA_ERR_INVALID_ARG;
  }
  if (!aligned(q_fp8, 16) || !aligned(kv_pages_fp8, 16) || !aligned(workspace, 256) ||
      !aligned(out_bf16, 8) || (out_f32_debug && !aligned(out_f32_debug, 16))) {
    set_error(w + ": q/kv need 16-byte, workspace 256-byte, outputs 8/16-byte alignment");
    return MLA_ERR_INVALID_ARG;
  }
  if (!(std::isfinite(q_scale) && std::isfinite(kv_scale) && std::isfinite(softmax_scale))) {
    set_error(w + ": scales must be finite");
    return MLA_ERR_INVALID_ARG;
  }
  const int64_t rows_total = static_cast<int64_t>(batch) * q_len * num_heads;
  const size_t need = ws_total(rows_total, max_splits);
  if (workspace_bytes < need) {
    set_error(w + ": workspace of " + std::to_string(workspace_bytes) + " bytes is below the " +
              std::to_string(need) + " required");
    return MLA_ERR_WORKSPACE_TOO_SMALL;
  }
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  dl->rg = row_groups_fp8(num_heads * q_len);
  dl->batch = batch;
  dl->kv_split = kv_split;
  dl->max_splits = max_splits;
  DecodeParams& prm = dl->prm;
  prm.page_table = page_table;
  prm.kv_lens = kv_lens;
  prm.splits = splits;
  prm.chunks = chunks;
  prm.num_pages = num_pages;
  prm.max_pages = max_pages_per_req;
  prm.max_splits = max_splits;
  prm.q_len = q_len;
  prm.num_heads = num_heads;
  prm.causal = causal ? 1 : 0;
  prm.rows_per_req = num_heads * q_len;
  prm.rows_per_group = dl->rg.rows;
  prm.c_log2 = static_cast<float>(static_cast<double>(softmax_scale) * q_scale * kv_scale *
                                  1.4426950408889634);
  prm.kv_scale = kv_scale;
  prm.q_scale_dev = nullptr;
  prm.kv_scale_dev = nullptr;
  prm.sm_scale_dev = nullptr;
  prm.q_scale_h = q_scale;
  prm.sm_scale_h = softmax_scale;
  prm.output_scale = 1.0f;
  prm.sinks = nullptr;
  prm.query_lens = nullptr;
  prm.kv_bounds = nullptr;
  prm.block_idx = nullptr;
  prm.topk = 0;
  prm.cta_items = nullptr;
  prm.num_items = 0;
  prm.batch = batch;
  dl->num_ctas = 0;
  {
    const long long w = g_wait_cycles.load();
    prm.wait_cycles = w > 0 ? w : kWaitLimitCycles;
  }
  prm.debug_expire = g_debug_expire.load();
  prm.status = reinterpret_cast<int*>(ws);
  prm.ws_ml = reinterpret_cast<float*>(ws + ws_ml_offset());
  prm.ws_o = reinterpret_cast<float*>(ws + ws_o_offset(rows_total, max_splits));
  prm.out = reinterpret_cast<__nv_bfloat16*>(out_bf16);
  prm.lse = lse_f32;
  prm.out_f32 = out_f32_debug;
  MergeParams& mp = dl->mp;
  mp.po = prm.ws_o;
  mp.pml = prm.ws_ml;
  mp.rows = static_cast<int32_t>(rows_total);
  mp.stride_s = max_splits;
  mp.uniform_s = max_splits;
  mp.splits = splits;
  mp.rows_per_req = num_heads * q_len;
  mp.num_heads = num_heads;
  mp.output_scale = 1.0f;
  mp.sinks = nullptr;
  mp.out = prm.out;
  mp.lse = lse_f32;
  mp.out_f32 = out_f32_debug;
  return MLA_OK;
}

// Options of mla_decode_ex / mla_decode_sparse (NULL = none).
static int apply_options(const mla_decode_options_t* o, const char* who, DecodeLaunch* dl) {
  if (!o) return MLA_OK;
  const std::string w(who);
  if (!std::isfinite(o->output_scale)) {
    set_error(w + ": output_scale must be finite");
    return MLA_ERR_INVALID_ARG;
  }
  if (o->cta_items) {
    const int64_t cap = static_cast<int64_t>(dl->batch) * dl->max_splits * dl->rg.groups;
    if (o->num_ctas < 1 || o->num_ctas > cap) {
      set_error(w + ": num_ctas must be in [1, batch * max_splits * row groups]");
      return MLA_ERR_INVALID_ARG;
    }
  }
  if (o->persistent_ctas < 0 || (o->persistent_ctas > 0 && !o->cta_items)) {
    set_error(w + ": persistent_ctas needs a CTA item list and must be >= 0");
    return MLA_ERR_INVALID_ARG;
  }
  if (o->phases != MLA_PHASE_ALL && o->phases != MLA_PHASE_SPLIT && o->phases != MLA_PHASE_MERGE) {
    set_error(w + ": phases must be MLA_PHASE_ALL, MLA_PHASE_SPLIT or MLA_PHASE_MERGE");
    return MLA_ERR_INVALID_ARG;
  }
  dl->phases = o->phases;
  dl->prm.q_scale_dev = o->q_scale_dev;
  dl->prm.kv_scale_dev = o->kv_scale_dev;
  dl->prm.sm_scale_dev = o->softmax_scale_dev;
  dl->prm.output_scale = o->output_scale;
  dl->prm.sinks = o->sinks;
  dl->prm.query_lens = o->query_lens;
  dl->prm.kv_bounds = o->kv_bounds;
  dl->prm.cta_items = o->cta_items;
  dl->prm.num_items = o->cta_items ? o->num_ctas : 0;
  // Persistent CTAs: at most one per item.
  dl->num_ctas = o->cta_items ? (o->persistent_ctas > 0 && o->persistent_ctas < o->num_ctas
                                     ? o->persistent_ctas
                                     : o->num_ctas)
                              : 0;
  dl->mp.output_scale = o->output_scale;
  dl->mp.sinks = o->sinks;
  return MLA_OK;
}

static int launch_decode_split(const void* q_fp8, const void* kv_pages_fp8, int64_t num_pages,
                               const DecodeLaunch& dl, cudaStream_t st) {
  cudaError_t e;
  const int b = dl.batch, g = dl.rg.groups;
  // Key windows and page selections take the masked-position variant.
  const bool gather = dl.prm.kv_bounds != nullptr || dl.prm.block_idx != nullptr;
  switch (dl.rg.nr) {
    case 16:
      e = gather ? launch_split<16, true>(q_fp8, kv_pages_fp8, num_pages, b, g, dl.num_ctas, dl.prm, st)
                 : launch_split<16, false>(q_fp8, kv_pages_fp8, num_pages, b, g, dl.num_ctas, dl.prm, st);
      break;
    case 32:
      e = gather ? launch_split<32, true>(q_fp8, kv_pages_fp8, num_pages, b, g, dl.num_ctas, dl.prm, st)
                 : launch_split<32, false>(q_fp8, kv_pages_fp8, num_pages, b, g, dl.num_ctas, dl.prm, st);
      break;
    case 48:
      e = gather ? launch_split<48, true>(q_fp8, kv_pages_fp8, num_pages, b, g, dl.num_ctas, dl.prm, st)
                 : launch_split<48, false>(q_fp8, kv_pages_fp8, num_pages, b, g, dl.num_ctas, dl.prm, st);
      break;
    case kMaxRowsPerCtaFp8:
      e = gather ? launch_split<kMaxRowsPerCtaFp8, true>(q_fp8, kv_pages_fp8, num_pages, b, g,
                                                         dl.num_ctas, dl.prm, st)
                 : launch_split<kMaxRowsPerCtaFp8, false>(q_fp8, kv_pages_fp8, num_pages, b, g,
                                                          dl.num_ctas, dl.prm, st);
      break;
    default:
      set_error("mla_decode: internal row grouping error");
      return MLA_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) return cuda_fail("mla_decode: split-KV launch", e);
  return MLA_OK;
}

static int launch_decode_merge(const DecodeLaunch& dl, cudaStream_t st) {
  if (dl.max_splits <= 1) return MLA_OK;  // every request was written directly
  cudaError_t e = launch_merge(dl.mp, dl.kv_split, st);
  if (e != cudaSuccess) return cuda_fail("mla_decode: merge launch", e);
  return MLA_OK;
}

// The phases an options structure asks for (both by default).
static int launch_decode_phases(const void* q_fp8, const void* kv_pages_fp8, int64_t num_pages,
                                const DecodeLaunch& dl, cudaStream_t st) {
  if (dl.phases != MLA_PHASE_MERGE) {
    const int rc = launch_decode_split(q_fp8, kv_pages_fp8, num_pages, dl, st);
    if (rc != MLA_OK) return rc;
  }
  return dl.phases == MLA_PHASE_SPLIT ? MLA_OK : launch_decode_merge(dl, st);
}

}  // namespace mla

#define MLA_DECODE_ARGS                                                                     \
  q_fp8, kv_pages_fp8, num_pages, page_table, max_pages_per_req, kv_lens, splits, chunks,   \
      max_splits, kv_split, batch, q_len, num_heads, causal, q_scale, kv_scale, softmax_scale, \
      workspace, workspace_bytes, out_bf16, lse_f32, out_f32_debug

extern "C" int mla_decode(const void* q_fp8, const void* kv_pages_fp8, int64_t num_pages,
                          const int32_t* page_table, int32_t max_pages_per_req,
                          const int32_t* kv_lens, const int32_t* splits, const int32_t* chunks,
                          int32_t max_splits, int32_t kv_split, int32_t batch, int32_t q_len,
                          int32_t num_heads, int32_t causal, float q_scale, float kv_scale,
                          float softmax_scale, void* workspace, size_t workspace_bytes,
                          void* out_bf16, float* lse_f32, float* out_f32_debug, void* stream) {
  DecodeLaunch dl;
  int rc = prepare_decode(MLA_DECODE_ARGS, "mla_decode", &dl);
  if (rc != MLA_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  rc = launch_decode_split(q_fp8, kv_pages_fp8, num_pages, dl, st);
  if (rc != MLA_OK) return rc;
  return launch_decode_merge(dl, st);
}

extern "C" int mla_decode_ex(const void* q_fp8, const void* kv_pages_fp8, int64_t num_pages,
                             const int32_t* page_table, int32_t max_pages_per_req,
                             const int32_t* kv_lens, const int32_t* splits, const int32_t* chunks,
                             int32_t max_splits, int32_t kv_split, int32_t batch, int32_t q_len,
                             int32_t num_heads, int32_t causal, float q_scale, float kv_scale,
                             float softmax_scale, void* workspace, size_t workspace_bytes,
                             void* out_bf16, float* lse_f32, float* out_f32_debug,
                             const mla_decode_options_t* options, void* stream) {
  DecodeLaunch dl;
  int rc = prepare_decode(MLA_DECODE_ARGS, "mla_decode_ex", &dl);
  if (rc != MLA_OK) return rc;
  rc = apply_options(options, "mla_decode_ex", &dl);
  if (rc != MLA_OK) return rc;
  return launch_decode_phases(q_fp8, kv_pages_fp8, num_pages, dl,
                              reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int mla_decode_sparse(const void* q_fp8, const void* kv_pages_fp8, int64_t num_pages,
                                 const int32_t* page_table, int32_t max_pages_per_req,
                                 const int32_t* kv_lens, const int32_t* block_idx, int32_t topk,
                                 const int32_t* splits, const int32_t* chunks, int32_t max_splits,
                                 int32_t kv_split, int32_t batch, int32_t q_len,
                                 int32_t num_heads, int32_t causal, float q_scale,
                                 float kv_scale, float softmax_scale, void* workspace,
                                 size_t workspace_bytes, void* out_bf16, float* lse_f32,
                                 float* out_f32_debug, const mla_decode_options_t* options,
                                 void* stream) {
  if (!block_idx) {
    set_error("mla_decode_sparse: null block_idx");
    return MLA_ERR_INVALID_ARG;
  }
  if (topk < 1 || static_cast<int64_t>(topk) * MLA_PAGE_SIZE > INT32_MAX / 2) {
    set_error("mla_decode_sparse: topk must be >= 1 and 32 * topk must fit in int32");
    return MLA_ERR_INVALID_ARG;
  }
  DecodeLaunch dl;
  int rc = prepare_decode(MLA_DECODE_ARGS, "mla_decode_sparse", &dl);
  if (rc != MLA_OK) return rc;
  dl.prm.block_idx = block_idx;
  dl.prm.topk = topk;
  rc = apply_options(options, "mla_decode_sparse", &dl);
  if (rc != MLA_OK) return rc;
  return launch_decode_phases(q_fp8, kv_pages_fp8, num_pages, dl,
                              reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int mla_decode_splitkv(const void* q_fp8, const void* kv_pages_fp8, int64_t num_pages,
                                  const int32_t* page_table, int32_t max_pages_per_req,
                                  const int32_t* kv_lens, const int32_t* splits,
                                  const int32_t* chunks, int32_t max_splits, int32_t kv_split,
                                  int32_t batch, int32_t q_len, int32_t num_heads, int32_t causal,
                                  float q_scale, float kv_scale, float softmax_scale,
                                  void* workspace, size_t workspace_bytes, void* out_bf16,
                                  float* lse_f32, float* out_f32_debug, void* stream) {
  DecodeLaunch dl;
  int rc = prepare_decode(MLA_DECODE_ARGS, "mla_decode_splitkv", &dl);
  if (rc != MLA_OK) return rc;
  return launch_decode_split(q_fp8, kv_pages_fp8, num_pages, dl,
                             reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int mla_decode_merge(const void* q_fp8, const void* kv_pages_fp8, int64_t num_pages,
                                const int32_t* page_table, int32_t max_pages_per_req,
                                const int32_t* kv_lens, const int32_t* splits,
                                const int32_t* chunks, int32_t max_splits, int32_t kv_split,
                                int32_t batch, int32_t q_len, int32_t num_heads, int32_t causal,
                                float q_scale, float kv_scale, float softmax_scale,
                                void* workspace, size_t workspace_bytes, void* out_bf16,
                                float* lse_f32, float* out_f32_debug, void* stream) {
  DecodeLaunch dl;
  int rc = prepare_decode(MLA_DECODE_ARGS, "mla_decode_merge", &dl);
  if (rc != MLA_OK) return rc;
  return launch_decode_merge(dl, reinterpret_cast<cudaStream_t>(stream));
}

namespace mla {

// ---------------------------------------------------------------------------
// Decode without a caller-provided workspace.
//
// Some callers cannot call cudaMalloc: code running inside a host runtime that
// owns every device allocation through its own planner and forbids side
// allocations, or a latency-critical path where cudaMalloc's implicit
// device-wide synchronisation is not acceptable.  For them this entry point
// takes its scratch (the status word and the split partials) from a fixed
// array that lives in the library image.  Every GPU that loads the library
// holds the array until the process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_static_ws[MLA_STATIC_WS_BYTES];

// Device address of g_static_ws on each device (host code cannot use the
// symbol itself as a device pointer), resolved at set-up: once per device and
// CUDA context.  The context id is kept with the address so that, after a
// cudaDeviceReset (which unloads the library's module and may reload it
// elsewhere), the next call resolves the address again instead of using a
// stale one.
static std::mutex g_static_ws_mu;
static void* g_static_ws_ptr[64] = {nullptr};
static unsigned long long g_static_ws_ctx[64] = {0};

typedef CUresult (*PfnCtxGetCurrent)(CUcontext*);
typedef CUresult (*PfnCtxGetId)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (0 if it cannot be read).
static unsigned long long current_ctx_id() {
  static PfnCtxGetCurrent get_cur = nullptr;
  static PfnCtxGetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PfnCtxGetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PfnCtxGetId>(f);
  });
  if (!get_cur || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_cur(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

static int static_ws_address(void** out, const char* who) {
  const std::string w(who);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail((w + ": cudaGetDevice").c_str(), e);
  if (dev < 0 || dev >= 64) {
    set_error(w + ": device ordinal above 63");
    return MLA_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_static_ws_mu);
  // Before the runtime's first use of the device no context is current yet
  // (id 0); cudaGetSymbolAddress below makes the primary context current.
  unsigned long long ctx = current_ctx_id();
  const bool stale = g_static_ws_ptr[dev] && ctx != 0 && ctx != g_static_ws_ctx[dev];
  if (!g_static_ws_ptr[dev] || stale) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_ws);
    if (e != cudaSuccess || !ptr) return cuda_fail((w + ": cudaGetSymbolAddress").c_str(), e);
    if (ctx == 0) ctx = current_ctx_id();  // the call above made the context current
    // The status header starts at zero on a fresh set-up (after that it is
    // only set by the device and cleared by mla_decode_static_ws_status).
    e = cudaMemset(ptr, 0, kStatusBytes);
    if (e != cudaSuccess) return cuda_fail((w + ": status header reset").c_str(), e);
    g_static_ws_ptr[dev] = ptr;
    g_static_ws_ctx[dev] = ctx;
  }
  *out = g_static_ws_ptr[dev];
  return MLA_OK;
}

}  // namespace mla

extern "C" int mla_decode_static_ws(const void* q_fp8, const void* kv_pages_fp8,
                                    int64_t num_pages, const int32_t* page_table,
                                    int32_t max_pages_per_req, const int32_t* kv_lens,
                                    const int32_t* splits, const int32_t* chunks,
                                    int32_t max_splits, int32_t kv_split, int32_t batch,
                                    int32_t q_len, int32_t num_heads, int32_t causal,
                                    float q_scale, float kv_scale, float softmax_scale,
                                    void* out_bf16, float* lse_f32, float* out_f32_debug,
                                    void* stream) {
  if (batch >= 1 && q_len >= 1 && num_heads >= 1 && max_splits >= 1) {
    const size_t need = ws_total(static_cast<int64_t>(batch) * q_len * num_heads, max_splits);
    if (need > MLA_STATIC_WS_BYTES) {
      set_error("mla_decode_static_ws: this call needs " + std::to_string(need) +
                " bytes of scratch, above the fixed MLA_STATIC_WS_BYTES (" +
                std::to_string(static_cast<size_t>(MLA_STATIC_WS_BYTES)) +
                "); use mla_decode with a caller-owned workspace");
      return MLA_ERR_WORKSPACE_TOO_SMALL;
    }
  }
  void* workspace = nullptr;
  int rc = static_ws_address(&workspace, "mla_decode_static_ws");
  if (rc != MLA_OK) return rc;
  const size_t workspace_bytes = MLA_STATIC_WS_BYTES;
  DecodeLaunch dl;
  rc = prepare_decode(MLA_DECODE_ARGS, "mla_decode_static_ws", &dl);
  if (rc != MLA_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The array keeps the previous call's partials; every partial the merge
  // reads is written by this call's split kernel first.  The status word is
  // sticky: a condition any call reports stays until
  // mla_decode_static_ws_status reads and clears it.
  rc = launch_decode_split(q_fp8, kv_pages_fp8, num_pages, dl, st);
  if (rc != MLA_OK) return rc;
  return launch_decode_merge(dl, st);
}

extern "C" int mla_decode_static_ws_status(void* stream) {
  void* workspace = nullptr;
  int rc = static_ws_address(&workspace, "mla_decode_static_ws_status");
  if (rc != MLA_OK) return rc;
  return mla_decode_status(workspace, stream);
}

extern "C" void mla_debug_set_wait_limit(long long cycles) {
  g_wait_cycles.store(cycles > 0 ? cycles : 0);
}

extern "C" void mla_debug_set_expire(int32_t role, int32_t tile) {
  g_debug_expire.store((role < 0 || role > 255 || tile < 0 || tile >= (1 << 24))
                           ? -1
                           : (role << 24) | tile);
}

extern "C" int mla_decode_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < kStatusBytes) {
    set_error("mla_decode_workspace_init: null or too small workspace");
    return MLA_ERR_INVALID_ARG;
  }
  cudaError_t e = cudaMemsetAsync(workspace, 0, kStatusBytes,
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("mla_decode_workspace_init", e);
  return MLA_OK;
}

extern "C" int mla_merge(const float* partial_o, const float* partial_ml, int32_t rows,
                         int32_t num_ctas_kv, int32_t kv_split, void* out_bf16, float* lse_f32,
                         float* out_f32_debug, void* stream) {
  if (!partial_o || !partial_ml || !out_bf16) {
    set_error("mla_merge: null pointer argument");
    return MLA_ERR_INVALID_ARG;
  }
  // Rows run on grid x (up to 2^31 - 1 CTAs); offsets are 64-bit.
  if (rows < 1 || num_ctas_kv < 1) {
    set_error("mla_merge: rows and num_ctas_kv must be >= 1");
    return MLA_ERR_INVALID_ARG;
  }
  if (kv_split != 1 && kv_split != 2 && kv_split != 4 && kv_split != 8 && kv_split != 16) {
    set_error("mla_merge: kv_split must be 1, 2, 4, 8 or 16");
    return MLA_ERR_INVALID_ARG;
  }
  if (!aligned(partial_o, 16) || !aligned(partial_ml, 8) || !aligned(out_bf16, 8) ||
      (out_f32_debug && !aligned(out_f32_debug, 16))) {
    set_error("mla_merge: partial_o/out_f32 need 16-byte, partial_ml/out 8-byte alignment");
    return MLA_ERR_INVALID_ARG;
  }
  MergeParams mp;
  mp.po = partial_o;
  mp.pml = partial_ml;
  mp.rows = rows;
  mp.stride_s = num_ctas_kv;
  mp.uniform_s = num_ctas_kv;
  mp.splits = nullptr;
  mp.rows_per_req = 1;
  mp.num_heads = 1;
  mp.output_scale = 1.0f;
  mp.sinks = nullptr;
  mp.out = reinterpret_cast<__nv_bfloat16*>(out_bf16);
  mp.lse = lse_f32;
  mp.out_f32 = out_f32_debug;
  cudaError_t e = launch_merge(mp, kv_split, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("mla_merge: launch", e);
  return MLA_OK;
}

extern "C" int mla_decode_status(const void* workspace, void* stream) {
  if (!workspace) {
    set_error("mla_decode_status: null workspace");
    return MLA_ERR_INVALID_ARG;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail("mla_decode_status: stream", e);
  int v = 0;
  e = cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail("mla_decode_status: read", e);
  e = cudaMemset(const_cast<void*>(workspace), 0, sizeof(int));
  if (e != cudaSuccess) return cuda_fail("mla_decode_status: clear", e);
  if (v == MLA_ERR_TIMEOUT) {
    set_error("mla_decode: a device wait ran out (timeout)");
    return MLA_ERR_TIMEOUT;
  }
  if (v != 0) {
    set_error("mla_decode: device detected a bad page id or inconsistent plan arrays");
    return MLA_ERR_INVALID_ARG;
  }
  return MLA_OK;
}
