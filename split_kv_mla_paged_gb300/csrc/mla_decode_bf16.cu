// Paged BF16-KV MLA decode for GB300 (sm_103a): the same split-KV method as
// the FP8 kernel with a BF16 cache (issue #20510 "CuTe DSL FP8 MLA decode
// regression", Repro 2 text: the BF16 kernel mla_decode_fp16.py, same
// geometry: 512 latent + 64 rope, page size 32, BF16 output).
//
// Differences from the FP8 kernel (mla_decode.cu):
//  * A token row is 1152 bytes, in nine 64-element blocks (8 latent + 1
//    rope) of 128 B, each staged with the 128-byte swizzle.
//  * QK and PV are tcgen05.mma kind::f16 (K = 16 elements per instruction;
//    A and B of one type, so Q is BF16 too and there are no q/kv scales).
//  * P is BF16 (8 mantissa bits, so one term is enough: |err| <= 2^-9 of a
//    weight).  Partials have the FP8 kernel's layout, so the merge is shared.
//  * Row groups of at most 16 rows (mla_split_kv_bf16_q16_kernel) keep Q in
//    TMEM and stream 64-token tiles (73,728 B) through three stages; 32- and
//    48-row groups (mla_split_kv_bf16_wide_kernel) use the FP8 kernel's
//    swapped layout with 128-token tiles (147,456 B: one stage, released
//    block by block).
//  * As in the FP8 kernel, warp 1 issues QK and warp 2 PV, and PV
//    completions alternate between two barriers by tile parity.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <string>

#include "mla_device.cuh"

namespace mla {

constexpr int kTokB = 64;                                   // tokens per tile
constexpr uint32_t kRowBytesB = MLA_HEAD_DIM * 2;           // 1152
constexpr uint32_t kTileBytesB = kTokB * kRowBytesB;        // 73728
constexpr uint32_t kBlkBytesB = kTokB * 128;                // 8192: one 64-element block
constexpr uint32_t kRopeOffB = 8 * kBlkBytesB;              // block 8 = rope
constexpr uint32_t kPageBlkBytesB = MLA_PAGE_SIZE * 128;    // 4096: one page of one block
constexpr uint32_t kPageBytesB = MLA_PAGE_SIZE * kRowBytesB;

// Instruction descriptor for kind::f16 with BF16 A and B, fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t M, uint32_t N, uint32_t a_mn,
                                                  uint32_t b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// tcgen05.mma kind::f16 with the A operand in TMEM (lane = row, two 16-bit
// elements per 32-bit column, element 2c in the low half; K = 16 elements =
// 8 columns per instruction).
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32"
      " [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);  // a in the low half
  return *reinterpret_cast<uint32_t*>(&v);
}

// Rows of a staged 64-token tile (two pages) that hold no loaded key: pages
// not loaded (past the split's end, outside a window, an unused selection
// slot) and the tail of a request's last page.  The warp zeroes all 1152
// bytes of such a row (nine 128-byte blocks) so V holds no stale or NaN
// values.  kGather: `info` holds the rows loaded per page (byte q for page
// q); otherwise the first `valid` rows of the tile are keys of the split.
template <bool kGather>
__device__ __forceinline__ void zero_unloaded_rows_bf16(uint8_t* kvp, int lane, uint32_t info,
                                                        int valid) {
  const uint4 z = make_uint4(0, 0, 0, 0);
  auto zero_rows = [&](int r0, int nrow) {
    for (int idx = lane; idx < nrow * 72; idx += 32) {
      const int r = r0 + idx / 72;
      const int c = idx % 72;
      *reinterpret_cast<uint4*>(kvp + (c / 8) * kBlkBytesB + r * 128 + (c % 8) * 16) = z;
    }
  };
  bool any = false;
  if constexpr (kGather) {
#pragma unroll 1
    for (int q = 0; q < 2; ++q) {
      const int nv = static_cast<int>((info >> (8 * q)) & 0xFFu);
      if (nv < MLA_PAGE_SIZE) {
        zero_rows(q * MLA_PAGE_SIZE + nv, MLA_PAGE_SIZE - nv);
        any = true;
      }
    }
  } else if (valid < kTokB) {
    zero_rows(valid, kTokB - valid);
    any = true;
  }
  if (any) {
    fence_proxy_async_smem();
    __syncwarp();
  }
}

// CTA coordinates of the split kernels: the (request, split x row group)
// grid, split-major, or an entry of the CTA item list (kItems).  Returns
// false (after reporting) for an item outside the batch or the row groups.
template <bool kItems>
__device__ __forceinline__ bool cta_coords(const DecodeParams& p, int ngroups, int& b, int& split,
                                           int& grp) {
  if constexpr (kItems) {
    const int it = p.cta_items[blockIdx.x];
    b = it >> MLA_ITEM_B_SHIFT;
    split = (it >> MLA_ITEM_S_SHIFT) & ((1 << (MLA_ITEM_B_SHIFT - MLA_ITEM_S_SHIFT)) - 1);
    grp = it & ((1 << MLA_ITEM_S_SHIFT) - 1);
    if (it < 0 || b >= p.batch || grp >= ngroups) {
      if (threadIdx.x == 0) report(p.status, MLA_ERR_INVALID_ARG);
      return false;
    }
  } else {
    split = blockIdx.y / ngroups;
    grp = blockIdx.y - split * ngroups;
    b = blockIdx.x;
  }
  return true;
}

// Key range of split `split` of request b for the BF16 kernels (64-token
// tiles): the plan checks (reported as MLA_ERR_INVALID_ARG), the split's
// token range in the planned space (positions, or the compact range of a
// page selection), the key window, and the first tile (whole tiles below a
// dense window are skipped; tiles stay aligned to the split start).
struct SplitRange {
  int L, nsplit, q_b, tok_begin, tok_end, t0, win_lo, win_hi;
  bool sparse;
};

template <bool kGather, int kTile = kTokB>
__device__ __forceinline__ bool split_range(const DecodeParams& p, int b, int split,
                                            SplitRange& r) {
  r.L = p.kv_lens[b];
  r.nsplit = p.splits[b];
  const int chunk = p.chunks[b];
  r.sparse = kGather && p.block_idx != nullptr;
  const int Lspace = r.sparse ? p.topk * MLA_PAGE_SIZE : r.L;
  r.q_b = p.query_lens ? p.query_lens[b] : p.q_len;
  const bool bad = r.L < 1 || r.q_b < 1 || r.q_b > p.q_len || (p.causal && r.L < r.q_b) ||
                   r.nsplit > p.max_splits || chunk < MLA_TILE_TOKENS ||
                   (chunk % MLA_TILE_TOKENS) != 0 ||
                   static_cast<int64_t>(r.nsplit) * chunk < Lspace ||
                   static_cast<int64_t>(r.nsplit - 1) * chunk >= Lspace ||
                   static_cast<int64_t>(r.L) > static_cast<int64_t>(p.max_pages) * MLA_PAGE_SIZE;
  if (bad) {
    if (threadIdx.x == 0) report(p.status, MLA_ERR_INVALID_ARG);
    return false;
  }
  r.tok_begin = split * chunk;
  r.tok_end = min(Lspace, r.tok_begin + chunk);
  r.win_lo = 0;
  r.win_hi = r.L;
  if (kGather && p.kv_bounds) {
    r.win_lo = max(0, p.kv_bounds[2 * b]);
    r.win_hi = min(r.L, p.kv_bounds[2 * b + 1]);
  }
  r.t0 = r.tok_begin;
  if (kGather && !r.sparse) {
    r.tok_end = min(r.tok_end, r.win_hi);
    if (r.win_lo >= r.tok_end)
      r.t0 = r.tok_end;
    else if (r.win_lo > r.tok_begin)
      r.t0 = r.tok_begin + (r.win_lo - r.tok_begin) / kTile * kTile;
  }
  return true;
}

// One lane's page of a producer window (32 pages = 16 tiles per window):
// compact page pi = page0 + w * 32 + lane maps to logical page lp (pi
// itself, or the selection's entry), loaded when it holds keys inside the
// window and before the end of the split (dense) or of the request
// (selection).  Returns the physical page (0 if none) and sets nv_out to the
// page's rows to load (0: not loaded).  Out-of-pool page ids and selection
// order violations are reported.
template <bool kGather>
__device__ __forceinline__ int bf16_window_page(const DecodeParams& p, const SplitRange& r,
                                                const int32_t* pt, int b, int page0,
                                                int page_end, int w, int lane, int& last_lp,
                                                int& nv_out) {
  const int pi = page0 + w * 32 + lane;
  int pg = 0;
  nv_out = 0;
  if constexpr (!kGather) {
    if (pi < page_end) {
      pg = pt[pi];
      if (pg < 0 || pg >= p.num_pages) {
        report(p.status, MLA_ERR_INVALID_ARG);
        pg = 0;
      }
      nv_out = MLA_PAGE_SIZE;
    }
  } else {
    int lp = -1;
    if (pi < page_end) {
      lp = pi;
      if (r.sparse) lp = (pi < p.topk) ? p.block_idx[static_cast<int64_t>(b) * p.topk + pi] : -1;
    }
    if (r.sparse) {
      int prev = __shfl_up_sync(0xffffffffu, lp, 1);
      if (lane == 0) prev = last_lp;
      if (lp >= 0 && prev >= 0 && lp <= prev) report(p.status, MLA_ERR_INVALID_ARG);
      last_lp = __shfl_sync(0xffffffffu, lp, 31);
    }
    const int64_t end_pos = r.sparse ? r.win_hi : r.tok_end;
    const int64_t first = static_cast<int64_t>(lp) * MLA_PAGE_SIZE;
    if (lp >= 0 && first < end_pos && first + MLA_PAGE_SIZE > r.win_lo) {
      pg = pt[lp];
      if (pg < 0 || pg >= p.num_pages) {
        report(p.status, MLA_ERR_INVALID_ARG);
        pg = 0;
      }
      nv_out = static_cast<int>(end_pos - first < MLA_PAGE_SIZE ? end_pos - first
                                                                 : MLA_PAGE_SIZE);
    }
  }
  return pg;
}

// ---------------------------------------------------------------------------
// Row groups of at most 16 rows (H12 q1, the common BF16 case): Q lives in
// TMEM as the A operand of a non-swapped QK, which frees the shared memory
// for three KV stages.
//  * TMEM: Q [128 lanes x 288 columns] (lane l holds row l % 16: eight copies
//    of the 16 rows, two BF16 values per column, element 2c in the low half),
//    S [128 x 64 tokens] x 2 buffers, O^T [128 dims x 16 rows] x 4 blocks.
//  * QK: S = Q K^T, M = 128 (the row copies), N = 64 tokens, K = 16 per
//    instruction, B = the K tile (K-major, 128-byte swizzle), 36 per tile.
//  * Softmax: thread (lane l of warp w) takes row l % 16 and the eight tokens
//    8 (2w + l / 16) .. +7, so all 128 threads work on distinct scores.
//  * P^T goes K-major (a row's 64 tokens = one 128-byte swizzled line) into
//    the consumed rope block; PV is the swapped O^T += V^T P^T as before.
// ---------------------------------------------------------------------------
namespace q16 {
constexpr int NR = 16;
constexpr int NST = 3;
constexpr int kThreads = 96 + 128;  // TMA, QK issuer, PV issuer, softmax warpgroup
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kQCol = 0;      // 288 columns
constexpr uint32_t kSCol = 288;    // 2 x 64 columns
constexpr uint32_t kOCol = 416;    // 4 x 16 columns
constexpr uint32_t kQStage = (NST - 1) * kTileBytesB;  // Q staged by TMA in the last stage
constexpr uint32_t kAux = NST * kTileBytesB;
constexpr uint32_t kBars = kAux;               // 17 x 8 B
constexpr uint32_t kTmemSlot = kAux + 136;
constexpr uint32_t kFlags = kAux + 144;
constexpr uint32_t kStageInfo = kAux + 160;    // NST x 4 B: rows loaded per page
constexpr uint32_t kRedMax = kAux + 176;       // 4 warps x 16 rows
constexpr uint32_t kRedSum = kRedMax + 256;    // 2 x 4 x 16
constexpr uint32_t kKref = kRedSum + 512;      // 16
constexpr uint32_t kAlpha = kKref + 64;        // 16
constexpr uint32_t kEnd = kAlpha + 64;
constexpr uint32_t kSmemBytes = kEnd + 1024;
static_assert(kSmemBytes <= 232448u, "shared memory");
constexpr int BAR_QTMEM = BAR_PFREE0;  // Q copied into TMEM (128 arrivals)
// PV(i) completion, alternating by tile parity (this kernel has no P^T
// buffer barriers): with QK and PV issued by different warps, a waiter is
// then never more than one phase away from the phase it waits for.
constexpr int BAR_ODONE_0 = BAR_ODONE;
constexpr int BAR_ODONE_1 = BAR_PFREE1;
}  // namespace q16

template <bool kGather, bool kItems>
__global__ void __launch_bounds__(q16::kThreads, 1)
    mla_split_kv_bf16_q16_kernel(const __grid_constant__ CUtensorMap tm_kv,
                                 const __grid_constant__ CUtensorMap tm_q, const DecodeParams p) {
  using namespace q16;
  const int ngroups = (p.rows_per_req + p.rows_per_group - 1) / p.rows_per_group;
  int b, split, grp;
  if (!cta_coords<kItems>(p, ngroups, b, split, grp)) return;
  if (split >= p.splits[b]) return;  // empty split slot of a shorter request
  SplitRange sr;
  if (!split_range<kGather>(p, b, split, sr)) return;
  const int L = sr.L, nsplit = sr.nsplit, q_b = sr.q_b, tok_end = sr.tok_end, t0 = sr.t0;
  const bool sparse = sr.sparse;
  const float c_log2 =
      p.sm_scale_dev ? *p.sm_scale_dev * 1.4426950408889634f : p.c_log2;
  const int row0 = grp * p.rows_per_group;
  const int rows_here = min(p.rows_per_group, p.rows_per_req - row0);
  // Rows of real query tokens (the others are padding slots of a shorter
  // query block: no key is visible to them).
  const int rows_valid = max(0, min(rows_here, q_b * p.num_heads - row0));
  const int n_tiles =
      (rows_valid > 0 && tok_end > t0) ? (tok_end - t0 + kTokB - 1) / kTokB : 0;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(base);
  auto bar = [&](int i) -> uint32_t { return sbase + kBars + 8u * i; };
  volatile int* flags = reinterpret_cast<volatile int*>(base + kFlags);
  volatile int* abort_flag = flags + 2;
  float* red_max = reinterpret_cast<float*>(base + kRedMax);
  float* red_sum = reinterpret_cast<float*>(base + kRedSum);
  float* kref = reinterpret_cast<float*>(base + kKref);
  float* alpha_s = reinterpret_cast<float*>(base + kAlpha);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int k = 0; k < NST; ++k) {
      mbar_init(bar(BAR_FULL0 + k), 1);
      mbar_init(bar(BAR_EMPTY0 + k), 1);
    }
    mbar_init(bar(BAR_QFULL), 1);
    mbar_init(bar(BAR_QTMEM), 128);
    mbar_init(bar(BAR_SFULL0), 1);
    mbar_init(bar(BAR_SFULL1), 1);
    mbar_init(bar(BAR_SFREE0), 128);
    mbar_init(bar(BAR_SFREE1), 128);
    mbar_init(bar(BAR_PFULL0), 128);
    mbar_init(bar(BAR_PFULL1), 128);
    mbar_init(bar(BAR_ODONE_0), 1);
    mbar_init(bar(BAR_ODONE_1), 1);
    mbar_init(bar(BAR_FINAL), 2);  // one commit from each MMA warp
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + kTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base + kTmemSlot);

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      tma_prefetch_desc(&tm_kv);
      tma_prefetch_desc(&tm_q);
      const int qrow = b * p.rows_per_req + row0;
      mbar_arrive_expect_tx(bar(BAR_QFULL), NR * kRowBytesB);
#pragma unroll
      for (int d = 0; d < 9; ++d)
        tma_load_2d(sbase + kQStage + d * NR * 128, &tm_q, d * 64, qrow, bar(BAR_QFULL));
    }
    const uint64_t pol = l2_policy_evict_first();
    const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.max_pages;
    const int page0 = t0 / MLA_PAGE_SIZE;
    const int page_end = (tok_end + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE;
    int last_lp = -1;
    int window_nv, window_next_nv;
    int window = bf16_window_page<kGather>(p, sr, pt, b, page0, page_end, 0, lane, last_lp,
                                           window_nv);
    int window_next = bf16_window_page<kGather>(p, sr, pt, b, page0, page_end, 1, lane, last_lp,
                                                window_next_nv);
    volatile uint32_t* stage_info = reinterpret_cast<volatile uint32_t*>(base + kStageInfo);
    int issued = 0;
    int st = 0, round = 0;
    for (int i = 0; i < n_tiles; ++i) {
      if (i > 0 && (i & 15) == 0) {
        window = window_next;
        window_nv = window_next_nv;
        window_next = bf16_window_page<kGather>(p, sr, pt, b, page0, page_end, (i >> 4) + 1,
                                                lane, last_lp, window_next_nv);
      }
      bool ok = !expired_here(p, WAIT_STAGE_FREE, i);
      if (ok && round > 0) {
        ok = mbar_wait_abort(bar(BAR_EMPTY0 + st), (round - 1) & 1, p.wait_cycles, abort_flag);
      } else if (ok && st == NST - 1) {
        // The last stage holds the staged Q until it has been copied to TMEM.
        ok = mbar_wait_abort(bar(BAR_QTMEM), 0, p.wait_cycles, abort_flag);
      }
      ok = __all_sync(0xffffffffu, ok && !*abort_flag);
      if (!ok) {
        if (lane == 0) {
          report(p.status, MLA_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      const int src = (i & 15) * 2 + (lane & 1);
      const int my_page = __shfl_sync(0xffffffffu, window, src);
      const int my_nv = __shfl_sync(0xffffffffu, window_nv, src);
      const int nv1 = __shfl_sync(0xffffffffu, my_nv, 1);
      const bool my_load = my_nv > 0;
      const int nload = __popc(__ballot_sync(0xffffffffu, lane < 2 && my_load));
      const uint32_t fb = bar(BAR_FULL0 + st);
      if (lane == 0) {
        if constexpr (kGather)
          stage_info[st] = static_cast<uint32_t>(my_nv) | (static_cast<uint32_t>(nv1) << 8);
        mbar_arrive_expect_tx(fb, nload * kPageBytesB);
      }
      __syncwarp();
      if (lane < 2 && my_load) {
        const uint32_t kv = sbase + st * kTileBytesB;
        const int row = my_page * MLA_PAGE_SIZE;
#pragma unroll
        for (int d = 0; d < 9; ++d)
          tma_load_2d_hint(kv + d * kBlkBytesB + lane * kPageBlkBytesB, &tm_kv, d * 64, row, fb,
                           pol);
      }
      __syncwarp();
      issued = i + 1;
      if (++st == NST) {
        st = 0;
        ++round;
      }
    }
    if (lane == 0) {
      for (int k = max(0, issued - NST); k < issued; ++k)
        mbar_wait(bar(BAR_FULL0 + k % NST), (k / NST) & 1, kWaitLimitCycles);
      mbar_wait(bar(BAR_QFULL), 0, kWaitLimitCycles);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ================= MMA issuers: warp 1 QK, warp 2 PV =================
    // Two issuing warps keep the tensor pipe fed with QK(i + 1) while PV(i)
    // goes out (one warp issuing both left ~30 % of the pipe's rate unused).
    constexpr uint32_t kIdQK = idesc_bf16(128, 64, 0, 0);
    constexpr uint32_t kIdPV = idesc_bf16(128, NR, 1, 0);
    bool ok = (warp == 1) ? mbar_wait(bar(BAR_QTMEM), 0, p.wait_cycles) : true;
    auto fail = [&]() {
      if (lane == 0) {
        report(p.status, MLA_ERR_TIMEOUT);
        *abort_flag = 1;
      }
    };
    auto issue_pv = [&](int j, int jst) {
      tc_fence_after();
      const uint32_t kv = sbase + jst * kTileBytesB;
      const uint32_t pbuf = kv + kRopeOffB;
#pragma unroll
      for (int d = 0; d < 4; ++d) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t a = smem_desc(kv + 2 * d * kBlkBytesB + ks * 2048, kBlkBytesB, 1024,
                                       kLayoutSW128);
          // B = P^T, K-major: a row's 64 tokens in one swizzled 128-byte line,
          // 16 tokens (32 B) per instruction, 8-row groups 1 KB apart.
          const uint64_t bd = smem_desc(pbuf + ks * 32, 16, 1024, kLayoutSW128);
          umma_bf16(tmem + kOCol + d * NR, a, bd, kIdPV, (j > 0 || ks > 0) ? 1u : 0u);
        }
      }
      umma_commit(bar(BAR_EMPTY0 + jst));
      umma_commit(bar((j & 1) ? BAR_ODONE_1 : BAR_ODONE_0));
    };
    auto issue_qk = [&](int ist, int sb) {
      tc_fence_after();
      const uint32_t kv = sbase + ist * kTileBytesB;
#pragma unroll
      for (int kk = 0; kk < 36; ++kk) {
        const int d = kk >> 2, sub = kk & 3;
        const uint64_t bd = smem_desc(kv + d * kBlkBytesB + sub * 32, 16, 1024, kLayoutSW128);
        umma_bf16_ta(tmem + kSCol + sb * 64, tmem + kQCol + kk * 8, bd, kIdQK, kk > 0 ? 1u : 0u);
      }
      umma_commit(bar(BAR_SFULL0 + sb));
    };
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) fail();
    tc_fence_after();
    // Each warp waits on one barrier at a time, in tile order.
    auto qk_step = [&](int j) -> bool {
      const int st = j % NST;
      bool w = !expired_here(p, WAIT_TILE_FULL, j) &&
               mbar_wait_abort(bar(BAR_FULL0 + st), (j / NST) & 1, p.wait_cycles, abort_flag);
      const int use = j >> 1;
      if (w && use >= 1)
        w = mbar_wait_abort(bar(BAR_SFREE0 + (j & 1)), (use - 1) & 1, p.wait_cycles, abort_flag);
      w = __all_sync(0xffffffffu, w && !*abort_flag);
      if (!w) return false;
      const uint32_t info =
          kGather ? *reinterpret_cast<volatile uint32_t*>(base + kStageInfo + 4 * st) : 0u;
      zero_unloaded_rows_bf16<kGather>(base + st * kTileBytesB, lane, info,
                                       tok_end - (t0 + j * kTokB));
      if (lane == 0) issue_qk(st, j & 1);
      __syncwarp();
      return true;
    };
    if (warp == 1) {
      // QK(j) once its tile has landed, its S^T buffer is free and PV(j - 2)
      // has completed (which keeps the softmax's wait for PV(j - 1) within
      // one phase of its barrier; QK(j) still overlaps PV(j - 1)).
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j >= 2) {
          bool w = mbar_wait_abort(bar(((j - 2) & 1) ? BAR_ODONE_1 : BAR_ODONE_0),
                                   ((j - 2) >> 1) & 1, p.wait_cycles, abort_flag);
          w = __all_sync(0xffffffffu, w && !*abort_flag);
          if (!w) {
            ok = false;
            break;
          }
        }
        ok = qk_step(j);
      }
    } else {
      for (int i = 0; ok && i < n_tiles; ++i) {
        bool w = !expired_here(p, WAIT_P_FULL, i) &&
                 mbar_wait_abort(bar(BAR_PFULL0 + (i & 1)), (i >> 1) & 1, p.wait_cycles,
                                 abort_flag);
        w = __all_sync(0xffffffffu, w && !*abort_flag);
        if (!w) {
          ok = false;
          break;
        }
        if (lane == 0) issue_pv(i, i % NST);
        __syncwarp();
      }
    }
    if (!ok) fail();
    if (lane == 0) umma_commit(bar(BAR_FINAL));
    __syncwarp();
    mbar_wait(bar(BAR_FINAL), 0, kWaitLimitCycles);
  } else {
    // ================= softmax warpgroup =================
    const int w = warp & 3;                 // TMEM lane quadrant this warp may access
    const int lidx = w * 32 + lane;         // TMEM lane
    const int row = lidx & 15;              // query row of this thread
    const int slot = lidx >> 4;             // tokens 8*slot .. 8*slot + 7 of a tile
    const bool hi = lane >= 16;
    const int sid = threadIdx.x - 96;       // 0..127; owner of row sid when < 16
    const uint32_t lane_addr = static_cast<uint32_t>(w * 32) << 16;
    bool ok = true;
    // ---- Q: staged rows -> TMEM (lane l gets row l % 16) ----
    ok = mbar_wait(bar(BAR_QFULL), 0, p.wait_cycles);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      const uint8_t* qs = base + kQStage;
#pragma unroll 1
      for (int d = 0; d < 9; ++d) {
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 v = *reinterpret_cast<const uint4*>(
              qs + d * NR * 128 + row * 128 + ((j ^ (row & 7)) * 16));
          r[4 * j + 0] = v.x;
          r[4 * j + 1] = v.y;
          r[4 * j + 2] = v.z;
          r[4 * j + 3] = v.w;
        }
        tmem_st32(tmem + lane_addr + kQCol + d * 32, r);
      }
      tmem_st_wait();
    }
    tc_fence_before();
    mbar_arrive(bar(BAR_QTMEM));

    float k_row = -INFINITY;  // owner state
    float l_row = 0.0f;
    float kreg = -INFINITY;   // this thread's row reference
    const float c = c_log2;
    const int qi = (row0 + row) / p.num_heads;
    const bool row_ok = row < rows_valid;
    const int lim = p.causal ? min(tok_end, L - q_b + qi + 1) : tok_end;
    // Selection: logical page ids of 16 tiles' compact pages, one per lane
    // (this thread's tokens lie in page slot / 4 of its tile).
    auto sel_window = [&](int wn) -> int {
      const int cp = t0 / MLA_PAGE_SIZE + wn * 32 + lane;
      return (cp < p.topk) ? p.block_idx[static_cast<int64_t>(b) * p.topk + cp] : -1;
    };
    int sel_cur = -1, sel_next = -1;
    if (sparse) {
      sel_cur = sel_window(0);
      sel_next = sel_window(1);
    }
    for (int i = 0; i < n_tiles; ++i) {
      const int sb = i & 1;
      const int use = i >> 1;
      if (ok)
        ok = !expired_here(p, WAIT_S_FULL, i) &&
             mbar_wait_abort(bar(BAR_SFULL0 + sb), use & 1, p.wait_cycles, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok && lane == 0) *abort_flag = 1;  // the other roles stop waiting
      float t[8];
      if (ok) {
        tc_fence_after();
        uint32_t r[16];
        tmem_ld16(tmem + lane_addr + kSCol + sb * 64 + w * 16, r);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 8; ++k) t[k] = __uint_as_float(hi ? r[8 + k] : r[k]);
        tc_fence_before();
        mbar_arrive(bar(BAR_SFREE0 + sb));
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) t[k] = 0.0f;
      }
      const int j0 = t0 + i * kTokB + slot * 8;
      if constexpr (kGather) {
        // Restricted key sets: the token's key position decides.
        int64_t pos0 = j0;
        bool page_ok = true;
        if (sparse) {
          if (i > 0 && (i & 15) == 0) {
            sel_cur = sel_next;
            sel_next = sel_window((i >> 4) + 1);
          }
          const int lp = __shfl_sync(0xffffffffu, sel_cur, (i & 15) * 2 + (slot >> 2));
          pos0 = static_cast<int64_t>(lp) * MLA_PAGE_SIZE + (slot & 3) * 8;
          page_ok = lp >= 0;
        }
        const int plim = p.causal ? min(sr.win_hi, L - q_b + qi + 1) : sr.win_hi;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const bool vis = row_ok && page_ok && j0 + k < tok_end && pos0 + k >= sr.win_lo &&
                           pos0 + k < plim;
          t[k] = vis ? t[k] * c : -INFINITY;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) t[k] = (row_ok && j0 + k < lim) ? t[k] * c : -INFINITY;
      }
      bool over = false;
#pragma unroll
      for (int k = 0; k < 8; ++k) over |= t[k] > kreg + 0.75f;
      const bool any_over = bar_sync_or(kVoteBarrier, 128, over);
      if (sid < NR && i > 0) {
        const float* rs = red_sum + ((i - 1) & 1) * 64;
        l_row += (rs[sid] + rs[16 + sid]) + (rs[32 + sid] + rs[48 + sid]);
      }
      if (any_over) {
        float m = t[0];
#pragma unroll
        for (int k = 1; k < 8; ++k) m = fmaxf(m, t[k]);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        if (!hi) red_max[w * 16 + row] = m;
        if (sid == 0) flags[0] = 0;
        named_bar_sync(kSoftmaxBarrier, 128);
        if (sid < NR) {
          const float mt = fmaxf(fmaxf(red_max[sid], red_max[16 + sid]),
                                 fmaxf(red_max[32 + sid], red_max[48 + sid]));
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
        named_bar_sync(kSoftmaxBarrier, 128);
        kreg = kref[row];
        const bool corr = flags[0] != 0;
        if (ok && corr && i > 0) {
          // PV(i - 1) done.  PV(i - 2) completed before QK(i) was issued and
          // PV(i + 1) needs this tile's P^T, so the barrier of PV(i - 1)'s
          // parity is within one phase of the awaited one.
          ok = mbar_wait_abort(bar(((i - 1) & 1) ? BAR_ODONE_1 : BAR_ODONE_0),
                               ((i - 1) >> 1) & 1, p.wait_cycles, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (ok) {
            tc_fence_after();
#pragma unroll 1
            for (int d = 0; d < 4; ++d) {
              uint32_t r[16];
              const uint32_t addr = tmem + lane_addr + kOCol + d * NR;
              tmem_ld16(addr, r);
              tmem_ld_wait();
#pragma unroll
              for (int k = 0; k < 16; ++k)
                r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha_s[k]);
              tmem_st16(addr, r);
            }
            tmem_st_wait();
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) t[k] = softmax_weight<false>(t[k], kreg);
      if (ok) {
        // P^T row `row`, tokens 8*slot..+7: one 16-byte chunk of the row's
        // swizzled 128-byte line in the rope block of this tile's stage.
        uint8_t* pbuf = base + (i % NST) * kTileBytesB + kRopeOffB;
        uint4 v;
        v.x = pack_bf16x2(t[0], t[1]);
        v.y = pack_bf16x2(t[2], t[3]);
        v.z = pack_bf16x2(t[4], t[5]);
        v.w = pack_bf16x2(t[6], t[7]);
        *reinterpret_cast<uint4*>(pbuf + (row >> 3) * 1024 + (row & 7) * 128 +
                                  ((slot ^ (row & 7)) * 16)) = v;
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(BAR_PFULL0 + (i & 1)));
      }
      float sum = ((t[0] + t[1]) + (t[2] + t[3])) + ((t[4] + t[5]) + (t[6] + t[7]));
      sum += __shfl_xor_sync(0xffffffffu, sum, 16);
      if (!hi) red_sum[(i & 1) * 64 + w * 16 + row] = sum;
    }
    if (!ok && lane == 0) {
      report(p.status, MLA_ERR_TIMEOUT);
      *abort_flag = 1;
    }
    // ---- epilogue ----
    named_bar_sync(kSoftmaxBarrier, 128);
    const bool single = (nsplit == 1);
    float* scale_s = alpha_s;
    if (sid < NR) {
      if (n_tiles > 0) {
        const float* rs = red_sum + ((n_tiles - 1) & 1) * 64;
        l_row += (rs[sid] + rs[16 + sid]) + (rs[32 + sid] + rs[48 + sid]);
      }
      const float m_s = (k_row == -INFINITY) ? -INFINITY : k_row - 8.0f;
      const int64_t grow = static_cast<int64_t>(b) * p.rows_per_req + row0 + sid;
      float sc = 0.0f;
      if (sid < rows_here) {
        if (single) {
          // A sink is one more (zero-valued) key: it joins the denominator.
          const float sink2 = p.sinks
                                  ? p.sinks[(row0 + sid) % p.num_heads] * 1.4426950408889634f
                                  : -INFINITY;
          const float mm = fmaxf(l_row > 0.0f ? m_s : -INFINITY, sink2);
          const float a = (l_row > 0.0f) ? exp2f(m_s - mm) : 0.0f;
          const float den = l_row * a + (sink2 == -INFINITY ? 0.0f : exp2f(sink2 - mm));
          if (p.lse)
            p.lse[grow] = (den > 0.0f) ? 0.6931471805599453f * (mm + log2f(den)) : -INFINITY;
          sc = (den > 0.0f) ? p.output_scale * a / den : 0.0f;
        } else {
          float* ml = p.ws_ml + (grow * p.max_splits + split) * 2;
          ml[0] = m_s;
          ml[1] = l_row;
          sc = 1.0f;
        }
      }
      scale_s[sid] = sc;
    }
    named_bar_sync(kSoftmaxBarrier, 128);
    bool fin = !expired_here(p, WAIT_FINAL, 0) && mbar_wait(bar(BAR_FINAL), 0, p.wait_cycles);
    fin = __all_sync(0xffffffffu, fin);
    if (!fin && lane == 0) report(p.status, MLA_ERR_TIMEOUT);
    if (ok && fin && n_tiles > 0) {
      tc_fence_after();
      // The rows' scales in registers, not re-read after every store.
      float sc_r[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) sc_r[k] = scale_s[k];
#pragma unroll 1
      for (int d = 0; d < 4; ++d) {
        const int dim = d * 128 + lidx;
        uint32_t r[16];
        tmem_ld16(tmem + lane_addr + kOCol + d * NR, r);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          if (k < rows_here) {
            const float v = __uint_as_float(r[k]) * sc_r[k];
            const int64_t grow = static_cast<int64_t>(b) * p.rows_per_req + row0 + k;
            if (single) {
              p.out[grow * MLA_LATENT_DIM + dim] = __float2bfloat16_rn(v);
              if (p.out_f32) p.out_f32[grow * MLA_LATENT_DIM + dim] = v;
            } else {
              p.ws_o[(grow * p.max_splits + split) * MLA_LATENT_DIM + dim] = v;
            }
          }
        }
      }
    } else if (ok && fin && n_tiles == 0 && single) {
      // Only padding query slots here: O = 0 (partials need only (-inf, 0)).
      for (int d = 0; d < 4; ++d) {
        const int dim = d * 128 + lidx;
        for (int k = 0; k < rows_here; ++k) {
          const int64_t grow = static_cast<int64_t>(b) * p.rows_per_req + row0 + k;
          p.out[grow * MLA_LATENT_DIM + dim] = __float2bfloat16_rn(0.0f);
          if (p.out_f32) p.out_f32[grow * MLA_LATENT_DIM + dim] = 0.0f;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// 32- and 48-row groups with 128-token tiles
// ---------------------------------------------------------------------------
// The swapped layout of the FP8 kernel (M = 128 tokens, TMEM lane = token,
// every lane of a softmax warp holds a token) with BF16 operands.  A 128-token
// BF16 tile is 147,456 B, so the CTA holds one KV stage next to Q^T and two
// P^T buffers, and releases it block by block: the rope block once QK has
// read it, latent blocks 2d and 2d + 1 once PV's latent group d has, with a
// full and an empty barrier per block; the producer refills each block for
// the next tile as soon as it is free and QK issues each block's steps as
// they land.  QK: 36 `kind::f16` instructions (K = 16) of N = NR per tile;
// PV: 4 latent groups x 8 token slices of N = NR; P in one BF16 term, in its
// own double buffer; S^T double-buffered in TMEM.
namespace bw {
constexpr int kTok = 128;                                  // tokens per tile
constexpr uint32_t kBlk = kTok * 128;                      // 16,384: one 64-element block
constexpr uint32_t kTile = 9 * kBlk;                       // 147,456: 8 latent blocks + rope
constexpr int kRopeBlk = 8;
}  // namespace bw

template <int NR>
struct CfgW {
  static_assert(NR == 32 || NR == 48, "NR");
  static constexpr int NS = 2;                     // S^T buffers
  static constexpr uint32_t kOCol = NS * NR;       // O^T: 4 latent groups x NR columns
  static constexpr uint32_t kTmemUsed = NS * NR + 4 * NR;
  static constexpr uint32_t kTmemCols = kTmemUsed <= 256 ? 256 : 512;
  static constexpr int SWG = 2;
  static constexpr int NRH = NR / SWG;
  static_assert(NRH % 8 == 0, "rows per softmax warpgroup");
  static constexpr int kThreads = 96 + 128 * SWG;
  static constexpr uint32_t kQBytes = NR * kRowBytesB;
  static constexpr uint32_t kPBytes = NR * bw::kTok * 2;  // one BF16 P^T buffer
  static constexpr uint32_t kKV = 0;
  static constexpr uint32_t kQ = bw::kTile;
  static constexpr uint32_t kP = kQ + kQBytes;            // two P^T buffers
  static constexpr uint32_t kAux = kP + 2 * kPBytes;
  static_assert(kQ % 1024 == 0 && kP % 1024 == 0 && kAux % 1024 == 0, "alignment");
  // aux: 19 mbarriers, TMEM slot, flags, rows loaded per page, reductions,
  // then 18 block barriers (full: 8 b, empty: 8 (9 + b)).
  static constexpr uint32_t kBars = kAux;
  static constexpr uint32_t kTmemSlot = kAux + 152;
  static constexpr uint32_t kFlags = kAux + 160;
  static constexpr uint32_t kStageInfo = kAux + 176;
  static constexpr uint32_t kRedMax = kAux + 192;  // 4 x NR floats (alpha reuses row 0)
  static constexpr uint32_t kAlpha = kRedMax;
  static constexpr uint32_t kRedSum = kRedMax + 16 * NR;  // 2 x 4 x NR floats
  static constexpr uint32_t kKref = kRedSum + 32 * NR;
  static constexpr uint32_t kBlkBars = kKref + 4 * NR;
  static_assert(kBlkBars % 8 == 0, "mbarrier alignment");
  static constexpr uint32_t kEnd = kBlkBars + 18 * 8;
  static constexpr uint32_t kSmemBytes = kEnd + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448u, "shared memory");
};
// PV completions alternate between BAR_ODONE and this slot (the stage's
// full/empty barriers are the block barriers).
constexpr int kBarOdone1W = BAR_FULL0;

// Rows of a staged 128-token tile (four pages) that hold no loaded key; the
// warp zeroes all 1152 bytes of each (nine 128-byte blocks, 16 KB apart).
// kGather: `info` holds the rows loaded per page (byte q for page q);
// otherwise the first `valid` rows of the tile are keys of the split.
template <bool kGather>
__device__ __forceinline__ void zero_unloaded_rows_w(uint8_t* kvp, int lane, uint32_t info,
                                                     int valid) {
  const uint4 z = make_uint4(0, 0, 0, 0);
  auto zero_rows = [&](int r0, int nrow) {
    for (int idx = lane; idx < nrow * 72; idx += 32) {
      const int r = r0 + idx / 72;
      const int c = idx % 72;
      *reinterpret_cast<uint4*>(kvp + (c / 8) * bw::kBlk + r * 128 + (c % 8) * 16) = z;
    }
  };
  bool any = false;
  if constexpr (kGather) {
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      const int nv = static_cast<int>((info >> (8 * q)) & 0xFFu);
      if (nv < MLA_PAGE_SIZE) {
        zero_rows(q * MLA_PAGE_SIZE + nv, MLA_PAGE_SIZE - nv);
        any = true;
      }
    }
  } else if (valid < bw::kTok) {
    zero_rows(valid, bw::kTok - valid);
    any = true;
  }
  if (any) {
    fence_proxy_async_smem();
    __syncwarp();
  }
}

template <int NR, bool kGather, bool kItems>
__global__ void __launch_bounds__(CfgW<NR>::kThreads, 1)
    mla_split_kv_bf16_wide_kernel(const __grid_constant__ CUtensorMap tm_kv,
                                  const __grid_constant__ CUtensorMap tm_q, const DecodeParams p) {
  using C = CfgW<NR>;
  using bw::kTok;
  const int ngroups = (p.rows_per_req + p.rows_per_group - 1) / p.rows_per_group;
  int b, split, grp;
  if (!cta_coords<kItems>(p, ngroups, b, split, grp)) return;
  if (split >= p.splits[b]) return;  // empty split slot of a shorter request
  SplitRange sr;
  if (!split_range<kGather, kTok>(p, b, split, sr)) return;
  const int L = sr.L, nsplit = sr.nsplit, q_b = sr.q_b, tok_end = sr.tok_end, t0 = sr.t0;
  const bool sparse = sr.sparse;
  const float c_log2 =
      p.sm_scale_dev ? *p.sm_scale_dev * 1.4426950408889634f : p.c_log2;
  const int row0 = grp * p.rows_per_group;
  const int rows_here = min(p.rows_per_group, p.rows_per_req - row0);
  // Rows of real query tokens (the others are padding slots of a shorter
  // query block: no key is visible to them).
  const int rows_valid = max(0, min(rows_here, q_b * p.num_heads - row0));
  const int n_tiles =
      (rows_valid > 0 && tok_end > t0) ? (tok_end - t0 + kTok - 1) / kTok : 0;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(base);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kBars + 8u * i; };
  // Block b of the stage: b = 0..7 latent blocks of 64 elements, 8 rope.
  auto full_blk = [&](int blk) -> uint32_t { return sbase + C::kBlkBars + 8u * blk; };
  auto empty_blk = [&](int blk) -> uint32_t { return sbase + C::kBlkBars + 8u * (9 + blk); };
  volatile int* flags = reinterpret_cast<volatile int*>(base + C::kFlags);
  volatile int* abort_flag = flags + 2;
  float* red_max = reinterpret_cast<float*>(base + C::kRedMax);
  float* red_sum = reinterpret_cast<float*>(base + C::kRedSum);
  float* kref = reinterpret_cast<float*>(base + C::kKref);
  float* alpha_s = reinterpret_cast<float*>(base + C::kAlpha);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int k = 0; k < 9; ++k) {
      mbar_init(full_blk(k), 1);
      mbar_init(empty_blk(k), 1);
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
    mbar_init(bar(kBarOdone1W), 1);
    mbar_init(bar(BAR_FINAL), 2);  // one commit from each MMA warp
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + C::kTmemSlot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base + C::kTmemSlot);

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      tma_prefetch_desc(&tm_kv);
      tma_prefetch_desc(&tm_q);
      const int qrow = b * p.rows_per_req + row0;
      mbar_arrive_expect_tx(bar(BAR_QFULL), C::kQBytes);
#pragma unroll
      for (int d = 0; d < 9; ++d)
        tma_load_2d(sbase + C::kQ + d * NR * 128, &tm_q, d * 64, qrow, bar(BAR_QFULL));
    }
    const uint64_t pol = l2_policy_evict_first();
    const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.max_pages;
    const int page0 = t0 / MLA_PAGE_SIZE;
    const int page_end = (tok_end + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE;  // exclusive
    // Page ids of 8 tiles (32 pages) per window, one per lane, fetched a
    // window ahead, with the rows of each page to load (0: not loaded).
    int last_lp = -1;
    int window_nv, window_next_nv;
    int window = bf16_window_page<kGather>(p, sr, pt, b, page0, page_end, 0, lane, last_lp,
                                           window_nv);
    int window_next = bf16_window_page<kGather>(p, sr, pt, b, page0, page_end, 1, lane, last_lp,
                                                window_next_nv);
    volatile uint32_t* stage_info = reinterpret_cast<volatile uint32_t*>(base + C::kStageInfo);
    int issued = 0;       // tiles whose nine blocks are out
    int armed_part = 0;   // blocks out of a tile cut short by a failed wait
    for (int i = 0; i < n_tiles; ++i) {
      if (i > 0 && (i & 7) == 0) {
        window = window_next;
        window_nv = window_next_nv;
        window_next = bf16_window_page<kGather>(p, sr, pt, b, page0, page_end, (i >> 3) + 1,
                                                lane, last_lp, window_next_nv);
      }
      bool ok = !expired_here(p, WAIT_STAGE_FREE, i);
      ok = __all_sync(0xffffffffu, ok && !*abort_flag);
      if (!ok) {
        if (lane == 0) {
          report(p.status, MLA_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      // Lane q (< 4) takes the id and the rows to load of the tile's page q;
      // the rows per page go to the QK warp (which zeroes the rest) with the
      // rope block's full barrier.
      const int src = (i & 7) * 4 + (lane & 3);
      const int my_page = __shfl_sync(0xffffffffu, window, src);
      const int my_nv = __shfl_sync(0xffffffffu, window_nv, src);
      const int nv1 = __shfl_sync(0xffffffffu, my_nv, 1);
      const int nv2 = __shfl_sync(0xffffffffu, my_nv, 2);
      const int nv3 = __shfl_sync(0xffffffffu, my_nv, 3);
      const bool my_load = my_nv > 0;
      const int nload = __popc(__ballot_sync(0xffffffffu, lane < 4 && my_load));
      const uint32_t kv = sbase + C::kKV;
      const int row = my_page * MLA_PAGE_SIZE;
      // Rope first (free once QK(i - 1) is done), then latent blocks 0-7
      // as PV(i - 1) releases them.
      int armed = 0;
#pragma unroll 1
      for (int bi = 0; bi < 9; ++bi) {
        const int blk = (bi == 0) ? bw::kRopeBlk : bi - 1;
        if (i > 0) {
          ok = mbar_wait_abort(empty_blk(blk), (i - 1) & 1, p.wait_cycles, abort_flag);
          ok = __all_sync(0xffffffffu, ok && !*abort_flag);
          if (!ok) break;
        }
        const uint32_t fb = full_blk(blk);
        if (lane == 0) {
          if (kGather && bi == 0)
            stage_info[0] = static_cast<uint32_t>(my_nv) | (static_cast<uint32_t>(nv1) << 8) |
                            (static_cast<uint32_t>(nv2) << 16) |
                            (static_cast<uint32_t>(nv3) << 24);
          mbar_arrive_expect_tx(fb, nload * (MLA_PAGE_SIZE * 128));
        }
        __syncwarp();
        if (lane < 4 && my_load)
          tma_load_2d_hint(kv + blk * bw::kBlk + lane * (MLA_PAGE_SIZE * 128), &tm_kv, blk * 64,
                           row, fb, pol);
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
      issued = i + 1;
    }
    // Before the CTA exits, the copies this warp issued land: the last full
    // tile's blocks (those a cut-short tile re-armed have landed for it: their
    // release needed them), then the cut-short tile's armed blocks.
    if (lane == 0) {
      if (issued > 0) {
        const int k = issued - 1;
        for (int bi = armed_part; bi < 9; ++bi)
          mbar_wait(full_blk(bi == 0 ? bw::kRopeBlk : bi - 1), k & 1, kWaitLimitCycles);
      }
      for (int bi = 0; bi < armed_part; ++bi)
        mbar_wait(full_blk(bi == 0 ? bw::kRopeBlk : bi - 1), issued & 1, kWaitLimitCycles);
      mbar_wait(bar(BAR_QFULL), 0, kWaitLimitCycles);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ================= MMA issuers: warp 1 QK, warp 2 PV =================
    constexpr uint32_t kIdQK = idesc_bf16(128, NR, 0, 0);
    constexpr uint32_t kIdPV = idesc_bf16(128, NR, 1, 1);
    bool ok = (warp == 1) ? mbar_wait(bar(BAR_QFULL), 0, p.wait_cycles) : true;
    auto fail = [&]() {
      if (lane == 0) {
        report(p.status, MLA_ERR_TIMEOUT);
        *abort_flag = 1;
      }
    };
    // Four K = 16 steps of QK over block blk of the stage into S buffer sb.
    auto qk_block = [&](int blk, int sb, bool first) {
      tc_fence_after();
#pragma unroll
      for (int sub = 0; sub < 4; ++sub) {
        const uint64_t a = smem_desc(sbase + C::kKV + blk * bw::kBlk + sub * 32, 16, 1024,
                                     kLayoutSW128);
        const uint64_t bd =
            smem_desc(sbase + C::kQ + blk * NR * 128 + sub * 32, 16, 1024, kLayoutSW128);
        umma_bf16(tmem + sb * NR, a, bd, kIdQK, (first && sub == 0) ? 0u : 1u);
      }
    };
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) fail();
    if (warp == 1) {
      // QK(j): the rope steps once the rope block has landed and S buffer
      // j & 1 is free, then each latent block's steps as it lands (all of
      // them first when the tile has rows to zero, which span every block).
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int sb = j & 1;
        const int use = j >> 1;
        bool w = !expired_here(p, WAIT_TILE_FULL, j) &&
                 mbar_wait_abort(full_blk(bw::kRopeBlk), j & 1, p.wait_cycles, abort_flag);
        if (w && use >= 1)
          w = mbar_wait_abort(bar(BAR_SFREE0 + sb), (use - 1) & 1, p.wait_cycles, abort_flag);
        w = __all_sync(0xffffffffu, w && !*abort_flag);
        if (!w) {
          ok = false;
          break;
        }
        const uint32_t info =
            kGather ? *reinterpret_cast<volatile uint32_t*>(base + C::kStageInfo) : 0u;
        const int valid = tok_end - (t0 + j * kTok);
        const bool partial = kGather ? (info != 0x20202020u) : (valid < kTok);
        if (partial) {
          for (int blk = 0; w && blk < 8; ++blk)
            w = mbar_wait_abort(full_blk(blk), j & 1, p.wait_cycles, abort_flag);
          w = __all_sync(0xffffffffu, w && !*abort_flag);
          if (!w) {
            ok = false;
            break;
          }
          zero_unloaded_rows_w<kGather>(base + C::kKV, lane, info, valid);
        }
        if (lane == 0) qk_block(bw::kRopeBlk, sb, true);
        __syncwarp();
        for (int blk = 0; blk < 8; ++blk) {
          if (!partial) {
            w = mbar_wait_abort(full_blk(blk), j & 1, p.wait_cycles, abort_flag);
            w = __all_sync(0xffffffffu, w && !*abort_flag);
            if (!w) break;
          }
          if (lane == 0) qk_block(blk, sb, false);
          __syncwarp();
        }
        if (!w) {
          ok = false;
          break;
        }
        // S^T is complete, and the rope block free, once these MMAs are.
        if (lane == 0) {
          umma_commit(bar(BAR_SFULL0 + sb));
          umma_commit(empty_blk(bw::kRopeBlk));
        }
        __syncwarp();
      }
    } else {
      // PV(i) as soon as its P^T is ready; latent group d (blocks 2d, 2d + 1)
      // is released when its MMAs complete.
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int pb = i & 1;
        bool w = !expired_here(p, WAIT_P_FULL, i) &&
                 mbar_wait_abort(bar(BAR_PFULL0 + pb), (i >> 1) & 1, p.wait_cycles,
                                 abort_flag);
        w = __all_sync(0xffffffffu, w && !*abort_flag);
        if (!w) {
          ok = false;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t pbuf = sbase + C::kP + pb * C::kPBytes;
#pragma unroll
          for (int d = 0; d < 4; ++d) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              // A = V^T, MN-major: 64-element atoms 16 KB apart (latent blocks
              // 2d, 2d + 1), 8-token groups 1 KB apart; 16 tokens per step.
              const uint64_t a = smem_desc(sbase + C::kKV + 2 * d * bw::kBlk + ks * 2048,
                                           bw::kBlk, 1024, kLayoutSW128);
              // B = P^T, MN-major, no swizzle: 8-row groups 2 KB apart, 8-token
              // groups 128 B apart.
              const uint64_t bd = smem_desc(pbuf + ks * 256, 128, 2048, kLayoutNone);
              umma_bf16(tmem + C::kOCol + d * NR, a, bd, kIdPV, (i > 0 || ks > 0) ? 1u : 0u);
            }
            umma_commit(empty_blk(2 * d));
            umma_commit(empty_blk(2 * d + 1));
          }
          umma_commit(bar(BAR_PFREE0 + pb));
          umma_commit(bar((i & 1) ? kBarOdone1W : BAR_ODONE));
        }
        __syncwarp();
      }
    }
    if (!ok) fail();
    if (lane == 0) umma_commit(bar(BAR_FINAL));
    __syncwarp();
    mbar_wait(bar(BAR_FINAL), 0, kWaitLimitCycles);
  } else {
    // ================= softmax warpgroups =================
    // As in the FP8 kernel's 32/48-row configurations: TMEM lane = token of
    // the tile, warpgroup g owns rows [g * NRH, (g + 1) * NRH) of every token.
    constexpr int NRH = C::NRH;
    constexpr int NT = 128 * C::SWG;
    const int quad = warp & 3;
    const int rbase = ((warp - 3) >> 2) * NRH;
    const int tok = quad * 32 + lane;  // token within the tile == TMEM lane == O^T lane
    const int sid = threadIdx.x - 96;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    float k_row = -INFINITY;
    float l_row = 0.0f;
    float kreg[NRH];
#pragma unroll
    for (int k = 0; k < NRH; ++k) kreg[k] = -INFINITY;
    const float c = c_log2;
    const int qi_first = row0 / p.num_heads;
    const int lim_min = p.causal ? min(tok_end, L - q_b + qi_first + 1) : tok_end;
    const int my_row0 = row0 + rbase;
    const int my_rows = max(0, min(NRH, rows_valid - rbase));
    // Selection: logical page ids of 8 tiles' compact pages, one per lane
    // (this warp's tokens are page `quad` of the tile).
    auto sel_window = [&](int w) -> int {
      const int cp = t0 / MLA_PAGE_SIZE + w * 32 + lane;
      return (cp < p.topk) ? p.block_idx[static_cast<int64_t>(b) * p.topk + cp] : -1;
    };
    int sel_cur = -1, sel_next = -1;
    if (sparse) {
      sel_cur = sel_window(0);
      sel_next = sel_window(1);
    }
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int sb = i & 1;
      const int use = i >> 1;
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
      const int tile_tok0 = t0 + i * kTok;
      const int j = tile_tok0 + tok;
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
        tok_ok = tok_ok && pos >= sr.win_lo && pos < sr.win_hi;
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
      } else if (tile_tok0 + kTok <= lim_min) {
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
      // Reference check and update as in the FP8 kernel (integer references
      // k with t <= k + 0.75; exact power-of-two rescales of l and O^T).
      bool over = false;
#pragma unroll
      for (int k = 0; k < NRH; ++k) over |= t[k] > kreg[k] + 0.75f;
      const bool any_over = bar_sync_or(kVoteBarrier, NT, over);
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
          // PV(i - 1) done (S^T(i) implies PV(i - 1) released every latent
          // block, so its completion barrier is within one phase).
          ok = mbar_wait_abort(bar(((i - 1) & 1) ? kBarOdone1W : BAR_ODONE), ((i - 1) >> 1) & 1,
                               p.wait_cycles, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (ok) {
            tc_fence_after();
#pragma unroll 1
            for (int d = 0; d < 4; ++d) {
#pragma unroll
              for (int cc = 0; cc < NRH / 8; ++cc) {
                uint32_t r[8];
                const uint32_t addr = tmem + lane_addr + C::kOCol + d * NR + rbase + cc * 8;
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
#pragma unroll
      for (int k = 0; k < NRH; ++k) t[k] = softmax_weight<true>(t[k], kreg[k]);
      // P^T buffer i & 1: free once PV(i - 2) is done.
      const int pb = i & 1;
      if (ok && expired_here(p, WAIT_P_FREE, i)) ok = false;
      if (ok && i >= 2)
        ok = mbar_wait_abort(bar(BAR_PFREE0 + pb), ((i >> 1) - 1) & 1, p.wait_cycles,
                             abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok && lane == 0) *abort_flag = 1;
      if (ok) {
        // P^T (BF16), MN-major: [NR/8 row groups][128 tokens][8 rows].
        uint8_t* pbuf = base + C::kP + pb * C::kPBytes;
#pragma unroll
        for (int g = 0; g < NRH / 8; ++g) {
          uint4 v;
          v.x = pack_bf16x2(t[g * 8 + 0], t[g * 8 + 1]);
          v.y = pack_bf16x2(t[g * 8 + 2], t[g * 8 + 3]);
          v.z = pack_bf16x2(t[g * 8 + 4], t[g * 8 + 5]);
          v.w = pack_bf16x2(t[g * 8 + 6], t[g * 8 + 7]);
          *reinterpret_cast<uint4*>(pbuf + ((rbase >> 3) + g) * 2048 + tok * 16) = v;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(BAR_PFULL0 + pb));
      }
      warp_reduce_rows<NRH, false>(t, lane, red_sum + (i & 1) * 4 * NR + quad * NR + rbase);
    }
    if (!ok && lane == 0) {
      report(p.status, MLA_ERR_TIMEOUT);
      *abort_flag = 1;
    }
    // ---- epilogue (as in the FP8 kernel; O^T has NR columns per group) ----
    named_bar_sync(kSoftmaxBarrier, NT);
    const bool single = (nsplit == 1);
    float* scale_s = alpha_s;
    if (sid < NR) {
      if (n_tiles > 0) {
        const float* rs = red_sum + ((n_tiles - 1) & 1) * 4 * NR;
        l_row += (rs[sid] + rs[NR + sid]) + (rs[2 * NR + sid] + rs[3 * NR + sid]);
      }
      const float m_s = (k_row == -INFINITY) ? -INFINITY : k_row - 8.0f;
      const int64_t grow = static_cast<int64_t>(b) * p.rows_per_req + row0 + sid;
      float sc = 0.0f;
      if (sid < rows_here) {
        if (single) {
          // A sink is one more (zero-valued) key: it joins the denominator.
          const float sink2 = p.sinks
                                  ? p.sinks[(row0 + sid) % p.num_heads] * 1.4426950408889634f
                                  : -INFINITY;
          const float mm = fmaxf(l_row > 0.0f ? m_s : -INFINITY, sink2);
          const float a = (l_row > 0.0f) ? exp2f(m_s - mm) : 0.0f;
          const float den = l_row * a + (sink2 == -INFINITY ? 0.0f : exp2f(sink2 - mm));
          if (p.lse)
            p.lse[grow] = (den > 0.0f) ? 0.6931471805599453f * (mm + log2f(den)) : -INFINITY;
          sc = (den > 0.0f) ? p.output_scale * a / den : 0.0f;
        } else {
          float* ml = p.ws_ml + (grow * p.max_splits + split) * 2;
          ml[0] = m_s;
          ml[1] = l_row;
          sc = 1.0f;
        }
      }
      scale_s[sid] = sc;
    }
    named_bar_sync(kSoftmaxBarrier, NT);
    bool fin = !expired_here(p, WAIT_FINAL, 0) && mbar_wait(bar(BAR_FINAL), 0, p.wait_cycles);
    fin = __all_sync(0xffffffffu, fin);
    if (!fin && lane == 0) report(p.status, MLA_ERR_TIMEOUT);
    if (ok && fin && n_tiles > 0) {
      tc_fence_after();
      // Per latent group: this warpgroup's NRH columns in one batch of TMEM
      // loads, then the stores (row k of the warpgroup at base + k * stride).
      const int64_t grow0 = static_cast<int64_t>(b) * p.rows_per_req + row0 + rbase;
      const int64_t stride = single ? MLA_LATENT_DIM
                                    : static_cast<int64_t>(p.max_splits) * MLA_LATENT_DIM;
      float* const obase =
          single ? nullptr : p.ws_o + (grow0 * p.max_splits + split) * MLA_LATENT_DIM;
      const int nrow = min(NRH, rows_here - rbase);
      // Each warp turns its 32 dims x 8 rows at a time around through 1 KB of
      // the P^T buffers (free after the last PV), so that a lane stores 4
      // contiguous dims of a row (16 B of a partial, 8 B of BF16 output).
      float* const scr = reinterpret_cast<float*>(base + C::kP) + (warp - 3) * 256;
      // The rows' scales in registers: read from shared memory inside the
      // store loop, each would wait behind the previous row's stores.
      float sc_r[NRH];
#pragma unroll
      for (int k = 0; k < NRH; ++k) sc_r[k] = scale_s[rbase + k];
#pragma unroll 1
      for (int d = 0; d < 4; ++d) {
        const int dim4 = d * 128 + quad * 32 + (lane & 7) * 4;  // this lane's 4 dims
        uint32_t r[NRH];
#pragma unroll
        for (int cc = 0; cc < NRH / 8; ++cc)
          tmem_ld8(tmem + lane_addr + C::kOCol + d * NR + rbase + cc * 8,
                   *reinterpret_cast<uint32_t(*)[8]>(&r[cc * 8]));
        tmem_ld_wait();
#pragma unroll
        for (int c8 = 0; c8 < NRH / 8; ++c8) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            scr[kk * 32 + lane] = __uint_as_float(r[c8 * 8 + kk]) * sc_r[c8 * 8 + kk];
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
      }
    } else if (ok && fin && n_tiles == 0 && single) {
      // No key of this split is visible to any row here: O = 0 (partials
      // need only (-inf, 0)).
      for (int d = 0; d < 4; ++d) {
        const int dim = d * 128 + tok;
        for (int row = rbase; row < min(rows_here, rbase + NRH); ++row) {
          const int64_t grow = static_cast<int64_t>(b) * p.rows_per_req + row0 + row;
          p.out[grow * MLA_LATENT_DIM + dim] = __float2bfloat16_rn(0.0f);
          if (p.out_f32) p.out_f32[grow * MLA_LATENT_DIM + dim] = 0.0f;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 2-D BF16 view [rows, 576] with a (64, box_y) box, 128-byte swizzle.
static bool make_map_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint32_t box_y) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {MLA_HEAD_DIM, rows};
  cuuint64_t strides[1] = {kRowBytesB};
  cuuint32_t box[2] = {64, box_y};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NR, bool kGather, bool kItems>
static cudaError_t launch_split_bf16_w_t(const void* q, const void* kv, int64_t num_pages,
                                         int batch, int groups, int num_ctas,
                                         const DecodeParams& prm, cudaStream_t stream) {
  using C = CfgW<NR>;
  static std::atomic<uint64_t> attr_done{0};
  {
    const cudaError_t e = ensure_smem_attr(mla_split_kv_bf16_wide_kernel<NR, kGather, kItems>,
                                           static_cast<int>(C::kSmemBytes), attr_done);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tm_kv, tm_q;
  if (!make_map_bf16(&tm_kv, kv, static_cast<uint64_t>(num_pages) * MLA_PAGE_SIZE,
                     MLA_PAGE_SIZE) ||
      !make_map_bf16(&tm_q, q, static_cast<uint64_t>(batch) * prm.rows_per_req, NR))
    return cudaErrorInvalidValue;
  const dim3 grid = kItems ? dim3(num_ctas) : dim3(batch, prm.max_splits * groups);
  mla_split_kv_bf16_wide_kernel<NR, kGather, kItems>
      <<<grid, C::kThreads, C::kSmemBytes, stream>>>(tm_kv, tm_q, prm);
  return cudaGetLastError();
}

template <bool kGather, bool kItems>
static cudaError_t launch_split_bf16_q16_t(const void* q, const void* kv, int64_t num_pages,
                                           int batch, int groups, int num_ctas,
                                           const DecodeParams& prm, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  {
    const cudaError_t e = ensure_smem_attr(mla_split_kv_bf16_q16_kernel<kGather, kItems>,
                                           static_cast<int>(q16::kSmemBytes), attr_done);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap tm_kv, tm_q;
  if (!make_map_bf16(&tm_kv, kv, static_cast<uint64_t>(num_pages) * MLA_PAGE_SIZE,
                     MLA_PAGE_SIZE) ||
      !make_map_bf16(&tm_q, q, static_cast<uint64_t>(batch) * prm.rows_per_req, q16::NR))
    return cudaErrorInvalidValue;
  const dim3 grid = kItems ? dim3(num_ctas) : dim3(batch, prm.max_splits * groups);
  mla_split_kv_bf16_q16_kernel<kGather, kItems>
      <<<grid, q16::kThreads, q16::kSmemBytes, stream>>>(tm_kv, tm_q, prm);
  return cudaGetLastError();
}

// Row-group configuration x (key windows or selections) x (item list): each
// combination is its own kernel instantiation, so the plain grid variant's
// code is what it is without the options.
template <int NR>
static cudaError_t launch_split_bf16(const void* q, const void* kv, int64_t num_pages, int batch,
                                     int groups, int num_ctas, const DecodeParams& prm,
                                     cudaStream_t stream) {
  const bool gather = prm.kv_bounds != nullptr || prm.block_idx != nullptr;
  const bool items = prm.cta_items != nullptr;
  if constexpr (NR == q16::NR) {
    if (gather)
      return items ? launch_split_bf16_q16_t<true, true>(q, kv, num_pages, batch, groups,
                                                          num_ctas, prm, stream)
                   : launch_split_bf16_q16_t<true, false>(q, kv, num_pages, batch, groups,
                                                           num_ctas, prm, stream);
    return items ? launch_split_bf16_q16_t<false, true>(q, kv, num_pages, batch, groups,
                                                         num_ctas, prm, stream)
                 : launch_split_bf16_q16_t<false, false>(q, kv, num_pages, batch, groups,
                                                          num_ctas, prm, stream);
  } else {
    if (gather)
      return items ? launch_split_bf16_w_t<NR, true, true>(q, kv, num_pages, batch, groups,
                                                            num_ctas, prm, stream)
                   : launch_split_bf16_w_t<NR, true, false>(q, kv, num_pages, batch, groups,
                                                             num_ctas, prm, stream);
    return items ? launch_split_bf16_w_t<NR, false, true>(q, kv, num_pages, batch, groups,
                                                           num_ctas, prm, stream)
                 : launch_split_bf16_w_t<NR, false, false>(q, kv, num_pages, batch, groups,
                                                            num_ctas, prm, stream);
  }
}

}  // namespace mla

using namespace mla;

static int decode_bf16(const void* q_bf16, const void* kv_pages_bf16, int64_t num_pages,
                       const int32_t* page_table, int32_t max_pages_per_req,
                       const int32_t* kv_lens, const int32_t* block_idx, int32_t topk,
                       const int32_t* splits, const int32_t* chunks,
                       int32_t max_splits, int32_t kv_split, int32_t batch, int32_t q_len,
                       int32_t num_heads, int32_t causal, float softmax_scale, void* workspace,
                       size_t workspace_bytes, void* out_bf16, float* lse_f32,
                       float* out_f32_debug, const mla_decode_options_t* options,
                       const char* who_c, void* stream) {
  const std::string who(who_c);
  if (!q_bf16 || !kv_pages_bf16 || !page_table || !kv_lens || !splits || !chunks || !workspace ||
      !out_bf16) {
    set_error(who + ": null pointer argument");
    return MLA_ERR_INVALID_ARG;
  }
  if (batch < 1 || q_len < 1 || num_heads < 1 || max_pages_per_req < 1 || num_pages < 1) {
    set_error(who + ": batch, q_len, num_heads, max_pages_per_req and num_pages must be >= 1");
    return MLA_ERR_INVALID_ARG;
  }
  if (static_cast<int64_t>(num_heads) * q_len > MLA_MAX_ROWS || batch > 65535) {
    set_error(who + ": num_heads * q_len above MLA_MAX_ROWS or batch above 65535");
    return MLA_ERR_UNSUPPORTED;
  }
  if (num_pages * MLA_PAGE_SIZE > INT32_MAX) {
    set_error(who + ": page pool too large for 32-bit TMA row coordinates");
    return MLA_ERR_UNSUPPORTED;
  }
  if (max_splits < 1 || max_splits > MLA_MAX_SPLITS ||
      (kv_split != 1 && kv_split != 2 && kv_split != 4 && kv_split != 8 && kv_split != 16)) {
    set_error(who + ": max_splits in [1, MLA_MAX_SPLITS], kv_split in {1,2,4,8,16}");
    return MLA_ERR_INVALID_ARG;
  }
  if (!aligned(q_bf16, 16) || !aligned(kv_pages_bf16, 16) || !aligned(workspace, 256) ||
      !aligned(out_bf16, 8) || (out_f32_debug && !aligned(out_f32_debug, 16))) {
    set_error(who + ": q/kv need 16-byte, workspace 256-byte, outputs 8/16-byte alignment");
    return MLA_ERR_INVALID_ARG;
  }
  if (!std::isfinite(softmax_scale)) {
    set_error(who + ": softmax_scale must be finite");
    return MLA_ERR_INVALID_ARG;
  }
  const int64_t rows_total = static_cast<int64_t>(batch) * q_len * num_heads;
  const size_t need = ws_total(rows_total, max_splits);
  if (workspace_bytes < need) {
    set_error(who + ": workspace of " + std::to_string(workspace_bytes) +
              " bytes is below the " + std::to_string(need) + " required");
    return MLA_ERR_WORKSPACE_TOO_SMALL;
  }
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  const RowGroups rg = row_groups(num_heads * q_len);
  DecodeParams prm = {};
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
  prm.rows_per_group = rg.rows;
  prm.c_log2 = static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634);
  prm.kv_scale = 1.0f;
  prm.output_scale = 1.0f;
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
  prm.block_idx = block_idx;
  prm.topk = topk;
  prm.batch = batch;
  int num_ctas = 0;
  int phases = MLA_PHASE_ALL;
  if (options) {
    if (!std::isfinite(options->output_scale)) {
      set_error(who + ": output_scale must be finite");
      return MLA_ERR_INVALID_ARG;
    }
    if (options->q_scale_dev || options->kv_scale_dev) {
      set_error(who + ": q/kv scales are FP8-only (BF16 Q and KV carry no scale)");
      return MLA_ERR_UNSUPPORTED;
    }
    if (options->persistent_ctas != 0) {
      set_error(who + ": persistent CTAs are FP8-only");
      return MLA_ERR_UNSUPPORTED;
    }
    phases = options->phases;
    if (phases != MLA_PHASE_ALL && phases != MLA_PHASE_SPLIT && phases != MLA_PHASE_MERGE) {
      set_error(who + ": phases must be MLA_PHASE_ALL, MLA_PHASE_SPLIT or MLA_PHASE_MERGE");
      return MLA_ERR_INVALID_ARG;
    }
    if (options->cta_items) {
      const int64_t cap = static_cast<int64_t>(batch) * max_splits * rg.groups;
      if (options->num_ctas < 1 || options->num_ctas > cap) {
        set_error(who + ": num_ctas must be in [1, batch * max_splits * row groups]");
        return MLA_ERR_INVALID_ARG;
      }
      num_ctas = options->num_ctas;
    }
    prm.sm_scale_dev = options->softmax_scale_dev;
    prm.output_scale = options->output_scale;
    prm.sinks = options->sinks;
    prm.query_lens = options->query_lens;
    prm.kv_bounds = options->kv_bounds;
    prm.cta_items = options->cta_items;
    prm.num_items = options->cta_items ? options->num_ctas : 0;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (phases != MLA_PHASE_MERGE) {
    switch (rg.nr) {
      case 16:
        e = launch_split_bf16<16>(q_bf16, kv_pages_bf16, num_pages, batch, rg.groups, num_ctas,
                                  prm, st);
        break;
      case 32:
        e = launch_split_bf16<32>(q_bf16, kv_pages_bf16, num_pages, batch, rg.groups, num_ctas,
                                  prm, st);
        break;
      case 48:
        e = launch_split_bf16<48>(q_bf16, kv_pages_bf16, num_pages, batch, rg.groups, num_ctas,
                                  prm, st);
        break;
      default:
        set_error(who + ": internal row grouping error");
        return MLA_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) return cuda_fail((who + ": split-KV launch").c_str(), e);
  }
  if (max_splits > 1 && phases != MLA_PHASE_SPLIT) {
    MergeParams mp = {};
    mp.po = prm.ws_o;
    mp.pml = prm.ws_ml;
    mp.rows = static_cast<int32_t>(rows_total);
    mp.stride_s = max_splits;
    mp.uniform_s = max_splits;
    mp.splits = splits;
    mp.rows_per_req = num_heads * q_len;
    mp.num_heads = num_heads;
    mp.output_scale = prm.output_scale;
    mp.sinks = prm.sinks;
    mp.out = prm.out;
    mp.lse = lse_f32;
    mp.out_f32 = out_f32_debug;
    e = launch_merge(mp, kv_split, st);
    if (e != cudaSuccess) return cuda_fail((who + ": merge launch").c_str(), e);
  }
  return MLA_OK;
}

extern "C" int mla_decode_bf16(const void* q_bf16, const void* kv_pages_bf16, int64_t num_pages,
                               const int32_t* page_table, int32_t max_pages_per_req,
                               const int32_t* kv_lens, const int32_t* splits,
                               const int32_t* chunks, int32_t max_splits, int32_t kv_split,
                               int32_t batch, int32_t q_len, int32_t num_heads, int32_t causal,
                               float softmax_scale, void* workspace, size_t workspace_bytes,
                               void* out_bf16, float* lse_f32, float* out_f32_debug,
                               void* stream) {
  return decode_bf16(q_bf16, kv_pages_bf16, num_pages, page_table, max_pages_per_req, kv_lens,
                     nullptr, 0, splits, chunks, max_splits, kv_split, batch, q_len, num_heads,
                     causal, softmax_scale, workspace, workspace_bytes, out_bf16, lse_f32,
                     out_f32_debug, nullptr, "mla_decode_bf16", stream);
}

extern "C" int mla_decode_bf16_ex(const void* q_bf16, const void* kv_pages_bf16,
                                  int64_t num_pages, const int32_t* page_table,
                                  int32_t max_pages_per_req, const int32_t* kv_lens,
                                  const int32_t* splits, const int32_t* chunks,
                                  int32_t max_splits, int32_t kv_split, int32_t batch,
                                  int32_t q_len, int32_t num_heads, int32_t causal,
                                  float softmax_scale, void* workspace, size_t workspace_bytes,
                                  void* out_bf16, float* lse_f32, float* out_f32_debug,
                                  const mla_decode_options_t* options, void* stream) {
  return decode_bf16(q_bf16, kv_pages_bf16, num_pages, page_table, max_pages_per_req, kv_lens,
                     nullptr, 0, splits, chunks, max_splits, kv_split, batch, q_len, num_heads,
                     causal, softmax_scale, workspace, workspace_bytes, out_bf16, lse_f32,
                     out_f32_debug, options, "mla_decode_bf16_ex", stream);
}

extern "C" int mla_decode_bf16_sparse(const void* q_bf16, const void* kv_pages_bf16,
                                      int64_t num_pages, const int32_t* page_table,
                                      int32_t max_pages_per_req, const int32_t* kv_lens,
                                      const int32_t* block_idx, int32_t topk,
                                      const int32_t* splits, const int32_t* chunks,
                                      int32_t max_splits, int32_t kv_split, int32_t batch,
                                      int32_t q_len, int32_t num_heads, int32_t causal,
                                      float softmax_scale, void* workspace,
                                      size_t workspace_bytes, void* out_bf16, float* lse_f32,
                                      float* out_f32_debug, const mla_decode_options_t* options,
                                      void* stream) {
  if (!block_idx) {
    set_error("mla_decode_bf16_sparse: null block_idx");
    return MLA_ERR_INVALID_ARG;
  }
  if (topk < 1 || static_cast<int64_t>(topk) * MLA_PAGE_SIZE > INT32_MAX / 2) {
    set_error("mla_decode_bf16_sparse: topk must be >= 1 and 32 * topk must fit in int32");
    return MLA_ERR_INVALID_ARG;
  }
  return decode_bf16(q_bf16, kv_pages_bf16, num_pages, page_table, max_pages_per_req, kv_lens,
                     block_idx, topk, splits, chunks, max_splits, kv_split, batch, q_len,
                     num_heads, causal, softmax_scale, workspace, workspace_bytes, out_bf16,
                     lse_f32, out_f32_debug, options, "mla_decode_bf16_sparse", stream);
}
