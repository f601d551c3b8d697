// Device-side pieces shared by the FP8 and BF16 split-KV kernels and the
// merge: launch parameters, the softmax weight, reductions, E4M3 packing.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>

#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {

constexpr long long kWaitLimitCycles = 4000000000LL;  // about 2 s at 2 GHz
constexpr uint32_t kSoftmaxBarrier = 1;
constexpr uint32_t kVoteBarrier = 2;
// 96-row configuration: per-warpgroup vote and reference barriers (3 each).
constexpr uint32_t kVoteBarrierWg0 = 3;
constexpr uint32_t kSoftmaxBarrierWg0 = 6;

struct DecodeParams {
  const int32_t* page_table;
  const int32_t* kv_lens;
  const int32_t* splits;
  const int32_t* chunks;
  int64_t num_pages;
  int32_t max_pages;
  int32_t max_splits;
  int32_t q_len;
  int32_t num_heads;
  int32_t causal;
  int32_t rows_per_req;    // R = q_len * num_heads
  int32_t rows_per_group;  // RG
  float c_log2;            // softmax_scale * q_scale * kv_scale * log2(e)
  float kv_scale;
  // Optional device-side scales (element 0 is read by the kernel, so a graph
  // replay picks up new values); NULL means the host value above.
  const float* q_scale_dev;
  const float* kv_scale_dev;
  const float* sm_scale_dev;
  float q_scale_h;
  float sm_scale_h;
  float output_scale;      // multiplies O (not the LSE)
  const float* sinks;      // optional per-head sink logits (natural-log units)
  // Restrictions of the visible keys (NULL = none): per-request query-token
  // counts in the padded q_len slots, key windows [lo, hi) (int32 [B][2]) and
  // selected logical pages (int32 [B][topk], ascending, negative = unused; the
  // split plan then covers the compact range of 32 * topk tokens).
  const int32_t* query_lens;
  const int32_t* kv_bounds;
  const int32_t* block_idx;
  int32_t topk;
  // Optional CTA item list (mla_decode_plan_items): CTA i works on item
  // cta_items[i] of a 1-D grid, or (persistent CTAs) on items i, i + gridDim.x,
  // ... < num_items; NULL = the (batch, splits x groups) grid.
  const int32_t* cta_items;
  int32_t num_items;
  int32_t batch;
  long long wait_cycles;   // limit of the pipeline waits (drains always use the long limit)
  // Test hook (mla_debug_set_expire): (role << 24) | tile makes that one
  // pipeline wait read as expired; -1 = off.
  int32_t debug_expire;
  int* status;
  float* ws_ml;
  float* ws_o;
  __nv_bfloat16* out;
  float* lse;
  float* out_f32;
};

// Barrier indices inside the aux block.  The BF16 kernels use the first 17;
// the FP8 kernel also has the per-item Q-free and O^T-free barriers of its
// persistent mode.
enum : int {
  BAR_FULL0 = 0, BAR_EMPTY0 = 3, BAR_QFULL = 6, BAR_SFULL0, BAR_SFULL1, BAR_SFREE0, BAR_SFREE1,
  BAR_PFULL0, BAR_PFULL1, BAR_PFREE0, BAR_PFREE1, BAR_ODONE, BAR_FINAL, BAR_QFREE, BAR_OFREE,
  BAR_COUNT
};
static_assert(BAR_FINAL < 17 && BAR_COUNT <= 19, "barrier slots");

__device__ __forceinline__ void report(int* status, int code) {
  atomicCAS(status, 0, code);
}

// Pipeline wait roles of the test hook: the producer's wait for a free stage,
// the QK issuer's wait for a landed tile, the PV issuer's wait for P^T, the
// softmax's waits for S^T and for a free P^T buffer, and the softmax's wait
// for the last MMAs before the epilogue (tile 0).
enum : int {
  WAIT_STAGE_FREE = 0, WAIT_TILE_FULL = 1, WAIT_P_FULL = 2, WAIT_S_FULL = 3, WAIT_P_FREE = 4,
  WAIT_FINAL = 5
};
__device__ __forceinline__ bool expired_here(const DecodeParams& p, int role, int i) {
  return p.debug_expire == ((role << 24) | i);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^i for an integer i in [-126, 127], exactly.
__device__ __forceinline__ float pow2i(int i) { return __int_as_float((i + 127) << 23); }

// 2^(t - k + 8) with exact power-of-two scaling (k integer-valued): split
// t = r + f with r = rint(t), then 2^f * 2^(r - k + 8), the second factor
// built from its exponent bits.  The rounding uses the 1.5 * 2^23 addition
// trick (FMA-pipe adds instead of rint and float-to-int conversions), exact
// for |t| < 2^21.  Two forms with the same values there, chosen per kernel
// configuration by measurement: kBranchFree clamps t to +-2^21 and flushes
// t far below k to 0 through the exponent clamp (-inf by a select), which
// keeps the many independent weights of a 24-row thread in flight; the other
// form takes an exact fallback branch for |t| >= 2^21 or -inf, which is
// faster for the 16-row kernel.  Scores above 2^21 in log2 units are outside
// the branch-free form's range.
template <bool kBranchFree>
__device__ __forceinline__ float softmax_weight(float t, float k) {
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  if constexpr (kBranchFree) {
    const float tc = fminf(fmaxf(t, -2097152.0f), 2097152.0f);
    const float tr = tc + kMagic;
    const float r = tr - kMagic;            // rint(tc)
    const float f = tc - r;                 // exact, |f| <= 0.5
    const float ef = fmaxf((r - k) + 8.0f, -200.0f);  // integer-valued; exact
    int e = __float_as_int(ef + kMagic) - 0x4B400000 + 127;
    e = max(e, 0);                          // below 2^-126 the weight is flushed to 0
    const float w = ex2_approx(f) * __int_as_float(e << 23);
    return t == -INFINITY ? 0.0f : w;       // masked (the row's k may still be -inf)
  } else {
    if (fabsf(t) < 2097152.0f) {
      const float tr = t + kMagic;
      const float r = tr - kMagic;          // rint(t)
      const float f = t - r;                // exact, |f| <= 0.5
      const float ef = (r - k) + 8.0f;      // integer-valued and exact
      int e = __float_as_int(ef + kMagic) - 0x4B400000 + 127;
      e = max(e, 0);
      return ex2_approx(f) * __int_as_float(e << 23);
    }
    if (t == -INFINITY) return 0.0f;
    const float a = rintf(t);
    const float f = t - a;
    const int sc = static_cast<int>(a) - static_cast<int>(k) + 8;
    if (sc < -126) return 0.0f;
    return ex2_approx(f) * pow2i(sc);
  }
}

// Named barrier over `nthreads` threads that also ORs a predicate across them.
__device__ __forceinline__ bool bar_sync_or(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred q, p;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, %2, %3, q;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// Two E4M3 codes (low byte = element 0) back to floats (exact).
__device__ __forceinline__ float2 unpack_e4m3x2(uint16_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// P as a two-term E4M3 sum: hi = e4m3(p), lo = e4m3(p - hi).  p - hi is exact
// in fp32, and hi + lo carries p to ~2^-8 relative (E4M3 keeps 3 mantissa bits).
__device__ __forceinline__ void split_e4m3x4(const float* p, uint32_t& hi, uint32_t& lo) {
  hi = pack_e4m3x4(p[0], p[1], p[2], p[3]);
  const float2 h01 = unpack_e4m3x2(static_cast<uint16_t>(hi & 0xFFFFu));
  const float2 h23 = unpack_e4m3x2(static_cast<uint16_t>(hi >> 16));
  lo = pack_e4m3x4(p[0] - h01.x, p[1] - h01.y, p[2] - h23.x, p[3] - h23.y);
}

// Two weights as E4M3 hi and lo terms through packed halves: h = f16x2(w0, w1)
// (round to nearest), hi = e4m3(h), lo = e4m3(h - hi).  h - hi is exact in
// f16 (both are multiples of h's f16 quantum and |h - hi| <= half an E4M3
// step), so hi + lo carries each weight to ~2^-8 relative like the fp32 form,
// in five conversions and subtractions per pair instead of seven per value.
// Byte / half 0 holds w0.
__device__ __forceinline__ void split_e4m3x2_h(float w0, float w1, uint32_t& hi, uint32_t& lo) {
  uint32_t h, hh, d;
  uint16_t h8, l8;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(w1), "f"(w0));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(h8) : "r"(h));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hh) : "h"(h8));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(h), "r"(hh));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(l8) : "r"(d));
  hi = h8;
  lo = l8;
}

// 2^(t - k + 8) for the 96-row softmax: the same value as softmax_weight (t
// split as rint(t) + f, exact power-of-two scaling) from a per-row integer
// kc = 135 - 0x4B400000 - k: the bits of t + 1.5 * 2^23 are 0x4B400000 +
// rint(t), so bits + kc is the biased exponent rint(t) - k + 8 + 127, clamped
// at 0 (weights below 2^-126 flush to 0).  A masked score (-inf) and a row
// without a reference (kc = kKcNone) give an exponent below 0, i.e. 0.
// Requires t <= k + 0.75 (the vote guarantees it), so the exponent stays
// below 255.
constexpr int kKcNone = -2130706432;  // -2^31 + 2^24: bits + kc < 0 for every t
__device__ __forceinline__ float softmax_weight_kc(float t, int kc) {
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  const float tc = fmaxf(t, -2097152.0f);
  const float tr = tc + kMagic;
  const float r = tr - kMagic;  // rint(tc)
  const float f = tc - r;       // exact, |f| <= 0.5
  const int e = max(__float_as_int(tr) + kc, 0);
  return ex2_approx(f) * __int_as_float(e << 23);
}

// Warp reduce-scatter over N per-lane values (one per row): afterwards lane
// `l` holds the warp-wide reduction of rows [base, base + final_n) in v[0..).
// Halving steps exchange half of the values with the partner lane; once N is
// odd the remaining lane bits are reduced in full.
template <int N, int OFF>
struct ReduceScatter {
  static constexpr int kFinal = (OFF == 0) ? N
                                : (N % 2 == 0) ? ReduceScatter<N / 2, OFF / 2>::kFinal
                                               : ReduceScatter<N, OFF / 2>::kFinal;
  template <bool MAX>
  static __device__ __forceinline__ void run(float* v, int lane, int& base, bool& writer) {
    if constexpr (OFF == 0) {
      return;
    } else if constexpr (N % 2 == 0) {
      constexpr int H = N / 2;
      const bool up = (lane & OFF) != 0;
#pragma unroll
      for (int k = 0; k < H; ++k) {
        const float send = up ? v[k] : v[k + H];
        const float keep = up ? v[k + H] : v[k];
        const float recv = __shfl_xor_sync(0xffffffffu, send, OFF);
        v[k] = MAX ? fmaxf(keep, recv) : keep + recv;
      }
      if (up) base += H;
      ReduceScatter<H, OFF / 2>::template run<MAX>(v, lane, base, writer);
    } else {
#pragma unroll
      for (int k = 0; k < N; ++k) {
        const float recv = __shfl_xor_sync(0xffffffffu, v[k], OFF);
        v[k] = MAX ? fmaxf(v[k], recv) : v[k] + recv;
      }
      if (lane & OFF) writer = false;
      ReduceScatter<N, OFF / 2>::template run<MAX>(v, lane, base, writer);
    }
  }
};
template <int N>
struct ReduceScatter<N, 0> {
  static constexpr int kFinal = N;
  template <bool MAX>
  static __device__ __forceinline__ void run(float*, int, int&, bool&) {}
};

template <int NR, bool MAX>
__device__ __forceinline__ void warp_reduce_rows(float* v, int lane, float* dst) {
  int base = 0;
  bool writer = true;
  ReduceScatter<NR, 16>::template run<MAX>(v, lane, base, writer);
  constexpr int F = ReduceScatter<NR, 16>::kFinal;
  if (writer) {
#pragma unroll
    for (int k = 0; k < F; ++k) dst[base + k] = v[k];
  }
}

// ---------------------------------------------------------------------------
// Merge (the kernels are defined in mla_merge.cu): one CTA per (128-dim quarter, row); G groups of 32 lanes, each lane
// owning 4 consecutive dims.  Group g folds partials g, g+G, g+2G, ... with an
// online softmax (4 loads in flight per step; slots past the end re-read the
// step's first slot with weight 0), then group 0 combines the G group states
// through shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float exp2_exact_int(float x) {
  // 2^x; exact when x is an integer (the split kernel's reference maxima).
  if (x == -INFINITY) return 0.0f;
  const float a = rintf(x);
  const int ia = static_cast<int>(a);
  if (ia < -126) return 0.0f;
  return ex2_approx(x - a) * pow2i(ia > 127 ? 127 : ia);
}

struct MergeParams {
  const float* po;
  const float* pml;
  int32_t rows;
  int32_t stride_s;      // slots per row in memory
  int32_t uniform_s;     // slots per row when splits == nullptr
  const int32_t* splits; // per-request slot counts (decode path) or nullptr
  int32_t rows_per_req;
  int32_t num_heads;       // row r belongs to head r % num_heads (for sinks)
  float output_scale;
  const float* sinks;      // optional per-head sink logits (natural-log units)
  __nv_bfloat16* out;
  float* lse;
  float* out_f32;
};

// Raise a kernel's dynamic shared-memory limit to `bytes` once per device
// (the attribute is per device; `done` holds one bit per device id < 64).
template <typename Kernel>
inline cudaError_t ensure_smem_attr(Kernel fn, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t{1} << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Launches the merge as a programmatic dependent of the preceding grid.
cudaError_t launch_merge(const MergeParams& mp, int kv_split, cudaStream_t stream);
// cuTensorMapEncodeTiled through the runtime's driver entry point.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();
bool aligned(const void* p, uintptr_t a);
int cuda_fail(const char* what, cudaError_t e);
// Test hook: limit of the pipeline waits for later launches (0 = default).
extern std::atomic<long long> g_wait_cycles;
// Test hook: the pipeline wait (role << 24) | tile that later launches treat
// as expired (-1 = none).
extern std::atomic<int> g_debug_expire;

}  // namespace mla
