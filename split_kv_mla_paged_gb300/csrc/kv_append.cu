// FP8 paged KV append: quantize new 576-value latent rows (BF16) to E4M3 with
// kv_scale and scatter them into the paged cache.  This is the step that fills
// the cache the decode reads (TensorRT-LLM PR #17273, "Fuse the DSv4 MLA
// prologue": one warp owns a latent row, quantizes it to FP8 and scatters it
// through the page table); the model-specific RMSNorm and RoPE of that kernel
// are not part of this library.
//
// One warp per row: the row's 1152 input bytes are read as 72 16-byte vectors
// (lanes stride by 32), each converted to 8 E4M3 codes and stored as 8 bytes,
// so loads and stores are coalesced within the row.  code = e4m3(x / kv_scale)
// with the correctly rounded fp32 quotient (formed without a division
// instruction for the usual scales, see DivMode) and round-to-nearest-even,
// saturating at 448.
#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>
#include <cstdint>
#include <string>

#include "mla_internal.h"

namespace mla {

constexpr int kAppendWarps = 8;

__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// How x / kv_scale is formed.  Every mode gives the correctly rounded fp32
// quotient (the one an IEEE division gives) for every BF16 input x.
enum DivMode : int {
  kDivIeee = 0,        // the IEEE division
  kDivPow2 = 1,        // kv_scale = +-2^k with a normal reciprocal: x * (1/kv_scale) is exact
  kDivReciprocal = 2,  // 2^-32 <= kv_scale <= 2^32: reciprocal and one correction
};

// Quotient from the correctly rounded reciprocal y = RN(1/b) with one
// correction step (Markstein's theorem; Muller et al., "Handbook of
// Floating-Point Arithmetic", section on Newton-Raphson division with an FMA):
// q = RN(x*y); the residual e = q*b - x is exact in one FMA; q' = RN(q - e*y)
// is the correctly rounded x/b.  The clamp on e only acts when q is +-inf
// (x = +-inf, or a quotient past fp32's range): e is then inf or NaN (inf -
// inf), the clamp makes it finite and q' stays +-inf, which encodes like the
// IEEE quotient (saturated).  Forming the residual as q*b - x (not x - q*b)
// keeps the sign of a zero quotient (-0/b = -0).  A quotient at or below
// 2^-10 encodes to a signed zero whatever its low bits, and the range limits
// on b keep the residual of every larger quotient away from fp32's
// subnormals.  Checked exhaustively against the IEEE division: fp32 bits over
// all 2^23 significands of b times all 128 BF16 significands of x, and E4M3
// codes over all 65,536 BF16 patterns for scales across the range.
__device__ __forceinline__ float div_by_reciprocal(float x, float b, float y) {
  const float q = x * y;
  float e = __fmaf_rn(q, b, -x);
  e = fminf(fmaxf(e, -FLT_MAX), FLT_MAX);
  return __fmaf_rn(-e, y, q);
}

template <int kMode>
__device__ __forceinline__ uint2 quantize8(uint4 v, float kv_scale, float inv_scale) {
  float x[8];
  x[0] = bf16_bits_to_float(v.x & 0xFFFFu);
  x[1] = bf16_bits_to_float(v.x >> 16);
  x[2] = bf16_bits_to_float(v.y & 0xFFFFu);
  x[3] = bf16_bits_to_float(v.y >> 16);
  x[4] = bf16_bits_to_float(v.z & 0xFFFFu);
  x[5] = bf16_bits_to_float(v.z >> 16);
  x[6] = bf16_bits_to_float(v.w & 0xFFFFu);
  x[7] = bf16_bits_to_float(v.w >> 16);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if constexpr (kMode == kDivPow2) {
      x[k] *= inv_scale;
    } else if constexpr (kMode == kDivReciprocal) {
      x[k] = div_by_reciprocal(x[k], kv_scale, inv_scale);
    } else {
      x[k] = __fdiv_rn(x[k], kv_scale);
    }
  }
  uint2 o;
  o.x = pack4_e4m3(x[0], x[1], x[2], x[3]);
  o.y = pack4_e4m3(x[4], x[5], x[6], x[7]);
  return o;
}

// One warp per row.  The row's three 16-byte vectors per lane are loaded
// together with its request and position, before the page-table lookup
// that depends on them: one DRAM round trip for the data, overlapped with
// the index chain, instead of one per vector.
template <int kMode>
__global__ void __launch_bounds__(32 * kAppendWarps)
    mla_kv_append_kernel(const uint16_t* __restrict__ rows, int64_t n,
                         const int32_t* __restrict__ req, const int32_t* __restrict__ pos,
                         const int32_t* __restrict__ page_table, int32_t max_pages,
                         int32_t batch, uint8_t* __restrict__ kv, int64_t num_pages,
                         float kv_scale, float inv_scale, int* status) {
  constexpr int kChunks = MLA_HEAD_DIM / 8;  // 72 vectors of 8 values: 32 + 32 + 8
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5);
  if (row >= n) return;
  const uint4* src = reinterpret_cast<const uint4*>(rows + row * MLA_HEAD_DIM);
  uint4 v0 = __ldg(src + lane);
  uint4 v1 = __ldg(src + lane + 32);
  uint4 v2 = make_uint4(0u, 0u, 0u, 0u);
  if (lane < kChunks - 64) v2 = __ldg(src + lane + 64);
  const int32_t b = __ldg(req + row);
  const int32_t j = __ldg(pos + row);
  if (b < 0 || b >= batch || j < 0 || j / MLA_PAGE_SIZE >= max_pages) {
    if (status && lane == 0) atomicCAS(status, 0, MLA_ERR_INVALID_ARG);
    return;
  }
  const int64_t page = __ldg(page_table + static_cast<int64_t>(b) * max_pages + j / MLA_PAGE_SIZE);
  if (page < 0 || page >= num_pages) {
    if (status && lane == 0) atomicCAS(status, 0, MLA_ERR_INVALID_ARG);
    return;
  }
  uint2* dst = reinterpret_cast<uint2*>(
      kv + (page * MLA_PAGE_SIZE + j % MLA_PAGE_SIZE) * MLA_HEAD_DIM);
  dst[lane] = quantize8<kMode>(v0, kv_scale, inv_scale);
  dst[lane + 32] = quantize8<kMode>(v1, kv_scale, inv_scale);
  if (lane < kChunks - 64) dst[lane + 64] = quantize8<kMode>(v2, kv_scale, inv_scale);
}

}  // namespace mla

using namespace mla;

extern "C" int mla_kv_append(const void* rows_bf16, int64_t n_tokens, const int32_t* req_idx,
                             const int32_t* positions, const int32_t* page_table,
                             int32_t max_pages_per_req, int32_t batch, void* kv_pages_fp8,
                             int64_t num_pages, float kv_scale, int32_t* status, void* stream) {
  if (n_tokens < 0 || batch < 1 || max_pages_per_req < 1 || num_pages < 1) {
    set_error("mla_kv_append: n_tokens >= 0, batch, max_pages_per_req and num_pages >= 1");
    return MLA_ERR_INVALID_ARG;
  }
  if (n_tokens == 0) return MLA_OK;
  if (!rows_bf16 || !req_idx || !positions || !page_table || !kv_pages_fp8) {
    set_error("mla_kv_append: null pointer argument");
    return MLA_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(rows_bf16) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(kv_pages_fp8) & 7u) != 0) {
    set_error("mla_kv_append: rows need 16-byte and the page pool 8-byte alignment");
    return MLA_ERR_INVALID_ARG;
  }
  if (!std::isfinite(kv_scale) || kv_scale == 0.0f) {
    set_error("mla_kv_append: kv_scale must be finite and nonzero");
    return MLA_ERR_INVALID_ARG;
  }
  const int64_t blocks = (n_tokens + kAppendWarps - 1) / kAppendWarps;
  if (blocks > 0x7FFFFFFF) {
    set_error("mla_kv_append: too many tokens for one launch");
    return MLA_ERR_UNSUPPORTED;
  }
  // The division mode for this scale (all give the IEEE quotient).
  int ex = 0;
  const float inv = 1.0f / kv_scale;  // correctly rounded
  const float mag = std::fabs(kv_scale);
  const bool normal = std::isnormal(kv_scale) && std::isnormal(inv);
  int mode = kDivIeee;
  if (normal && std::fabs(std::frexp(kv_scale, &ex)) == 0.5f)
    mode = kDivPow2;
  else if (kv_scale > 0.0f && mag >= 0x1p-32f && mag <= 0x1p32f)
    mode = kDivReciprocal;
  const auto kernel = mode == kDivPow2        ? mla_kv_append_kernel<kDivPow2>
                      : mode == kDivReciprocal ? mla_kv_append_kernel<kDivReciprocal>
                                               : mla_kv_append_kernel<kDivIeee>;
  kernel<<<static_cast<unsigned>(blocks), 32 * kAppendWarps, 0,
           reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint16_t*>(rows_bf16), n_tokens, req_idx, positions, page_table,
      max_pages_per_req, batch, reinterpret_cast<uint8_t*>(kv_pages_fp8), num_pages, kv_scale,
      inv, reinterpret_cast<int*>(status));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error(std::string("mla_kv_append: launch: ") + cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}
