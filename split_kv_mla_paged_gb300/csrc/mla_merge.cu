// Online-softmax merge of split-KV partials for the paged MLA decode (GB300,
// sm_103a): per query row, the partials (m in log2 units, l, unnormalised
// O[512]) of its splits are combined into BF16 O and the natural-log LSE.
// The method follows TensorRT-LLM PR #20380 ("Description"): KvSplit thread
// groups over a row's partials, a shared-memory combine rescaled by
// exp2(group max - max), empty groups skipped, weight-0 padded loads.  The
// split kernels (mla_decode.cu, mla_decode_bf16.cu) write the partials and
// launch this kernel as their programmatic dependent.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "mla_device.cuh"

namespace mla {

// The merge of one (row, quarter of the latent dims): G thread groups over
// the row's partials, U loads in flight per group.  kMaxFirst: each group
// first takes the maximum m over its slots and then accumulates
// exp2(m_s - max) O_s with no running rescale, so its loads carry no
// dependence on the previous slot (the same numbers as the running form:
// every rescale there is an exact power of two for the split kernel's
// integer maxima); it pays one more round trip per group and serves rows
// whose groups hold many slots.
template <int G, int U, bool kMaxFirst>
__device__ __forceinline__ void merge_body(const MergeParams& p) {
  __shared__ float sm_m[G];
  __shared__ float sm_l[G];
  __shared__ float4 sm_o[G][32];
  // Partials are written by the preceding (programmatically dependent) grid.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int row = blockIdx.x;
  const int quarter = blockIdx.y;
  const int g = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int ns = p.uniform_s;
  if (p.splits) {
    ns = min(p.splits[row / p.rows_per_req], p.stride_s);
    if (ns <= 1) return;  // the split kernel wrote this row directly
  }
  const int dim = quarter * 128 + lane * 4;
  const float* pml = p.pml + static_cast<int64_t>(row) * p.stride_s * 2;
  const float* po = p.po + static_cast<int64_t>(row) * p.stride_s * MLA_LATENT_DIM + dim;
  float m = -INFINITY, l = 0.0f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  if constexpr (kMaxFirst) {
    // Lane k reads the (m, l) of slots g + G k, g + G (k + 32), ...
    for (int s = g + G * lane; s < ns; s += G * 32) {
      const float2 ml = *reinterpret_cast<const float2*>(pml + s * 2);
      if (ml.y > 0.0f) m = fmaxf(m, ml.x);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  }
  for (int s0 = g; (!kMaxFirst || m != -INFINITY) && s0 < ns; s0 += G * U) {
    float mu[U], lu[U];
    float4 ou[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int s = s0 + u * G;
      const bool in = s < ns;
      const int slot = in ? s : s0;  // weight-0 padded load of a valid slot
      const float2 ml = *reinterpret_cast<const float2*>(pml + slot * 2);
      ou[u] = *reinterpret_cast<const float4*>(po + static_cast<int64_t>(slot) * MLA_LATENT_DIM);
      mu[u] = (in && ml.y > 0.0f) ? ml.x : -INFINITY;
      lu[u] = ml.y;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (mu[u] == -INFINITY) continue;  // empty slot or padding: weight 0 (O unread)
      if constexpr (kMaxFirst) {
        const float w = exp2_exact_int(mu[u] - m);
        l += lu[u] * w;
        o.x += ou[u].x * w;
        o.y += ou[u].y * w;
        o.z += ou[u].z * w;
        o.w += ou[u].w * w;
      } else {
        const float m_new = fmaxf(m, mu[u]);
        const float a = exp2_exact_int(m - m_new);
        const float w = exp2_exact_int(mu[u] - m_new);
        l = l * a + lu[u] * w;
        o.x = o.x * a + ou[u].x * w;
        o.y = o.y * a + ou[u].y * w;
        o.z = o.z * a + ou[u].z * w;
        o.w = o.w * a + ou[u].w * w;
        m = m_new;
      }
    }
  }
  if (G > 1) {
    if (lane == 0) {
      sm_m[g] = m;
      sm_l[g] = l;
    }
    sm_o[g][lane] = o;
    __syncthreads();
    if (g != 0) return;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < G; ++k)
      if (sm_l[k] > 0.0f) M = fmaxf(M, sm_m[k]);
    l = 0.0f;
    o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int k = 0; k < G; ++k) {
        if (!(sm_l[k] > 0.0f)) continue;  // empty group
        const float w = exp2_exact_int(sm_m[k] - M);
        const float4 v = sm_o[k][lane];
        l += sm_l[k] * w;
        o.x += v.x * w;
        o.y += v.y * w;
        o.z += v.z * w;
        o.w += v.w * w;
      }
    }
    m = M;
  }
  if (!(l > 0.0f)) m = -INFINITY;
  // A sink is one more (zero-valued) key: it joins the denominator.
  const float sink2 = p.sinks ? p.sinks[row % p.num_heads] * 1.4426950408889634f : -INFINITY;
  const float mm = fmaxf(m, sink2);
  const float a = (m == -INFINITY) ? 0.0f : exp2_exact_int(m - mm);
  const float den = l * a + (sink2 == -INFINITY ? 0.0f : exp2f(sink2 - mm));
  const bool empty = !(den > 0.0f);
  const float inv = empty ? 0.0f : p.output_scale * a / den;
  const float4 r = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
  const int64_t off = static_cast<int64_t>(row) * MLA_LATENT_DIM + dim;
  __nv_bfloat162 lo = __floats2bfloat162_rn(r.x, r.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(r.z, r.w);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&lo);
  packed.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p.out + off) = packed;
  if (p.out_f32) *reinterpret_cast<float4*>(p.out_f32 + off) = r;
  if (p.lse && quarter == 0 && lane == 0)
    p.lse[row] = empty ? -INFINITY : 0.6931471805599453f * (mm + log2f(den));
}

template <int G, bool kMaxFirst>
__global__ void __launch_bounds__(32 * G) mla_merge_kernel(const MergeParams p) {
  merge_body<G, 4, kMaxFirst>(p);
}

// Grids of more than two 512-thread CTAs per SM: three per SM (at most 40
// registers, two loads in flight per group instead of four), so that the
// grid fits one wave.
__global__ void __launch_bounds__(512, 3) mla_merge_many_kernel(const MergeParams p) {
  merge_body<16, 2, false>(p);
}

// The merge is launched as a programmatic dependent of whatever precedes it
// on the stream (the split-KV kernel in mla_decode): its CTAs may be scheduled
// while the split kernel drains and wait in griddepcontrol.wait until the
// partials are visible.  Launched after anything else, the wait returns at once.
// kMany (16 groups only): the one-wave kernel for many-row grids.
template <int G, bool kMany = false>
static cudaError_t launch_merge_g(const MergeParams& mp, cudaStream_t stream) {
  // The max-first form where groups hold at least 8 slots and the grid has at
  // least 96 rows: on the GB300 merge-only sweep and the decode workloads it
  // is faster there (MTP B2 128K 6.9 -> 5.9 us, sparse q8 8.8 -> 7.8 us) and
  // slower for short groups or few rows (12 rows x 147 splits 5.0 -> 5.3 us).
  const bool max_first = mp.rows >= 96 && mp.stride_s >= 8 * G;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(mp.rows, 4);  // rows on x: no 65535 limit
  cfg.blockDim = dim3(32 * G);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static_assert(!kMany || G == 16, "the many-row merge has 16 groups");
  if constexpr (kMany) {
    return cudaLaunchKernelEx(&cfg, mla_merge_many_kernel, mp);
  } else {
    return max_first ? cudaLaunchKernelEx(&cfg, mla_merge_kernel<G, true>, mp)
                     : cudaLaunchKernelEx(&cfg, mla_merge_kernel<G, false>, mp);
  }
}

cudaError_t launch_merge(const MergeParams& mp, int kv_split, cudaStream_t stream) {
  cudaError_t e;
  switch (kv_split) {
    case 1: e = launch_merge_g<1>(mp, stream); break;
    case 2: e = launch_merge_g<2>(mp, stream); break;
    case 4: e = launch_merge_g<4>(mp, stream); break;
    case 8: e = launch_merge_g<8>(mp, stream); break;
    case 16: {
      int dev = 0, sms = 0;
      e = cudaGetDevice(&dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      e = (static_cast<int64_t>(mp.rows) * 4 > 2 * static_cast<int64_t>(sms))
              ? launch_merge_g<16, true>(mp, stream)
              : launch_merge_g<16, false>(mp, stream);
      break;
    }
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
