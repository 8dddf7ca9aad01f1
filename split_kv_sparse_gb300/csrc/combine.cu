// Log-sum-exp combine of split-KV partials ("The Split-K Dispatch", "The LSE
// Combine Strategy"; FlashMLA PR #25, "What changes": the combine owns the
// attention sink and the final cast; cuDNN-frontend PR #768: it also owns the
// amax of the recombined output).
//
// One warp per (output row, 128-wide column slice) at a time, so even one decode
// token (64 rows x 4 slices of the 512-wide O) spreads over 32 CTAs: the lanes read
// the row's split LSEs, take M = max_s LSE_s and w_s = 2^(LSE_s - M), then
// stream their slice of the fp32 partials as float4 loads, 8 or 16 splits in
// flight at a time (the first batch requested together with the LSEs), skipping
// every split with w_s = 0 (empty).
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"

namespace skv {
namespace {

constexpr int kWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// kBatch: splits' slices in flight at a time. 8 keeps a thread within 64
// registers, so 32 warps fit an SM and a few thousand rows run in one wave; 16
// (more registers) serves combines over more than 8 splits.
// A lane's four consecutive values of split s's slice: one 16-byte load of
// fp32 partials, or one 8-byte load of bf16 partials widened exactly.
template <bool kBf16>
__device__ __forceinline__ float4 load_slice(const float* o_acc, size_t off, int lane) {
  if constexpr (kBf16) {
    const uint2 w = __ldcs(reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(o_acc) + off) + lane);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
  } else {
    return __ldcs(reinterpret_cast<const float4*>(o_acc + off) + lane);
  }
}

template <int D, int kBatch, bool kBf16>
__global__ void __launch_bounds__(kWarps * 32, kBatch == 8 ? 4 : 1) combine_kernel(const CombineArgs a) {
  constexpr int kSlices = D / 128;   // 128 floats = one float4 per lane
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int items = a.rows * kSlices;
  const size_t rows = static_cast<size_t>(a.rows);
  grid_dependency_wait();      // the split pass has finished writing the partials
  float amax_l = 0.f;
  // A grid of a few CTAs per SM walks all (row, slice) items: a combine over
  // many tokens (or one that leaves most of them alone, as the balanced schedule
  // does) runs in one wave instead of many waves of short-lived CTAs.
#pragma unroll 1
  for (int item = blockIdx.x * kWarps + warp; item < items; item += gridDim.x * kWarps) {
    const int row = item / kSlices;
    const int slice = item - row * kSlices;
    int S = a.num_splits;
    if (a.bal_ctas > 0) {
      const int t = row / a.heads;
      const int pa = bal_cta_of(t * a.bal_nb, a.bal_units, a.bal_ctas);
      S = bal_cta_of((t + 1) * a.bal_nb - 1, a.bal_units, a.bal_ctas) - pa + 1;
      if (S == 1) continue;      // a whole token: the decode kernel wrote its final rows
    }
    auto load = [&](int s) {
      return load_slice<kBf16>(a.o_acc, (static_cast<size_t>(s) * rows + row) * D + slice * 128, lane);
    };
    // The first kBatch splits' slices are requested together with the LSEs, before
    // the weights are known (one memory round trip for S <= kBatch); a split whose
    // weight turns out 0 (empty) is then skipped, whatever its slice holds.
    // (With sparse splits — a plan whose slots are mostly empty for most rows —
    // the slices are requested only once the weights are known.)
    float4 x[kBatch];
    if (!a.sparse_splits) {
#pragma unroll
      for (int u = 0; u < kBatch; ++u) x[u] = u < S ? load(u) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float l0 = lane < S ? a.lse_acc[static_cast<size_t>(lane) * rows + row] : -INFINITY;
    const float l1 = lane + 32 < S ? a.lse_acc[static_cast<size_t>(lane + 32) * rows + row] : -INFINITY;
    const float M = warp_max(fmaxf(l0, l1));
    const bool empty = (M == -INFINITY);
    const float w0 = (l0 == -INFINITY) ? 0.f : exp2f(l0 - M);
    const float w1 = (l1 == -INFINITY) ? 0.f : exp2f(l1 - M);
    const float wsum = warp_sum(w0 + w1);
    auto weight = [&](int s) { return __shfl_sync(0xffffffffu, s < 32 ? w0 : w1, s & 31); };
    if (a.sparse_splits) {
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        x[u] = (u < S && weight(u) != 0.f) ? load(u) : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // acc = sum over s, in split order, of w_s * O_s
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto fold = [&](float w, const float4& v) {
      if (w != 0.f) {
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
    };
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (u < S) fold(weight(u), x[u]);
#pragma unroll 1
    for (int s0 = kBatch; s0 < S; s0 += kBatch) {
      float ws[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        ws[u] = s0 + u < S ? weight(s0 + u) : 0.f;
        x[u] = ws[u] != 0.f ? load(s0 + u) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) fold(ws[u], x[u]);
    }
    float inv = 0.f;
    if (!empty) {
      float den = wsum;
      if (a.sink != nullptr) den += exp2f(a.sink[row % a.heads] * kLog2e - M);
      inv = 1.f / den;
    }
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    amax_l = fmaxf(amax_l, fmaxf(fmaxf(fabsf(acc.x), fabsf(acc.y)), fmaxf(fabsf(acc.z), fabsf(acc.w))));
    const size_t base = static_cast<size_t>(row) * D + slice * 128;
    const int e = 4 * lane;
    if (a.out_dtype == 0) {
      reinterpret_cast<float4*>(static_cast<float*>(a.out) + base)[lane] = acc;
    } else if (a.out_dtype == 1) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + base + e) = pk;
    } else {
      const float2 lo = make_float2(acc.x * a.inv_scale, acc.y * a.inv_scale);
      const float2 hi = make_float2(acc.z * a.inv_scale, acc.w * a.inv_scale);
      const uint32_t c01 = __nv_cvt_float2_to_fp8x2(lo, __NV_SATFINITE, __NV_E4M3);
      const uint32_t c23 = __nv_cvt_float2_to_fp8x2(hi, __NV_SATFINITE, __NV_E4M3);
      *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(a.out) + base + e) = (c01 & 0xFFFFu) | (c23 << 16);
    }
    if (slice == 0 && lane == 0 && a.lse_out != nullptr) a.lse_out[row] = empty ? -INFINITY : M + log2f(wsum);
  }
  if (a.amax != nullptr) {
    amax_l = warp_max(amax_l);
    if (lane == 0 && amax_l > 0.f) atomicMax(reinterpret_cast<int*>(a.amax), __float_as_int(amax_l));
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, bool zero_amax, bool pdl, cudaStream_t stream) {
  if (zero_amax && a.amax != nullptr) {
    const cudaError_t e = cudaMemsetAsync(a.amax, 0, sizeof(float), stream);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  const int items = a.rows * (a.d / 128);
  const bool wide = a.num_splits > 8;
  // at most the CTAs that are resident at once (4 per SM for the narrow form's
  // register budget, 2 for the wide one); each warp then walks several items
  const int cap = a.num_sms > 0 ? a.num_sms * (wide ? 2 : 4) : 0x7fffffff;
  cfg.gridDim = dim3(static_cast<unsigned>(std::min((items + kWarps - 1) / kWarps, cap)));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (a.d == 512 && a.partial_bf16)
    return cudaLaunchKernelEx(&cfg, wide ? combine_kernel<512, 16, true> : combine_kernel<512, 8, true>, a);
  if (a.d == 512) return cudaLaunchKernelEx(&cfg, wide ? combine_kernel<512, 16, false> : combine_kernel<512, 8, false>, a);
  if (a.d == 128 && !a.partial_bf16)
    return cudaLaunchKernelEx(&cfg, wide ? combine_kernel<128, 16, false> : combine_kernel<128, 8, false>, a);
  return cudaErrorInvalidValue;
}

}  // namespace skv
