// Per-lane input loads of the token-order backwards (token_bwd.cu,
// value_beta_bwd.cu): runs of consecutive key-row elements and pairs of value
// columns, converted to fp32. Every address is aligned to the load's width: the
// tensors are 16-byte aligned, a run starts at a multiple of its length (4, 8 or
// 16 elements) and a pair at an even column.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

namespace gdr {
namespace {

// N consecutive elements from p as floats, by 16- or 8-byte loads
template <int N>
__device__ __forceinline__ void load_run(const float* p, float (&x)[N]) {
  static_assert(N % 4 == 0, "float4 loads");
#pragma unroll
  for (int i = 0; i < N; i += 4) {
    const float4 f = *reinterpret_cast<const float4*>(p + i);
    x[i] = f.x; x[i + 1] = f.y; x[i + 2] = f.z; x[i + 3] = f.w;
  }
}
template <int N>
__device__ __forceinline__ void load_run(const __nv_bfloat16* p, float (&x)[N]) {
  static_assert(N % 4 == 0, "8-byte loads at least");
  if constexpr (N % 8 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 8) {
      const uint4 u = *reinterpret_cast<const uint4*>(p + i);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {   // bf16 -> fp32 is the high half of the word
        x[i + 2 * j] = __uint_as_float(w[j] << 16);
        x[i + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; i += 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(p + i);
      x[i] = __uint_as_float(u.x << 16);
      x[i + 1] = __uint_as_float(u.x & 0xffff0000u);
      x[i + 2] = __uint_as_float(u.y << 16);
      x[i + 3] = __uint_as_float(u.y & 0xffff0000u);
    }
  }
}

// two consecutive elements (an aligned pair)
__device__ __forceinline__ float2 load_pair(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}
__device__ __forceinline__ float2 load_pair(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}

}  // namespace
}  // namespace gdr
