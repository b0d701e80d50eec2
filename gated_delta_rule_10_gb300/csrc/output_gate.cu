// Output epilogue: RMSNorm over the value channels, gain, SiLU output gate.
//
// Gated DeltaNet-2 notes, overall framework (the last stage of its flow chart),
// and LLMs-from-scratch ch. 11, section 11.3 (the module after its time loop):
// each (token, head) row o of d_v channels read out of the state becomes
//   y = o * rsqrt(mean_c(o_c^2) + eps) * weight * z * sigmoid(z),
// with weight the per-channel gain and z the output-gate input.
//
// Streaming and HBM-bound: every row of o and z is read once and y written
// once, 3 d_v elements per row, nothing reused. A row is spread over L lanes
// with one 16-byte vector of o and one of z per lane and step (L = d_v * elem /
// 16, capped at 32; a wider row gives each lane several vectors); the row's sum
// of squares is a butterfly over those L lanes. Rows stay packed in registers
// until used, which keeps the kernel near 40 registers and so about 1,500
// resident threads per SM, enough loads in flight to cover HBM latency; the
// grid is the number of blocks resident on all SMs at once, walking the rows
// with a grid stride.
// Loads and stores carry the streaming cache hint. y may be o itself (or z
// itself): a thread reads all of its row's elements before it writes any.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"

namespace gdr {
namespace {

constexpr int kGateThreads = 256;
constexpr int kRowsInFlight = 1;  // 1, 2 and 4 measured the same; 1 takes fewest registers

template <typename T>
struct RowShape;

template <>
struct RowShape<float> {
  using Vec = float4;
  static constexpr int kElem = 4;
};
template <>
struct RowShape<__nv_bfloat16> {
  using Vec = uint4;
  static constexpr int kElem = 8;
};

template <typename T, int DV>
struct RowSplit {
  static constexpr int kElem = RowShape<T>::kElem;
  static constexpr int kVecs = DV / kElem;                  // 16-byte vectors per row
  static constexpr int kLanes = kVecs < 32 ? kVecs : 32;    // lanes sharing a row
  static constexpr int kPerLane = kVecs / kLanes;           // vectors per lane
  static constexpr int kRowsPerWarp = 32 / kLanes;
  static_assert(DV % kElem == 0 && kVecs % kLanes == 0 && (kLanes & (kLanes - 1)) == 0,
                "row width must split evenly over a power-of-two lane group");
};

__device__ __forceinline__ void unpack(const float4& v, float (&x)[4]) {
  x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void unpack(const uint4& v, float (&x)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ float4 pack(const float (&x)[4]) {
  return make_float4(x[0], x[1], x[2], x[3]);
}
__device__ __forceinline__ uint4 pack(const float (&x)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// z sigmoid(z); the fast divide is exact enough here (2 ulp) and returns 0
// when 1 + exp(-z) overflows, the limit of z sigmoid(z) as z -> -inf
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

template <typename T, int DV>
__global__ void __launch_bounds__(kGateThreads)
    rmsnorm_gate_kernel(const T* o, const T* z, const float* weight, float eps, T* y,
                        long long rows) {
  using S = RowSplit<T, DV>;
  using Vec = typename RowShape<T>::Vec;
  constexpr int E = S::kElem;
  const int lane = threadIdx.x & 31;
  const int sub = lane / S::kLanes;  // which of the warp's rows
  const int col = lane % S::kLanes;  // position within the row's lane group

  // this lane's channels: vector p covers channels (p * kLanes + col) * E ..
  float wv[S::kPerLane][E];
#pragma unroll
  for (int p = 0; p < S::kPerLane; ++p) {
    const float* wp = weight + (p * S::kLanes + col) * E;
#pragma unroll
    for (int e = 0; e < E; e += 4) {
      const float4 g = __ldg(reinterpret_cast<const float4*>(wp + e));
      wv[p][e] = g.x; wv[p][e + 1] = g.y; wv[p][e + 2] = g.z; wv[p][e + 3] = g.w;
    }
  }

  const long long warps = static_cast<long long>(gridDim.x) * (kGateThreads / 32);
  const long long step = warps * S::kRowsPerWarp;  // rows covered by one sweep of the grid
  const long long first =
      (static_cast<long long>(blockIdx.x) * (kGateThreads / 32) + threadIdx.x / 32) *
      S::kRowsPerWarp;
  const float inv_dv = 1.0f / DV;
  // `base` is warp-uniform, so every lane reaches the shuffles below
  for (long long base = first; base < rows; base += step * kRowsInFlight) {
    // the rows stay packed in registers until they are used
    Vec ra[kRowsInFlight][S::kPerLane];
    Vec rb[kRowsInFlight][S::kPerLane];
#pragma unroll
    for (int i = 0; i < kRowsInFlight; ++i) {
      const long long row = base + sub + i * step;
      const bool live = row < rows;
      const size_t off = static_cast<size_t>(live ? row : 0) * DV;
#pragma unroll
      for (int p = 0; p < S::kPerLane; ++p) {
        const size_t at = off + static_cast<size_t>(p * S::kLanes + col) * E;
        ra[i][p] = Vec{};
        rb[i][p] = Vec{};
        if (live) {
          ra[i][p] = __ldcs(reinterpret_cast<const Vec*>(o + at));
          rb[i][p] = __ldcs(reinterpret_cast<const Vec*>(z + at));
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kRowsInFlight; ++i) {
      float ss = 0.f;
#pragma unroll
      for (int p = 0; p < S::kPerLane; ++p) {
        float a[E];
        unpack(ra[i][p], a);
#pragma unroll
        for (int e = 0; e < E; ++e) ss = fmaf(a[e], a[e], ss);
      }
#pragma unroll
      for (int m = S::kLanes / 2; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
      const float r = rsqrtf(fmaf(ss, inv_dv, eps));
      const long long row = base + sub + i * step;
      if (row < rows) {
        const size_t off = static_cast<size_t>(row) * DV;
#pragma unroll
        for (int p = 0; p < S::kPerLane; ++p) {
          float a[E], b[E];
          unpack(ra[i][p], a);
          unpack(rb[i][p], b);
#pragma unroll
          for (int e = 0; e < E; ++e) a[e] = a[e] * r * wv[p][e] * silu(b[e]);
          __stcs(reinterpret_cast<Vec*>(y + off + static_cast<size_t>(p * S::kLanes + col) * E),
                 pack(a));
        }
      }
    }
  }
}

template <typename T, int DV>
cudaError_t launch_typed(const void* o, const void* z, const float* weight, float eps, void* y,
                         long long rows, cudaStream_t stream) {
  using S = RowSplit<T, DV>;
  int dev = 0, sms = 0;
  cudaError_t err;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return err;
  // resident blocks per SM of this instantiation (the same on every GB300)
  static const int per_sm = [] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, rmsnorm_gate_kernel<T, DV>,
                                                      kGateThreads, 0) != cudaSuccess || n < 1)
      n = 1;
    return n;
  }();
  const long long rows_per_block = (kGateThreads / 32) * S::kRowsPerWarp * kRowsInFlight;
  const long long need = (rows + rows_per_block - 1) / rows_per_block;
  const long long cap = static_cast<long long>(sms) * per_sm;
  const unsigned grid = static_cast<unsigned>(need < cap ? need : cap);
  rmsnorm_gate_kernel<T, DV><<<grid, kGateThreads, 0, stream>>>(
      static_cast<const T*>(o), static_cast<const T*>(z), weight, eps, static_cast<T*>(y), rows);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dv(int dv, const void* o, const void* z, const float* weight, float eps,
                      void* y, long long rows, cudaStream_t stream) {
  switch (dv) {
    case 64: return launch_typed<T, 64>(o, z, weight, eps, y, rows, stream);
    case 128: return launch_typed<T, 128>(o, z, weight, eps, y, rows, stream);
    case 256: return launch_typed<T, 256>(o, z, weight, eps, y, rows, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_rmsnorm_gate(const void* o, const void* z, const float* weight, float eps,
                                void* y, long long rows, int dv, bool f32,
                                cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  return f32 ? launch_dv<float>(dv, o, z, weight, eps, y, rows, stream)
             : launch_dv<__nv_bfloat16>(dv, o, z, weight, eps, y, rows, stream);
}

}  // namespace gdr
