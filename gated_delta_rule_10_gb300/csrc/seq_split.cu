// Start states of the runs of a split sequence (fp32).
//
// Each run p of a (batch, head) maps its start state to its end state by
// S_end = M_p S_start + H_p: the delta-rule update is affine in the state, and
// affine maps of consecutive runs compose in order (LLMs from scratch ch. 11,
// section 11.4, on why the recurrence can be split into blocks). The scan
// kernel gives M_p (its identity slices) and H_p (the run from a zero state);
// this kernel walks the runs in order,
//   S_start[0] = h0 (or zero),  S_start[p] = M_{p-1} S_start[p-1] + H_{p-1},
// one CTA per (batch, head, 8 value columns) so that even B * H = 1 spreads
// over d_v / 8 SMs, 256 threads, each owning 4 rows of one column of the
// d_k x 8 product. M_{p-1} is staged in shared memory with 16-byte loads, its
// rows padded by four floats so that the row groups a warp reads fall in
// different banks.
#include "kernels.h"

namespace gdr {
namespace {

constexpr int kCombCols = 8;
constexpr int kCombThreads = 256;
constexpr int kCombPad = 4;

template <int DK>
__global__ void __launch_bounds__(kCombThreads)
    segment_combine_kernel(const float* __restrict__ M, const float* __restrict__ Hl,
                           const float* __restrict__ h0, float* __restrict__ S, int P, int dv) {
  constexpr int RPT = DK * kCombCols / kCombThreads;   // rows per thread (4 or 2)
  constexpr int LD = DK + kCombPad;
  extern __shared__ __align__(16) float smc[];
  float* sM = smc;                           // [DK][LD]
  float* sS = sM + DK * LD;                  // [DK][kCombCols]
  const int tid = threadIdx.x;
  const size_t bh = blockIdx.y;
  const int c0 = blockIdx.x * kCombCols;
  const int cc = tid % kCombCols, r0 = (tid / kCombCols) * RPT;   // column, first row

  // S_start[0]
  for (int e = tid; e < DK * kCombCols; e += kCombThreads) {
    const int i = e / kCombCols, c = e % kCombCols;
    const float x = h0 ? h0[(bh * DK + i) * dv + c0 + c] : 0.f;
    sS[e] = x;
    S[((bh * P) * DK + i) * dv + c0 + c] = x;
  }
  for (int p = 1; p < P; ++p) {
    const size_t run = bh * P + (p - 1);
    const float4* src = reinterpret_cast<const float4*>(M + run * DK * DK);
    for (int e = tid; e < DK * DK / 4; e += kCombThreads) {
      const int i = e / (DK / 4), j = (e % (DK / 4)) * 4;
      *reinterpret_cast<float4*>(sM + i * LD + j) = __ldg(src + e);
    }
    float acc[RPT];
#pragma unroll
    for (int a = 0; a < RPT; ++a) acc[a] = Hl[(run * DK + r0 + a) * dv + c0 + cc];
    __syncthreads();
#pragma unroll 4
    for (int j = 0; j < DK; j += 4) {
      float s4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) s4[u] = sS[(j + u) * kCombCols + cc];
#pragma unroll
      for (int a = 0; a < RPT; ++a) {
        const float4 m = *reinterpret_cast<const float4*>(sM + (r0 + a) * LD + j);
        acc[a] = fmaf(m.x, s4[0], fmaf(m.y, s4[1], fmaf(m.z, s4[2], fmaf(m.w, s4[3], acc[a]))));
      }
    }
    __syncthreads();   // every thread has read sS and sM of this step
#pragma unroll
    for (int a = 0; a < RPT; ++a) {
      sS[(r0 + a) * kCombCols + cc] = acc[a];
      S[((bh * P + p) * DK + r0 + a) * dv + c0 + cc] = acc[a];
    }
    __syncthreads();
  }
}

template <int DK>
cudaError_t launch_combine(const float* M, const float* Hl, const float* h0, float* S, int B,
                           int H, int P, int dv, cudaStream_t stream) {
  const size_t bytes = (static_cast<size_t>(DK) * (DK + kCombPad) + DK * kCombCols) * sizeof(float);
  auto kern = segment_combine_kernel<DK>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bytes));
  if (err != cudaSuccess) return err;
  const dim3 grid(dv / kCombCols, static_cast<unsigned>(B) * H);
  kern<<<grid, kCombThreads, bytes, stream>>>(M, Hl, h0, S, P, dv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_segment_combine(const float* M, const float* Hl, const float* h0, float* S,
                                   int B, int H, int P, int dk, int dv, cudaStream_t stream) {
  if (dv % kCombCols != 0) return cudaErrorInvalidValue;
  if (dk == 64) return launch_combine<64>(M, Hl, h0, S, B, H, P, dv, stream);
  if (dk == 128) return launch_combine<128>(M, Hl, h0, S, B, H, P, dv, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdr
