// Start states of the runs of a split sequence (fp32).
//
// Each run p of a (batch, head) maps its start state to its end state by
// S_end = M_p S_start + H_p: the delta-rule update is affine in the state, and
// affine maps of consecutive runs compose in order (LLMs from scratch ch. 11,
// section 11.4, on why the recurrence can be split into blocks). The scan
// kernel gives M_p (its identity slices) and H_p (the run from a zero state);
// this kernel walks the runs in order,
//   S_start[0] = h0 (or zero),  S_start[p] = M_{p-1} S_start[p-1] + H_{p-1},
// one CTA per (batch, head, 32 value columns), 2 d_k threads, each owning a
// 4 x 4 block of the d_k x 32 product. M_{p-1} is staged in shared memory with
// its rows padded by one float, so the four row groups a warp reads fall in
// different banks.
#include "kernels.h"

namespace gdr {
namespace {

constexpr int kCombCols = 32;

template <int DK>
__global__ void __launch_bounds__(2 * DK)
    segment_combine_kernel(const float* __restrict__ M, const float* __restrict__ Hl,
                           const float* __restrict__ h0, float* __restrict__ S, int P, int dv) {
  extern __shared__ float smc[];
  float* sM = smc;                           // [DK][DK + 1]
  float* sS = sM + DK * (DK + 1);            // [DK][kCombCols]
  const int tid = threadIdx.x;
  const size_t bh = blockIdx.y;
  const int c0 = blockIdx.x * kCombCols;
  const int r0 = (tid / 8) * 4, cc = (tid % 8) * 4;   // this thread's 4 x 4 block

  // S_start[0]
  for (int e = tid; e < DK * kCombCols; e += 2 * DK) {
    const int i = e / kCombCols, c = e % kCombCols;
    const float x = h0 ? h0[(bh * DK + i) * dv + c0 + c] : 0.f;
    sS[e] = x;
    S[((bh * P) * DK + i) * dv + c0 + c] = x;
  }
  for (int p = 1; p < P; ++p) {
    const size_t run = bh * P + (p - 1);
    for (int e = tid; e < DK * DK; e += 2 * DK) {
      const int i = e / DK, j = e % DK;
      sM[i * (DK + 1) + j] = M[(run * DK + i) * DK + j];
    }
    __syncthreads();
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = Hl[(run * DK + r0 + a) * dv + c0 + cc + b];
    for (int j = 0; j < DK; ++j) {
      const float4 s = *reinterpret_cast<const float4*>(sS + j * kCombCols + cc);
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const float m = sM[(r0 + a) * (DK + 1) + j];
        acc[a][0] = fmaf(m, s.x, acc[a][0]);
        acc[a][1] = fmaf(m, s.y, acc[a][1]);
        acc[a][2] = fmaf(m, s.z, acc[a][2]);
        acc[a][3] = fmaf(m, s.w, acc[a][3]);
      }
    }
    __syncthreads();   // every thread has read sS and sM of this step
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      *reinterpret_cast<float4*>(sS + (r0 + a) * kCombCols + cc) =
          make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
      *reinterpret_cast<float4*>(S + ((bh * P + p) * DK + r0 + a) * dv + c0 + cc) =
          make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    }
    __syncthreads();
  }
}

template <int DK>
cudaError_t launch_combine(const float* M, const float* Hl, const float* h0, float* S, int B,
                           int H, int P, int dv, cudaStream_t stream) {
  const size_t bytes = (static_cast<size_t>(DK) * (DK + 1) + DK * kCombCols) * sizeof(float);
  auto kern = segment_combine_kernel<DK>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bytes));
  if (err != cudaSuccess) return err;
  const dim3 grid(dv / kCombCols, static_cast<unsigned>(B) * H);
  kern<<<grid, 2 * DK, bytes, stream>>>(M, Hl, h0, S, P, dv);
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
