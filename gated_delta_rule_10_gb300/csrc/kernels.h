// Launch interface between the C ABI (gdr_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>

namespace gdr {

constexpr int kChunkLen = 64;  // C, the chunk length of the WY/UT algorithm

// Arguments of the chunkwise forward; pointers as documented in include/gdr.h.
struct ChunkArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* lam;
  const void* b;
  const void* w;
  const float* h0;
  void* o;
  float* hT;
  int B, T, H, dv;
  unsigned flags;
  float scale;
};

// Arguments of the single-token recurrent step.
struct StepArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* lam;
  const void* b;
  const void* w;
  float* state;
  void* o;
  int N, H;
  unsigned flags;
  float scale;
};

// Value-column slice width of one chunk-forward CTA for this problem.
int chunk_fwd_slice_width(int B, int H, int dk, int dv, bool f32);

cudaError_t launch_chunk_fwd(const ChunkArgs& a, int dk, int nv, bool f32,
                             cudaStream_t stream);
cudaError_t launch_recurrent_step(const StepArgs& a, int dk, int dv, bool f32,
                                  cudaStream_t stream);
cudaError_t launch_gate_cumsum(const float* g, float* G, int B, int T, int X,
                               cudaStream_t stream);

}  // namespace gdr
