// Chunk-local inclusive prefix sum of the log-decay (fp32).
//
// Gated DeltaNet-2 notes, key design 2: gamma_r = exp(sum_{i<=r} g_i) restarts
// at every chunk of C = 64 tokens; the training-strategy paragraph of the same
// notes keeps this cumulative sum in fp32. For g, G of shape [B, T, X] each
// thread owns four adjacent columns x of one (batch, chunk) and walks the
// chunk's tokens in order: every token row is read and written once, with
// 16-byte accesses coalesced along x (X = H for scalar gates, H * d_k for
// per-channel gates). The chunked forward computes the same sums on chip;
// this kernel serves callers that want G itself.
#include "common.cuh"
#include "kernels.h"

namespace gdr {
namespace {

constexpr int kCumThreads = 128;

__global__ void __launch_bounds__(kCumThreads) gate_cumsum_vec4(const float* g, float* G, int T,
                                                                int X, int n_chunks,
                                                                int groups) {
  const long long id = static_cast<long long>(blockIdx.x) * kCumThreads + threadIdx.x;
  const int xg = static_cast<int>(id % groups);
  if (id / groups >= n_chunks) return;
  const int chunk = static_cast<int>(id / groups);
  const int b = blockIdx.y;
  const int t0 = chunk * kChunk;
  const int t1 = min(T, t0 + kChunk);
  const size_t base = (static_cast<size_t>(b) * T + t0) * X + static_cast<size_t>(xg) * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int t = t0; t < t1; ++t) {
    const size_t off = base + static_cast<size_t>(t - t0) * X;
    const float4 x = *reinterpret_cast<const float4*>(g + off);
    acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
    *reinterpret_cast<float4*>(G + off) = acc;
  }
}

__global__ void __launch_bounds__(kCumThreads) gate_cumsum_scalar(const float* g, float* G, int T,
                                                                  int X, int n_chunks) {
  const long long id = static_cast<long long>(blockIdx.x) * kCumThreads + threadIdx.x;
  const int x = static_cast<int>(id % X);
  if (id / X >= n_chunks) return;
  const int chunk = static_cast<int>(id / X);
  const int b = blockIdx.y;
  const int t0 = chunk * kChunk;
  const int t1 = min(T, t0 + kChunk);
  const size_t base = (static_cast<size_t>(b) * T + t0) * X + x;
  float acc = 0.f;
  for (int t = t0; t < t1; ++t) {
    const size_t off = base + static_cast<size_t>(t - t0) * X;
    acc += g[off];
    G[off] = acc;
  }
}

}  // namespace

cudaError_t launch_gate_cumsum(const float* g, float* G, int B, int T, int X,
                               cudaStream_t stream) {
  const int n_chunks = (T + kChunk - 1) / kChunk;
  const bool vec = (X % 4 == 0) && (reinterpret_cast<uintptr_t>(g) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(G) % 16 == 0);
  const long long per_batch = static_cast<long long>(n_chunks) * (vec ? X / 4 : X);
  const long long blocks_x = (per_batch + kCumThreads - 1) / kCumThreads;
  // blockIdx.y is the batch; blockIdx.x covers (chunk, column group) pairs
  dim3 grid(static_cast<unsigned>(blocks_x), static_cast<unsigned>(B));
  if (vec) {
    gate_cumsum_vec4<<<grid, kCumThreads, 0, stream>>>(g, G, T, X, n_chunks, X / 4);
  } else {
    gate_cumsum_scalar<<<grid, kCumThreads, 0, stream>>>(g, G, T, X, n_chunks);
  }
  return cudaGetLastError();
}

}  // namespace gdr
