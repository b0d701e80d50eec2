// Token-order scan of the gated delta rule for every gate flag (bf16 or fp32
// inputs, fp32 state): the recurrence of LLMs from scratch ch. 11, section
// 11.2, in the general form of the Gated DeltaNet-2 notes, key design 1,
//   S~ = Diag(alpha_t) S_{t-1},  r = S~^T e_t,  u = z_t - r,  S_t = S~ + k_t u^T,
//   o_t = S_t^T (s q_t) = S~^T (s q_t) + (k_t . s q_t) u,
// walked token by token with the state in registers. Unlike the chunkwise form
// it factors no decay (alpha_t multiplies S directly), so any log-decay is
// exact in fp32; it is the path for inputs past the chunked path's range
// (GDR_ERR_RANGE) at the price of a sequential pass over the tokens.
//
// One CTA per (batch, head, 32 value columns), 256 threads: thread (rg, cg)
// holds d_k / 32 rows (rg, rg + 32, ...) of one float4 of value columns cg, so
// the two column sums per token are a reduction over the 32 row groups in
// shared memory. Per token the gates of the next token are read while the
// current one is applied.
#include "common.cuh"
#include "kernels.h"

namespace gdr {
namespace {

constexpr int kScanThreads = 256;
constexpr int kCols = 32;                 // value columns per CTA
constexpr int kCG = kCols / 4;            // float4 column groups
constexpr int kRG = kScanThreads / kCG;   // row groups (32)

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(kScanThreads) token_scan_kernel(const ChunkArgs a) {
  constexpr int RPT = DK / kRG;           // state rows per thread
  // every array 16-byte aligned: z is read as float4
  __shared__ __align__(16) float s_alpha[2][DK];
  __shared__ __align__(16) float s_e[2][DK];
  __shared__ __align__(16) float s_k[2][DK];
  __shared__ __align__(16) float s_q[2][DK];
  __shared__ __align__(16) float s_z[2][kCols];
  __shared__ float4 s_red[2][kRG][kCG];
  __shared__ float s_kq[2][kScanThreads / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cg = tid % kCG, rg = tid / kCG;
  const int c0 = blockIdx.x * kCols;      // first value column of this CTA
  const int h = blockIdx.y, bb = blockIdx.z;
  const int T = a.T, H = a.H;
  const bool CH = a.flags & 1u, ER = a.flags & 2u, WR = a.flags & 4u, QM = a.flags & 8u;
  const size_t bh = size_t(bb) * H + h;

  float4 S[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    S[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.h0)
      S[i] = *reinterpret_cast<const float4*>(a.h0 + (bh * DK + rg + i * kRG) * DV + c0 + cg * 4);
  }

  // token t's vectors into buffer t % 2 (all threads), with its k . s q partial
  auto stage = [&](int t) {
    const int buf = t & 1;
    const size_t tok = (size_t(bb) * T + t) * H + h;
    const TIn* q = static_cast<const TIn*>(a.q) + tok * DK;
    const TIn* k = static_cast<const TIn*>(a.k) + tok * DK;
    const float beta = (a.beta && !(ER && WR)) ? a.beta[tok] : 0.f;
    const float lam = QM ? a.lam[tok] : 0.f;
    float kq = 0.f;
    for (int i = tid; i < DK; i += kScanThreads) {
      const float qi = static_cast<float>(q[i]), ki = static_cast<float>(k[i]);
      const float x = QM ? ki + lam * qi : ki;
      const float e = ER ? static_cast<float>(static_cast<const TIn*>(a.b)[tok * DK + i]) * x
                         : beta * x;
      s_alpha[buf][i] = expf(CH ? a.g[tok * DK + i] : a.g[tok]);
      s_e[buf][i] = e;
      s_k[buf][i] = ki;
      s_q[buf][i] = a.scale * qi;
      kq += ki * a.scale * qi;
    }
    for (int j = tid; j < kCols; j += kScanThreads) {
      const float vj = static_cast<float>(static_cast<const TIn*>(a.v)[tok * DV + c0 + j]);
      s_z[buf][j] = WR ? static_cast<float>(static_cast<const TIn*>(a.w)[tok * DV + c0 + j]) * vj
                       : beta * vj;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
    if (lane == 0) s_kq[buf][warp] = kq;
  };

  if (T > 0) stage(0);
  __syncthreads();
  for (int t = 0; t < T; ++t) {
    const int buf = t & 1;
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f), p = r;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int row = rg + i * kRG;
      const float al = s_alpha[buf][row], e = s_e[buf][row], sq = s_q[buf][row];
      S[i].x *= al; S[i].y *= al; S[i].z *= al; S[i].w *= al;
      r.x += S[i].x * e; r.y += S[i].y * e; r.z += S[i].z * e; r.w += S[i].w * e;
      p.x += S[i].x * sq; p.y += S[i].y * sq; p.z += S[i].z * sq; p.w += S[i].w * sq;
    }
    s_red[0][rg][cg] = r;
    s_red[1][rg][cg] = p;
    if (t + 1 < T) stage(t + 1);   // the next token's vectors meanwhile
    __syncthreads();
    float4 rt = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int g = 0; g < kRG; ++g) {
      const float4 x = s_red[0][g][cg];
      rt.x += x.x; rt.y += x.y; rt.z += x.z; rt.w += x.w;
    }
    const float4 z = *reinterpret_cast<const float4*>(s_z[buf] + cg * 4);
    const float4 u = make_float4(z.x - rt.x, z.y - rt.y, z.z - rt.z, z.w - rt.w);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float ki = s_k[buf][rg + i * kRG];
      S[i].x += ki * u.x; S[i].y += ki * u.y; S[i].z += ki * u.z; S[i].w += ki * u.w;
    }
    if (rg == 0) {
      float kq_all = 0.f;
#pragma unroll
      for (int w = 0; w < kScanThreads / 32; ++w) kq_all += s_kq[buf][w];
      float4 pt = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
      for (int g = 0; g < kRG; ++g) {
        const float4 x = s_red[1][g][cg];
        pt.x += x.x; pt.y += x.y; pt.z += x.z; pt.w += x.w;
      }
      TIn* o = static_cast<TIn*>(a.o) + ((size_t(bb) * T + t) * H + h) * DV + c0 + cg * 4;
      store2(o, pt.x + kq_all * u.x, pt.y + kq_all * u.y);
      store2(o + 2, pt.z + kq_all * u.z, pt.w + kq_all * u.w);
    }
    __syncthreads();   // s_red and buffer t % 2 are free again
  }
  if (a.hT) {
#pragma unroll
    for (int i = 0; i < RPT; ++i)
      *reinterpret_cast<float4*>(a.hT + (bh * DK + rg + i * kRG) * DV + c0 + cg * 4) = S[i];
  }
}

template <int DK, int DV>
cudaError_t launch_scan(const ChunkArgs& a, bool f32, cudaStream_t stream) {
  const dim3 grid(DV / kCols, a.H, a.B);
  if (f32)
    token_scan_kernel<DK, DV, float><<<grid, kScanThreads, 0, stream>>>(a);
  else
    token_scan_kernel<DK, DV, __nv_bfloat16><<<grid, kScanThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_token_scan(const ChunkArgs& a, int dk, bool f32, cudaStream_t stream) {
  if (a.B > 65535 || a.H > 65535) return cudaErrorInvalidValue;
  if (dk == 64 && a.dv == 64) return launch_scan<64, 64>(a, f32, stream);
  if (dk == 64 && a.dv == 128) return launch_scan<64, 128>(a, f32, stream);
  if (dk == 128 && a.dv == 64) return launch_scan<128, 64>(a, f32, stream);
  if (dk == 128 && a.dv == 128) return launch_scan<128, 128>(a, f32, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdr
