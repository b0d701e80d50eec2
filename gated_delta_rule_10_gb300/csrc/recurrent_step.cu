// Single-token recurrent step of the gated delta rule (decode).
//
// LLMs from scratch ch. 11, section 11.2, in the general form of the
// Gated DeltaNet-2 notes, key design 1 (state S in R^{d_k x d_v}):
//   S~ = Diag(alpha) S,  r = S~^T e,  u = z - r,  S <- S~ + k u^T,
//   o  = S^T (s q) = S~^T (s q) + (k . s q) u.
// The step is bound by reading and writing S once (2 * d_k * d_v * 4 bytes per
// sequence and head). One CTA per (sequence, head); each thread owns 4
// consecutive value columns (one float4) of d_k / RG rows, so a warp reads
// whole 512-byte rows and S stays in registers between the read and the write.
#include "common.cuh"
#include "kernels.h"

namespace gdr {
namespace {

constexpr int kStepThreads = 256;

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(kStepThreads) recurrent_step_kernel(const StepArgs a) {
  constexpr int CG = DV / 4;               // float4 column groups
  constexpr int RG = kStepThreads / CG;    // row groups
  constexpr int RPT = DK / RG;             // state rows per thread
  __shared__ float s_alpha[DK], s_e[DK], s_k[DK], s_q[DK], s_z[DV];
  __shared__ float4 s_red[2][RG][CG];
  __shared__ float s_kq[kStepThreads / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cg = tid % CG, rg = tid / CG;
  const size_t tok = blockIdx.x;  // sequence * H + head
  const bool CH = a.flags & 1u, ER = a.flags & 2u, WR = a.flags & 4u, QM = a.flags & 8u;

  float* st = a.state + tok * DK * DV;
  float4 S[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    S[i] = *reinterpret_cast<const float4*>(st + size_t(rg + i * RG) * DV + cg * 4);

  const TIn* q = static_cast<const TIn*>(a.q) + tok * DK;
  const TIn* k = static_cast<const TIn*>(a.k) + tok * DK;
  const TIn* v = static_cast<const TIn*>(a.v) + tok * DV;
  const float beta = (a.beta && !(ER && WR)) ? a.beta[tok] : 0.f;
  const float lam = QM ? a.lam[tok] : 0.f;
  float kq = 0.f;
  for (int i = tid; i < DK; i += kStepThreads) {
    const float qi = static_cast<float>(q[i]), ki = static_cast<float>(k[i]);
    const float x = QM ? ki + lam * qi : ki;
    const float e = ER ? static_cast<float>(static_cast<const TIn*>(a.b)[tok * DK + i]) * x
                       : beta * x;
    s_alpha[i] = expf(CH ? a.g[tok * DK + i] : a.g[tok]);
    s_e[i] = e;
    s_k[i] = ki;
    s_q[i] = a.scale * qi;
    kq += ki * a.scale * qi;
  }
  for (int j = tid; j < DV; j += kStepThreads) {
    const float vj = static_cast<float>(v[j]);
    s_z[j] = WR ? static_cast<float>(static_cast<const TIn*>(a.w)[tok * DV + j]) * vj : beta * vj;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
  if (lane == 0) s_kq[warp] = kq;
  __syncthreads();

  float4 r = make_float4(0.f, 0.f, 0.f, 0.f), p = r;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int row = rg + i * RG;
    const float al = s_alpha[row], e = s_e[row], sq = s_q[row];
    S[i].x *= al; S[i].y *= al; S[i].z *= al; S[i].w *= al;
    r.x += S[i].x * e; r.y += S[i].y * e; r.z += S[i].z * e; r.w += S[i].w * e;
    p.x += S[i].x * sq; p.y += S[i].y * sq; p.z += S[i].z * sq; p.w += S[i].w * sq;
  }
  s_red[0][rg][cg] = r;
  s_red[1][rg][cg] = p;
  __syncthreads();

  float4 rt = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int g = 0; g < RG; ++g) {
    const float4 x = s_red[0][g][cg];
    rt.x += x.x; rt.y += x.y; rt.z += x.z; rt.w += x.w;
  }
  const float4 z = *reinterpret_cast<const float4*>(s_z + cg * 4);
  const float4 u = make_float4(z.x - rt.x, z.y - rt.y, z.z - rt.z, z.w - rt.w);
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int row = rg + i * RG;
    const float ki = s_k[row];
    float4 s = S[i];
    s.x += ki * u.x; s.y += ki * u.y; s.z += ki * u.z; s.w += ki * u.w;
    *reinterpret_cast<float4*>(st + size_t(row) * DV + cg * 4) = s;
  }
  if (rg == 0) {
    float kq_all = 0.f;
#pragma unroll
    for (int w = 0; w < kStepThreads / 32; ++w) kq_all += s_kq[w];
    float4 pt = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int g = 0; g < RG; ++g) {
      const float4 x = s_red[1][g][cg];
      pt.x += x.x; pt.y += x.y; pt.z += x.z; pt.w += x.w;
    }
    TIn* o = static_cast<TIn*>(a.o) + tok * DV + cg * 4;
    store2(o, pt.x + kq_all * u.x, pt.y + kq_all * u.y);
    store2(o + 2, pt.z + kq_all * u.z, pt.w + kq_all * u.w);
  }
}

template <int DK, int DV>
cudaError_t launch_step(const StepArgs& a, bool f32, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>(a.N) * static_cast<unsigned>(a.H);
  if (f32)
    recurrent_step_kernel<DK, DV, float><<<blocks, kStepThreads, 0, stream>>>(a);
  else
    recurrent_step_kernel<DK, DV, __nv_bfloat16><<<blocks, kStepThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent_step(const StepArgs& a, int dk, int dv, bool f32,
                                  cudaStream_t stream) {
  if (dk == 64 && dv == 64) return launch_step<64, 64>(a, f32, stream);
  if (dk == 64 && dv == 128) return launch_step<64, 128>(a, f32, stream);
  if (dk == 128 && dv == 64) return launch_step<128, 64>(a, f32, stream);
  if (dk == 128 && dv == 128) return launch_step<128, 128>(a, f32, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdr
