// Single-token recurrent step of the gated delta rule (decode).
//
// LLMs from scratch ch. 11, section 11.2, in the general form of the
// Gated DeltaNet-2 notes, key design 1 (state S in R^{d_k x d_v}):
//   S~ = Diag(alpha) S,  r = S~^T e,  u = z - r,  S <- S~ + k u^T,
//   o  = S^T (s q) = S~^T (s q) + (k . s q) u.
// The step is bound by reading and writing S once (2 * d_k * d_v * 4 bytes per
// sequence and head), so it is written as a stream: one persistent CTA per SM
// walks the (sequence, head) items with a stride of the grid, and each item's
// state moves by plain bulk copies through a ring of three shared-memory
// stages, two loads ahead of the item being updated, while the updated state
// of the previous item drains back to global memory by a bulk store. The
// update itself: each thread owns 4 consecutive value columns (one float4) of
// d_k / RG rows of the stage, so a warp reads whole rows, and S stays in
// registers between the two reductions over the rows and the write-back.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace gdr {
namespace {

constexpr int kStepThreads = 256;
constexpr int kStepStages = 3;

// The static shared data of one CTA, laid out by construction: the mbarriers
// padded to 32 bytes, then float arrays whose sizes are multiples of 16
// bytes, so that the float4 reads of z and of the reduction buffer are
// 16-byte aligned whatever the compiler's placement.
template <int DK, int DV, int RG, int CG>
struct __align__(16) StepShared {
  uint64_t full[4];   // kStepStages used
  float alpha[DK], e[DK], k[DK], q[DK], z[DV];
  float4 red[2][RG][CG];
  float kq[kStepThreads / 32];
};

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(kStepThreads, 1) recurrent_step_kernel(const StepArgs a) {
  constexpr int CG = DV / 4;               // float4 column groups
  constexpr int RG = kStepThreads / CG;    // row groups
  constexpr int RPT = DK / RG;             // state rows per thread
  constexpr uint32_t kBytes = DK * DV * 4;
  static_assert(kStepStages <= 4 && DK % 4 == 0 && DV % 4 == 0, "shared layout");
  extern __shared__ __align__(128) unsigned char ring[];   // kStepStages states
  __shared__ StepShared<DK, DV, RG, CG> sh;
  uint64_t* full = sh.full;
  float *s_alpha = sh.alpha, *s_e = sh.e, *s_k = sh.k, *s_q = sh.q, *s_z = sh.z;
  float4 (*s_red)[RG][CG] = sh.red;
  float* s_kq = sh.kq;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cg = tid % CG, rg = tid / CG;
  const bool CH = a.flags & 1u, ER = a.flags & 2u, WR = a.flags & 4u, QM = a.flags & 8u;
  const int items = a.N * a.H, stride = static_cast<int>(gridDim.x);
  const int cnt = (items - static_cast<int>(blockIdx.x) + stride - 1) / stride;
  const uint32_t rb = smem_u32(ring), fb = smem_u32(full);
  auto item = [&](int j) { return static_cast<size_t>(blockIdx.x) + static_cast<size_t>(j) * stride; };

  if (tid == 0) {
    for (int s = 0; s < kStepStages; ++s) tc::mbar_init(fb + 8 * s, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  int issued = 0;   // (thread 0) states requested so far
  auto load = [&](int j) {
    const uint32_t s = j % kStepStages;
    tc::mbar_arrive_expect_tx(fb + 8 * s, kBytes);
    tc::bulk_load(rb + s * kBytes, a.state + item(j) * DK * DV, kBytes, fb + 8 * s);
    issued = j + 1;
  };
  if (tid == 0)
    for (int j = 0; j < kStepStages - 1 && j < cnt; ++j) load(j);

  // the token's vector elements of this thread (key channel and value column
  // tid), loaded one item ahead and first used (converted) in the next item
  static_assert(DK <= kStepThreads && DV <= kStepThreads, "one element per thread");
  struct Token {
    TIn q, k, b, v, w;
    float g, beta, lam;
  };
  auto fetch = [&](int jj, Token& x) {
    const size_t tok = item(jj);
    if (tid < DK) {
      x.q = static_cast<const TIn*>(a.q)[tok * DK + tid];
      x.k = static_cast<const TIn*>(a.k)[tok * DK + tid];
      if (ER) x.b = static_cast<const TIn*>(a.b)[tok * DK + tid];
      x.g = CH ? a.g[tok * DK + tid] : a.g[tok];
    }
    if (tid < DV) {
      x.v = static_cast<const TIn*>(a.v)[tok * DV + tid];
      if (WR) x.w = static_cast<const TIn*>(a.w)[tok * DV + tid];
    }
    x.beta = (a.beta && !(ER && WR)) ? a.beta[tok] : 0.f;
    x.lam = QM ? a.lam[tok] : 0.f;
  };
  Token cur{}, nxt{};
  fetch(0, cur);

  int j = 0;
  for (; j < cnt; ++j) {
    const size_t tok = item(j);   // sequence * H + head
    float kq = 0.f;
    if (tid < DK) {
      const float qi = static_cast<float>(cur.q), ki = static_cast<float>(cur.k);
      const float x = QM ? ki + cur.lam * qi : ki;
      const float e = ER ? static_cast<float>(cur.b) * x : cur.beta * x;
      s_alpha[tid] = expf(cur.g);
      s_e[tid] = e;
      s_k[tid] = ki;
      s_q[tid] = a.scale * qi;
      kq = ki * a.scale * qi;
    }
    if (tid < DV) {
      const float vc = static_cast<float>(cur.v);
      s_z[tid] = WR ? static_cast<float>(cur.w) * vc : cur.beta * vc;
    }
    if (j + 1 < cnt) fetch(j + 1, nxt);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
    if (lane == 0) s_kq[warp] = kq;
    const uint32_t s = j % kStepStages;
    if (__syncthreads_or(!tc::mbar_wait(fb + 8 * s, (j / kStepStages) & 1))) break;

    float4* st = reinterpret_cast<float4*>(ring + s * kBytes);
    float4 S[RPT];
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f), p = r;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int row = rg + i * RG;
      S[i] = st[row * CG + cg];
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
      float4 x = S[i];
      x.x += ki * u.x; x.y += ki * u.y; x.z += ki * u.z; x.w += ki * u.w;
      st[row * CG + cg] = x;
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
    // the updated state back to global memory; its stage takes the state two
    // items ahead once the store before this one has read its own stage
    tc::fence_proxy_async();
    __syncthreads();
    if (tid == 0) {
      tc::bulk_store(a.state + tok * DK * DV, rb + s * kBytes, kBytes);
      tc::bulk_commit();
      if (j + kStepStages - 1 < cnt) {
        tc::bulk_wait_read<1>();
        load(j + kStepStages - 1);
      }
    }
    cur = nxt;
  }
  if (j < cnt) {
    // a state did not land within the bounded wait: this CTA's remaining
    // outputs read NaN (their states stay as they were), and no copy it
    // started may still be writing its shared memory when it exits
    const float nan = __int_as_float(0x7fc00000);
    for (int jj = j; jj < cnt; ++jj)
      for (int c = tid; c < DV; c += kStepThreads)
        static_cast<TIn*>(a.o)[item(jj) * DV + c] = static_cast<TIn>(nan);
    if (tid == 0)
      for (int jj = j; jj < issued; ++jj)
        tc::mbar_wait(fb + 8 * (jj % kStepStages), (jj / kStepStages) & 1);
  }
  if (tid == 0) tc::bulk_wait_all<0>();
}

// The kernel's shared-memory opt-in and the SM count, set and read once per
// device and instance, so that a launch inside a CUDA graph capture makes no
// other runtime call than the launch itself.
constexpr int kMaxDevices = 64;

template <int DK, int DV, typename TIn>
cudaError_t launch_step_t(const StepArgs& a, cudaStream_t stream) {
  constexpr int kSmem = kStepStages * DK * DV * 4;
  auto kern = recurrent_step_kernel<DK, DV, TIn>;
  static int sms_of[kMaxDevices] = {};   // 0: not yet set up on that device
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 0 && dev < kMaxDevices && sms_of[dev] > 0) {
    sms = sms_of[dev];
  } else {
    if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem)) !=
            cudaSuccess ||
        (err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return err;
    if (dev >= 0 && dev < kMaxDevices) sms_of[dev] = sms;
  }
  const long long items = static_cast<long long>(a.N) * a.H;
  const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);   // one CTA per SM
  kern<<<grid, kStepThreads, kSmem, stream>>>(a);
  err = cudaGetLastError();
  if (err == cudaErrorInvalidValue && dev >= 0 && dev < kMaxDevices && sms_of[dev] > 0) {
    // the opt-in is gone (the device was reset since): set it up again, once
    sms_of[dev] = 0;
    if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem)) !=
        cudaSuccess)
      return err;
    sms_of[dev] = sms;
    kern<<<grid, kStepThreads, kSmem, stream>>>(a);
    err = cudaGetLastError();
  }
  return err;
}

template <int DK, int DV>
cudaError_t launch_step(const StepArgs& a, bool f32, cudaStream_t stream) {
  return f32 ? launch_step_t<DK, DV, float>(a, stream)
             : launch_step_t<DK, DV, __nv_bfloat16>(a, stream);
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
