// Gradients of the token-order recurrence with a write strength per value
// channel (LLMs from scratch ch. 11, section 11.3; the forward is
// value_beta_scan.cu):
//   S~ = alpha_t S_{t-1},  r = S~^T k_t,  u = beta_t (.) (v_t - r),
//   S_t = S~ + k_t u^T,    o_t = S_t^T (s q_t),   alpha_t = exp(g_t)
// for L = <dO, o> + <dhT, S_T>. The reverse-mode step of token t, with dS
// holding dL/dS_t on entry and dL/dS_{t-1} on exit:
//   dS  += s q_t do_t^T,        dq_t  = s S_t do_t
//   du   = dS^T k_t,            dk_t  = dS u
//   dbeta_t = du (.) (v_t - r), dv_t  = du (.) beta_t,   dr = -du (.) beta_t
//   dS~  = dS + k_t dr^T,       dk_t += S~ dr
//   dg_t = <dS~, S~>,           dS   <- alpha_t dS~
// Given the keys every column of S follows its own map, so one CTA takes 32
// value columns of one (batch, head) and walks the tokens: forward first,
// keeping the state entering every 64-token chunk (checkpoints), then the
// chunks in reverse, each re-run from its checkpoint while the state entering
// each token is kept in a scratch slice, then walked backward. Checkpoints and
// scratch are stored in each thread's own order and read back only by the
// thread that wrote them. dv and dbeta are whole per column; dq, dk and dg sum
// over the column blocks of a (batch, head): the warps reduce in shared memory
// and add into the outputs (zeroed first) with atomics, so the last bits of
// those three depend on the order the CTAs arrive in.
//
// Layout: four warps of four groups of eight lanes; a group holds CL = 2
// columns, lane i of a group key rows i R .. i R + R - 1 (R = d_k / 8); sums
// over the key rows are three-step butterflies inside the group. The next
// token's inputs are loaded while the current one is processed.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"
#include "token_io.cuh"

namespace gdr {
namespace {

constexpr int kVbNW = 4;                  // warps per CTA
constexpr int kVbCL = 2;                  // columns per group of eight lanes
constexpr int kVbCols = 4 * kVbNW * kVbCL;   // value columns per CTA (32)
constexpr int kVbThreads = 32 * kVbNW;
constexpr int kVbChunk = 64;              // tokens between checkpoints

template <int R>
struct VbToken {
  float k[R], q[R];
  float v[kVbCL], be[kVbCL], dO[kVbCL];
  float al;
};

template <typename TIn, int DK>
__global__ void __launch_bounds__(kVbThreads)
    value_beta_bwd_kernel(const ValueBetaBwdArgs a, float* ckpt, float* scratch) {
  constexpr int R = DK / 8;
  constexpr int NS = R * kVbCL;   // state floats per thread
  __shared__ __align__(16) float red[2][kVbNW][2][DK];
  __shared__ float red_g[2][kVbNW];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gi = lane >> 3, li = lane & 7;
  const int h = blockIdx.y, bb = blockIdx.z;
  const int c0 = blockIdx.x * kVbCols + (warp * 4 + gi) * kVbCL;   // this group's columns
  const int r0 = li * R;                                            // this lane's key rows
  const int T = a.T, H = a.H, DV = a.nv;
  const int nc = (T + kVbChunk - 1) / kVbChunk;
  const size_t cta = (static_cast<size_t>(bb) * H + h) * gridDim.x + blockIdx.x;
  float* my_ckpt = ckpt + (cta * nc * kVbThreads + tid) * NS;        // + n * kVbThreads * NS
  float* my_scr = scratch + (cta * kVbChunk * kVbThreads + tid) * NS;   // + j * kVbThreads * NS
  const TIn* qg = static_cast<const TIn*>(a.q);
  const TIn* kg = static_cast<const TIn*>(a.k);
  const TIn* vg = static_cast<const TIn*>(a.v);
  const TIn* dOg = static_cast<const TIn*>(a.dO);

  auto fetch = [&](int t, VbToken<R>& x) {
    const size_t tk = (static_cast<size_t>(bb) * T + t) * H + h;
    static_assert(kVbCL == 2, "column pairs");
    load_run<R>(kg + tk * DK + r0, x.k);
    load_run<R>(qg + tk * DK + r0, x.q);
    const float2 v2 = load_pair(vg + tk * DV + c0), b2 = load_pair(a.beta + tk * DV + c0),
                 o2 = load_pair(dOg + tk * DV + c0);
    x.v[0] = v2.x; x.v[1] = v2.y;
    x.be[0] = b2.x; x.be[1] = b2.y;
    x.dO[0] = o2.x; x.dO[1] = o2.y;
    x.al = expf(a.g[tk]);
  };
  auto group_sum = [&](float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    return x;
  };
  // S~ = alpha S, r, u; S becomes S_t (forward step)
  auto step = [&](float (&S)[R][kVbCL], const VbToken<R>& x, float (&r)[kVbCL],
                  float (&u)[kVbCL]) {
#pragma unroll
    for (int c = 0; c < kVbCL; ++c) {
      float p = 0.f;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        S[i][c] *= x.al;
        p = fmaf(S[i][c], x.k[i], p);
      }
      r[c] = group_sum(p);
      u[c] = x.be[c] * (x.v[c] - r[c]);
#pragma unroll
      for (int i = 0; i < R; ++i) S[i][c] = fmaf(x.k[i], u[c], S[i][c]);
    }
  };
  auto save = [&](float* dst, const float (&S)[R][kVbCL]) {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int e = 0; e < NS; e += 4)
      d4[e / 4] = make_float4(S[e / kVbCL][e % kVbCL], S[(e + 1) / kVbCL][(e + 1) % kVbCL],
                              S[(e + 2) / kVbCL][(e + 2) % kVbCL], S[(e + 3) / kVbCL][(e + 3) % kVbCL]);
  };
  auto restore = [&](const float* src, float (&S)[R][kVbCL]) {
    const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
    for (int e = 0; e < NS; e += 4) {
      const float4 x = s4[e / 4];
      S[e / kVbCL][e % kVbCL] = x.x;
      S[(e + 1) / kVbCL][(e + 1) % kVbCL] = x.y;
      S[(e + 2) / kVbCL][(e + 2) % kVbCL] = x.z;
      S[(e + 3) / kVbCL][(e + 3) % kVbCL] = x.w;
    }
  };

  // ---- forward: the state entering every chunk ----
  float S[R][kVbCL];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int c = 0; c < kVbCL; ++c)
      S[i][c] = a.h0 ? a.h0[((static_cast<size_t>(bb) * H + h) * DK + r0 + i) * DV + c0 + c] : 0.f;
  {
    VbToken<R> cur, nxt;
    fetch(0, cur);
    for (int t = 0; t < T; ++t) {
      if (t % kVbChunk == 0) save(my_ckpt + static_cast<size_t>(t / kVbChunk) * kVbThreads * NS, S);
      if (t + 1 < T) fetch(t + 1, nxt);
      float r[kVbCL], u[kVbCL];
      step(S, cur, r, u);
      cur = nxt;
    }
  }

  // ---- reverse: every chunk re-run from its checkpoint, then walked backward ----
  float dS[R][kVbCL];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int c = 0; c < kVbCL; ++c)
      dS[i][c] = a.dhT ? a.dhT[((static_cast<size_t>(bb) * H + h) * DK + r0 + i) * DV + c0 + c] : 0.f;
  int par = 0;
  for (int n = nc - 1; n >= 0; --n) {
    const int t0 = n * kVbChunk, Lc = min(kVbChunk, T - t0);
    restore(my_ckpt + static_cast<size_t>(n) * kVbThreads * NS, S);
    {
      VbToken<R> cur, nxt;
      fetch(t0, cur);
      for (int j = 0; j < Lc; ++j) {
        save(my_scr + static_cast<size_t>(j) * kVbThreads * NS, S);
        if (j + 1 < Lc) fetch(t0 + j + 1, nxt);
        float r[kVbCL], u[kVbCL];
        step(S, cur, r, u);
        cur = nxt;
      }
    }
    VbToken<R> cur, nxt;
    fetch(t0 + Lc - 1, cur);
    for (int j = Lc - 1; j >= 0; --j) {
      const int t = t0 + j;
      const size_t tk = (static_cast<size_t>(bb) * T + t) * H + h;
      if (j > 0) fetch(t - 1, nxt);
      float St[R][kVbCL];   // S~, then (a copy of) S_t
      restore(my_scr + static_cast<size_t>(j) * kVbThreads * NS, St);
      float r[kVbCL], u[kVbCL];
      // S~ and r, u (the forward step, keeping S~)
      float Sw[R][kVbCL];
#pragma unroll
      for (int c = 0; c < kVbCL; ++c) {
        float p = 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i) {
          Sw[i][c] = St[i][c] * cur.al;   // S~
          p = fmaf(Sw[i][c], cur.k[i], p);
        }
        r[c] = group_sum(p);
        u[c] = cur.be[c] * (cur.v[c] - r[c]);
      }
      float dq[R], dk[R], gpart = 0.f;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        dq[i] = 0.f;
        dk[i] = 0.f;
      }
      float du[kVbCL];
#pragma unroll
      for (int c = 0; c < kVbCL; ++c) {
        float p = 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const float st = fmaf(cur.k[i], u[c], Sw[i][c]);   // S_t
          dq[i] = fmaf(st, cur.dO[c], dq[i]);
          dS[i][c] = fmaf(a.scale * cur.q[i], cur.dO[c], dS[i][c]);
          p = fmaf(dS[i][c], cur.k[i], p);
          dk[i] = fmaf(dS[i][c], u[c], dk[i]);
        }
        du[c] = group_sum(p);
      }
#pragma unroll
      for (int c = 0; c < kVbCL; ++c) {
        const float dr = -du[c] * cur.be[c];
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const float dst = fmaf(cur.k[i], dr, dS[i][c]);   // dS~
          dk[i] = fmaf(Sw[i][c], dr, dk[i]);
          gpart = fmaf(dst, Sw[i][c], gpart);
          dS[i][c] = cur.al * dst;
        }
        if (li == 0) {
          a.dv[tk * DV + c0 + c] = du[c] * cur.be[c];
          a.dbeta[tk * DV + c0 + c] = du[c] * (cur.v[c] - r[c]);
        }
      }
      // row sums over the group's columns -> over the warp's groups -> shared
#pragma unroll
      for (int i = 0; i < R; ++i) {
        dq[i] += __shfl_xor_sync(0xffffffffu, dq[i], 8);
        dq[i] += __shfl_xor_sync(0xffffffffu, dq[i], 16);
        dk[i] += __shfl_xor_sync(0xffffffffu, dk[i], 8);
        dk[i] += __shfl_xor_sync(0xffffffffu, dk[i], 16);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) gpart += __shfl_xor_sync(0xffffffffu, gpart, o);
      if (gi == 0) {
#pragma unroll
        for (int i = 0; i < R; ++i) {
          red[par][warp][0][r0 + i] = a.scale * dq[i];
          red[par][warp][1][r0 + i] = dk[i];
        }
      }
      if (lane == 0) red_g[par][warp] = gpart;
      __syncthreads();   // (the buffer of parity par is written again two tokens on)
      for (int i = tid; i < 2 * DK; i += kVbThreads) {
        const int which = i / DK, row = i % DK;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kVbNW; ++w) s += red[par][w][which][row];
        atomicAdd((which ? a.dk : a.dq) + tk * DK + row, s);
      }
      if (tid == 0) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kVbNW; ++w) s += red_g[par][w];
        atomicAdd(a.dg + tk, s);
      }
      par ^= 1;
      cur = nxt;
    }
  }
  if (a.dh0) {
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int c = 0; c < kVbCL; ++c)
        a.dh0[((static_cast<size_t>(bb) * H + h) * DK + r0 + i) * DV + c0 + c] = dS[i][c];
  }
}

template <typename T, int DK>
cudaError_t launch_vb_bwd(const ValueBetaBwdArgs& a, float* ckpt, float* scratch,
                          cudaStream_t stream) {
  const dim3 grid(a.nv / kVbCols, a.H, a.B);
  value_beta_bwd_kernel<T, DK><<<grid, kVbThreads, 0, stream>>>(a, ckpt, scratch);
  return cudaGetLastError();
}

}  // namespace

size_t value_beta_bwd_workspace_bytes(int B, int T, int H, int dk, int dv) {
  const size_t ctas = static_cast<size_t>(B) * H * (dv / kVbCols);
  const size_t nc = static_cast<size_t>((T + kVbChunk - 1) / kVbChunk);
  const size_t per = static_cast<size_t>(dk) * kVbCols * sizeof(float);   // one state slice
  return kChunkWorkspaceBytes + ctas * nc * per + ctas * kVbChunk * per;
}

cudaError_t launch_value_beta_bwd(const ValueBetaBwdArgs& a, bool f32, cudaStream_t stream) {
  if (a.nk != 64 && a.nk != 128) return cudaErrorInvalidValue;
  if (a.nv % kVbCols != 0) return cudaErrorInvalidValue;
  const size_t ctas = static_cast<size_t>(a.B) * a.H * (a.nv / kVbCols);
  const size_t nc = static_cast<size_t>((a.T + kVbChunk - 1) / kVbChunk);
  const size_t per = static_cast<size_t>(a.nk) * kVbCols;
  float* ckpt = reinterpret_cast<float*>(static_cast<unsigned char*>(a.workspace) +
                                         kChunkWorkspaceBytes);
  float* scratch = ckpt + ctas * nc * per;
  cudaError_t err;
  // dq, dk and dg are sums over the column blocks
  if ((err = cudaMemsetAsync(a.dq, 0, static_cast<size_t>(a.B) * a.T * a.H * a.nk * 4, stream)) != cudaSuccess ||
      (err = cudaMemsetAsync(a.dk, 0, static_cast<size_t>(a.B) * a.T * a.H * a.nk * 4, stream)) != cudaSuccess ||
      (err = cudaMemsetAsync(a.dg, 0, static_cast<size_t>(a.B) * a.T * a.H * 4, stream)) != cudaSuccess)
    return err;
  if (a.nk == 64)
    return f32 ? launch_vb_bwd<float, 64>(a, ckpt, scratch, stream)
               : launch_vb_bwd<__nv_bfloat16, 64>(a, ckpt, scratch, stream);
  return f32 ? launch_vb_bwd<float, 128>(a, ckpt, scratch, stream)
             : launch_vb_bwd<__nv_bfloat16, 128>(a, ckpt, scratch, stream);
}

}  // namespace gdr
