// Gradients of the gated delta rule walked token by token (every flag but the
// per-value-channel write strength, which has value_beta_bwd.cu): the
// backward counterpart of token_scan.cu, with no decay factoring and so no
// range limit. The recurrence, in the general form of the Gated DeltaNet-2
// notes, key design 1 (LLMs from scratch ch. 11, section 11.2):
//   S~ = Diag(alpha_t) S_{t-1},  r = S~^T e_t,  u = z_t - r,
//   S_t = S~ + k_t u^T,          o_t = S_t^T (s q_t)
// with x = k + lam q (QMIX) or k, e = b (.) x (erase gate) or beta x,
// z = w (.) v (write gate) or beta v, alpha = exp(g) per key channel or per
// head. The reverse step of token t (dS: dL/dS_t on entry, dL/dS_{t-1} on exit):
//   dS += s q do^T,  dq = s S_t do,  du = dS^T k,  dk = dS u,  dz = du,
//   dr = -du,  de = S~ dr,  dS~ = dS + e dr^T,  dg = <dS~, S~> (per key row
//   or summed),  dS <- Diag(alpha) dS~,
// then through the gates: dv = w (.) dz or beta dz, dw = v (.) dz,
// dx = b (.) de or beta de, db = x (.) de, dbeta = <v, dz> + <x, de> (the
// scalar gates that apply), dk += dx, dq += lam dx, dlam = <q, dx>.
// Given the keys and gates every column of S evolves on its own, so a CTA
// takes 16 value columns of one (batch, head): forward first, keeping the
// state entering every 64-token chunk, then the chunks in reverse, each re-run
// from its checkpoint with the state entering each token in a scratch slice
// (both stored and read back by the thread that owns them), and walked
// backward. Everything but dv and dw sums over the column blocks of a (batch,
// head), linearly in each block's share of du and de: the warps reduce in
// shared memory and add into the outputs (zeroed first) with atomics.
//
// Layout: four warps of two groups of sixteen lanes; a group holds CL = 2
// columns, lane i of a group key rows i R .. i R + R - 1 (R = d_k / 16); sums
// over the key rows are four-step butterflies inside the group. The next
// token's inputs are loaded while the current one is processed.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"
#include "token_io.cuh"

namespace gdr {
namespace {

constexpr int kTbNW = 4;
constexpr int kTbCL = 2;
constexpr int kTbCols = 2 * kTbNW * kTbCL;   // value columns per CTA (16)
constexpr int kTbThreads = 32 * kTbNW;
constexpr int kTbChunk = 64;

template <int R>
struct TbToken {
  float k[R], q[R], b[R], g[R];
  float v[kTbCL], w[kTbCL], dO[kTbCL];
  float gs, beta, lam;
};

template <typename TIn, int DK>
__global__ void __launch_bounds__(kTbThreads)
    token_bwd_kernel(const ChunkBwdArgs a, float* ckpt, float* scratch) {
  constexpr int R = DK / 16;
  constexpr int NS = R * kTbCL;
  __shared__ __align__(16) float red[2][kTbNW][4][DK];   // dq, dk, db, dg rows
  __shared__ float red_s[2][kTbNW][3];                    // dg (per head), dbeta, dlam

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gi = lane >> 4, li = lane & 15;
  const int h = blockIdx.y, bb = blockIdx.z;
  const int c0 = blockIdx.x * kTbCols + (warp * 2 + gi) * kTbCL;
  const int r0 = li * R;
  const int T = a.T, H = a.H, DV = a.dv_dim;
  const bool CH = a.flags & 1u, ER = a.flags & 2u, WR = a.flags & 4u, QM = a.flags & 8u;
  const bool use_beta = a.beta != nullptr && !(ER && WR);
  const int nc = (T + kTbChunk - 1) / kTbChunk;
  const size_t cta = (static_cast<size_t>(bb) * H + h) * gridDim.x + blockIdx.x;
  float* my_ckpt = ckpt + (cta * nc * kTbThreads + tid) * NS;
  float* my_scr = scratch + (cta * kTbChunk * kTbThreads + tid) * NS;
  const TIn* qg = static_cast<const TIn*>(a.q);
  const TIn* kg = static_cast<const TIn*>(a.k);
  const TIn* vg = static_cast<const TIn*>(a.v);
  const TIn* bg = static_cast<const TIn*>(a.b);
  const TIn* wg = static_cast<const TIn*>(a.w);
  const TIn* dOg = static_cast<const TIn*>(a.dO);

  auto fetch = [&](int t, TbToken<R>& x) {
    const size_t tk = (static_cast<size_t>(bb) * T + t) * H + h;
    static_assert(kTbCL == 2, "column pairs");
    load_run<R>(kg + tk * DK + r0, x.k);
    load_run<R>(qg + tk * DK + r0, x.q);
    if (ER) {
      load_run<R>(bg + tk * DK + r0, x.b);
    } else {
#pragma unroll
      for (int i = 0; i < R; ++i) x.b[i] = 0.f;
    }
    if (CH) {
      load_run<R>(a.g + tk * DK + r0, x.g);
    } else {
#pragma unroll
      for (int i = 0; i < R; ++i) x.g[i] = 0.f;
    }
    const float2 v2 = load_pair(vg + tk * DV + c0), o2 = load_pair(dOg + tk * DV + c0);
    const float2 w2 = WR ? load_pair(wg + tk * DV + c0) : make_float2(0.f, 0.f);
    x.v[0] = v2.x; x.v[1] = v2.y;
    x.w[0] = w2.x; x.w[1] = w2.y;
    x.dO[0] = o2.x; x.dO[1] = o2.y;
    x.gs = CH ? 0.f : a.g[tk];
    x.beta = use_beta ? a.beta[tk] : 0.f;
    x.lam = QM ? a.lam[tk] : 0.f;
  };
  // the token's decay factors, erase input and erase vector (this lane's rows)
  auto keys = [&](const TbToken<R>& x, float (&al)[R], float (&xe)[R], float (&e)[R]) {
    const float as = CH ? 0.f : expf(x.gs);
#pragma unroll
    for (int i = 0; i < R; ++i) {
      al[i] = CH ? expf(x.g[i]) : as;
      xe[i] = QM ? fmaf(x.lam, x.q[i], x.k[i]) : x.k[i];
      e[i] = ER ? x.b[i] * xe[i] : x.beta * xe[i];
    }
  };
  auto group_sum = [&](float s) {
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    s += __shfl_xor_sync(0xffffffffu, s, 8);
    return s;
  };
  auto save = [&](float* dst, const float (&S)[R][kTbCL]) {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int e4 = 0; e4 < NS; e4 += 4)
      d4[e4 / 4] = make_float4(S[e4 / kTbCL][e4 % kTbCL], S[(e4 + 1) / kTbCL][(e4 + 1) % kTbCL],
                               S[(e4 + 2) / kTbCL][(e4 + 2) % kTbCL],
                               S[(e4 + 3) / kTbCL][(e4 + 3) % kTbCL]);
  };
  auto restore = [&](const float* src, float (&S)[R][kTbCL]) {
    const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
    for (int e4 = 0; e4 < NS; e4 += 4) {
      const float4 x = s4[e4 / 4];
      S[e4 / kTbCL][e4 % kTbCL] = x.x;
      S[(e4 + 1) / kTbCL][(e4 + 1) % kTbCL] = x.y;
      S[(e4 + 2) / kTbCL][(e4 + 2) % kTbCL] = x.z;
      S[(e4 + 3) / kTbCL][(e4 + 3) % kTbCL] = x.w;
    }
  };
  auto step = [&](float (&S)[R][kTbCL], const TbToken<R>& x) {
    float al[R], xe[R], e[R];
    keys(x, al, xe, e);
#pragma unroll
    for (int c = 0; c < kTbCL; ++c) {
      float p = 0.f;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        S[i][c] *= al[i];
        p = fmaf(S[i][c], e[i], p);
      }
      const float z = WR ? x.w[c] * x.v[c] : x.beta * x.v[c];
      const float u = z - group_sum(p);
#pragma unroll
      for (int i = 0; i < R; ++i) S[i][c] = fmaf(x.k[i], u, S[i][c]);
    }
  };

  // ---- forward: the state entering every chunk ----
  float S[R][kTbCL];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int c = 0; c < kTbCL; ++c)
      S[i][c] = a.h0 ? a.h0[((static_cast<size_t>(bb) * H + h) * DK + r0 + i) * DV + c0 + c] : 0.f;
  {
    TbToken<R> cur, nxt;
    fetch(0, cur);
    for (int t = 0; t < T; ++t) {
      if (t % kTbChunk == 0) save(my_ckpt + static_cast<size_t>(t / kTbChunk) * kTbThreads * NS, S);
      if (t + 1 < T) fetch(t + 1, nxt);
      step(S, cur);
      cur = nxt;
    }
  }

  // ---- reverse ----
  float dS[R][kTbCL];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int c = 0; c < kTbCL; ++c)
      dS[i][c] = a.dhT ? a.dhT[((static_cast<size_t>(bb) * H + h) * DK + r0 + i) * DV + c0 + c] : 0.f;
  int par = 0;
  for (int n = nc - 1; n >= 0; --n) {
    const int t0 = n * kTbChunk, Lc = min(kTbChunk, T - t0);
    restore(my_ckpt + static_cast<size_t>(n) * kTbThreads * NS, S);
    {
      TbToken<R> cur, nxt;
      fetch(t0, cur);
      for (int j = 0; j < Lc; ++j) {
        save(my_scr + static_cast<size_t>(j) * kTbThreads * NS, S);
        if (j + 1 < Lc) fetch(t0 + j + 1, nxt);
        step(S, cur);
        cur = nxt;
      }
    }
    TbToken<R> cur, nxt;
    fetch(t0 + Lc - 1, cur);
    for (int j = Lc - 1; j >= 0; --j) {
      const int t = t0 + j;
      const size_t tk = (static_cast<size_t>(bb) * T + t) * H + h;
      if (j > 0) fetch(t - 1, nxt);
      float Sw[R][kTbCL];
      restore(my_scr + static_cast<size_t>(j) * kTbThreads * NS, Sw);
      float al[R], xe[R], e[R];
      keys(cur, al, xe, e);
      float u[kTbCL];
#pragma unroll
      for (int c = 0; c < kTbCL; ++c) {
        float p = 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i) {
          Sw[i][c] *= al[i];   // S~
          p = fmaf(Sw[i][c], e[i], p);
        }
        const float z = WR ? cur.w[c] * cur.v[c] : cur.beta * cur.v[c];
        u[c] = z - group_sum(p);
      }
      float dq[R], dk[R], de[R], dg[R];
#pragma unroll
      for (int i = 0; i < R; ++i) {
        dq[i] = 0.f;
        dk[i] = 0.f;
        de[i] = 0.f;
        dg[i] = 0.f;
      }
      float du[kTbCL];
#pragma unroll
      for (int c = 0; c < kTbCL; ++c) {
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
      float gsum = 0.f, bpart = 0.f, lpart = 0.f;
#pragma unroll
      for (int c = 0; c < kTbCL; ++c) {
        const float dr = -du[c];
#pragma unroll
        for (int i = 0; i < R; ++i) {
          de[i] = fmaf(Sw[i][c], dr, de[i]);
          const float dst = fmaf(e[i], dr, dS[i][c]);   // dS~
          dg[i] = fmaf(dst, Sw[i][c], dg[i]);
          dS[i][c] = al[i] * dst;
        }
        if (li == 0) {
          a.dv[tk * DV + c0 + c] = WR ? du[c] * cur.w[c] : cur.beta * du[c];
          if (WR) a.dw[tk * DV + c0 + c] = du[c] * cur.v[c];
          if (use_beta && !WR) bpart = fmaf(du[c], cur.v[c], bpart);
        }
      }
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const float dx = ER ? cur.b[i] * de[i] : cur.beta * de[i];
        if (use_beta && !ER) bpart = fmaf(xe[i], de[i], bpart);
        dq[i] = a.scale * dq[i] + (QM ? cur.lam * dx : 0.f);
        if (QM) lpart = fmaf(cur.q[i], dx, lpart);
        dk[i] += dx;
        de[i] *= xe[i];   // db (erase gate)
        gsum += dg[i];
      }
      // rows: over the warp's two groups, then shared; scalars: over the warp
#pragma unroll
      for (int i = 0; i < R; ++i) {
        dq[i] += __shfl_xor_sync(0xffffffffu, dq[i], 16);
        dk[i] += __shfl_xor_sync(0xffffffffu, dk[i], 16);
        de[i] += __shfl_xor_sync(0xffffffffu, de[i], 16);
        dg[i] += __shfl_xor_sync(0xffffffffu, dg[i], 16);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        gsum += __shfl_xor_sync(0xffffffffu, gsum, o);
        bpart += __shfl_xor_sync(0xffffffffu, bpart, o);
        lpart += __shfl_xor_sync(0xffffffffu, lpart, o);
      }
      if (gi == 0) {
#pragma unroll
        for (int i = 0; i < R; ++i) {
          red[par][warp][0][r0 + i] = dq[i];
          red[par][warp][1][r0 + i] = dk[i];
          red[par][warp][2][r0 + i] = de[i];
          red[par][warp][3][r0 + i] = dg[i];
        }
      }
      if (lane == 0) {
        red_s[par][warp][0] = gsum;
        red_s[par][warp][1] = bpart;
        red_s[par][warp][2] = lpart;
      }
      __syncthreads();   // (the buffer of parity par is written again two tokens on)
      for (int i = tid; i < 4 * DK; i += kTbThreads) {
        const int which = i / DK, row = i % DK;
        if ((which == 2 && !ER) || (which == 3 && !CH)) continue;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kTbNW; ++w) s += red[par][w][which][row];
        float* dst = which == 0 ? a.dq : which == 1 ? a.dk : which == 2 ? a.db : a.dg;
        atomicAdd(dst + tk * DK + row, s);
      }
      if (tid < 3) {
        const bool live = tid == 0 ? !CH : tid == 1 ? (use_beta && a.dbeta) : QM;
        if (live) {
          float s = 0.f;
#pragma unroll
          for (int w = 0; w < kTbNW; ++w) s += red_s[par][w][tid];
          atomicAdd((tid == 0 ? a.dg : tid == 1 ? a.dbeta : a.dlam) + tk, s);
        }
      }
      par ^= 1;
      cur = nxt;
    }
  }
  if (a.dh0) {
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int c = 0; c < kTbCL; ++c)
        a.dh0[((static_cast<size_t>(bb) * H + h) * DK + r0 + i) * DV + c0 + c] = dS[i][c];
  }
}

template <typename TIn, int DK>
cudaError_t launch_tb(const ChunkBwdArgs& a, float* ckpt, float* scratch, cudaStream_t stream) {
  const dim3 grid(a.dv_dim / kTbCols, a.H, a.B);
  token_bwd_kernel<TIn, DK><<<grid, kTbThreads, 0, stream>>>(a, ckpt, scratch);
  return cudaGetLastError();
}

}  // namespace

size_t token_bwd_workspace_bytes(int B, int T, int H, int dk, int dv) {
  const size_t ctas = static_cast<size_t>(B) * H * (dv / kTbCols);
  const size_t nc = static_cast<size_t>((T + kTbChunk - 1) / kTbChunk);
  const size_t per = static_cast<size_t>(dk) * kTbCols * sizeof(float);
  return kChunkWorkspaceBytes + ctas * nc * per + ctas * kTbChunk * per;
}

cudaError_t launch_token_bwd(const ChunkBwdArgs& a, bool f32, cudaStream_t stream) {
  if ((a.dk_dim != 64 && a.dk_dim != 128) || a.dv_dim % kTbCols != 0) return cudaErrorInvalidValue;
  const size_t ctas = static_cast<size_t>(a.B) * a.H * (a.dv_dim / kTbCols);
  const size_t nc = static_cast<size_t>((a.T + kTbChunk - 1) / kTbChunk);
  const size_t per = static_cast<size_t>(a.dk_dim) * kTbCols;
  float* ckpt = reinterpret_cast<float*>(static_cast<unsigned char*>(a.workspace) +
                                         kChunkWorkspaceBytes);
  float* scratch = ckpt + ctas * nc * per;
  const size_t rows = static_cast<size_t>(a.B) * a.T * a.H;
  const bool CH = a.flags & 1u, ER = a.flags & 2u, WR = a.flags & 4u, QM = a.flags & 8u;
  cudaError_t err = cudaSuccess;
  // everything that sums over the column blocks starts from zero
  auto zero = [&](void* p, size_t bytes) {
    if (err == cudaSuccess && p) err = cudaMemsetAsync(p, 0, bytes, stream);
  };
  zero(a.dq, rows * a.dk_dim * 4);
  zero(a.dk, rows * a.dk_dim * 4);
  zero(a.dg, rows * (CH ? a.dk_dim : 1) * 4);
  if (ER) zero(a.db, rows * a.dk_dim * 4);
  if (!(ER && WR)) zero(a.dbeta, rows * 4);
  if (QM) zero(a.dlam, rows * 4);
  (void)WR;
  if (err != cudaSuccess) return err;
  if (a.dk_dim == 64)
    return f32 ? launch_tb<float, 64>(a, ckpt, scratch, stream)
               : launch_tb<__nv_bfloat16, 64>(a, ckpt, scratch, stream);
  return f32 ? launch_tb<float, 128>(a, ckpt, scratch, stream)
             : launch_tb<__nv_bfloat16, 128>(a, ckpt, scratch, stream);
}

}  // namespace gdr
