// Token-order scan for the write strength per value channel (the README
// variant of LLMs from scratch ch. 11, section 11.3), bf16 or fp32 inputs:
//
//   S~  = alpha_t S_{t-1}                          alpha_t = exp(g_t), one per head
//   r   = S~^T k_t                                 (d_v)
//   S_t = S~ + k_t (beta_t (.) (v_t - r))^T         beta_t in R^{d_v}
//   o_t = S_t^T (scale q_t)
//
// With beta per value channel every column of S follows its own affine map
// (section 11.4), so no (I + T)^{-1} is shared by the columns of a chunk; the
// state stays in fp32 registers and the tokens are walked in order. The work
// is a few d_k x d_v products per token-head on the FP32 pipe.
//
// Layout: one CTA per (batch, head, 4 * NW * CL value columns), NW warps. Eight
// lanes share a column: lane i of the group holds key rows i*R .. i*R+R-1
// (R = d_k / 8) of CL columns, and the column sums (S^T k, S^T q) are
// three-step butterflies inside the group. One pass over the state per token
// does the write and both sums that read the new state (o_t and the next
// token's prediction), so each token waits on one butterfly, not two. Tokens
// come in blocks of kTB: the next block's q, k, v, beta and g are loaded into
// registers while
// the current one is processed from shared memory (fp32, q and k padded so the
// eight lanes of a group read eight different bank quads), and o goes out one
// block at a time with 16-byte stores. Tokens past T are zero-filled with
// alpha = 1, which leaves S unchanged.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"

namespace gdr {
namespace {

constexpr int kTB = 32;  // tokens per block

template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kPerVec = 4;
  __device__ static void to_f32(const uint4& u, float* x) {
    x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
  }
  __device__ static uint4 from_f32(const float* x) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                      __float_as_uint(x[3]));
  }
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kPerVec = 8;
  __device__ static void to_f32(const uint4& u, float* x) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static uint4 from_f32(const float* x) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <typename T, int DK, int CL, int NW>
struct VBLayout {
  static constexpr int kThreads = 32 * NW;
  static constexpr int R = DK / 8;               // key rows per lane
  static constexpr int kSeg = R + 4;             // padded floats per lane segment
  static constexpr int kRow = 8 * kSeg;          // one token's q or k
  static constexpr int kCols = 4 * NW * CL;      // value columns per CTA
  static constexpr int E = Elem<T>::kPerVec;
  // per-thread 16-byte loads of one block
  static constexpr int kQKVecs = kTB * DK / E;                // per tensor
  static constexpr int kQKPer = (kQKVecs + kThreads - 1) / kThreads;
  static constexpr int kVVecs = kTB * kCols / E;
  static constexpr int kBVecs = kTB * kCols / 4;              // beta is fp32
  static constexpr int kVPer = (kVVecs + kThreads - 1) / kThreads;
  static constexpr int kBPer = (kBVecs + kThreads - 1) / kThreads;
  // shared memory (floats)
  static constexpr int oK = 0;
  static constexpr int oQ = oK + kTB * kRow;
  static constexpr int oV = oQ + kTB * kRow;
  static constexpr int oB = oV + kTB * kCols;
  static constexpr int oO = oB + kTB * kCols;
  static constexpr int oA = oO + kTB * kCols;
  static constexpr int floats = oA + kTB;
  static constexpr size_t bytes = static_cast<size_t>(floats) * 4;
};

template <typename T, int DK, int DV, int CL, int NW>
__global__ void __launch_bounds__(32 * NW)
    value_beta_scan_kernel(const T* __restrict__ q, const T* __restrict__ k,
                           const T* __restrict__ v, const float* __restrict__ g,
                           const float* __restrict__ beta, const float* h0, T* __restrict__ o,
                           float* hT, int Tn, int H, float scale) {
  using L = VBLayout<T, DK, CL, NW>;
  using EL = Elem<T>;
  constexpr int kVBThreads = L::kThreads;
  constexpr int R = L::R, E = L::E;
  extern __shared__ __align__(16) float sm[];
  float* sK = sm + L::oK;
  float* sQ = sm + L::oQ;
  float* sV = sm + L::oV;
  float* sB = sm + L::oB;
  float* sO = sm + L::oO;
  float* sA = sm + L::oA;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = lane >> 3, li = lane & 7;
  // this lane's R key rows of token t's q or k (fp32, padded segment)
  auto load_row = [&](const float* base, int t, float (&x)[R]) {
    const float* p = base + t * L::kRow + li * L::kSeg;
#pragma unroll
    for (int i = 0; i < R; i += 4) {
      const float4 a = *reinterpret_cast<const float4*>(p + i);
      x[i] = a.x; x[i + 1] = a.y; x[i + 2] = a.z; x[i + 3] = a.w;
    }
  };
  // sum over the eight lanes of a group (every lane gets it)
  auto group_sum = [](float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    return x;
  };
  const int bh = blockIdx.y, bb = bh / H, h = bh % H;
  const int col0 = blockIdx.x * L::kCols;
  const int my_col = (warp * 4 + grp) * CL;   // first of this group's columns in the CTA
  const int row0 = li * R;
  const int n_blocks = (Tn + kTB - 1) / kTB;

  // state: rows row0 .. row0+R-1, columns col0 + my_col .. +CL-1
  float S[R][CL];
  {
    const float* src = h0 ? h0 + (static_cast<size_t>(bh) * DK + row0) * DV + col0 + my_col : nullptr;
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int c = 0; c < CL; ++c) S[i][c] = src ? src[static_cast<size_t>(i) * DV + c] : 0.f;
  }

  // raw block loads (16 bytes each) kept in registers until the block is staged
  uint4 rk[L::kQKPer], rq[L::kQKPer], rv[L::kVPer];
  float4 rb[L::kBPer];
  float rg = 0.f;
  auto load_block = [&](int blk) {
    const int t0 = blk * kTB;
#pragma unroll
    for (int u = 0; u < L::kQKPer; ++u) {
      const int id = tid + u * kVBThreads, t = id / (DK / E), c = (id % (DK / E)) * E;
      rk[u] = make_uint4(0, 0, 0, 0);
      rq[u] = make_uint4(0, 0, 0, 0);
      if (id < L::kQKVecs && t0 + t < Tn) {
        const size_t off = ((static_cast<size_t>(bb) * Tn + t0 + t) * H + h) * DK + c;
        rk[u] = __ldg(reinterpret_cast<const uint4*>(k + off));
        rq[u] = __ldg(reinterpret_cast<const uint4*>(q + off));
      }
    }
#pragma unroll
    for (int u = 0; u < L::kVPer; ++u) {
      const int id = tid + u * kVBThreads, t = id / (L::kCols / E), c = (id % (L::kCols / E)) * E;
      rv[u] = make_uint4(0, 0, 0, 0);
      if (id < L::kVVecs && t0 + t < Tn)
        rv[u] = __ldg(reinterpret_cast<const uint4*>(
            v + ((static_cast<size_t>(bb) * Tn + t0 + t) * H + h) * DV + col0 + c));
    }
#pragma unroll
    for (int u = 0; u < L::kBPer; ++u) {
      const int id = tid + u * kVBThreads, t = id / (L::kCols / 4), c = (id % (L::kCols / 4)) * 4;
      rb[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (id < L::kBVecs && t0 + t < Tn)
        rb[u] = __ldg(reinterpret_cast<const float4*>(
            beta + ((static_cast<size_t>(bb) * Tn + t0 + t) * H + h) * DV + col0 + c));
    }
    rg = 0.f;
    if (tid < kTB && t0 + tid < Tn) rg = __ldg(g + (static_cast<size_t>(bb) * Tn + t0 + tid) * H + h);
  };
  auto stage_block = [&]() {
#pragma unroll
    for (int u = 0; u < L::kQKPer; ++u) {
      const int id = tid + u * kVBThreads, t = id / (DK / E), c = (id % (DK / E)) * E;
      if (id < L::kQKVecs) {
        float xk[E], xq[E];
        EL::to_f32(rk[u], xk);
        EL::to_f32(rq[u], xq);
        // channel c + j lives in lane segment (c + j) / R at position (c + j) % R;
        // E divides R, so one vector stays inside one segment
        const int at = t * L::kRow + (c / R) * L::kSeg + c % R;
#pragma unroll
        for (int j = 0; j < E; j += 4) {
          *reinterpret_cast<float4*>(sK + at + j) = make_float4(xk[j], xk[j + 1], xk[j + 2], xk[j + 3]);
          *reinterpret_cast<float4*>(sQ + at + j) = make_float4(xq[j], xq[j + 1], xq[j + 2], xq[j + 3]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < L::kVPer; ++u) {
      const int id = tid + u * kVBThreads, t = id / (L::kCols / E), c = (id % (L::kCols / E)) * E;
      if (id < L::kVVecs) {
        float x[E];
        EL::to_f32(rv[u], x);
#pragma unroll
        for (int j = 0; j < E; j += 4)
          *reinterpret_cast<float4*>(sV + t * L::kCols + c + j) =
              make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
      }
    }
#pragma unroll
    for (int u = 0; u < L::kBPer; ++u) {
      const int id = tid + u * kVBThreads, t = id / (L::kCols / 4), c = (id % (L::kCols / 4)) * 4;
      if (id < L::kBVecs) *reinterpret_cast<float4*>(sB + t * L::kCols + c) = rb[u];
    }
    if (tid < kTB) sA[tid] = expf(rg);   // zero-filled tokens get alpha = 1
  };

  load_block(0);
  for (int blk = 0; blk < n_blocks; ++blk) {
    __syncthreads();   // the previous block is done with shared memory
    stage_block();
    __syncthreads();
    if (blk + 1 < n_blocks) load_block(blk + 1);

    // r = S^T k of the block's first token; inside the block one pass over the
    // state per token does the write of token t and both column sums that
    // follow it (S_t^T q_t for o_t and S_t^T k_{t+1} for the next token)
    float r[CL], kr[R];
    load_row(sK, 0, kr);
#pragma unroll
    for (int c = 0; c < CL; ++c) {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int i = 0; i < R; i += 2) {
        a0 = fmaf(kr[i], S[i][c], a0);
        a1 = fmaf(kr[i + 1], S[i + 1][c], a1);
      }
      r[c] = group_sum(a0 + a1);
    }
#pragma unroll 2
    for (int t = 0; t < kTB; ++t) {
      float kn[R], qr[R];
      load_row(sQ, t, qr);
      const bool more = t + 1 < kTB;
      load_row(sK, more ? t + 1 : t, kn);
      const float alpha = sA[t];
#pragma unroll
      for (int c = 0; c < CL; ++c) {
        // S~^T k = alpha S^T k
        const float d = sB[t * L::kCols + my_col + c] * (sV[t * L::kCols + my_col + c] - alpha * r[c]);
        float y0 = 0.f, y1 = 0.f, n0 = 0.f, n1 = 0.f;
#pragma unroll
        for (int i = 0; i < R; i += 2) {
          S[i][c] = fmaf(alpha, S[i][c], kr[i] * d);
          S[i + 1][c] = fmaf(alpha, S[i + 1][c], kr[i + 1] * d);
          y0 = fmaf(qr[i], S[i][c], y0);
          y1 = fmaf(qr[i + 1], S[i + 1][c], y1);
          n0 = fmaf(kn[i], S[i][c], n0);
          n1 = fmaf(kn[i + 1], S[i + 1][c], n1);
        }
        float y = y0 + y1, n = n0 + n1;
#pragma unroll
        for (int m = 1; m < 8; m <<= 1) {
          y += __shfl_xor_sync(0xffffffffu, y, m);
          n += __shfl_xor_sync(0xffffffffu, n, m);
        }
        r[c] = n;   // unused after the block's last token
        if (li == 0) sO[t * L::kCols + my_col + c] = scale * y;
      }
#pragma unroll
      for (int i = 0; i < R; ++i) kr[i] = kn[i];
    }
    __syncthreads();
    // o of this block: [kTB][kCols] from shared memory, 16-byte stores
    const int t0 = blk * kTB;
#pragma unroll
    for (int u = 0; u < L::kVPer; ++u) {
      const int id = tid + u * kVBThreads, t = id / (L::kCols / E), c = (id % (L::kCols / E)) * E;
      if (id < L::kVVecs && t0 + t < Tn) {
        float x[E];
#pragma unroll
        for (int j = 0; j < E; ++j) x[j] = sO[t * L::kCols + c + j];
        *reinterpret_cast<uint4*>(o + ((static_cast<size_t>(bb) * Tn + t0 + t) * H + h) * DV +
                                  col0 + c) = EL::from_f32(x);
      }
    }
  }

  if (hT) {
    float* dst = hT + (static_cast<size_t>(bh) * DK + row0) * DV + col0 + my_col;
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int c = 0; c < CL; ++c) dst[static_cast<size_t>(i) * DV + c] = S[i][c];
  }
}

template <typename T, int DK, int DV, int CL, int NW>
cudaError_t launch_shape(const ValueBetaArgs& a, cudaStream_t stream) {
  using L = VBLayout<T, DK, CL, NW>;
  static_assert(DV % L::kCols == 0, "value columns split evenly over CTAs");
  auto kern = value_beta_scan_kernel<T, DK, DV, CL, NW>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L::bytes));
  if (err != cudaSuccess) return err;
  const dim3 grid(DV / L::kCols, static_cast<unsigned>(a.B) * a.H);
  kern<<<grid, L::kThreads, L::bytes, stream>>>(
      static_cast<const T*>(a.q), static_cast<const T*>(a.k), static_cast<const T*>(a.v), a.g,
      a.beta, a.h0, static_cast<T*>(a.o), a.hT, a.T, a.H, a.scale);
  return cudaGetLastError();
}

// Two columns per lane group and four warps per CTA (32 value columns): of
// 1/2/4 columns and 2/4/8 warps this measured fastest on 4 x 4096 x 16 x 128.
template <typename T, int DK, int DV>
cudaError_t launch_typed(const ValueBetaArgs& a, cudaStream_t stream) {
  return launch_shape<T, DK, DV, 2, 4>(a, stream);
}

template <typename T>
cudaError_t launch_dims(const ValueBetaArgs& a, int dk, int dv, cudaStream_t stream) {
  if (dk == 64 && dv == 64) return launch_typed<T, 64, 64>(a, stream);
  if (dk == 64 && dv == 128) return launch_typed<T, 64, 128>(a, stream);
  if (dk == 128 && dv == 64) return launch_typed<T, 128, 64>(a, stream);
  if (dk == 128 && dv == 128) return launch_typed<T, 128, 128>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_value_beta_scan(const ValueBetaArgs& a, int dk, int dv, bool f32,
                                   cudaStream_t stream) {
  return f32 ? launch_dims<float>(a, dk, dv, stream)
             : launch_dims<__nv_bfloat16>(a, dk, dv, stream);
}

}  // namespace gdr
