// Chunkwise backward of the gated delta rule (Gated DeltaNet-2 notes, key design
// 3), every flag but the write strength per value channel, fp32 arithmetic.
//
// For loss gradients dO (and dS_T) it returns dq, dk, dv, dg, dbeta, dlam, db,
// dw and dh0 through four kernels over fp32 records in the workspace:
//   1. bwd_chunk_prep  (one CTA per chunk): the chunk's forward quantities as
//      the chunk algebra defines them -- G (in-chunk cumsum of g), gamma, the
//      erase / write vectors E, Z, K_bar = k / gamma, E_bar = gamma E,
//      T = tril(E_bar K_bar^T, -1), A = (I + T)^{-1} (forward substitution),
//      Y = A E_bar, U = A Z, Q_gamma = s gamma q, K_tail = gamma_C / gamma k,
//      A_qk = tril(Q_gamma K_bar^T, 0);
//   2. bwd_state_pass  (one CTA per (batch, head, 32 value columns)): S_n and
//      W_n = U - Y S_n of every chunk, S_{n+1} = Diag(gamma_C) S_n + K_tail^T W_n;
//   3. bwd_dstate_pass (same grid, chunks in reverse): dW_n = A_qk^T dO_n +
//      K_tail dS_{n+1}, dS_n = Diag(gamma_C) dS_{n+1} + Q_gamma^T dO_n - Y^T dW_n,
//      keeping dS_{n+1} and dW_n of every chunk; dh0 = dS_0;
//   4. bwd_chunk_grad  (one CTA per chunk): dA_qk, dQ_gamma, dK_bar, dK_tail,
//      dY, the notes' gate-aware dA = dU Z^T + dY E_bar^T, dZ, dE_bar, the
//      notes' adjoint of the triangular inverse dT = -tril(A^T dA A^T, -1), then
//      the chain through the decay factors, the cumulative sum and the erase /
//      write vectors to the inputs.
// The products run on the FP32 pipe from the records (each CTA's operands stay
// in L2 while it works); chunks past the end are zero-filled, which leaves every
// product and the reverse cumulative sum exact for the valid rows.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"

namespace gdr {
namespace {

constexpr int kC = 64;            // chunk length
constexpr int kBwdThreads = 256;

// C (m, n) = alpha sum_k A(m, k) B(k, n) + beta C (m, n), every thread of the
// CTA; operands by strides (a transpose is a stride swap). mask: 0 none,
// 1 keep n <= m, 2 keep n < m (others written as zero).
__device__ void block_gemm(float* C, int ldc, const float* A, int sam, int sak, const float* B,
                           int sbk, int sbn, int M, int N, int K, float alpha, float beta,
                           int mask = 0) {
  for (int idx = threadIdx.x; idx < M * N; idx += blockDim.x) {
    const int m = idx / N, n = idx % N;
    float acc = 0.f;
    if (!(mask == 1 && n > m) && !(mask == 2 && n >= m)) {
      const float* a = A + static_cast<size_t>(m) * sam;
      const float* b = B + static_cast<size_t>(n) * sbn;
#pragma unroll 4
      for (int k = 0; k < K; ++k) acc = fmaf(a[static_cast<size_t>(k) * sak], b[static_cast<size_t>(k) * sbk], acc);
    }
    float* c = C + static_cast<size_t>(m) * ldc + n;
    *c = alpha * acc + (beta != 0.f ? beta * *c : 0.f);
  }
  __syncthreads();
}

template <typename T>
__device__ __forceinline__ float ldx(const T* p, size_t i);
template <>
__device__ __forceinline__ float ldx<float>(const float* p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ldx<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}

// offsets (floats) of one chunk's record
struct Rec {
  int dk, dv;
  __host__ __device__ size_t mk() const { return static_cast<size_t>(kC) * dk; }
  __host__ __device__ size_t mv() const { return static_cast<size_t>(kC) * dv; }
  __host__ __device__ size_t oG() const { return 0; }
  __host__ __device__ size_t oGam() const { return oG() + mk(); }
  __host__ __device__ size_t oE() const { return oGam() + mk(); }
  __host__ __device__ size_t oKb() const { return oE() + mk(); }
  __host__ __device__ size_t oEb() const { return oKb() + mk(); }
  __host__ __device__ size_t oQg() const { return oEb() + mk(); }
  __host__ __device__ size_t oKt() const { return oQg() + mk(); }
  __host__ __device__ size_t oY() const { return oKt() + mk(); }
  __host__ __device__ size_t oX() const { return oY() + mk(); }       // the erase input x
  __host__ __device__ size_t oZ() const { return oX() + mk(); }
  __host__ __device__ size_t oU() const { return oZ() + mv(); }
  __host__ __device__ size_t oA() const { return oU() + mv(); }
  __host__ __device__ size_t oAqk() const { return oA() + kC * kC; }
  __host__ __device__ size_t oT() const { return oAqk() + kC * kC; }
  __host__ __device__ size_t size() const { return oT() + kC * kC; }
};

struct BwdPtrs {
  const void *q, *k, *v, *dO;
  const float *g, *beta, *lam;
  const void *b, *w;
  const float *h0, *dhT;
  float *d_q, *d_k, *d_v, *d_g, *d_beta, *d_lam, *d_b, *d_w, *d_h0;   // outputs
  float* rec;      // [chunks] records
  float* S;        // [B, H, Nc, dk, dv] state entering each chunk
  float* W;        // [B, H, Nc, 64, dv]
  float* dS;       // [B, H, Nc, dk, dv] gradient leaving each chunk (dS_{n+1})
  float* dW;       // [B, H, Nc, 64, dv]
  float* scr;      // [chunks] per-chunk scratch of the gradient kernel
  int B, T, H, dk, dv, Nc;
  unsigned flags;
  float scale;
};

__device__ __forceinline__ size_t chunk_id(const BwdPtrs& p, int bb, int h, int n) {
  return (static_cast<size_t>(bb) * p.H + h) * p.Nc + n;
}

// ---------------------------------------------------------------- 1. records
template <typename T>
__global__ void __launch_bounds__(kBwdThreads) bwd_chunk_prep(const BwdPtrs p) {
  const Rec R{p.dk, p.dv};
  const int cid = blockIdx.x;
  const int n = cid % p.Nc, bh = cid / p.Nc, h = bh % p.H, bb = bh / p.H;
  const int t0 = n * kC, Lr = min(kC, p.T - t0);
  const int dk = p.dk, dv = p.dv, tid = threadIdx.x;
  float* r = p.rec + static_cast<size_t>(cid) * R.size();
  const bool CH = p.flags & 1u, ER = p.flags & 2u, WR = p.flags & 4u, QM = p.flags & 8u;
  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  const T* v = static_cast<const T*>(p.v);
  const T* bg = static_cast<const T*>(p.b);
  const T* wg = static_cast<const T*>(p.w);
  auto tok = [&](int i) { return (static_cast<size_t>(bb) * p.T + t0 + i) * p.H + h; };
  // G: in-chunk inclusive cumsum per key channel (scalar gates broadcast)
  for (int c = tid; c < dk; c += blockDim.x) {
    float acc = 0.f;
    for (int i = 0; i < kC; ++i) {
      if (i < Lr) acc += CH ? p.g[tok(i) * dk + c] : p.g[tok(i)];
      r[R.oG() + i * dk + c] = acc;
      r[R.oGam() + i * dk + c] = expf(acc);
    }
  }
  __syncthreads();
  // E, x (erase input), K_bar, E_bar, Q_gamma, K_tail
  for (int e = tid; e < kC * dk; e += blockDim.x) {
    const int i = e / dk, c = e % dk;
    float qv = 0.f, kv = 0.f, x = 0.f, E = 0.f;
    if (i < Lr) {
      qv = ldx(q, tok(i) * dk + c);
      kv = ldx(k, tok(i) * dk + c);
      x = QM ? kv + p.lam[tok(i)] * qv : kv;
      E = ER ? ldx(bg, tok(i) * dk + c) * x : p.beta[tok(i)] * x;
    }
    const float gam = r[R.oGam() + e], gC = r[R.oGam() + (kC - 1) * dk + c];
    r[R.oX() + e] = x;
    r[R.oE() + e] = E;
    r[R.oKb() + e] = kv / gam;
    r[R.oEb() + e] = gam * E;
    r[R.oQg() + e] = p.scale * gam * qv;
    r[R.oKt() + e] = gC / gam * kv;
  }
  for (int e = tid; e < kC * dv; e += blockDim.x) {
    const int i = e / dv, c = e % dv;
    float z = 0.f;
    if (i < Lr) {
      const float vv = ldx(v, tok(i) * dv + c);
      z = WR ? ldx(wg, tok(i) * dv + c) * vv : p.beta[tok(i)] * vv;
    }
    r[R.oZ() + e] = z;
  }
  __syncthreads();
  // T = tril(E_bar K_bar^T, -1), A_qk = tril(Q_gamma K_bar^T, 0)
  block_gemm(r + R.oT(), kC, r + R.oEb(), dk, 1, r + R.oKb(), 1, dk, kC, kC, dk, 1.f, 0.f, 2);
  block_gemm(r + R.oAqk(), kC, r + R.oQg(), dk, 1, r + R.oKb(), 1, dk, kC, kC, dk, 1.f, 0.f, 1);
  // A = (I + T)^{-1}: row r of (I + T) A = I gives A_r = e_r - sum_{i<r} T_ri A_i;
  // thread c owns column c
  if (tid < kC) {
    float* A = r + R.oA();
    const float* Tm = r + R.oT();
    for (int i = 0; i < kC; ++i) {
      float acc = (i == tid) ? 1.f : 0.f;
      for (int j = 0; j < i; ++j) acc = fmaf(-Tm[i * kC + j], A[j * kC + tid], acc);
      A[i * kC + tid] = acc;
    }
  }
  __syncthreads();
  // Y = A E_bar, U = A Z
  block_gemm(r + R.oY(), dk, r + R.oA(), kC, 1, r + R.oEb(), dk, 1, kC, dk, kC, 1.f, 0.f);
  block_gemm(r + R.oU(), dv, r + R.oA(), kC, 1, r + R.oZ(), dv, 1, kC, dv, kC, 1.f, 0.f);
}

// ------------------------------------------------------- 2. forward states
constexpr int kSlice = 32;

__global__ void __launch_bounds__(kBwdThreads) bwd_state_pass(const BwdPtrs p) {
  const Rec R{p.dk, p.dv};
  const int col0 = blockIdx.x * kSlice, h = blockIdx.y, bb = blockIdx.z;
  const int dk = p.dk, dv = p.dv, tid = threadIdx.x;
  extern __shared__ float sm[];
  float* S = sm;                       // [dk][kSlice]
  float* Wl = S + dk * kSlice;         // [64][kSlice]
  for (int e = tid; e < dk * kSlice; e += blockDim.x) {
    const int i = e / kSlice, c = e % kSlice;
    S[e] = p.h0 ? p.h0[((static_cast<size_t>(bb) * p.H + h) * dk + i) * dv + col0 + c] : 0.f;
  }
  __syncthreads();
  for (int n = 0; n < p.Nc; ++n) {
    const size_t cid = chunk_id(p, bb, h, n);
    const float* r = p.rec + cid * R.size();
    float* Sg = p.S + cid * dk * dv;
    float* Wg = p.W + cid * kC * dv;
    for (int e = tid; e < dk * kSlice; e += blockDim.x)
      Sg[(e / kSlice) * dv + col0 + e % kSlice] = S[e];
    // W = U - Y S
    for (int e = tid; e < kC * kSlice; e += blockDim.x) {
      const int i = e / kSlice, c = e % kSlice;
      float acc = r[R.oU() + i * dv + col0 + c];
      for (int j = 0; j < dk; ++j) acc = fmaf(-r[R.oY() + i * dk + j], S[j * kSlice + c], acc);
      Wl[e] = acc;
      Wg[i * dv + col0 + c] = acc;
    }
    __syncthreads();
    // S' = Diag(gamma_C) S + K_tail^T W
    for (int e = tid; e < dk * kSlice; e += blockDim.x) {
      const int i = e / kSlice, c = e % kSlice;
      float acc = r[R.oGam() + (kC - 1) * dk + i] * S[e];
      for (int j = 0; j < kC; ++j) acc = fmaf(r[R.oKt() + j * dk + i], Wl[j * kSlice + c], acc);
      S[e] = acc;   // each thread owns its elements; W is read from Wl only
    }
    __syncthreads();
  }
}

// ------------------------------------------------------- 3. reverse states
template <typename T>
__global__ void __launch_bounds__(kBwdThreads) bwd_dstate_pass(const BwdPtrs p) {
  const Rec R{p.dk, p.dv};
  const int col0 = blockIdx.x * kSlice, h = blockIdx.y, bb = blockIdx.z;
  const int dk = p.dk, dv = p.dv, tid = threadIdx.x;
  const T* dO = static_cast<const T*>(p.dO);
  extern __shared__ float sm[];
  float* dS = sm;                      // [dk][kSlice]
  float* dWl = dS + dk * kSlice;       // [64][kSlice]
  float* dOl = dWl + kC * kSlice;      // [64][kSlice]
  for (int e = tid; e < dk * kSlice; e += blockDim.x) {
    const int i = e / kSlice, c = e % kSlice;
    dS[e] = p.dhT ? p.dhT[((static_cast<size_t>(bb) * p.H + h) * dk + i) * dv + col0 + c] : 0.f;
  }
  __syncthreads();
  for (int n = p.Nc - 1; n >= 0; --n) {
    const size_t cid = chunk_id(p, bb, h, n);
    const float* r = p.rec + cid * R.size();
    const int t0 = n * kC, Lr = min(kC, p.T - t0);
    float* dSg = p.dS + cid * dk * dv;
    float* dWg = p.dW + cid * kC * dv;
    for (int e = tid; e < dk * kSlice; e += blockDim.x)
      dSg[(e / kSlice) * dv + col0 + e % kSlice] = dS[e];
    for (int e = tid; e < kC * kSlice; e += blockDim.x) {
      const int i = e / kSlice, c = e % kSlice;
      dOl[e] = i < Lr ? ldx(dO, ((static_cast<size_t>(bb) * p.T + t0 + i) * p.H + h) * dv + col0 + c)
                      : 0.f;
    }
    __syncthreads();
    // dW = A_qk^T dO + K_tail dS'
    for (int e = tid; e < kC * kSlice; e += blockDim.x) {
      const int i = e / kSlice, c = e % kSlice;
      float acc = 0.f;
      for (int j = 0; j < kC; ++j) acc = fmaf(r[R.oAqk() + j * kC + i], dOl[j * kSlice + c], acc);
      for (int j = 0; j < dk; ++j) acc = fmaf(r[R.oKt() + i * dk + j], dS[j * kSlice + c], acc);
      dWl[e] = acc;
      dWg[i * dv + col0 + c] = acc;
    }
    __syncthreads();
    // dS = Diag(gamma_C) dS' + Q_gamma^T dO - Y^T dW
    for (int e = tid; e < dk * kSlice; e += blockDim.x) {
      const int i = e / kSlice, c = e % kSlice;
      float acc = r[R.oGam() + (kC - 1) * dk + i] * dS[e];
      for (int j = 0; j < kC; ++j) {
        acc = fmaf(r[R.oQg() + j * dk + i], dOl[j * kSlice + c], acc);
        acc = fmaf(-r[R.oY() + j * dk + i], dWl[j * kSlice + c], acc);
      }
      dS[e] = acc;
    }
    __syncthreads();
  }
  if (p.d_h0)
    for (int e = tid; e < dk * kSlice; e += blockDim.x)
      p.d_h0[((static_cast<size_t>(bb) * p.H + h) * dk + e / kSlice) * dv + col0 + e % kSlice] = dS[e];
}

// ------------------------------------------------------- 4. gradients
struct Scr {
  int dk, dv;
  __host__ __device__ size_t mk() const { return static_cast<size_t>(kC) * dk; }
  __host__ __device__ size_t mv() const { return static_cast<size_t>(kC) * dv; }
  __host__ __device__ size_t oDAqk() const { return 0; }
  __host__ __device__ size_t oDA() const { return oDAqk() + kC * kC; }
  __host__ __device__ size_t oX() const { return oDA() + kC * kC; }
  __host__ __device__ size_t oDT() const { return oX() + kC * kC; }
  __host__ __device__ size_t oDQg() const { return oDT() + kC * kC; }
  __host__ __device__ size_t oDKb() const { return oDQg() + mk(); }
  __host__ __device__ size_t oDKt() const { return oDKb() + mk(); }
  __host__ __device__ size_t oDY() const { return oDKt() + mk(); }
  __host__ __device__ size_t oDEb() const { return oDY() + mk(); }
  __host__ __device__ size_t oDG() const { return oDEb() + mk(); }
  __host__ __device__ size_t oDZ() const { return oDG() + mk(); }
  __host__ __device__ size_t oDO() const { return oDZ() + mv(); }
  __host__ __device__ size_t oDgC() const { return oDO() + mv(); }
  __host__ __device__ size_t size() const { return oDgC() + dk; }
};

template <typename T>
__global__ void __launch_bounds__(kBwdThreads) bwd_chunk_grad(const BwdPtrs p) {
  const Rec R{p.dk, p.dv};
  const Scr Q{p.dk, p.dv};
  const int cid = blockIdx.x;
  const int n = cid % p.Nc, bh = cid / p.Nc, h = bh % p.H, bb = bh / p.H;
  const int t0 = n * kC, Lr = min(kC, p.T - t0);
  const int dk = p.dk, dv = p.dv, tid = threadIdx.x;
  const bool CH = p.flags & 1u, ER = p.flags & 2u, WR = p.flags & 4u, QM = p.flags & 8u;
  const float* r = p.rec + static_cast<size_t>(cid) * R.size();
  float* s = p.scr + static_cast<size_t>(cid) * Q.size();
  const float* S = p.S + static_cast<size_t>(cid) * dk * dv;
  const float* dSn = p.dS + static_cast<size_t>(cid) * dk * dv;
  const float* W = p.W + static_cast<size_t>(cid) * kC * dv;
  const float* dW = p.dW + static_cast<size_t>(cid) * kC * dv;
  const T* dOg = static_cast<const T*>(p.dO);
  auto tok = [&](int i) { return (static_cast<size_t>(bb) * p.T + t0 + i) * p.H + h; };
  float* dO = s + Q.oDO();
  for (int e = tid; e < kC * dv; e += blockDim.x) {
    const int i = e / dv, c = e % dv;
    dO[e] = i < Lr ? ldx(dOg, tok(i) * dv + c) : 0.f;
  }
  // dgamma_C = rowsum(dS' (.) S)
  for (int c = tid; c < dk; c += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < dv; ++j) acc = fmaf(dSn[c * dv + j], S[c * dv + j], acc);
    s[Q.oDgC() + c] = acc;
  }
  __syncthreads();
  // dA_qk = tril(dO W^T, 0); dQ_gamma = dO S^T + dA_qk K_bar; dK_bar = dA_qk^T Q_gamma
  block_gemm(s + Q.oDAqk(), kC, dO, dv, 1, W, 1, dv, kC, kC, dv, 1.f, 0.f, 1);
  block_gemm(s + Q.oDQg(), dk, dO, dv, 1, S, 1, dv, kC, dk, dv, 1.f, 0.f);
  block_gemm(s + Q.oDQg(), dk, s + Q.oDAqk(), kC, 1, r + R.oKb(), dk, 1, kC, dk, kC, 1.f, 1.f);
  block_gemm(s + Q.oDKb(), dk, s + Q.oDAqk(), 1, kC, r + R.oQg(), dk, 1, kC, dk, kC, 1.f, 0.f);
  // dK_tail = W dS'^T; dY = -dW S^T
  block_gemm(s + Q.oDKt(), dk, W, dv, 1, dSn, 1, dv, kC, dk, dv, 1.f, 0.f);
  block_gemm(s + Q.oDY(), dk, dW, dv, 1, S, 1, dv, kC, dk, dv, -1.f, 0.f);
  // the notes' gate-aware dA = dU Z^T + dY E_bar^T (dU = dW)
  block_gemm(s + Q.oDA(), kC, dW, dv, 1, r + R.oZ(), 1, dv, kC, kC, dv, 1.f, 0.f);
  block_gemm(s + Q.oDA(), kC, s + Q.oDY(), dk, 1, r + R.oEb(), 1, dk, kC, kC, dk, 1.f, 1.f);
  // dZ = A^T dU; dE_bar = A^T dY
  block_gemm(s + Q.oDZ(), dv, r + R.oA(), 1, kC, dW, dv, 1, kC, dv, kC, 1.f, 0.f);
  block_gemm(s + Q.oDEb(), dk, r + R.oA(), 1, kC, s + Q.oDY(), dk, 1, kC, dk, kC, 1.f, 0.f);
  // the notes' adjoint of the inverse: dT = -tril(A^T dA A^T, -1)
  block_gemm(s + Q.oX(), kC, r + R.oA(), 1, kC, s + Q.oDA(), kC, 1, kC, kC, kC, 1.f, 0.f);
  block_gemm(s + Q.oDT(), kC, s + Q.oX(), kC, 1, r + R.oA(), 1, kC, kC, kC, kC, -1.f, 0.f, 2);
  // dE_bar += dT K_bar; dK_bar += dT^T E_bar
  block_gemm(s + Q.oDEb(), dk, s + Q.oDT(), kC, 1, r + R.oKb(), dk, 1, kC, dk, kC, 1.f, 1.f);
  block_gemm(s + Q.oDKb(), dk, s + Q.oDT(), 1, kC, r + R.oEb(), dk, 1, kC, dk, kC, 1.f, 1.f);
  // the decay factors: dG = gamma dgamma (+ gamma_C dgamma_C on the last row), with
  // dgamma = dE_bar E - dK_bar K_bar / gamma - dK_tail K_tail / gamma + dQ_gamma Q_gamma / gamma
  // and dgamma_C += sum_r dK_tail k / gamma; dq, dk, dE per element
  for (int c = tid; c < dk; c += blockDim.x) {
    float dgc = s[Q.oDgC() + c];
    const float gC = r[R.oGam() + (kC - 1) * dk + c];
    for (int i = 0; i < kC; ++i) {
      const size_t e = static_cast<size_t>(i) * dk + c;
      const float gam = r[R.oGam() + e];
      const float kv = r[R.oKb() + e] * gam;     // k = K_bar gamma
      dgc = fmaf(s[Q.oDKt() + e], kv / gam, dgc);
      const float dgam = s[Q.oDEb() + e] * r[R.oE() + e] - s[Q.oDKb() + e] * r[R.oKb() + e] / gam -
                         s[Q.oDKt() + e] * r[R.oKt() + e] / gam + s[Q.oDQg() + e] * r[R.oQg() + e] / gam;
      s[Q.oDG() + e] = gam * dgam;
    }
    s[Q.oDG() + (kC - 1) * dk + c] += gC * dgc;
    // reverse cumulative sum within the chunk: dg_i = sum_{r >= i} dG_r
    float acc = 0.f;
    for (int i = kC - 1; i >= 0; --i) {
      acc += s[Q.oDG() + static_cast<size_t>(i) * dk + c];
      s[Q.oDG() + static_cast<size_t>(i) * dk + c] = acc;
    }
  }
  __syncthreads();
  // key-side outputs per (row, channel)
  for (int e = tid; e < kC * dk; e += blockDim.x) {
    const int i = e / dk, c = e % dk;
    if (i >= Lr) continue;
    const float gam = r[R.oGam() + e], gC = r[R.oGam() + (kC - 1) * dk + c];
    const float dE = gam * s[Q.oDEb() + e];
    const float x = r[R.oX() + e];
    const float bta = p.beta ? p.beta[tok(i)] : 0.f;
    const float dx = ER ? ldx(static_cast<const T*>(p.b), tok(i) * dk + c) * dE : bta * dE;
    float dkv = s[Q.oDKb() + e] / gam + gC / gam * s[Q.oDKt() + e] + dx;
    float dqv = p.scale * gam * s[Q.oDQg() + e];
    if (QM) dqv += p.lam[tok(i)] * dx;
    p.d_k[tok(i) * dk + c] = dkv;
    p.d_q[tok(i) * dk + c] = dqv;
    if (ER) p.d_b[tok(i) * dk + c] = x * dE;
    if (CH) p.d_g[tok(i) * dk + c] = s[Q.oDG() + e];
  }
  // value-side outputs
  for (int e = tid; e < kC * dv; e += blockDim.x) {
    const int i = e / dv, c = e % dv;
    if (i >= Lr) continue;
    const float dZ = s[Q.oDZ() + e];
    const float vv = ldx(static_cast<const T*>(p.v), tok(i) * dv + c);
    if (WR) {
      p.d_v[tok(i) * dv + c] = ldx(static_cast<const T*>(p.w), tok(i) * dv + c) * dZ;
      p.d_w[tok(i) * dv + c] = vv * dZ;
    } else {
      p.d_v[tok(i) * dv + c] = p.beta[tok(i)] * dZ;
    }
  }
  // per-row outputs: scalar dg, dbeta, dlam
  if (tid < kC && tid < Lr) {
    const int i = tid;
    float dgs = 0.f, dbe = 0.f, dla = 0.f;
    for (int c = 0; c < dk; ++c) {
      const size_t e = static_cast<size_t>(i) * dk + c;
      dgs += s[Q.oDG() + e];
      const float dE = r[R.oGam() + e] * s[Q.oDEb() + e];
      if (!ER) dbe = fmaf(r[R.oX() + e], dE, dbe);
      if (QM) {
        const float dx = ER ? ldx(static_cast<const T*>(p.b), tok(i) * dk + c) * dE
                            : p.beta[tok(i)] * dE;
        dla = fmaf(ldx(static_cast<const T*>(p.q), tok(i) * dk + c), dx, dla);
      }
    }
    if (!WR)
      for (int c = 0; c < dv; ++c)
        dbe = fmaf(ldx(static_cast<const T*>(p.v), tok(i) * dv + c), s[Q.oDZ() + static_cast<size_t>(i) * dv + c], dbe);
    if (!CH) p.d_g[tok(i)] = dgs;
    if (p.d_beta) p.d_beta[tok(i)] = dbe;
    if (QM) p.d_lam[tok(i)] = dla;
  }
}

template <typename T>
cudaError_t launch_all(const BwdPtrs& p, cudaStream_t stream) {
  const int chunks = p.B * p.H * p.Nc;
  bwd_chunk_prep<T><<<chunks, kBwdThreads, 0, stream>>>(p);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const dim3 sgrid(p.dv / kSlice, p.H, p.B);
  const size_t sm2 = (static_cast<size_t>(p.dk) + kC) * kSlice * sizeof(float);
  bwd_state_pass<<<sgrid, kBwdThreads, sm2, stream>>>(p);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  const size_t sm3 = (static_cast<size_t>(p.dk) + 2 * kC) * kSlice * sizeof(float);
  bwd_dstate_pass<T><<<sgrid, kBwdThreads, sm3, stream>>>(p);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  bwd_chunk_grad<T><<<chunks, kBwdThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t chunk_bwd_workspace_bytes(int B, int T, int H, int dk, int dv) {
  const size_t nc = static_cast<size_t>((T + kC - 1) / kC);
  const size_t chunks = static_cast<size_t>(B) * H * nc;
  const Rec R{dk, dv};
  const Scr Q{dk, dv};
  const size_t floats = chunks * (R.size() + Q.size() + 2 * static_cast<size_t>(dk) * dv +
                                  2 * static_cast<size_t>(kC) * dv);
  return floats * sizeof(float);
}

cudaError_t launch_chunk_bwd(const ChunkBwdArgs& a, bool f32, cudaStream_t stream) {
  BwdPtrs p;
  p.q = a.q; p.k = a.k; p.v = a.v; p.dO = a.dO;
  p.g = a.g; p.beta = a.beta; p.lam = a.lam; p.b = a.b; p.w = a.w;
  p.h0 = a.h0; p.dhT = a.dhT;
  p.d_q = a.dq; p.d_k = a.dk; p.d_v = a.dv; p.d_g = a.dg; p.d_beta = a.dbeta; p.d_lam = a.dlam;
  p.d_b = a.db; p.d_w = a.dw; p.d_h0 = a.dh0;
  p.B = a.B; p.T = a.T; p.H = a.H; p.dk = a.dk_dim; p.dv = a.dv_dim;
  p.Nc = (a.T + kC - 1) / kC;
  p.flags = a.flags; p.scale = a.scale;
  const size_t chunks = static_cast<size_t>(p.B) * p.H * p.Nc;
  const Rec R{p.dk, p.dv};
  const Scr Q{p.dk, p.dv};
  float* base = static_cast<float*>(a.workspace);
  p.rec = base;
  p.scr = p.rec + chunks * R.size();
  p.S = p.scr + chunks * Q.size();
  p.dS = p.S + chunks * p.dk * p.dv;
  p.W = p.dS + chunks * p.dk * p.dv;
  p.dW = p.W + chunks * kC * p.dv;
  return f32 ? launch_all<float>(p, stream) : launch_all<__nv_bfloat16>(p, stream);
}

}  // namespace gdr
