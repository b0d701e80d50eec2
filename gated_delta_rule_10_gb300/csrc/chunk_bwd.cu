// Chunkwise backward of the gated delta rule (Gated DeltaNet-2 notes, key design
// 3), every flag but the write strength per value channel, fp32 arithmetic.
//
// For loss gradients dO (and dS_T) it returns dq, dk, dv, dg, dbeta, dlam, db,
// dw and dh0 through four kernels over fp32 records in the workspace:
//   1. bwd_chunk_prep  (one CTA per chunk): the chunk's forward quantities as
//      the chunk algebra defines them -- gamma = exp(in-chunk cumsum of g), the
//      erase / write vectors E, Z, K_bar = k / gamma, E_bar = gamma E,
//      T = tril(E_bar K_bar^T, -1), A = (I + T)^{-1} (forward substitution),
//      Y = A E_bar, U = A Z, Q_gamma = s gamma q, K_tail = gamma_C / gamma k,
//      A_qk = tril(Q_gamma K_bar^T, 0);
//   2. bwd_state_pass  (one CTA per (batch, head, 64 value columns)): S_n and
//      W_n = U - Y S_n of every chunk, S_{n+1} = Diag(gamma_C) S_n + K_tail^T W_n;
//   3. bwd_dstate_pass (same grid, chunks in reverse): dW_n = A_qk^T dO_n +
//      K_tail dS_{n+1}, dS_n = Diag(gamma_C) dS_{n+1} + Q_gamma^T dO_n - Y^T dW_n,
//      keeping dS_{n+1} and dW_n of every chunk; dh0 = dS_0;
//   4. bwd_chunk_grad  (one CTA per chunk): dA_qk, dQ_gamma, dK_bar, dK_tail,
//      dY, the notes' gate-aware dA = dU Z^T + dY E_bar^T, dZ, dE_bar, the
//      notes' adjoint of the triangular inverse dT = -tril(A^T dA A^T, -1), then
//      the chain through the decay factors, the cumulative sum and the erase /
//      write vectors to the inputs.
// The per-chunk kernels run their products on the tensor cores (warp-level MMA;
// for fp32 inputs every fp32 operand is split into tf32 hi + lo, about fp32
// accuracy; for bf16 inputs one tf32 product), their operands staged through
// shared memory a 32-wide K slice at a time; the state
// passes keep the state in MMA accumulators and multiply on warp-level MMAs
// with bf16 hi + lo split operands, the next chunk's operands copied in while
// the current one is used. Chunks
// past the end are zero-filled, which leaves every product and the reverse
// cumulative sum exact for the valid rows.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"

namespace gdr {
namespace {

constexpr int kC = 64;            // chunk length
constexpr int kBwdThreads = 256;
// The records hold K_bar = k / gamma and E_bar = gamma E with gamma = e^{G} taken
// from the chunk's first row, so an in-chunk log-decay sum below this leaves
// 1 / gamma outside the fp32 range (e^{88.7}) with margin; such a chunk is
// reported as GDR_ERR_RANGE in the status words ([1] = batch * H + head,
// [2] = chunk; the first report wins) and its gradients are not to be used.
constexpr float kBwdDecayFloor = -80.f;

constexpr int kKT = 32;           // K slice of the staged products
constexpr int kU = 4;             // elements per thread whose loads are issued together

__device__ __forceinline__ uint32_t sa32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 16-byte asynchronous copy global -> shared (both 16-byte aligned)
__device__ __forceinline__ void cp16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa32(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// fp32 -> tf32 hi + lo with x ~= hi + lo to ~2^-22 relative (round to nearest each)
__device__ __forceinline__ uint32_t tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = tf32_rna(x);
  lo = tf32_rna(x - __uint_as_float(hi));
}
// warp-level MMA, D = A (16 x 8, row) B (8 x 8, col) + D, tf32 operands, fp32 accumulation
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// C (m, n) = alpha sum_k A(m, k) B(k, n) + beta C (m, n) for M = 64 rows and
// N = 16 TN columns (64 or 128), by the whole CTA (256 threads = 8 warps, each a
// 16 WM x 32 tile of C in MMA accumulators). A and B are staged through shared
// memory one 32-wide K slice at a time with asynchronous 16-byte copies, the
// next slice in flight while the current one is used. Each operand keeps its
// global layout in shared memory: AK / BK say that A / B is contiguous along k
// (else along m / n); every base, stride and offset is a multiple of 4 floats.
// The products run on the tensor cores. With NP = 3 each fp32 operand is split
// into tf32 hi + lo and the three products lo*hi + hi*lo + hi*hi are accumulated
// in fp32, which keeps about fp32 accuracy (the dropped lo*lo term is ~2^-22
// relative); with NP = 1 the operands are rounded to tf32 (2^-11 relative) and
// hi*hi alone is accumulated.
// mask: 0 none, 1 keep n <= m, 2 keep n < m (others written as 0).
// Kept out of line: one body per layout instead of one per call site keeps the
// per-chunk kernels' code small enough for the instruction cache.
template <int NP, int TN, bool AK, bool BK>
__device__ __noinline__ void gemm64_t(float* C, int ldc, const float* A, int sam, int sak, const float* B,
                         int sbk, int sbn, int K, float alpha, float beta, int mask,
                         float* sbuf) {
  constexpr int M = 64, N = 16 * TN;
  constexpr int WM = N == 128 ? 2 : 1, WN = 4;     // 16-row and 8-column tiles per warp
  constexpr int WARPS_N = N / (8 * WN);
  static_assert((M / (16 * WM)) * WARPS_N == kBwdThreads / 32, "one tile per warp");
  // A slice: AK ? [M][kKT + 4] : [kKT][M + 8];  B slice: BK ? [N][kKT + 4] : [kKT][N + 8]
  // (the paddings put the 32 lanes of every fragment load in 32 different banks)
  constexpr int LA = AK ? kKT + 4 : M + 8, LB = BK ? kKT + 4 : N + 8;
  constexpr int SA = AK ? M * LA : kKT * LA, SB = BK ? N * LB : kKT * LB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int m0 = (warp / WARPS_N) * 16 * WM, n0 = (warp % WARPS_N) * 8 * WN;
  auto stage = [&](int buf, int k0) {
    float* As = sbuf + buf * (SA + SB);
    float* Bs = As + SA;
    for (int idx = tid; idx < M * kKT / 4; idx += blockDim.x) {
      if (AK) {
        const int m = idx / (kKT / 4), kk = (idx % (kKT / 4)) * 4;
        cp16(As + m * LA + kk, A + static_cast<size_t>(m) * sam + k0 + kk);
      } else {
        const int m = (idx % (M / 4)) * 4, kk = idx / (M / 4);
        cp16(As + kk * LA + m, A + static_cast<size_t>(k0 + kk) * sak + m);
      }
    }
    for (int idx = tid; idx < N * kKT / 4; idx += blockDim.x) {
      if (BK) {
        const int n = idx / (kKT / 4), kk = (idx % (kKT / 4)) * 4;
        cp16(Bs + n * LB + kk, B + static_cast<size_t>(n) * sbn + k0 + kk);
      } else {
        const int n = (idx % (N / 4)) * 4, kk = idx / (N / 4);
        cp16(Bs + kk * LB + n, B + static_cast<size_t>(k0 + kk) * sbk + n);
      }
    }
    cp_commit();
  };
  float acc[WM][WN][4];
#pragma unroll
  for (int i = 0; i < WM; ++i)
#pragma unroll
    for (int j = 0; j < WN; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;
  const int slices = K / kKT;
  stage(0, 0);
  for (int sl = 0; sl < slices; ++sl) {
    if (sl + 1 < slices) {
      stage((sl + 1) & 1, (sl + 1) * kKT);
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    const float* As = sbuf + (sl & 1) * (SA + SB);
    const float* Bs = As + SA;
    auto a_at = [&](int m, int k) { return AK ? As[m * LA + k] : As[k * LA + m]; };
    auto b_at = [&](int k, int n) { return BK ? Bs[n * LB + k] : Bs[k * LB + n]; };
#pragma unroll
    for (int k8 = 0; k8 < kKT; k8 += 8) {
      // fragments: A rows g, g + 8 and columns t, t + 4; B rows t, t + 4 and column g
      uint32_t ah[WM][4], al[WM][4], bh[WN][2], bl[WN][2];
      auto split = [](float x, uint32_t& hi, uint32_t& lo) {
        if constexpr (NP == 3) {
          split_tf32(x, hi, lo);
        } else {
          hi = tf32_rna(x);
          lo = 0u;
        }
      };
#pragma unroll
      for (int i = 0; i < WM; ++i) {
        const int r = m0 + 16 * i + g, k = k8 + t;
        split(a_at(r, k), ah[i][0], al[i][0]);
        split(a_at(r + 8, k), ah[i][1], al[i][1]);
        split(a_at(r, k + 4), ah[i][2], al[i][2]);
        split(a_at(r + 8, k + 4), ah[i][3], al[i][3]);
      }
#pragma unroll
      for (int j = 0; j < WN; ++j) {
        const int n = n0 + 8 * j + g, k = k8 + t;
        split(b_at(k, n), bh[j][0], bl[j][0]);
        split(b_at(k + 4, n), bh[j][1], bl[j][1]);
      }
#pragma unroll
      for (int i = 0; i < WM; ++i)
#pragma unroll
        for (int j = 0; j < WN; ++j) {
          if constexpr (NP == 3) {
            mma_tf32(acc[i][j], al[i], bh[j][0], bh[j][1]);
            mma_tf32(acc[i][j], ah[i], bl[j][0], bl[j][1]);
          }
          mma_tf32(acc[i][j], ah[i], bh[j][0], bh[j][1]);
        }
    }
    __syncthreads();   // the buffer is restaged two slices on
  }
  // accumulator e of a tile: row g (+ 8 for e >= 2), column 2 t (+ 1 for odd e)
#pragma unroll
  for (int i = 0; i < WM; ++i)
#pragma unroll
    for (int j = 0; j < WN; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int m = m0 + 16 * i + g + 8 * hf, n = n0 + 8 * j + 2 * t;
        float2* c = reinterpret_cast<float2*>(C + static_cast<size_t>(m) * ldc + n);
        float2 v = make_float2(alpha * acc[i][j][2 * hf], alpha * acc[i][j][2 * hf + 1]);
        if (beta != 0.f) {
          const float2 o = *c;
          v.x = fmaf(beta, o.x, v.x);
          v.y = fmaf(beta, o.y, v.y);
        }
        if ((mask == 1 && n > m) || (mask == 2 && n >= m)) v.x = 0.f;
        if ((mask == 1 && n + 1 > m) || (mask == 2 && n + 1 >= m)) v.y = 0.f;
        *c = v;
      }
  __syncthreads();
}

template <int NP, int TN>
__device__ void gemm64_n(float* C, int ldc, const float* A, int sam, int sak, const float* B,
                         int sbk, int sbn, int K, float alpha, float beta, int mask, float* sbuf) {
  if (sak == 1) {
    if (sbk == 1) gemm64_t<NP, TN, true, true>(C, ldc, A, sam, sak, B, sbk, sbn, K, alpha, beta, mask, sbuf);
    else gemm64_t<NP, TN, true, false>(C, ldc, A, sam, sak, B, sbk, sbn, K, alpha, beta, mask, sbuf);
  } else {
    if (sbk == 1) gemm64_t<NP, TN, false, true>(C, ldc, A, sam, sak, B, sbk, sbn, K, alpha, beta, mask, sbuf);
    else gemm64_t<NP, TN, false, false>(C, ldc, A, sam, sak, B, sbk, sbn, K, alpha, beta, mask, sbuf);
  }
}

// M = 64 products with N = 64 or 128 (the only shapes of the chunk algebra).
template <int NP>
__device__ void gemm64(float* C, int ldc, const float* A, int sam, int sak, const float* B,
                       int sbk, int sbn, int N, int K, float alpha, float beta, float* sbuf,
                       int mask = 0) {
  if (N == 128)
    gemm64_n<NP, 8>(C, ldc, A, sam, sak, B, sbk, sbn, K, alpha, beta, mask, sbuf);
  else
    gemm64_n<NP, 4>(C, ldc, A, sam, sak, B, sbk, sbn, K, alpha, beta, mask, sbuf);
}

// tf32 products per product of the per-chunk kernels: three (split operands,
// about fp32 accuracy) for fp32 inputs; one for bf16 inputs, whose 2^-8
// rounding already bounds the result's accuracy well above tf32's 2^-11
template <typename T>
constexpr int kProducts = 3;
template <>
constexpr int kProducts<__nv_bfloat16> = 1;

// two stages of the largest slices: A [64][36] (or [kKT][72]), B [128][36] (or [kKT][136])
constexpr size_t kGemmSmem = static_cast<size_t>(2) * (64 * 36 + 128 * 36) * sizeof(float);
static_assert(64 * 36 >= kKT * 72 && 128 * 36 >= kKT * 136, "stage sizes cover every layout");

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
  __host__ __device__ size_t oGam() const { return 0; }
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
  int* status;     // kStatusWords status words (the start of the workspace)
  int B, T, H, dk, dv, Nc;
  unsigned flags;
  float scale;
};

__device__ __forceinline__ size_t chunk_id(const BwdPtrs& p, int bb, int h, int n) {
  return (static_cast<size_t>(bb) * p.H + h) * p.Nc + n;
}

// ---------------------------------------------------------------- 1. records
template <typename T>
__global__ void __launch_bounds__(kBwdThreads, 3) bwd_chunk_prep(const BwdPtrs p) {
  constexpr int kNP = kProducts<T>;
  const Rec R{p.dk, p.dv};
  const int cid = blockIdx.x;
  const int n = cid % p.Nc, bh = cid / p.Nc, h = bh % p.H, bb = bh / p.H;
  const int t0 = n * kC, Lr = min(kC, p.T - t0);
  const int dk = p.dk, dv = p.dv, tid = threadIdx.x;
  float* r = p.rec + static_cast<size_t>(cid) * R.size();
  const bool CH = p.flags & 1u, ER = p.flags & 2u, WR = p.flags & 4u, QM = p.flags & 8u;
  extern __shared__ __align__(16) float sg[];
  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  const T* v = static_cast<const T*>(p.v);
  const T* bg = static_cast<const T*>(p.b);
  const T* wg = static_cast<const T*>(p.w);
  auto tok = [&](int i) { return (static_cast<size_t>(bb) * p.T + t0 + i) * p.H + h; };
  const int bd = blockDim.x;
  // G: in-chunk inclusive cumsum of the log-decay (per key channel, or one per row
  // broadcast over the channels), in shared memory; rows past the end add nothing
  float* sG = sg;                  // [64][dk] (per channel) or [64]
  float* sGC = sg + kC * dk;       // [dk] gamma_C
  if (CH) {
    for (int e0 = tid; e0 < kC * dk; e0 += kU * bd) {
      float x[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int e = e0 + u * bd, i = e / dk;
        x[u] = (e < kC * dk && i < Lr) ? p.g[tok(i) * dk + e % dk] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (e0 + u * bd < kC * dk) sG[e0 + u * bd] = x[u];
    }
  } else if (tid < kC) {
    sG[tid] = tid < Lr ? p.g[tok(tid)] : 0.f;
  }
  __syncthreads();
  bool low = false;   // some G below the range of the records (kBwdDecayFloor)
  if (CH) {
    for (int c = tid; c < dk; c += bd) {
      float acc = 0.f;
      for (int i = 0; i < kC; ++i) {
        acc += sG[i * dk + c];
        sG[i * dk + c] = acc;
        low |= acc < kBwdDecayFloor;
      }
      sGC[c] = expf(acc);
    }
  } else if (tid == 0) {
    float acc = 0.f;
    for (int i = 0; i < kC; ++i) {
      acc += sG[i];
      sG[i] = acc;
      low |= acc < kBwdDecayFloor;
    }
  }
  if (low && atomicCAS(p.status, 0, 6) == 0) {   // GDR_ERR_RANGE
    p.status[1] = bh;
    p.status[2] = n;
  }
  __syncthreads();
  if (!CH)
    for (int c = tid; c < dk; c += bd) sGC[c] = expf(sG[kC - 1]);
  __syncthreads();
  // gamma, x (erase input), E, K_bar, E_bar, Q_gamma, K_tail; loads batched ahead
  // of the stores so that they overlap
  for (int e0 = tid; e0 < kC * dk; e0 += kU * bd) {
    float qv[kU], kv[kU], bv[kU], rb[kU], rl[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * bd, i = e / dk, c = e % dk;
      const bool ok = e < kC * dk && i < Lr;
      qv[u] = ok ? ldx(q, tok(i) * dk + c) : 0.f;
      kv[u] = ok ? ldx(k, tok(i) * dk + c) : 0.f;
      bv[u] = ok && ER ? ldx(bg, tok(i) * dk + c) : 0.f;
      rb[u] = ok && !ER ? p.beta[tok(i)] : 0.f;
      rl[u] = ok && QM ? p.lam[tok(i)] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * bd, i = e / dk, c = e % dk;
      if (e >= kC * dk) continue;
      const float gam = expf(CH ? sG[e] : sG[i]), gC = sGC[c];
      const float x = QM ? kv[u] + rl[u] * qv[u] : kv[u];
      const float E = ER ? bv[u] * x : rb[u] * x;
      r[R.oGam() + e] = gam;
      r[R.oX() + e] = x;
      r[R.oE() + e] = E;
      r[R.oKb() + e] = kv[u] / gam;
      r[R.oEb() + e] = gam * E;
      r[R.oQg() + e] = p.scale * gam * qv[u];
      r[R.oKt() + e] = gC / gam * kv[u];
    }
  }
  for (int e0 = tid; e0 < kC * dv; e0 += kU * bd) {
    float vv[kU], sc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * bd, i = e / dv;
      const bool ok = e < kC * dv && i < Lr;
      vv[u] = ok ? ldx(v, tok(i) * dv + e % dv) : 0.f;
      sc[u] = !ok ? 0.f : WR ? ldx(wg, tok(i) * dv + e % dv) : p.beta[tok(i)];
    }
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (e0 + u * bd < kC * dv) r[R.oZ() + e0 + u * bd] = sc[u] * vv[u];
  }
  __syncthreads();
  // T = tril(E_bar K_bar^T, -1), A_qk = tril(Q_gamma K_bar^T, 0)
  gemm64<kNP>(r + R.oT(), kC, r + R.oEb(), dk, 1, r + R.oKb(), 1, dk, kC, dk, 1.f, 0.f, sg, 2);
  gemm64<kNP>(r + R.oAqk(), kC, r + R.oQg(), dk, 1, r + R.oKb(), 1, dk, kC, dk, 1.f, 0.f, sg, 1);
  // A = (I + T)^{-1}: row i of (I + T) A = I gives A_i = e_i - sum_{j<i} T_ij A_j.
  // T and A sit in shared memory; thread c owns column c (two accumulators).
  {
    float* sT = sg;              // [64][64]
    float* sA = sg + kC * kC;    // [64][65]
    for (int e = tid * 4; e < kC * kC; e += blockDim.x * 4) cp16(sT + e, r + R.oT() + e);
    cp_commit();
    cp_wait<0>();
    __syncthreads();
    if (tid < kC) {
      for (int i = 0; i < kC; ++i) {
        float a0 = (i == tid) ? 1.f : 0.f, a1 = 0.f;
        const float* Ti = sT + i * kC;
        int j = 0;
        for (; j + 4 <= i; j += 4) {
          const float4 t4 = *reinterpret_cast<const float4*>(Ti + j);
          a0 = fmaf(-t4.x, sA[j * 65 + tid], a0);
          a1 = fmaf(-t4.y, sA[(j + 1) * 65 + tid], a1);
          a0 = fmaf(-t4.z, sA[(j + 2) * 65 + tid], a0);
          a1 = fmaf(-t4.w, sA[(j + 3) * 65 + tid], a1);
        }
        for (; j < i; ++j) a0 = fmaf(-Ti[j], sA[j * 65 + tid], a0);
        sA[i * 65 + tid] = a0 + a1;
      }
    }
    __syncthreads();
    for (int e = tid; e < kC * kC; e += blockDim.x) r[R.oA() + e] = sA[(e / kC) * 65 + e % kC];
    __syncthreads();
  }
  // Y = A E_bar, U = A Z
  gemm64<kNP>(r + R.oY(), dk, r + R.oA(), kC, 1, r + R.oEb(), dk, 1, dk, kC, 1.f, 0.f, sg);
  gemm64<kNP>(r + R.oU(), dv, r + R.oA(), kC, 1, r + R.oZ(), dv, 1, dv, kC, 1.f, 0.f, sg);
}

// ------------------------------------------------------- 2. forward states
// Warp-level MMA on bf16 operands (m16n8k16, fp32 accumulation). An fp32
// operand x is split into bf16 hi = rn(x) and lo = rn(x - hi); with NP = 3 the
// three products lo*hi + hi*lo + hi*hi are accumulated, which leaves a relative
// error of about 2^-17 per term (the dropped lo*lo is below it); NP = 1 keeps
// hi*hi only. Operands are fp32 (or the input type) in shared memory, split as
// the fragments are loaded.
__device__ __forceinline__ uint32_t pack_bf16(float lo_idx, float hi_idx) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi_idx), "f"(lo_idx));
  return r;
}
template <int NP>
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(x0, x1);
  if (NP == 3)
    lo = pack_bf16(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <int NP>
struct FragA {
  uint32_t h[4], l[4];
  __device__ __forceinline__ void negate() {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      h[i] ^= 0x80008000u;
      if (NP == 3) l[i] ^= 0x80008000u;
    }
  }
};
template <int NP>
struct FragB {
  uint32_t h[2], l[2];
};
__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// A fragment (16 x 16 at rows m0, columns k0) of a(m, k) = X[m ld + k] (KC) or
// X[k ld + m] (!KC). Conflict-free shared-memory reads need ld = 8 (mod 32)
// for KC and ld = 4 (mod 32) otherwise.
template <bool KC, int NP>
__device__ __forceinline__ void load_a(FragA<NP>& f, const float* X, int ld, int m0, int k0) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int r0 = m0 + g, c0 = k0 + 2 * t;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int r = r0 + (q & 1) * 8, c = c0 + (q >> 1) * 8;
    float x0, x1;
    if (KC) {
      const float2 v = *reinterpret_cast<const float2*>(X + r * ld + c);
      x0 = v.x;
      x1 = v.y;
    } else {
      x0 = X[c * ld + r];
      x1 = X[(c + 1) * ld + r];
    }
    split_pair<NP>(x0, x1, f.h[q], f.l[q]);
  }
}
// B fragment (16 x 8 at rows k0, columns n0) of b(k, n) = X[n ld + k] (KC) or
// X[k ld + n] (!KC); same padding rule as load_a.
template <bool KC, int NP, typename T>
__device__ __forceinline__ void load_b(FragB<NP>& f, const T* X, int ld, int k0, int n0) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int n = n0 + g, k = k0 + 2 * t;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int kk = k + q * 8;
    float x0, x1;
    if (KC) {
      x0 = ldf(X + n * ld + kk);
      x1 = ldf(X + n * ld + kk + 1);
    } else {
      x0 = ldf(X + kk * ld + n);
      x1 = ldf(X + (kk + 1) * ld + n);
    }
    split_pair<NP>(x0, x1, f.h[q], f.l[q]);
  }
}
template <int NP>
__device__ __forceinline__ void mma_split(float (&d)[4], const FragA<NP>& a, const FragB<NP>& b) {
  if (NP == 3) {
    mma_bf16(d, a.l, b.h[0], b.h[1]);
    mma_bf16(d, a.h, b.l[0], b.l[1]);
  }
  mma_bf16(d, a.h, b.h[0], b.h[1]);
}

// 16-byte asynchronous copy that reads src_bytes (0 or 16) and zero-fills the rest
__device__ __forceinline__ void cp16z(void* smem, const void* gmem, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(sa32(smem)), "l"(gmem),
               "r"(src_bytes)
               : "memory");
}

constexpr int kSlice = 64;          // value columns per state-pass CTA
constexpr int kPassThreads = 256;   // 8 warps
constexpr int kLS = kSlice + 4;     // row pitch of the state / W tiles (floats)

// The accumulator tile of a warp in a [rows x 64] product with 8 warps:
// rows 16 mt.., n-tiles nt0 .. nt0 + NT - 1 (NT = rows / 16 of 8-column tiles).
template <int ROWS>
struct WarpTile {
  static constexpr int NT = ROWS / 16;            // n-tiles per warp
  static constexpr int WPM = 8 / (ROWS / 16);     // warps per 16-row tile
  int mt, nt0;
  __device__ WarpTile(int warp) : mt(warp / WPM), nt0((warp % WPM) * NT) {}
};

// Forward state pass. One CTA per (batch, head, 64 value columns), chunks in
// order: W_n = U_n - Y_n S_n, S_{n+1} = Diag(gamma_C) S_n + K_tail^T W_n, S_n
// and W_n written out for the gradient kernel. S_n lives in the warps'
// accumulators (and as the MMA operand in shared memory); the next chunk's
// Y, U, K_tail and gamma_C are copied in while the current one is used.
template <int DK>
struct StatePassSmem {
  static constexpr int LY = DK + 8, LU = kSlice, LKT = DK + 4;
  static constexpr int STAGE = kC * LY + kC * LU + kC * LKT + DK;
  static constexpr size_t floats = 2 * STAGE + DK * kLS + kC * kLS;
};

template <int DK, int NP>
__global__ void __launch_bounds__(kPassThreads, 1) bwd_state_pass(const BwdPtrs p) {
  using L = StatePassSmem<DK>;
  const Rec R{DK, p.dv};
  const int col0 = blockIdx.x * kSlice, h = blockIdx.y, bb = blockIdx.z;
  const int dv = p.dv, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  extern __shared__ __align__(16) float sm[];
  float* S = sm + 2 * L::STAGE;        // [DK][kLS]
  float* Wl = S + DK * kLS;            // [64][kLS]
  auto stage = [&](int n) {
    float* st = sm + (n & 1) * L::STAGE;
    float* Ys = st;
    float* Us = Ys + kC * L::LY;
    float* Kts = Us + kC * L::LU;
    float* gC = Kts + kC * L::LKT;
    const float* r = p.rec + chunk_id(p, bb, h, n) * R.size();
    for (int e = tid * 4; e < kC * DK; e += kPassThreads * 4) {
      const int i = e / DK, c = e % DK;
      cp16(Ys + i * L::LY + c, r + R.oY() + e);
      cp16(Kts + i * L::LKT + c, r + R.oKt() + e);
    }
    for (int e = tid * 4; e < kC * kSlice; e += kPassThreads * 4) {
      const int i = e / kSlice, c = e % kSlice;
      cp16(Us + i * L::LU + c, r + R.oU() + static_cast<size_t>(i) * dv + col0 + c);
    }
    for (int e = tid * 4; e < DK; e += kPassThreads * 4) cp16(gC + e, r + R.oGam() + (kC - 1) * DK + e);
    cp_commit();
  };
  // S accumulators: rows 16 ts.mt + g (+ 8), columns 8 (ts.nt0 + j) + 2 t (+ 1)
  const WarpTile<DK> ts(warp);
  float acc[WarpTile<DK>::NT][4];
  const size_t bh = static_cast<size_t>(bb) * p.H + h;
#pragma unroll
  for (int j = 0; j < WarpTile<DK>::NT; ++j)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int r = 16 * ts.mt + g + 8 * hf, c = 8 * (ts.nt0 + j) + 2 * t;
      float2 v = make_float2(0.f, 0.f);
      if (p.h0) v = *reinterpret_cast<const float2*>(p.h0 + (bh * DK + r) * dv + col0 + c);
      acc[j][2 * hf] = v.x;
      acc[j][2 * hf + 1] = v.y;
      *reinterpret_cast<float2*>(S + r * kLS + c) = v;
    }
  stage(0);
  for (int n = 0; n < p.Nc; ++n) {
    const size_t cid = chunk_id(p, bb, h, n);
    float* Sg = p.S + cid * DK * dv;
#pragma unroll
    for (int j = 0; j < WarpTile<DK>::NT; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = 16 * ts.mt + g + 8 * hf, c = 8 * (ts.nt0 + j) + 2 * t;
        *reinterpret_cast<float2*>(Sg + static_cast<size_t>(r) * dv + col0 + c) =
            make_float2(acc[j][2 * hf], acc[j][2 * hf + 1]);
      }
    if (n + 1 < p.Nc) stage(n + 1);
    else cp_commit();
    cp_wait<1>();
    __syncthreads();   // chunk n's operands landed; S_n complete in shared memory
    const float* st = sm + (n & 1) * L::STAGE;
    const float* Ys = st;
    const float* Us = Ys + kC * L::LY;
    const float* Kts = Us + kC * L::LU;
    const float* gC = Kts + kC * L::LKT;
    // W = U - Y S: warp -> rows 16 (warp & 3), n-tiles 4 (warp >> 2) .. + 3
    {
      const int mt = warp & 3, nt0 = (warp >> 2) * 4;
      float w[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w[j][e] = Us[(16 * mt + g + 8 * (e >> 1)) * L::LU + 8 * (nt0 + j) + 2 * t + (e & 1)];
#pragma unroll 2
      for (int ks = 0; ks < DK / 16; ++ks) {
        FragA<NP> a;
        load_a<true, NP>(a, Ys, L::LY, 16 * mt, 16 * ks);
        a.negate();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          FragB<NP> b;
          load_b<false, NP>(b, S, kLS, 16 * ks, 8 * (nt0 + j));
          mma_split<NP>(w[j], a, b);
        }
      }
      float* Wg = p.W + cid * kC * dv;
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int r = 16 * mt + g + 8 * hf, c = 8 * (nt0 + j) + 2 * t;
          const float2 v = make_float2(w[j][2 * hf], w[j][2 * hf + 1]);
          *reinterpret_cast<float2*>(Wl + r * kLS + c) = v;
          *reinterpret_cast<float2*>(Wg + static_cast<size_t>(r) * dv + col0 + c) = v;
        }
    }
    __syncthreads();   // W complete; S no longer read
    // S' = Diag(gamma_C) S + K_tail^T W
    {
      const float g0 = gC[16 * ts.mt + g], g1 = gC[16 * ts.mt + g + 8];
#pragma unroll
      for (int j = 0; j < WarpTile<DK>::NT; ++j) {
        acc[j][0] *= g0;
        acc[j][1] *= g0;
        acc[j][2] *= g1;
        acc[j][3] *= g1;
      }
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks) {
        FragA<NP> a;
        load_a<false, NP>(a, Kts, L::LKT, 16 * ts.mt, 16 * ks);
#pragma unroll
        for (int j = 0; j < WarpTile<DK>::NT; ++j) {
          FragB<NP> b;
          load_b<false, NP>(b, Wl, kLS, 16 * ks, 8 * (ts.nt0 + j));
          mma_split<NP>(acc[j], a, b);
        }
      }
#pragma unroll
      for (int j = 0; j < WarpTile<DK>::NT; ++j)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int r = 16 * ts.mt + g + 8 * hf, c = 8 * (ts.nt0 + j) + 2 * t;
          *reinterpret_cast<float2*>(S + r * kLS + c) = make_float2(acc[j][2 * hf], acc[j][2 * hf + 1]);
        }
    }
    __syncthreads();   // S_{n+1} complete; this stage's buffers free
  }
  cp_wait<0>();
}

// ------------------------------------------------------- 3. reverse states
// Reverse state pass, chunks in reverse order: dW_n = A_qk^T dO_n + K_tail
// dS_{n+1}, dS_n = Diag(gamma_C) dS_{n+1} + Q_gamma^T dO_n - Y^T dW_n, with
// dS_{n+1} and dW_n written out. dS lives in the accumulators. The operands of
// the dW product (A_qk, K_tail, dO) and of the dS product (Q_gamma, Y,
// gamma_C) are two copy groups: each is refilled for the previous chunk as
// soon as its product is done, so it lands while the other product runs (dO,
// read by both, is double-buffered).
template <int DK, typename T>
struct DStateSmem {
  static constexpr int LAQ = kC + 4, LKT = DK + 8, LQ = DK + 4;
  // dO rows: 68 floats or 72 bf16 (a row pitch of 4 banks mod 32 either way)
  static constexpr int LO = sizeof(T) == 4 ? kSlice + 4 : kSlice + 8;
  static constexpr size_t f_aq = 0, f_kt = f_aq + kC * LAQ, f_do = f_kt + kC * LKT;
  static constexpr size_t do_floats = (static_cast<size_t>(kC) * LO * sizeof(T) + 15) / 16 * 4;
  static constexpr size_t f_qg = f_do + 2 * do_floats, f_y = f_qg + kC * LQ, f_gc = f_y + kC * LQ;
  static constexpr size_t f_ds = f_gc + DK, f_dw = f_ds + DK * kLS;
  static constexpr size_t floats = f_dw + kC * kLS;
};

template <int DK, int NP, typename T>
__global__ void __launch_bounds__(kPassThreads, 1) bwd_dstate_pass(const BwdPtrs p) {
  using L = DStateSmem<DK, T>;
  const Rec R{DK, p.dv};
  const int col0 = blockIdx.x * kSlice, h = blockIdx.y, bb = blockIdx.z;
  const int dv = p.dv, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const T* dO = static_cast<const T*>(p.dO);
  extern __shared__ __align__(16) float sm[];
  float* Aq = sm + L::f_aq;
  float* Kt = sm + L::f_kt;
  float* Qg = sm + L::f_qg;
  float* Ys = sm + L::f_y;
  float* gC = sm + L::f_gc;
  float* dS = sm + L::f_ds;
  float* dWl = sm + L::f_dw;
  auto dO_buf = [&](int n) { return reinterpret_cast<T*>(sm + L::f_do + (n & 1) * L::do_floats); };
  auto stage_a = [&](int n) {
    const float* r = p.rec + chunk_id(p, bb, h, n) * R.size();
    for (int e = tid * 4; e < kC * kC; e += kPassThreads * 4) cp16(Aq + (e / kC) * L::LAQ + e % kC, r + R.oAqk() + e);
    for (int e = tid * 4; e < kC * DK; e += kPassThreads * 4) cp16(Kt + (e / DK) * L::LKT + e % DK, r + R.oKt() + e);
    constexpr int V = 16 / sizeof(T);   // elements per 16-byte copy
    T* ob = dO_buf(n);
    const int t0 = n * kC, Lr = min(kC, p.T - t0);
    for (int e = tid * V; e < kC * kSlice; e += kPassThreads * V) {
      const int i = e / kSlice, c = e % kSlice;
      const bool ok = i < Lr;
      const size_t src = ((static_cast<size_t>(bb) * p.T + t0 + (ok ? i : 0)) * p.H + h) * dv + col0 + c;
      cp16z(ob + i * L::LO + c, dO + src, ok ? 16 : 0);
    }
    cp_commit();
  };
  auto stage_b = [&](int n) {
    const float* r = p.rec + chunk_id(p, bb, h, n) * R.size();
    for (int e = tid * 4; e < kC * DK; e += kPassThreads * 4) {
      const int i = e / DK, c = e % DK;
      cp16(Qg + i * L::LQ + c, r + R.oQg() + e);
      cp16(Ys + i * L::LQ + c, r + R.oY() + e);
    }
    for (int e = tid * 4; e < DK; e += kPassThreads * 4) cp16(gC + e, r + R.oGam() + (kC - 1) * DK + e);
    cp_commit();
  };
  const WarpTile<DK> ts(warp);
  float acc[WarpTile<DK>::NT][4];
  const size_t bh = static_cast<size_t>(bb) * p.H + h;
#pragma unroll
  for (int j = 0; j < WarpTile<DK>::NT; ++j)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int r = 16 * ts.mt + g + 8 * hf, c = 8 * (ts.nt0 + j) + 2 * t;
      float2 v = make_float2(0.f, 0.f);
      if (p.dhT) v = *reinterpret_cast<const float2*>(p.dhT + (bh * DK + r) * dv + col0 + c);
      acc[j][2 * hf] = v.x;
      acc[j][2 * hf + 1] = v.y;
      *reinterpret_cast<float2*>(dS + r * kLS + c) = v;
    }
  stage_a(p.Nc - 1);
  stage_b(p.Nc - 1);
  for (int n = p.Nc - 1; n >= 0; --n) {
    const size_t cid = chunk_id(p, bb, h, n);
    float* dSg = p.dS + cid * DK * dv;
#pragma unroll
    for (int j = 0; j < WarpTile<DK>::NT; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = 16 * ts.mt + g + 8 * hf, c = 8 * (ts.nt0 + j) + 2 * t;
        *reinterpret_cast<float2*>(dSg + static_cast<size_t>(r) * dv + col0 + c) =
            make_float2(acc[j][2 * hf], acc[j][2 * hf + 1]);
      }
    cp_wait<1>();
    __syncthreads();   // A_qk, K_tail, dO of chunk n landed; dS_{n+1} complete
    const T* ob = dO_buf(n);
    // dW = A_qk^T dO + K_tail dS': warp -> rows 16 (warp & 3), n-tiles 4 (warp >> 2) .. + 3
    {
      const int mt = warp & 3, nt0 = (warp >> 2) * 4;
      float w[4][4] = {};
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks) {
        FragA<NP> a;
        load_a<false, NP>(a, Aq, L::LAQ, 16 * mt, 16 * ks);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          FragB<NP> b;
          load_b<false, NP>(b, ob, L::LO, 16 * ks, 8 * (nt0 + j));
          mma_split<NP>(w[j], a, b);
        }
      }
#pragma unroll 2
      for (int ks = 0; ks < DK / 16; ++ks) {
        FragA<NP> a;
        load_a<true, NP>(a, Kt, L::LKT, 16 * mt, 16 * ks);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          FragB<NP> b;
          load_b<false, NP>(b, dS, kLS, 16 * ks, 8 * (nt0 + j));
          mma_split<NP>(w[j], a, b);
        }
      }
      float* dWg = p.dW + cid * kC * dv;
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int r = 16 * mt + g + 8 * hf, c = 8 * (nt0 + j) + 2 * t;
          const float2 v = make_float2(w[j][2 * hf], w[j][2 * hf + 1]);
          *reinterpret_cast<float2*>(dWl + r * kLS + c) = v;
          *reinterpret_cast<float2*>(dWg + static_cast<size_t>(r) * dv + col0 + c) = v;
        }
    }
    __syncthreads();   // dW complete; A_qk, K_tail and dS' no longer read
    if (n > 0) stage_a(n - 1);
    else cp_commit();
    cp_wait<1>();
    __syncthreads();   // Q_gamma, Y, gamma_C of chunk n landed
    // dS = Diag(gamma_C) dS' + Q_gamma^T dO - Y^T dW
    {
      const float g0 = gC[16 * ts.mt + g], g1 = gC[16 * ts.mt + g + 8];
#pragma unroll
      for (int j = 0; j < WarpTile<DK>::NT; ++j) {
        acc[j][0] *= g0;
        acc[j][1] *= g0;
        acc[j][2] *= g1;
        acc[j][3] *= g1;
      }
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks) {
        FragA<NP> aq, ay;
        load_a<false, NP>(aq, Qg, L::LQ, 16 * ts.mt, 16 * ks);
        load_a<false, NP>(ay, Ys, L::LQ, 16 * ts.mt, 16 * ks);
        ay.negate();
#pragma unroll
        for (int j = 0; j < WarpTile<DK>::NT; ++j) {
          FragB<NP> b;
          load_b<false, NP>(b, ob, L::LO, 16 * ks, 8 * (ts.nt0 + j));
          mma_split<NP>(acc[j], aq, b);
          load_b<false, NP>(b, dWl, kLS, 16 * ks, 8 * (ts.nt0 + j));
          mma_split<NP>(acc[j], ay, b);
        }
      }
#pragma unroll
      for (int j = 0; j < WarpTile<DK>::NT; ++j)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int r = 16 * ts.mt + g + 8 * hf, c = 8 * (ts.nt0 + j) + 2 * t;
          *reinterpret_cast<float2*>(dS + r * kLS + c) = make_float2(acc[j][2 * hf], acc[j][2 * hf + 1]);
        }
    }
    __syncthreads();   // dS_n complete; Q_gamma, Y, gamma_C and dW no longer read
    if (n > 0) stage_b(n - 1);
    else cp_commit();
  }
  cp_wait<0>();
  if (p.d_h0)
#pragma unroll
    for (int j = 0; j < WarpTile<DK>::NT; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = 16 * ts.mt + g + 8 * hf, c = 8 * (ts.nt0 + j) + 2 * t;
        *reinterpret_cast<float2*>(p.d_h0 + (bh * DK + r) * dv + col0 + c) =
            make_float2(acc[j][2 * hf], acc[j][2 * hf + 1]);
      }
}

// ------------------------------------------------------- 4. gradients
// Buffers whose lifetimes do not overlap share space (every product ends on a
// CTA barrier, so a buffer's next occupant is written only after its last
// reader): dA_qk -> dA -> dT in one 64 x 64 region, the fp32 copy of dO ->
// dY -> X in one 64 x max(d_k, d_v) region.
struct Scr {
  int dk, dv;
  __host__ __device__ size_t mk() const { return static_cast<size_t>(kC) * dk; }
  __host__ __device__ size_t mv() const { return static_cast<size_t>(kC) * dv; }
  __host__ __device__ size_t oR1() const { return 0; }
  __host__ __device__ size_t oR2() const { return oR1() + kC * kC; }
  __host__ __device__ size_t oDAqk() const { return oR1(); }
  __host__ __device__ size_t oDA() const { return oR1(); }
  __host__ __device__ size_t oDT() const { return oR1(); }
  __host__ __device__ size_t oDO() const { return oR2(); }
  __host__ __device__ size_t oDY() const { return oR2(); }
  __host__ __device__ size_t oX() const { return oR2(); }
  __host__ __device__ size_t oDQg() const { return oR2() + (mk() > mv() ? mk() : mv()); }
  __host__ __device__ size_t oDKb() const { return oDQg() + mk(); }
  __host__ __device__ size_t oDKt() const { return oDKb() + mk(); }
  __host__ __device__ size_t oDEb() const { return oDKt() + mk(); }
  __host__ __device__ size_t oDZ() const { return oDEb() + mk(); }
  __host__ __device__ size_t oDgC() const { return oDZ() + mv(); }
  __host__ __device__ size_t size() const { return oDgC() + dk; }
};

template <typename T>
__global__ void __launch_bounds__(kBwdThreads, 3) bwd_chunk_grad(const BwdPtrs p) {
  constexpr int kNP = kProducts<T>;
  const Rec R{p.dk, p.dv};
  const Scr Q{p.dk, p.dv};
  const int cid = blockIdx.x;
  const int n = cid % p.Nc, bh = cid / p.Nc, h = bh % p.H, bb = bh / p.H;
  const int t0 = n * kC, Lr = min(kC, p.T - t0);
  const int dk = p.dk, dv = p.dv, tid = threadIdx.x;
  const bool CH = p.flags & 1u, ER = p.flags & 2u, WR = p.flags & 4u, QM = p.flags & 8u;
  const float* r = p.rec + static_cast<size_t>(cid) * R.size();
  float* s = p.scr + static_cast<size_t>(cid) * Q.size();
  extern __shared__ __align__(16) float sg[];
  const float* S = p.S + static_cast<size_t>(cid) * dk * dv;
  const float* dSn = p.dS + static_cast<size_t>(cid) * dk * dv;
  const float* W = p.W + static_cast<size_t>(cid) * kC * dv;
  const float* dW = p.dW + static_cast<size_t>(cid) * kC * dv;
  const T* dOg = static_cast<const T*>(p.dO);
  auto tok = [&](int i) { return (static_cast<size_t>(bb) * p.T + t0 + i) * p.H + h; };
  float* dO = s + Q.oDO();
  const int bd = blockDim.x, warp = tid >> 5, lane = tid & 31, nw = bd >> 5;
  for (int e0 = tid; e0 < kC * dv; e0 += kU * bd) {
    float x[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * bd, i = e / dv;
      x[u] = (e < kC * dv && i < Lr) ? ldx(dOg, tok(i) * dv + e % dv) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (e0 + u * bd < kC * dv) dO[e0 + u * bd] = x[u];
  }
  // dgamma_C = rowsum(dS' (.) S): one warp per row, 16-byte loads; lane l keeps
  // the sum of the warp's l-th row and stores it after the loop
  {
    float keep = 0.f;
    for (int l = 0; warp + nw * l < dk; ++l) {
      const int c = warp + nw * l;
      float acc = 0.f;
      for (int j = lane * 4; j < dv; j += 128) {
        const float4 x = *reinterpret_cast<const float4*>(dSn + static_cast<size_t>(c) * dv + j);
        const float4 y = *reinterpret_cast<const float4*>(S + static_cast<size_t>(c) * dv + j);
        acc = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, acc))));
      }
      acc = warp_sum(acc);
      if (lane == l) keep = acc;
    }
    if (warp + nw * lane < dk) s[Q.oDgC() + warp + nw * lane] = keep;
  }
  __syncthreads();
  // dA_qk = tril(dO W^T, 0); dQ_gamma = dO S^T + dA_qk K_bar; dK_bar = dA_qk^T Q_gamma
  gemm64<kNP>(s + Q.oDAqk(), kC, dO, dv, 1, W, 1, dv, kC, dv, 1.f, 0.f, sg, 1);
  gemm64<kNP>(s + Q.oDQg(), dk, dO, dv, 1, S, 1, dv, dk, dv, 1.f, 0.f, sg);
  gemm64<kNP>(s + Q.oDQg(), dk, s + Q.oDAqk(), kC, 1, r + R.oKb(), dk, 1, dk, kC, 1.f, 1.f, sg);
  gemm64<kNP>(s + Q.oDKb(), dk, s + Q.oDAqk(), 1, kC, r + R.oQg(), dk, 1, dk, kC, 1.f, 0.f, sg);
  // dK_tail = W dS'^T; dY = -dW S^T
  gemm64<kNP>(s + Q.oDKt(), dk, W, dv, 1, dSn, 1, dv, dk, dv, 1.f, 0.f, sg);
  gemm64<kNP>(s + Q.oDY(), dk, dW, dv, 1, S, 1, dv, dk, dv, -1.f, 0.f, sg);
  // the notes' gate-aware dA = dU Z^T + dY E_bar^T (dU = dW)
  gemm64<kNP>(s + Q.oDA(), kC, dW, dv, 1, r + R.oZ(), 1, dv, kC, dv, 1.f, 0.f, sg);
  gemm64<kNP>(s + Q.oDA(), kC, s + Q.oDY(), dk, 1, r + R.oEb(), 1, dk, kC, dk, 1.f, 1.f, sg);
  // dZ = A^T dU; dE_bar = A^T dY
  gemm64<kNP>(s + Q.oDZ(), dv, r + R.oA(), 1, kC, dW, dv, 1, dv, kC, 1.f, 0.f, sg);
  gemm64<kNP>(s + Q.oDEb(), dk, r + R.oA(), 1, kC, s + Q.oDY(), dk, 1, dk, kC, 1.f, 0.f, sg);
  // the notes' adjoint of the inverse: dT = -tril(A^T dA A^T, -1)
  gemm64<kNP>(s + Q.oX(), kC, r + R.oA(), 1, kC, s + Q.oDA(), kC, 1, kC, kC, 1.f, 0.f, sg);
  gemm64<kNP>(s + Q.oDT(), kC, s + Q.oX(), kC, 1, r + R.oA(), 1, kC, kC, kC, -1.f, 0.f, sg, 2);
  // dE_bar += dT K_bar; dK_bar += dT^T E_bar
  gemm64<kNP>(s + Q.oDEb(), dk, s + Q.oDT(), kC, 1, r + R.oKb(), dk, 1, dk, kC, 1.f, 1.f, sg);
  gemm64<kNP>(s + Q.oDKb(), dk, s + Q.oDT(), 1, kC, r + R.oEb(), dk, 1, dk, kC, 1.f, 1.f, sg);
  // the decay factors: dG = gamma dgamma with
  //   dgamma = dE_bar E - dK_bar K_bar / gamma - dK_tail K_tail / gamma + dQ_gamma Q_gamma / gamma,
  // dgamma_C += sum_r dK_tail k / gamma (= dK_tail K_bar), and dG of the last row
  // gains gamma_C dgamma_C; dg is the reverse cumulative sum of dG within the
  // chunk. Thread (channel c, part) owns rows [part RPT, part RPT + RPT) of
  // channel c: pass A forms dG in shared memory with per-part column sums and
  // writes dq, dk, db; pass B adds the later parts and gamma_C dgamma_C and runs
  // the cumulative sum up its rows.
  float* sDG = sg;                 // [64][dk]
  float* sP = sDG + kC * dk;       // [parts][dk] column sums of dG
  float* sQ = sP + 4 * dk;         // [parts][dk] column sums of dK_tail K_bar
  const int parts = bd / dk, RPT = kC / parts;
  const int c = tid % dk, part = tid / dk, i0 = part * RPT;
  const float gC = r[R.oGam() + (kC - 1) * dk + c];
  {
    float psum = 0.f, pdgc = 0.f;
    for (int ii = 0; ii < RPT; ii += kU) {
      float gam[kU], kb[kU], E[kU], kt[kU], qg[kU], x[kU], deb[kU], dkb[kU], dkt[kU], dqg[kU];
      float bv[kU], rb[kU], rl[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + ii + u;
        const size_t e = static_cast<size_t>(i) * dk + c;
        gam[u] = r[R.oGam() + e];
        kb[u] = r[R.oKb() + e];
        E[u] = r[R.oE() + e];
        kt[u] = r[R.oKt() + e];
        qg[u] = r[R.oQg() + e];
        x[u] = r[R.oX() + e];
        deb[u] = s[Q.oDEb() + e];
        dkb[u] = s[Q.oDKb() + e];
        dkt[u] = s[Q.oDKt() + e];
        dqg[u] = s[Q.oDQg() + e];
        const bool ok = i < Lr;
        bv[u] = ok && ER ? ldx(static_cast<const T*>(p.b), tok(i) * dk + c) : 0.f;
        rb[u] = ok && !ER ? p.beta[tok(i)] : 0.f;
        rl[u] = ok && QM ? p.lam[tok(i)] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + ii + u;
        const float dgam = deb[u] * E[u] - dkb[u] * kb[u] / gam[u] - dkt[u] * kt[u] / gam[u] +
                           dqg[u] * qg[u] / gam[u];
        const float dG = gam[u] * dgam;
        sDG[i * dk + c] = dG;
        psum += dG;
        pdgc = fmaf(dkt[u], kb[u], pdgc);
        if (i < Lr) {
          const float dE = gam[u] * deb[u];
          const float dx = ER ? bv[u] * dE : rb[u] * dE;
          p.d_k[tok(i) * dk + c] = dkb[u] / gam[u] + gC / gam[u] * dkt[u] + dx;
          p.d_q[tok(i) * dk + c] = p.scale * gam[u] * dqg[u] + (QM ? rl[u] * dx : 0.f);
          if (ER) p.d_b[tok(i) * dk + c] = x[u] * dE;
        }
      }
    }
    sP[part * dk + c] = psum;
    sQ[part * dk + c] = pdgc;
  }
  __syncthreads();
  {
    float dgc = s[Q.oDgC() + c];
    for (int q2 = 0; q2 < parts; ++q2) dgc += sQ[q2 * dk + c];
    float acc = gC * dgc;
    for (int q2 = part + 1; q2 < parts; ++q2) acc += sP[q2 * dk + c];
    for (int i = i0 + RPT - 1; i >= i0; --i) {
      acc += sDG[i * dk + c];
      sDG[i * dk + c] = acc;
      if (CH && i < Lr) p.d_g[tok(i) * dk + c] = acc;
    }
  }
  // value-side outputs per (row, channel)
  for (int e0 = tid; e0 < kC * dv; e0 += kU * bd) {
    float dZ[kU], vv[kU], sc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * bd, i = e / dv;
      const bool ok = e < kC * dv && i < Lr;
      dZ[u] = ok ? s[Q.oDZ() + e] : 0.f;
      vv[u] = ok ? ldx(static_cast<const T*>(p.v), tok(i) * dv + e % dv) : 0.f;
      sc[u] = !ok ? 0.f : WR ? ldx(static_cast<const T*>(p.w), tok(i) * dv + e % dv) : p.beta[tok(i)];
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * bd, i = e / dv;
      if (e >= kC * dv || i >= Lr) continue;
      p.d_v[tok(i) * dv + e % dv] = sc[u] * dZ[u];
      if (WR) p.d_w[tok(i) * dv + e % dv] = vv[u] * dZ[u];
    }
  }
  __syncthreads();
  // per-row outputs: scalar dg (sum of dg over the channels), dbeta, dlam; one
  // warp per row, the channels over the lanes
  for (int i = warp; i < Lr; i += nw) {
    float dgs = 0.f, dbe = 0.f, dla = 0.f;
    const float bt = p.beta ? p.beta[tok(i)] : 0.f;
    for (int c2 = lane; c2 < dk; c2 += 32) {
      const size_t e = static_cast<size_t>(i) * dk + c2;
      dgs += sDG[e];
      const float dE = r[R.oGam() + e] * s[Q.oDEb() + e];
      if (!ER) dbe = fmaf(r[R.oX() + e], dE, dbe);
      if (QM) {
        const float dx = ER ? ldx(static_cast<const T*>(p.b), tok(i) * dk + c2) * dE : bt * dE;
        dla = fmaf(ldx(static_cast<const T*>(p.q), tok(i) * dk + c2), dx, dla);
      }
    }
    if (!WR)
      for (int c2 = lane; c2 < dv; c2 += 32)
        dbe = fmaf(ldx(static_cast<const T*>(p.v), tok(i) * dv + c2),
                   s[Q.oDZ() + static_cast<size_t>(i) * dv + c2], dbe);
    dgs = warp_sum(dgs);
    dbe = warp_sum(dbe);
    dla = warp_sum(dla);
    if (lane == 0) {
      if (!CH) p.d_g[tok(i)] = dgs;
      if (p.d_beta) p.d_beta[tok(i)] = dbe;
      if (QM) p.d_lam[tok(i)] = dla;
    }
  }
}

// the forward and reverse state passes: one CTA per (batch, head, 64 value columns)
template <int DK, typename T>
cudaError_t launch_passes(const BwdPtrs& p, cudaStream_t stream) {
  constexpr int NP = 3;
  const dim3 grid(p.dv / kSlice, p.H, p.B);
  const size_t sm2 = StatePassSmem<DK>::floats * sizeof(float);
  const size_t sm3 = DStateSmem<DK, T>::floats * sizeof(float);
  cudaError_t err;
  if ((err = cudaFuncSetAttribute(bwd_state_pass<DK, NP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(sm2))) != cudaSuccess ||
      (err = cudaFuncSetAttribute(bwd_dstate_pass<DK, NP, T>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(sm3))) != cudaSuccess)
    return err;
  bwd_state_pass<DK, NP><<<grid, kPassThreads, sm2, stream>>>(p);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  bwd_dstate_pass<DK, NP, T><<<grid, kPassThreads, sm3, stream>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_all(const BwdPtrs& p, cudaStream_t stream) {
  const int chunks = p.B * p.H * p.Nc;
  cudaError_t err;
  if ((err = cudaFuncSetAttribute(bwd_chunk_prep<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(kGemmSmem))) != cudaSuccess ||
      (err = cudaFuncSetAttribute(bwd_chunk_grad<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(kGemmSmem))) != cudaSuccess)
    return err;
  bwd_chunk_prep<T><<<chunks, kBwdThreads, kGemmSmem, stream>>>(p);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if ((err = (p.dk == 128 ? launch_passes<128, T>(p, stream) : launch_passes<64, T>(p, stream))) !=
      cudaSuccess)
    return err;
  bwd_chunk_grad<T><<<chunks, kBwdThreads, kGemmSmem, stream>>>(p);
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
  return kChunkWorkspaceBytes + floats * sizeof(float);   // status words, then the records
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
  p.status = static_cast<int*>(a.workspace);
  cudaError_t err = cudaMemsetAsync(p.status, 0, kStatusWords * sizeof(int), stream);
  if (err != cudaSuccess) return err;
  float* base = reinterpret_cast<float*>(static_cast<unsigned char*>(a.workspace) +
                                         kChunkWorkspaceBytes);
  p.rec = base;
  p.scr = p.rec + chunks * R.size();
  p.S = p.scr + chunks * Q.size();
  p.dS = p.S + chunks * p.dk * p.dv;
  p.W = p.dS + chunks * p.dk * p.dv;
  p.dW = p.W + chunks * kC * p.dv;
  return f32 ? launch_all<float>(p, stream) : launch_all<__nv_bfloat16>(p, stream);
}

}  // namespace gdr
