// Chunkwise-parallel forward of the gated delta rule for fp32 inputs, fused
// into one kernel (bf16 inputs take the tcgen05 kernel of chunk_fwd_tc.cu).
//
// Algorithm: Gated DeltaNet-2 notes, key design 2 (the chunkwise WY form with
// the cumulative decay absorbed into the rank-one factors), which the Q-Delta
// notes (key design 3) reuse with the mixed erase input. One CTA owns one
// (batch, head) and a slice of NV value columns of the state S (d_k x d_v):
// the value columns of S evolve independently, so slicing d_v multiplies the
// number of independent sequential scans. Per chunk of C = 64 tokens:
//
//   gates   G_r = sum_{i<=r} g_i (fp32, in-chunk), gamma_r = exp(G_r)
//   factors E_bar = gamma (.) E, K_bar = gamma^{-1} (.) K  (rebased, below)
//   T       = tril(E_bar K_bar^T, -1),  A_qk = tril(Q_gamma K_bar^T, 0)
//   A       = (I + T)^{-1}   (forward substitution, fp32, 16x16 blocks)
//   Y = A E_abs, U = A Z     (E_abs_r = gamma_r (.) e_r, Z rows z_r)
//   W       = U - Y S_n
//   O_n     = Q_gamma S_n + A_qk W
//   S_{n+1} = Diag(gamma_C) S_n + K_tail^T W,  K_tail_r = gamma_C/gamma_r (.) k_r
//
// The products run on warp-level tensor-core MMA with bf16 operands and fp32
// accumulation. Every fp32 operand is split into a bf16 pair hi + lo and each
// product takes hi*hi + hi*lo + lo*hi, which keeps ~2^-16 relative accuracy
// (the template keeps a one-plane mode, SPLIT = false, for bf16 operands).
// S stays fp32 in registers across all chunks of the scan.
//
// Decay factors of T and A_qk. Scalar gates: T_ri = (e_r . k_i) exp(G_r - G_i)
// and A_qk_ri = s (q_r . k_i) exp(G_r - G_i), the factor (<= 1) applied per
// element after the product, so any finite g works. Per-channel gates cannot
// be factored out of the product; there E_bar and K_bar carry
// exp(+-(G_r - rho)) with rho = G_C / 2 per key channel instead of
// exp(+-G_r): the products are unchanged (the rho factors cancel) while the
// largest exponent halves. The smaller factor must stay a normal fp32/bf16
// number (about 1e-38) with room for the size of e and k, which holds for an
// in-chunk log-decay sum down to about -140 per channel.
#include "common.cuh"
#include "kernels.h"

namespace gdr {
namespace {

constexpr int kThreads = 128;  // 4 warps; warp w owns chunk rows 16w..16w+15

template <int DK, int NV, bool SPLIT>
struct ChunkSmem {
  static constexpr int P = SPLIT ? 2 : 1;  // bf16 planes (hi, lo)
  static constexpr int LDK = DK + 8;      // row stride of [64 x DK] tiles (bf16)
  static constexpr int LDC = 64 + 8;      // [64 x 64]
  static constexpr int LDN = NV + 8;      // [64 x NV] and [DK x NV]
  static constexpr int LDT = 65;          // fp32 [64 x 64]
  static constexpr size_t kX = size_t(P) * 64 * LDK * 2;
  static constexpr size_t kC = size_t(P) * 64 * LDC * 2;
  static constexpr size_t kZ = size_t(P) * 64 * LDN * 2;
  static constexpr size_t kS = size_t(P) * DK * LDN * 2;
  static constexpr size_t kT = size_t(64) * LDT * 4;
  static constexpr size_t kG = size_t(64) * DK * 4;
  static constexpr size_t kGA = kG > kT ? kG : kT;
  static constexpr size_t kP = size_t(3) * 256 * 4;
  static constexpr size_t oX0 = 0;
  static constexpr size_t oX1 = oX0 + kX;
  static constexpr size_t oX2 = oX1 + kX;
  static constexpr size_t oAqk = oX2 + kX;
  static constexpr size_t oA = oAqk + kC;
  static constexpr size_t oZ = oA + kC;
  static constexpr size_t oW = oZ + kZ;
  static constexpr size_t oS = oW + kZ;
  static constexpr size_t oT = oS + kS;
  static constexpr size_t oGA = oT + kT;
  static constexpr size_t oP = oGA + kGA;
  static constexpr size_t oVec = oP + kP;
  static constexpr size_t kVec = size_t(3 * 64 + 2 * DK) * 4;
  static constexpr size_t bytes = oVec + kVec;
};

// A bf16 tile in shared memory, row-major with stride ld; with SPLIT a second
// plane `plane` elements further holds the low-order parts.
struct Tile {
  __nv_bfloat16* hi;
  int ld;
  int plane;
  __device__ __forceinline__ __nv_bfloat16* lo() const { return hi + plane; }
};

template <bool SPLIT>
__device__ __forceinline__ void put8(const Tile& t, int r, int c0, const float (&x)[8]) {
  uint4 h;
  uint32_t* hp = reinterpret_cast<uint32_t*>(&h);
#pragma unroll
  for (int i = 0; i < 4; ++i) hp[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
  *reinterpret_cast<uint4*>(t.hi + r * t.ld + c0) = h;
  if (SPLIT) {
    const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&h);
    uint4 l;
    uint32_t* lp = reinterpret_cast<uint32_t*>(&l);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(hb[i]);
      lp[i] = pack_bf16x2(x[2 * i] - f.x, x[2 * i + 1] - f.y);
    }
    *reinterpret_cast<uint4*>(t.lo() + r * t.ld + c0) = l;
  }
}

template <bool SPLIT>
__device__ __forceinline__ void put2(const Tile& t, int r, int c, float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  *reinterpret_cast<__nv_bfloat162*>(t.hi + r * t.ld + c) = h;
  if (SPLIT) {
    float2 f = __bfloat1622float2(h);
    *reinterpret_cast<__nv_bfloat162*>(t.lo() + r * t.ld + c) =
        __floats2bfloat162_rn(a - f.x, b - f.y);
  }
}

// acc[16 x 8NT] += A[16 x K] * B[K x 8NT] for one warp.
//  A rows r0..r0+15: AT=false reads a row-major [M x K] tile, AT=true the
//  transpose of a row-major [K x M] tile.
//  B columns n0..: BT=false reads a row-major [N x K] tile (B^T stored),
//  BT=true a row-major [K x N] tile.
template <int K, int NT, bool AT, bool BT, bool SPLIT>
__device__ __forceinline__ void warp_gemm(float (&acc)[NT][4], const Tile& A, int r0,
                                          const Tile& B, int n0) {
  static_assert(NT % 2 == 0, "n-tiles are loaded in pairs");
  const int lane = threadIdx.x & 31;
  const int mi = lane >> 3, mj = lane & 7;
#pragma unroll
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t ah[4], al[4];
    const int aoff = AT ? (k0 + (mi >> 1) * 8 + mj) * A.ld + r0 + (mi & 1) * 8
                        : (r0 + (lane & 15)) * A.ld + k0 + (lane >> 4) * 8;
    if (AT) ldsm_x4_t(ah, A.hi + aoff); else ldsm_x4(ah, A.hi + aoff);
    if (SPLIT) {
      if (AT) ldsm_x4_t(al, A.lo() + aoff); else ldsm_x4(al, A.lo() + aoff);
    }
#pragma unroll
    for (int nt = 0; nt < NT; nt += 2) {
      const int n = n0 + nt * 8;
      const int boff = BT ? (k0 + (mi & 1) * 8 + mj) * B.ld + n + (mi >> 1) * 8
                          : (n + (mi >> 1) * 8 + mj) * B.ld + k0 + (mi & 1) * 8;
      uint32_t bh[4];
      if (BT) ldsm_x4_t(bh, B.hi + boff); else ldsm_x4(bh, B.hi + boff);
      mma_bf16_16816(acc[nt], ah, bh[0], bh[1]);
      mma_bf16_16816(acc[nt + 1], ah, bh[2], bh[3]);
      if (SPLIT) {
        uint32_t bl[4];
        if (BT) ldsm_x4_t(bl, B.lo() + boff); else ldsm_x4(bl, B.lo() + boff);
        mma_bf16_16816(acc[nt], ah, bl[0], bl[1]);
        mma_bf16_16816(acc[nt + 1], ah, bl[2], bl[3]);
        mma_bf16_16816(acc[nt], al, bh[0], bh[1]);
        mma_bf16_16816(acc[nt + 1], al, bh[2], bh[3]);
      }
    }
  }
}

template <bool ACCURATE>
__device__ __forceinline__ float gexp(float x) {
  return ACCURATE ? expf(x) : __expf(x);
}

template <typename TIn>
__device__ __forceinline__ void load8_or_zero(const TIn* p, bool valid, float (&x)[8]) {
  if (valid) {
    load8(p, x);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = 0.f;
  }
}

template <int DK, int NV, bool SPLIT, typename TIn>
__global__ void __launch_bounds__(kThreads, 1) chunk_fwd_kernel(const ChunkArgs a) {
  using L = ChunkSmem<DK, NV, SPLIT>;
  constexpr int RS = DK / 4;      // state rows per warp
  constexpr int MTS = RS / 16;    // state m-tiles per warp
  constexpr int NT = NV / 8;      // n-tiles of a value slice
  constexpr int VK = DK / 8;      // 8-wide vectors per key row
  constexpr int VN = NV / 8;      // 8-wide vectors per value-slice row
  extern __shared__ __align__(128) unsigned char smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slice = blockIdx.x, h = blockIdx.y, bb = blockIdx.z;
  const int T = a.T, H = a.H, DV = a.dv;
  const bool CH = a.flags & 1u, ER = a.flags & 2u, WR = a.flags & 4u, QM = a.flags & 8u;
  const int col0 = slice * NV;
  const int fr = lane >> 2, fc = (lane & 3) * 2;  // accumulator fragment row / column

  const Tile X0{reinterpret_cast<__nv_bfloat16*>(smem + L::oX0), L::LDK, 64 * L::LDK};
  const Tile X1{reinterpret_cast<__nv_bfloat16*>(smem + L::oX1), L::LDK, 64 * L::LDK};
  const Tile X2{reinterpret_cast<__nv_bfloat16*>(smem + L::oX2), L::LDK, 64 * L::LDK};
  const Tile tAqk{reinterpret_cast<__nv_bfloat16*>(smem + L::oAqk), L::LDC, 64 * L::LDC};
  const Tile tA{reinterpret_cast<__nv_bfloat16*>(smem + L::oA), L::LDC, 64 * L::LDC};
  const Tile tZ{reinterpret_cast<__nv_bfloat16*>(smem + L::oZ), L::LDN, 64 * L::LDN};
  const Tile tW{reinterpret_cast<__nv_bfloat16*>(smem + L::oW), L::LDN, 64 * L::LDN};
  const Tile tS{reinterpret_cast<__nv_bfloat16*>(smem + L::oS), L::LDN, DK * L::LDN};
  float* sT = reinterpret_cast<float*>(smem + L::oT);    // [64][65]: T
  float* sG = reinterpret_cast<float*>(smem + L::oGA);   // [64][DK]: G (channel gates)
  float* sAf = sG;                                       // [64][65]: A, after the gates are used
  float* sP = reinterpret_cast<float*>(smem + L::oP);    // [3][16][16]
  float* sBeta = reinterpret_cast<float*>(smem + L::oVec);
  float* sLam = sBeta + 64;
  float* sGs = sLam + 64;     // [64] G for scalar gates
  float* sGL = sGs + 64;      // [DK] G at the chunk's last row
  float* sGC = sGL + DK;      // [DK] gamma_C = exp(G_last)

  const TIn* q = static_cast<const TIn*>(a.q);
  const TIn* k = static_cast<const TIn*>(a.k);
  const TIn* v = static_cast<const TIn*>(a.v);
  const TIn* gb = static_cast<const TIn*>(a.b);
  const TIn* gw = static_cast<const TIn*>(a.w);
  TIn* o = static_cast<TIn*>(a.o);

  // ---- initial state of this (batch, head, slice), fp32 in registers ----
  float accS[MTS][NT][4];
  const size_t state_base = (size_t(bb) * H + h) * DK * DV + col0;
#pragma unroll
  for (int mt = 0; mt < MTS; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = warp * RS + mt * 16 + fr + hf * 8, c = nt * 8 + fc;
        float2 s = make_float2(0.f, 0.f);
        if (a.h0) s = *reinterpret_cast<const float2*>(a.h0 + state_base + size_t(r) * DV + c);
        accS[mt][nt][2 * hf] = s.x;
        accS[mt][nt][2 * hf + 1] = s.y;
        put2<SPLIT>(tS, r, c, s.x, s.y);
      }

  const int n_chunks = (T + kChunk - 1) / kChunk;
  for (int n = 0; n < n_chunks; ++n) {
    const int t0 = n * kChunk;
    const int Lr = min(kChunk, T - t0);
    const size_t row0 = size_t(bb) * T + t0;  // (batch, token) row of the chunk's first token
    __syncthreads();  // the previous chunk is done with every tile

    // ---- gates: in-chunk inclusive cumsum of g (fp32), beta, lam ----
    if (CH) {
      for (int c = tid; c < DK; c += kThreads) {
        const float* gp = a.g + (row0 * H + h) * DK + c;
        float acc = 0.f;
#pragma unroll 8
        for (int r = 0; r < kChunk; ++r) {
          const float gv = r < Lr ? __ldg(gp + size_t(r) * H * DK) : 0.f;
          acc += gv;
          sG[r * DK + c] = acc;
        }
        sGL[c] = acc;
        sGC[c] = gexp<SPLIT>(acc);
      }
    } else if (warp == 0) {
      float g0 = lane < Lr ? __ldg(a.g + (row0 + lane) * H + h) : 0.f;
      float g1 = lane + 32 < Lr ? __ldg(a.g + (row0 + lane + 32) * H + h) : 0.f;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float u0 = __shfl_up_sync(0xffffffffu, g0, off);
        const float u1 = __shfl_up_sync(0xffffffffu, g1, off);
        if (lane >= off) { g0 += u0; g1 += u1; }
      }
      g1 += __shfl_sync(0xffffffffu, g0, 31);
      sGs[lane] = g0;
      sGs[lane + 32] = g1;
      const float tot = __shfl_sync(0xffffffffu, g1, 31);
      const float gc = gexp<SPLIT>(tot);
      for (int c = lane; c < DK; c += 32) { sGL[c] = tot; sGC[c] = gc; }
    }
    if (tid < kChunk) {
      const size_t ti = (row0 + tid) * H + h;
      sBeta[tid] = (tid < Lr && a.beta) ? __ldg(a.beta + ti) : 0.f;
      sLam[tid] = (tid < Lr && QM) ? __ldg(a.lam + ti) : 0.f;
    }
    __syncthreads();

    // ---- prep 1: rebased E_bar, K_bar, Q' and the write rows Z ----
    for (int it = tid; it < kChunk * VK; it += kThreads) {
      const int r = it / VK, c0 = (it % VK) * 8;
      const bool valid = r < Lr;
      const size_t off = ((row0 + r) * H + h) * DK + c0;
      float qv[8], kv[8], bv[8];
      load8_or_zero(q + off, valid, qv);
      load8_or_zero(k + off, valid, kv);
      if (ER) load8_or_zero(gb + off, valid, bv);
      float Eb[8], Kb[8], Qr[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = c0 + j;
        const float G = CH ? sG[r * DK + c] : sGs[r];
        const float rho = 0.5f * sGL[c];
        const float x = QM ? kv[j] + sLam[r] * qv[j] : kv[j];
        const float e = ER ? bv[j] * x : sBeta[r] * x;
        // scalar gates: raw factors here, the decay exp(G_r - G_i) <= 1 is
        // applied per element of T and A_qk in step 1
        const float f = CH ? gexp<SPLIT>(G - rho) : 1.f;
        const float fi = CH ? gexp<SPLIT>(rho - G) : 1.f;
        Eb[j] = f * e;
        Kb[j] = fi * kv[j];
        Qr[j] = a.scale * f * qv[j];
      }
      put8<SPLIT>(X0, r, c0, Eb);
      put8<SPLIT>(X1, r, c0, Kb);
      put8<SPLIT>(X2, r, c0, Qr);
    }
    for (int it = tid; it < kChunk * VN; it += kThreads) {
      const int r = it / VN, c0 = (it % VN) * 8;
      const bool valid = r < Lr;
      const size_t off = ((row0 + r) * H + h) * DV + col0 + c0;
      float vv[8], wv[8], z[8];
      load8_or_zero(v + off, valid, vv);
      if (WR) load8_or_zero(gw + off, valid, wv);
#pragma unroll
      for (int j = 0; j < 8; ++j) z[j] = WR ? wv[j] * vv[j] : sBeta[r] * vv[j];
      put8<SPLIT>(tZ, r, c0, z);
    }
    __syncthreads();

    // ---- step 1: T = tril(E_bar K_bar^T, -1) and A_qk = tril(Q' K_bar^T, 0) ----
    {
      float accT[8][4], accQ[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) { accT[nt][i] = 0.f; accQ[nt][i] = 0.f; }
      warp_gemm<DK, 8, false, false, SPLIT>(accT, X0, warp * 16, X1, 0);
      warp_gemm<DK, 8, false, false, SPLIT>(accQ, X2, warp * 16, X1, 0);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int r = warp * 16 + fr + hf * 8, c = nt * 8 + fc;
          float d0 = 1.f, d1 = 1.f;  // exp(G_r - G_i) for scalar gates
          if (!CH) {
            d0 = c <= r ? gexp<SPLIT>(sGs[r] - sGs[c]) : 0.f;
            d1 = c + 1 <= r ? gexp<SPLIT>(sGs[r] - sGs[c + 1]) : 0.f;
          }
          sT[r * L::LDT + c] = c < r ? d0 * accT[nt][2 * hf] : 0.f;
          sT[r * L::LDT + c + 1] = c + 1 < r ? d1 * accT[nt][2 * hf + 1] : 0.f;
          put2<SPLIT>(tAqk, r, c, c <= r ? d0 * accQ[nt][2 * hf] : 0.f,
                      c + 1 <= r ? d1 * accQ[nt][2 * hf + 1] : 0.f);
        }
    }
    __syncthreads();

    // ---- prep 2: E_abs = gamma (.) E, Q_gamma = s gamma (.) q, K_tail ----
    for (int it = tid; it < kChunk * VK; it += kThreads) {
      const int r = it / VK, c0 = (it % VK) * 8;
      const bool valid = r < Lr;
      const size_t off = ((row0 + r) * H + h) * DK + c0;
      float qv[8], kv[8], bv[8];
      load8_or_zero(q + off, valid, qv);
      load8_or_zero(k + off, valid, kv);
      if (ER) load8_or_zero(gb + off, valid, bv);
      float Ea[8], Qg[8], Kt[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = c0 + j;
        const float G = CH ? sG[r * DK + c] : sGs[r];
        const float x = QM ? kv[j] + sLam[r] * qv[j] : kv[j];
        const float e = ER ? bv[j] * x : sBeta[r] * x;
        const float f = gexp<SPLIT>(G);
        Ea[j] = f * e;
        Qg[j] = a.scale * f * qv[j];
        Kt[j] = gexp<SPLIT>(sGL[c] - G) * kv[j];
      }
      put8<SPLIT>(X0, r, c0, Ea);
      put8<SPLIT>(X1, r, c0, Qg);
      put8<SPLIT>(X2, r, c0, Kt);
    }
    __syncthreads();

    // ---- step 2: A = (I + T)^{-1} by forward substitution, fp32 ----
    // Diagonal 16x16 blocks: warp w inverts block w; lane c < 16 owns column c.
    if (lane < 16) {
      const int base = warp * 16;
      float col[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < r; ++i) acc += sT[(base + r) * L::LDT + base + i] * col[i];
        col[r] = (r == lane ? 1.f : 0.f) - acc;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) sAf[(base + r) * L::LDT + base + lane] = col[r];
    }
    __syncthreads();
    // Off-diagonal blocks by distance d = I - J:
    //   A_IJ = -A_II * sum_{K=J}^{I-1} T_IK A_KJ
#pragma unroll 1
    for (int d = 1; d < 4; ++d) {
      const int nb = 4 - d;
      for (int e = tid; e < nb * 256; e += kThreads) {
        const int J = e >> 8, r = (e >> 4) & 15, c = e & 15, I = J + d;
        float acc = 0.f;
        for (int Kb = J; Kb < I; ++Kb) {
#pragma unroll
          for (int m = 0; m < 16; ++m)
            acc += sT[(16 * I + r) * L::LDT + 16 * Kb + m] * sAf[(16 * Kb + m) * L::LDT + 16 * J + c];
        }
        sP[J * 256 + r * 16 + c] = acc;
      }
      __syncthreads();
      for (int e = tid; e < nb * 256; e += kThreads) {
        const int J = e >> 8, r = (e >> 4) & 15, c = e & 15, I = J + d;
        float acc = 0.f;
        for (int m = 0; m <= r; ++m)
          acc += sAf[(16 * I + r) * L::LDT + 16 * I + m] * sP[J * 256 + m * 16 + c];
        sAf[(16 * I + r) * L::LDT + 16 * J + c] = -acc;
      }
      __syncthreads();
    }
    for (int it = tid; it < 64 * 8; it += kThreads) {
      const int r = it >> 3, c0 = (it & 7) * 8;
      float x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = (c0 + j <= r) ? sAf[r * L::LDT + c0 + j] : 0.f;
      put8<SPLIT>(tA, r, c0, x);
    }
    __syncthreads();

    // ---- step 3: Y = A E_abs (kept as the next A operand), U = A Z ----
    float accU[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) accU[nt][i] = 0.f;
    warp_gemm<64, NT, false, true, SPLIT>(accU, tA, warp * 16, tZ, 0);
    {
      float accY[DK / 8][4];
#pragma unroll
      for (int nt = 0; nt < DK / 8; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) accY[nt][i] = 0.f;
      warp_gemm<64, DK / 8, false, true, SPLIT>(accY, tA, warp * 16, X0, 0);
      __syncthreads();  // every warp is done reading E_abs
#pragma unroll
      for (int nt = 0; nt < DK / 8; ++nt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          put2<SPLIT>(X0, warp * 16 + fr + hf * 8, nt * 8 + fc, accY[nt][2 * hf],
                      accY[nt][2 * hf + 1]);
    }
    __syncthreads();

    // ---- step 4: the state pass across chunks ----
    float accO[NT][4];
    {
      float accYS[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) { accYS[nt][i] = 0.f; accO[nt][i] = 0.f; }
      warp_gemm<DK, NT, false, true, SPLIT>(accYS, X0, warp * 16, tS, 0);  // Y S_n
      warp_gemm<DK, NT, false, true, SPLIT>(accO, X1, warp * 16, tS, 0);   // Q_gamma S_n
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          put2<SPLIT>(tW, warp * 16 + fr + hf * 8, nt * 8 + fc,
                      accU[nt][2 * hf] - accYS[nt][2 * hf],
                      accU[nt][2 * hf + 1] - accYS[nt][2 * hf + 1]);
    }
    __syncthreads();
    warp_gemm<64, NT, false, true, SPLIT>(accO, tAqk, warp * 16, tW, 0);  // + A_qk W
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = warp * 16 + fr + hf * 8;
        if (r < Lr)
          store2(o + ((row0 + r) * H + h) * DV + col0 + nt * 8 + fc, accO[nt][2 * hf],
                 accO[nt][2 * hf + 1]);
      }
    // S_{n+1} = Diag(gamma_C) S_n + K_tail^T W
#pragma unroll
    for (int mt = 0; mt < MTS; ++mt) {
      const int rb = warp * RS + mt * 16;
      const float g0 = sGC[rb + fr], g1 = sGC[rb + fr + 8];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        accS[mt][nt][0] *= g0;
        accS[mt][nt][1] *= g0;
        accS[mt][nt][2] *= g1;
        accS[mt][nt][3] *= g1;
      }
      warp_gemm<64, NT, true, true, SPLIT>(accS[mt], X2, rb, tW, 0);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        put2<SPLIT>(tS, rb + fr, nt * 8 + fc, accS[mt][nt][0], accS[mt][nt][1]);
        put2<SPLIT>(tS, rb + fr + 8, nt * 8 + fc, accS[mt][nt][2], accS[mt][nt][3]);
      }
    }
  }

  if (a.hT) {
#pragma unroll
    for (int mt = 0; mt < MTS; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int r = warp * RS + mt * 16 + fr + hf * 8, c = nt * 8 + fc;
          store2(a.hT + state_base + size_t(r) * DV + c, accS[mt][nt][2 * hf],
                 accS[mt][nt][2 * hf + 1]);
        }
  }
}

template <int DK, int NV, bool SPLIT, typename TIn>
cudaError_t launch_one(const ChunkArgs& a, cudaStream_t stream) {
  using L = ChunkSmem<DK, NV, SPLIT>;
  static_assert(L::bytes <= 232448, "shared memory budget of one CTA");
  auto kern = chunk_fwd_kernel<DK, NV, SPLIT, TIn>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L::bytes));
  if (err != cudaSuccess) return err;
  dim3 grid(a.dv / NV, a.H, a.B);
  kern<<<grid, kThreads, L::bytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_fwd_f32(const ChunkArgs& a, int dk, cudaStream_t stream) {
  // value slices of 16 (d_k = 128) or 32 (d_k = 64) columns keep the hi/lo
  // operand planes within one CTA's shared memory
  if (dk == 64 && a.dv % 32 == 0) return launch_one<64, 32, true, float>(a, stream);
  if (dk == 128 && a.dv % 16 == 0) return launch_one<128, 16, true, float>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdr
