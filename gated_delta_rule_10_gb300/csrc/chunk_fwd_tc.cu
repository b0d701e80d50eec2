// Chunkwise forward of the gated delta rule on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory), bf16 inputs.
//
// Algorithm: Gated DeltaNet-2 notes, key design 2 (chunkwise WY form with the
// cumulative decay absorbed into the rank-one factors); Q-Delta notes, key
// design 3 reuse it with the mixed erase input. One CTA owns one (batch,
// head) and a 64-wide slice of value columns; it walks the chunks of C = 64
// tokens in order. Per chunk, with S_n the state slice (d_k x 64, fp32):
//
//   M1  D1  = [E_bar ; Q'] K_bar^T            (M=128, N=64, K=d_k)
//           rows 0..63 -> T = tril(., -1) (fp32, shared memory)
//           rows 64..127 -> A_qk = tril(., 0) (bf16 operand)
//       A   = (I + T)^{-1}                    (fp32 forward substitution)
//   M2  D_Y = A E_abs,  D_U = A Z             (M=64)
//   M3  D_U += (-Y) S_n   -> W = U - Y S_n,   D_O = Q_gamma S_n   (M=64, K=d_k)
//   M4  D_O += A_qk W     -> O_n,             D_S = K_tail^T W    (M=d_k, K=64)
//       S_{n+1} = Diag(gamma_C) S_n + D_S     (fp32, one state row per thread)
//
// Operands live in shared memory in the 128-byte-swizzled layout of tc.cuh;
// one thread issues each group of MMAs and commits it to an mbarrier that the
// CTA waits on with a bounded poll. If a wait gives up, the CTA records
// GDR_ERR_TIMEOUT (and where) in the workspace status words, releases its
// tensor memory and returns.
//
// Decay factors of T and A_qk: for scalar gates the factor exp(G_r - G_i) <= 1
// multiplies each element after the product (no range limit); for per-channel
// gates E_bar, K_bar and Q' carry exp(+-(G_r - rho)) with rho = G_C / 2 per
// key channel (the rho factors cancel in the products).
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tri_inverse.cuh"

namespace gdr {
namespace {

constexpr int kTcThreads = 128;
constexpr int kNV = 64;                    // value columns per CTA
constexpr uint32_t kTmemCols = 512;

template <int DK>
struct TcLayout {
  // bf16 operand tiles, each a multiple of 1024 bytes
  static constexpr uint32_t oEQ = 0;                       // [E_bar; Q']  128 x DK (A, K-major)
  static constexpr uint32_t oKb = oEQ + 128 * DK * 2;      // K_bar        64 x DK  (B, K-major)
  static constexpr uint32_t oA = oKb + 64 * DK * 2;        // A            64 x 64  (A, K-major)
  static constexpr uint32_t oAqk = oA + 64 * 64 * 2;       // A_qk         64 x 64  (A, K-major)
  static constexpr uint32_t oEa = oAqk + 64 * 64 * 2;      // E_abs     K=64 x DK   (B, MN-major)
  static constexpr uint32_t oZ = oEa + 64 * DK * 2;        // Z         K=64 x 64   (B, MN-major)
  static constexpr uint32_t oY = oZ + 64 * kNV * 2;        // -Y           64 x DK  (A, K-major)
  static constexpr uint32_t oQg = oY + 64 * DK * 2;        // Q_gamma      64 x DK  (A, K-major)
  static constexpr uint32_t oKt = oQg + 64 * DK * 2;       // K_tail    K=64 x DK   (A, MN-major)
  static constexpr uint32_t oS = oKt + 64 * DK * 2;        // S_n      K=DK x 64    (B, MN-major)
  static constexpr uint32_t oW = oS + DK * kNV * 2;        // W        K=64 x 64    (B, MN-major)
  // fp32 work areas
  static constexpr uint32_t oT = oW + 64 * kNV * 2;        // [64][65] T
  static constexpr uint32_t kG = 64 * DK * 4;              // [64][DK] G (channel gates)
  static constexpr uint32_t kAf = 64 * 65 * 4;             // [64][65] A (aliases G)
  static constexpr uint32_t oGA = oT + 64 * 65 * 4;
  static constexpr uint32_t oP = oGA + (kG > kAf ? kG : kAf);  // [4][256] inverse scratch
  static constexpr uint32_t oVec = oP + 4 * 256 * 4;       // beta, lam, Gs, eG, eGL [64] each
  static constexpr uint32_t oCh = oVec + 5 * 64 * 4;       // GL, gC, e^rho [DK] each
  static constexpr uint32_t oBar = (oCh + 3 * DK * 4 + 7) & ~7u;  // 4 mbarriers
  static constexpr uint32_t oSlot = oBar + 4 * 8;          // TMEM base address
  static constexpr uint32_t bytes = oSlot + 16;
  static constexpr uint32_t launch_bytes = bytes + 1024;   // slack to align the base
};

// TMEM column map (fp32 accumulators, lanes = rows)
template <int DK>
struct TmemMap {
  static constexpr uint32_t D1 = 0;                 // 64 columns
  static constexpr uint32_t DY = 64;                // DK columns
  static constexpr uint32_t DU = 64 + DK;           // 64
  static constexpr uint32_t DO = DU + kNV;          // 64
  static constexpr uint32_t DS = DO + kNV;          // 64
};

__device__ __forceinline__ void st_shared_16(unsigned char* base, uint32_t off, uint4 v) {
  *reinterpret_cast<uint4*>(base + off) = v;
}

__device__ __forceinline__ uint4 pack8(const float* x) {
  uint4 u;
  u.x = pack_bf16x2(x[0], x[1]);
  u.y = pack_bf16x2(x[2], x[3]);
  u.z = pack_bf16x2(x[4], x[5]);
  u.w = pack_bf16x2(x[6], x[7]);
  return u;
}

// Operand tiles of one chunk from the raw rows (flags as template parameters,
// so no per-element branch on them). Each thread takes 8-channel vectors of
// rows it, it + 16, ...; all its global loads are issued before any use.
// Channel gates: f = e^{G-rho}, fi = e^{rho-G} per element and, with
// rho = G_C / 2, e^G = f e^rho and e^{G_C - G} = fi e^rho (two exps each).
template <int DK, bool CH, bool ER, bool QM>
__device__ __forceinline__ void prep_tiles(unsigned char* smem, const ChunkArgs& a,
                                           const __nv_bfloat16* q, const __nv_bfloat16* k,
                                           const __nv_bfloat16* gb, size_t row0, int H, int h,
                                           int Lr, const float* sG, const float* sGL,
                                           const float* sER, const float* sBeta,
                                           const float* sLam, const float* sEG,
                                           const float* sEGL) {
  using L = TcLayout<DK>;
  constexpr int VK = DK / 8;
  constexpr int kIter = 4;                                  // vectors in flight per thread
  constexpr int kPasses = kChunk * VK / kTcThreads / kIter;
  const int tid = threadIdx.x;
#pragma unroll 1
  for (int pass = 0; pass < kPasses; ++pass) {
  float qv[kIter][8], kv[kIter][8], bv[ER ? kIter : 1][8];
#pragma unroll
  for (int u = 0; u < kIter; ++u) {
    const int it = tid + (pass * kIter + u) * kTcThreads;
    const int r = it / VK, c0 = (it % VK) * 8;
    const size_t off = ((row0 + r) * H + h) * DK + c0;
    if (r < Lr) {
      load8(q + off, qv[u]);
      load8(k + off, kv[u]);
      if (ER) load8(gb + off, bv[ER ? u : 0]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        qv[u][j] = 0.f;
        kv[u][j] = 0.f;
        if (ER) bv[ER ? u : 0][j] = 0.f;
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kIter; ++u) {
    const int it = tid + (pass * kIter + u) * kTcThreads;
    const int r = it / VK, c0 = (it % VK) * 8;
    const float lam = sLam[r], beta = sBeta[r];
    const float ear = CH ? 0.f : sEG[r], ktr = CH ? 0.f : sEGL[r];
    float Eb[8], Qr[8], Kb[8], Ea[8], Qg[8], Kt[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = c0 + j;
      const float x = QM ? kv[u][j] + lam * qv[u][j] : kv[u][j];
      const float e = ER ? bv[ER ? u : 0][j] * x : beta * x;
      float f = 1.f, fi = 1.f, ea = ear, kt = ktr;
      if (CH) {
        const float G = sG[r * DK + c], rho = 0.5f * sGL[c], er = sER[c];
        f = __expf(G - rho);
        fi = __expf(rho - G);
        ea = f * er;
        kt = fi * er;
      }
      Eb[j] = f * e;
      Qr[j] = a.scale * f * qv[u][j];
      Kb[j] = fi * kv[u][j];
      Ea[j] = ea * e;
      Qg[j] = a.scale * ea * qv[u][j];
      Kt[j] = kt * kv[u][j];
    }
    st_shared_16(smem, L::oEQ + tc::tile_off(128, r, c0), pack8(Eb));
    st_shared_16(smem, L::oEQ + tc::tile_off(128, 64 + r, c0), pack8(Qr));
    st_shared_16(smem, L::oKb + tc::tile_off(64, r, c0), pack8(Kb));
    st_shared_16(smem, L::oEa + tc::tile_off(64, r, c0), pack8(Ea));
    st_shared_16(smem, L::oQg + tc::tile_off(64, r, c0), pack8(Qg));
    st_shared_16(smem, L::oKt + tc::tile_off(64, r, c0), pack8(Kt));
  }
  }
}

template <int DK, bool WR>
__device__ __forceinline__ void prep_z(unsigned char* smem, const __nv_bfloat16* v,
                                       const __nv_bfloat16* gw, size_t row0, int H, int h,
                                       int DV, int col0, int Lr, const float* sBeta) {
  using L = TcLayout<DK>;
  constexpr int kIter = kChunk * (kNV / 8) / kTcThreads;
  const int tid = threadIdx.x;
  float vv[kIter][8], wv[WR ? kIter : 1][8];
#pragma unroll
  for (int u = 0; u < kIter; ++u) {
    const int it = tid + u * kTcThreads;
    const int r = it / (kNV / 8), c0 = (it % (kNV / 8)) * 8;
    const size_t off = ((row0 + r) * H + h) * DV + col0 + c0;
    if (r < Lr) {
      load8(v + off, vv[u]);
      if (WR) load8(gw + off, wv[WR ? u : 0]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        vv[u][j] = 0.f;
        if (WR) wv[WR ? u : 0][j] = 0.f;
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kIter; ++u) {
    const int it = tid + u * kTcThreads;
    const int r = it / (kNV / 8), c0 = (it % (kNV / 8)) * 8;
    const float beta = sBeta[r];
    float z[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) z[j] = WR ? wv[WR ? u : 0][j] * vv[u][j] : beta * vv[u][j];
    st_shared_16(smem, L::oZ + tc::tile_off(64, r, c0), pack8(z));
  }
}

template <int DK>
__global__ void __launch_bounds__(kTcThreads, 1)
    chunk_fwd_tc_kernel(const ChunkArgs a, int* status) {
  using L = TcLayout<DK>;
  using TM = TmemMap<DK>;
  extern __shared__ unsigned char smem_raw[];
  // aligned by pointer arithmetic on the shared array, so the compiler keeps
  // every access below in the shared state space
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slice = blockIdx.x, h = blockIdx.y, bb = blockIdx.z;
  const int T = a.T, H = a.H, DV = a.dv;
  const bool CH = a.flags & 1u, WR = a.flags & 4u, QM = a.flags & 8u;
  const int col0 = slice * kNV;

  float* sT = reinterpret_cast<float*>(smem + L::oT);
  float* sG = reinterpret_cast<float*>(smem + L::oGA);
  float* sAf = sG;
  float* sP = reinterpret_cast<float*>(smem + L::oP);
  float* sBeta = reinterpret_cast<float*>(smem + L::oVec);
  float* sLam = sBeta + 64;
  float* sGs = sLam + 64;    // scalar gates: G_r
  float* sEG = sGs + 64;     // scalar gates: exp(G_r)
  float* sEGL = sEG + 64;    // scalar gates: exp(G_C - G_r)
  float* sGL = reinterpret_cast<float*>(smem + L::oCh);  // [DK] G_C
  float* sGC = sGL + DK;                                 // [DK] gamma_C
  float* sER = sGC + DK;                                 // [DK] e^{rho}, rho = G_C / 2
  const uint32_t bar0 = sbase + L::oBar;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L::oSlot);

  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(a.v);
  const __nv_bfloat16* gb = static_cast<const __nv_bfloat16*>(a.b);
  const __nv_bfloat16* gw = static_cast<const __nv_bfloat16*>(a.w);
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.o);

  if (warp == 0) tc::tmem_alloc(smem_u32(tslot), kTmemCols);
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) tc::mbar_init(bar0 + 8 * i, 1);
    tc::fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tlane = tmem + (static_cast<uint32_t>(warp * 32) << 16);  // this warp's lanes

  // ---- state rows: thread -> key channel s_row (all NV value columns) ----
  const bool s_owner = (DK == 128) || (lane < 16);
  const int s_row = (DK == 128) ? tid : warp * 16 + (lane & 15);
  float S[kNV];
  {
    const size_t base = ((size_t(bb) * H + h) * DK + s_row) * DV + col0;
#pragma unroll
    for (int j = 0; j < kNV; j += 4) {
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (a.h0 && s_owner) x = *reinterpret_cast<const float4*>(a.h0 + base + j);
      S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
    }
    if (s_owner) {
#pragma unroll
      for (int j = 0; j < kNV; j += 8)
        st_shared_16(smem, L::oS + tc::tile_off(DK, s_row, j), pack8(S + j));
    }
  }

  int fail_at = -1;
  const int n_chunks = (T + kChunk - 1) / kChunk;
  for (int n = 0; n < n_chunks; ++n) {
    const int t0 = n * kChunk;
    const int Lr = min(kChunk, T - t0);
    const size_t row0 = size_t(bb) * T + t0;
    const uint32_t par = static_cast<uint32_t>(n & 1);
    tc::fence_before_sync();
    __syncthreads();

    // ---- gates: in-chunk cumsum of g (fp32), beta, lam ----
    if (CH) {
      for (int c = tid; c < DK; c += kTcThreads) {
        const float* gp = a.g + (row0 * H + h) * DK + c;
        float acc = 0.f;
#pragma unroll 8
        for (int r = 0; r < kChunk; ++r) {
          const float gv = r < Lr ? __ldg(gp + size_t(r) * H * DK) : 0.f;
          acc += gv;
          sG[r * DK + c] = acc;
        }
        sGL[c] = acc;
        sGC[c] = __expf(acc);
        sER[c] = __expf(0.5f * acc);
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
      const float tot = __shfl_sync(0xffffffffu, g1, 31);
      sGs[lane] = g0;
      sGs[lane + 32] = g1;
      sEG[lane] = __expf(g0);
      sEG[lane + 32] = __expf(g1);
      sEGL[lane] = __expf(tot - g0);
      sEGL[lane + 32] = __expf(tot - g1);
      const float gc = __expf(tot);
      for (int c = lane; c < DK; c += 32) { sGL[c] = tot; sGC[c] = gc; }
    }
    if (tid < kChunk) {
      const size_t ti = (row0 + tid) * H + h;
      sBeta[tid] = (tid < Lr && a.beta) ? __ldg(a.beta + ti) : 0.f;
      sLam[tid] = (tid < Lr && QM) ? __ldg(a.lam + ti) : 0.f;
    }
    __syncthreads();

    // ---- operand tiles of the chunk ----
    switch (a.flags & 11u) {   // CH | ER | QM select the key-side tiles
#define GDR_PREP(F)                                                                        \
  case F:                                                                                  \
    prep_tiles<DK, (F & 1u) != 0, (F & 2u) != 0, (F & 8u) != 0>(smem, a, q, k, gb, row0, H, h, \
                                                                Lr, sG, sGL, sER, sBeta, sLam, \
                                                                sEG, sEGL);                \
    break;
      GDR_PREP(0) GDR_PREP(1) GDR_PREP(2) GDR_PREP(3)
      GDR_PREP(8) GDR_PREP(9) GDR_PREP(10) GDR_PREP(11)
#undef GDR_PREP
      default: break;
    }
    if (WR)
      prep_z<DK, true>(smem, v, gw, row0, H, h, DV, col0, Lr, sBeta);
    else
      prep_z<DK, false>(smem, v, gw, row0, H, h, DV, col0, Lr, sBeta);
    tc::fence_proxy_async();
    __syncthreads();

    // ---- M1: [E_bar; Q'] K_bar^T ----
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t id = tc::idesc_bf16(128, 64, 0, 0);
      const uint64_t dEQ = tc::smem_desc(sbase + L::oEQ, 16, 1024);
      const uint64_t dKb = tc::smem_desc(sbase + L::oKb, 16, 1024);
#pragma unroll
      for (int k0 = 0; k0 < DK; k0 += 16) {
        const uint32_t ka = (k0 >> 6) * (128 * 128) + (k0 & 63) * 2;
        const uint32_t kb = (k0 >> 6) * (64 * 128) + (k0 & 63) * 2;
        tc::mma_bf16(tmem + TM::D1, dEQ + (ka >> 4), dKb + (kb >> 4), id, k0 > 0);
      }
      tc::commit(bar0);
    }
    if (__syncthreads_or(!tc::mbar_wait(bar0, par))) { fail_at = 4 * n; break; }
    tc::fence_after_sync();

    // ---- T (fp32) and A_qk (bf16 operand) with masks and scalar decay ----
    {
      const int r = tid & 63;
      const bool isT = tid < 64;
      const float Gr = CH ? 0.f : sGs[r];
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
        float x[16];
        tc::tmem_ld16(tlane + TM::D1 + c, x);
        const int lim = isT ? r : r + 1;   // T strictly lower, A_qk with diagonal
        if (CH) {
#pragma unroll
          for (int j = 0; j < 16; ++j) x[j] = select_f32(c + j < lim, x[j], 0.f);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            x[j] = select_f32(c + j < lim, __expf(fminf(Gr - sGs[c + j], 0.f)) * x[j], 0.f);
        }
        if (isT) {
#pragma unroll
          for (int j = 0; j < 16; ++j) sT[r * 65 + c + j] = x[j];
        } else {
          st_shared_16(smem, L::oAqk + tc::tile_off(64, r, c), pack8(x));
          st_shared_16(smem, L::oAqk + tc::tile_off(64, r, c + 8), pack8(x + 8));
        }
      }
    }
    __syncthreads();

    // ---- A = (I + T)^{-1} ----
    invert_unit_lower_64(sT, sAf, sP, warp, lane, [] { __syncthreads(); });
    for (int it = tid; it < 64 * 8; it += kTcThreads) {
      const int r = it >> 3, c0 = (it & 7) * 8;
      float x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = select_f32(c0 + j <= r, sAf[r * 65 + c0 + j], 0.f);
      st_shared_16(smem, L::oA + tc::tile_off(64, r, c0), pack8(x));
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();

    // ---- M2: Y = A E_abs, U = A Z; and Q_gamma S_n ----
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t idY = tc::idesc_bf16(64, DK, 0, 1);
      constexpr uint32_t idN = tc::idesc_bf16(64, kNV, 0, 1);
      const uint64_t dA = tc::smem_desc(sbase + L::oA, 16, 1024);
      const uint64_t dEa = tc::smem_desc(sbase + L::oEa, 64 * 128, 1024);
      const uint64_t dZ = tc::smem_desc(sbase + L::oZ, 64 * 128, 1024);
      const uint64_t dQg = tc::smem_desc(sbase + L::oQg, 16, 1024);
      const uint64_t dS = tc::smem_desc(sbase + L::oS, DK * 128, 1024);
#pragma unroll
      for (int k0 = 0; k0 < 64; k0 += 16) {
        const uint32_t kr = ((k0 / 8) * 1024) >> 4;
        tc::mma_bf16(tmem + TM::DY, dA + ((k0 * 2) >> 4), dEa + kr, idY, k0 > 0);
        tc::mma_bf16(tmem + TM::DU, dA + ((k0 * 2) >> 4), dZ + kr, idN, k0 > 0);
      }
#pragma unroll
      for (int k0 = 0; k0 < DK; k0 += 16) {
        const uint32_t ka = (k0 >> 6) * (64 * 128) + (k0 & 63) * 2;
        tc::mma_bf16(tmem + TM::DO, dQg + (ka >> 4), dS + (((k0 / 8) * 1024) >> 4), idN, k0 > 0);
      }
      tc::commit(bar0 + 8);
    }
    if (__syncthreads_or(!tc::mbar_wait(bar0 + 8, par))) { fail_at = 4 * n + 1; break; }
    tc::fence_after_sync();

    // ---- -Y to shared memory (M=64 accumulator: lanes 0..15 of each quadrant) ----
#pragma unroll
    for (int c = 0; c < DK; c += 16) {
      float x[16];
      tc::tmem_ld16(tlane + TM::DY + c, x);
#pragma unroll
      for (int j = 0; j < 16; ++j) x[j] = -x[j];
      if (lane < 16) {
        const int r = warp * 16 + lane;
        st_shared_16(smem, L::oY + tc::tile_off(64, r, c), pack8(x));
        st_shared_16(smem, L::oY + tc::tile_off(64, r, c + 8), pack8(x + 8));
      }
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();

    // ---- M3: W = U - Y S_n (accumulated onto U) ----
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t idN = tc::idesc_bf16(64, kNV, 0, 1);
      const uint64_t dY = tc::smem_desc(sbase + L::oY, 16, 1024);
      const uint64_t dS = tc::smem_desc(sbase + L::oS, DK * 128, 1024);
#pragma unroll
      for (int k0 = 0; k0 < DK; k0 += 16) {
        const uint32_t ka = (k0 >> 6) * (64 * 128) + (k0 & 63) * 2;
        tc::mma_bf16(tmem + TM::DU, dY + (ka >> 4), dS + (((k0 / 8) * 1024) >> 4), idN, 1);
      }
      tc::commit(bar0 + 16);
    }
    if (__syncthreads_or(!tc::mbar_wait(bar0 + 16, par))) { fail_at = 4 * n + 2; break; }
    tc::fence_after_sync();

#pragma unroll
    for (int c = 0; c < kNV; c += 16) {
      float x[16];
      tc::tmem_ld16(tlane + TM::DU + c, x);
      if (lane < 16) {
        const int r = warp * 16 + lane;
        st_shared_16(smem, L::oW + tc::tile_off(64, r, c), pack8(x));
        st_shared_16(smem, L::oW + tc::tile_off(64, r, c + 8), pack8(x + 8));
      }
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();

    // ---- M4: O_n = Q_gamma S_n + A_qk W; D_S = K_tail^T W ----
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t idO = tc::idesc_bf16(64, kNV, 0, 1);
      constexpr uint32_t idS = tc::idesc_bf16(DK, kNV, 1, 1);
      const uint64_t dW = tc::smem_desc(sbase + L::oW, 64 * 128, 1024);
      const uint64_t dAqk = tc::smem_desc(sbase + L::oAqk, 16, 1024);
      const uint64_t dKt = tc::smem_desc(sbase + L::oKt, 64 * 128, 1024);
#pragma unroll
      for (int k0 = 0; k0 < 64; k0 += 16) {
        const uint32_t kr = ((k0 / 8) * 1024) >> 4;
        tc::mma_bf16(tmem + TM::DO, dAqk + ((k0 * 2) >> 4), dW + kr, idO, 1);
        tc::mma_bf16(tmem + TM::DS, dKt + kr, dW + kr, idS, k0 > 0);
      }
      tc::commit(bar0 + 24);
    }
    if (__syncthreads_or(!tc::mbar_wait(bar0 + 24, par))) { fail_at = 4 * n + 3; break; }
    tc::fence_after_sync();

    // ---- outputs and the next state ----
    {
      const int r = warp * 16 + (lane & 15);
      __nv_bfloat16* orow = o + ((row0 + r) * H + h) * DV + col0;
#pragma unroll
      for (int c = 0; c < kNV; c += 16) {
        float x[16];
        tc::tmem_ld16(tlane + TM::DO + c, x);
        if (lane < 16 && r < Lr) {
          *reinterpret_cast<uint4*>(orow + c) = pack8(x);
          *reinterpret_cast<uint4*>(orow + c + 8) = pack8(x + 8);
        }
      }
    }
    {
      const float gc = sGC[s_row];
#pragma unroll
      for (int c = 0; c < kNV; c += 16) {
        float x[16];
        tc::tmem_ld16(tlane + TM::DS + c, x);
#pragma unroll
        for (int j = 0; j < 16; ++j) S[c + j] = gc * S[c + j] + x[j];
        if (s_owner) {
          st_shared_16(smem, L::oS + tc::tile_off(DK, s_row, c), pack8(S + c));
          st_shared_16(smem, L::oS + tc::tile_off(DK, s_row, c + 8), pack8(S + c + 8));
        }
      }
    }
    tc::fence_proxy_async();
  }

  if (fail_at < 0 && a.hT && s_owner) {
    const size_t base = ((size_t(bb) * H + h) * DK + s_row) * DV + col0;
#pragma unroll
    for (int j = 0; j < kNV; j += 4)
      *reinterpret_cast<float4*>(a.hT + base + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
  }
  if (fail_at >= 0 && tid == 0 && status) {
    if (atomicCAS(status, 0, 5) == 0) {  // GDR_ERR_TIMEOUT
      status[1] = static_cast<int>((blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x);
      status[2] = fail_at;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

template <int DK>
cudaError_t launch_tc(const ChunkArgs& a, int* status, cudaStream_t stream) {
  using L = TcLayout<DK>;
  static_assert(L::launch_bytes <= 232448, "shared memory budget of one CTA");
  auto kern = chunk_fwd_tc_kernel<DK>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L::launch_bytes));
  if (err != cudaSuccess) return err;
  dim3 grid(a.dv / kNV, a.H, a.B);
  kern<<<grid, kTcThreads, L::launch_bytes, stream>>>(a, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_fwd_tc(const ChunkArgs& a, int dk, int* status, cudaStream_t stream) {
  if (dk == 64) return launch_tc<64>(a, status, stream);
  if (dk == 128) return launch_tc<128>(a, status, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdr
