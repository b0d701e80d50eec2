// Chunk preparation kernel of the two-kernel chunkwise forward (bf16 inputs,
// every gate variant): the intra-chunk half of the WY/UT algorithm of the
// Gated DeltaNet-2 notes, key design 2 (Q-Delta notes, key design 3, for the
// mixed erase input), for all chunks of all (batch, head) pairs at once. Only
// the state pass is sequential in the chunk index, so this half has
// B * H * ceil(T / 64) independent CTAs and fills the GPU even when B * H is
// small.
//
// One CTA takes one chunk (128 threads, two CTAs per SM):
//   gates   G = in-chunk cumsum of g (per key channel or per row), gamma_C
//   tiles   E_bar = f (.) e, Q' = s f (.) q, K_bar = f^-1 (.) k, E_abs = gamma (.) e,
//           Z = z, and for the packet Q_gamma = s gamma (.) q, K_tail = gamma_C / gamma (.) k
//           (channel gates: f = e^{G - rho}, rho = G_C / 2, so every factor stays in range;
//           scalar gates: f = 1 and exp(G_r - G_i) <= 1 multiplies T and A_qk afterwards)
//   M1      D1 = [E_bar; Q'] K_bar^T            (tcgen05, M=128, N=64, K=d_k)
//           T = tril(D1[0:64], -1) (fp32), A_qk = tril(D1[64:128], 0) -> packet
//   UT      A = (I + T)^{-1}                   (blocked forward substitution)
//   M2      Y = A E_abs, U = A Z                (M=64, N=d_k and d_v) -> packet (-Y, U)
// The packet layout is in packet.h.
// Operands live in shared memory in the 128-byte swizzle of tc.cuh; packet
// tiles go from registers straight to global memory in the same byte layout.
#include "common.cuh"
#include "kernels.h"
#include "packet.h"
#include "tc.cuh"
#include "tri_inverse.cuh"

namespace gdr {
namespace {

constexpr int kThreads = 128;

constexpr uint32_t align1k(uint32_t x) { return (x + 1023u) & ~1023u; }

template <int DK, int DV>
struct PrepLayout {
  // region 1: [E_bar; Q'] and K_bar until M1 completes, then T and A (fp32)
  static constexpr uint32_t kInv = 2 * 64 * 65 * 4;
  static constexpr uint32_t kR1 = align1k(384 * DK > kInv ? 384 * DK : kInv);
  static constexpr uint32_t oEQ = 0;                 // 128 x DK  (A, K-major)
  static constexpr uint32_t oKb = 256 * DK;          // 64 x DK   (B, K-major)
  static constexpr uint32_t oT = 0;                  // [64][65]
  static constexpr uint32_t oAf = 64 * 65 * 4;       // [64][65]
  static constexpr uint32_t oEa = kR1;               // K=64 x DK (B, MN-major)
  static constexpr uint32_t oZ = oEa + 128 * DK;     // K=64 x DV (B, MN-major)
  static constexpr uint32_t oA = oZ + 128 * DV;      // 64 x 64   (A, K-major)
  static constexpr uint32_t oP = oA + 8192;          // [4][256] inverse scratch
  static constexpr uint32_t oPart = oP + 4096;       // per-row-block gate sums
  static constexpr uint32_t oVec = oPart + 4096;     // beta, lam, G, e^G, e^{G_C-G} [64]
  static constexpr uint32_t oBar = oVec + 5 * 64 * 4;
  static constexpr uint32_t oSlot = oBar + 16;
  static constexpr uint32_t bytes = oSlot + 16;
  static constexpr uint32_t launch_bytes = bytes + 1024;
  static constexpr uint32_t kTmemCols = (DK + DV) > 128 ? 256 : 128;
};

__device__ __forceinline__ uint4 pack8(const float* x) {
  uint4 u;
  u.x = pack_bf16x2(x[0], x[1]);
  u.y = pack_bf16x2(x[2], x[3]);
  u.z = pack_bf16x2(x[4], x[5]);
  u.w = pack_bf16x2(x[6], x[7]);
  return u;
}

__device__ __forceinline__ void st16(unsigned char* base, uint32_t off, uint4 v) {
  *reinterpret_cast<uint4*>(base + off) = v;
}

// Key-side tiles of the chunk. Thread t owns channels c0 = 8 (t % VK) .. +7 of
// the RPB consecutive rows from r0 = RPB (t / VK). With channel gates the
// in-chunk cumsum is a two-step scan: per-thread sums over its rows, then a
// prefix over row blocks through shared memory; G is never stored whole.
template <int DK, int DV, bool CH, bool ER, bool QM>
__device__ __forceinline__ void prep_keys(unsigned char* smem, unsigned char* pkt,
                                          const ChunkArgs& a, size_t row0, int h, int Lr,
                                          const float* sBeta, const float* sLam,
                                          const float* sEG, const float* sEGL, float* sPart) {
  using L = PrepLayout<DK, DV>;
  using P = Packet<DK, DV>;
  constexpr int VK = DK / 8, RB = kThreads / VK, RPB = kChunk / RB;
  const int tid = threadIdx.x, rb = tid / VK, c0 = (tid % VK) * 8, r0 = rb * RPB;
  const int H = a.H;
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* gb = static_cast<const __nv_bfloat16*>(a.b);

  float gv[CH ? RPB : 1][8];
  if (CH) {
    float ps[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) ps[j] = 0.f;
#pragma unroll
    for (int i = 0; i < RPB; ++i) {
      const int r = r0 + i;
      float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
      if (r < Lr) {
        const float4* p = reinterpret_cast<const float4*>(a.g + ((row0 + r) * H + h) * DK + c0);
        x0 = __ldg(p);
        x1 = __ldg(p + 1);
      }
      gv[i][0] = x0.x; gv[i][1] = x0.y; gv[i][2] = x0.z; gv[i][3] = x0.w;
      gv[i][4] = x1.x; gv[i][5] = x1.y; gv[i][6] = x1.z; gv[i][7] = x1.w;
#pragma unroll
      for (int j = 0; j < 8; ++j) ps[j] += gv[i][j];
    }
    float4* dst = reinterpret_cast<float4*>(sPart + rb * DK + c0);
    dst[0] = make_float4(ps[0], ps[1], ps[2], ps[3]);
    dst[1] = make_float4(ps[4], ps[5], ps[6], ps[7]);
  }
  __syncthreads();
  float G[8], rho[8], er[8];
  if (CH) {
    float tot[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) { G[j] = 0.f; tot[j] = 0.f; }
#pragma unroll
    for (int b = 0; b < RB; ++b) {
      const float4* src = reinterpret_cast<const float4*>(sPart + b * DK + c0);
      const float4 x0 = src[0], x1 = src[1];
      const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        tot[j] += x[j];
        G[j] += select_f32(b < rb, x[j], 0.f);
      }
    }
    float gc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      rho[j] = 0.5f * tot[j];
      er[j] = __expf(rho[j]);
      gc[j] = __expf(tot[j]);
    }
    if (rb == 0) {
      float4* dst = reinterpret_cast<float4*>(pkt + P::oGc + c0 * 4);
      dst[0] = make_float4(gc[0], gc[1], gc[2], gc[3]);
      dst[1] = make_float4(gc[4], gc[5], gc[6], gc[7]);
    }
  }

  // rows, in two batches with every global load of a batch issued first
  constexpr int kBatch = RPB >= 4 ? 4 : RPB;
#pragma unroll
  for (int i0 = 0; i0 < RPB; i0 += kBatch) {
    float qv[kBatch][8], kv[kBatch][8], bv[ER ? kBatch : 1][8];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int r = r0 + i0 + u;
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
    for (int u = 0; u < kBatch; ++u) {
      const int r = r0 + i0 + u;
      const float lam = sLam[r], beta = sBeta[r];
      const float ear = CH ? 0.f : sEG[r], ktr = CH ? 0.f : sEGL[r];
      float Eb[8], Qr[8], Kb[8], Ea[8], Qg[8], Kt[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float x = QM ? kv[u][j] + lam * qv[u][j] : kv[u][j];
        const float e = ER ? bv[ER ? u : 0][j] * x : beta * x;
        float f = 1.f, fi = 1.f, ea = ear, kt = ktr;
        if (CH) {
          G[j] += gv[CH ? i0 + u : 0][j];
          f = __expf(G[j] - rho[j]);
          fi = __expf(rho[j] - G[j]);
          ea = f * er[j];
          kt = fi * er[j];
        }
        Eb[j] = f * e;
        Qr[j] = a.scale * f * qv[u][j];
        Kb[j] = fi * kv[u][j];
        Ea[j] = ea * e;
        Qg[j] = a.scale * ea * qv[u][j];
        Kt[j] = kt * kv[u][j];
      }
      st16(smem, L::oEQ + tc::tile_off(128, r, c0), pack8(Eb));
      st16(smem, L::oEQ + tc::tile_off(128, 64 + r, c0), pack8(Qr));
      st16(smem, L::oKb + tc::tile_off(64, r, c0), pack8(Kb));
      st16(smem, L::oEa + tc::tile_off(64, r, c0), pack8(Ea));
      st16(pkt, P::oQY + tc::tile_off(128, r, c0), pack8(Qg));
      st16(pkt, P::oKt + tc::tile_off(64, r, c0), pack8(Kt));
    }
  }
}

// Z = beta v (or w (.) v with the write gate), all d_v columns.
template <int DK, int DV, bool WR>
__device__ __forceinline__ void prep_z(unsigned char* smem, const ChunkArgs& a, size_t row0,
                                       int h, int Lr, const float* sBeta) {
  using L = PrepLayout<DK, DV>;
  constexpr int VV = DV / 8, kIter = kChunk * VV / kThreads;
  const int tid = threadIdx.x;
  const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(a.v);
  const __nv_bfloat16* gw = static_cast<const __nv_bfloat16*>(a.w);
  float vv[kIter][8], wv[WR ? kIter : 1][8];
#pragma unroll
  for (int u = 0; u < kIter; ++u) {
    const int it = tid + u * kThreads, r = it / VV, c0 = (it % VV) * 8;
    const size_t off = ((row0 + r) * a.H + h) * DV + c0;
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
    const int it = tid + u * kThreads, r = it / VV, c0 = (it % VV) * 8;
    const float beta = sBeta[r];
    float z[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) z[j] = WR ? wv[WR ? u : 0][j] * vv[u][j] : beta * vv[u][j];
    st16(smem, L::oZ + tc::tile_off(64, r, c0), pack8(z));
  }
}

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 2)
    chunk_prep_kernel(const ChunkArgs a, unsigned char* packets, int* status) {
  using L = PrepLayout<DK, DV>;
  using P = Packet<DK, DV>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = blockIdx.x, h = blockIdx.y, bb = blockIdx.z;
  const int T = a.T, H = a.H;
  const int n_chunks = gridDim.x;
  const int t0 = n * kChunk, Lr = min(kChunk, T - t0);
  const size_t row0 = size_t(bb) * T + t0;
  const bool CH = a.flags & 1u, QM = a.flags & 8u;
  unsigned char* pkt = packets + ((size_t(bb) * H + h) * n_chunks + n) * P::bytes;

  float* sT = reinterpret_cast<float*>(smem + L::oT);
  float* sAf = reinterpret_cast<float*>(smem + L::oAf);
  float* sP = reinterpret_cast<float*>(smem + L::oP);
  float* sPart = reinterpret_cast<float*>(smem + L::oPart);
  float* sBeta = reinterpret_cast<float*>(smem + L::oVec);
  float* sLam = sBeta + 64;
  float* sGs = sLam + 64;
  float* sEG = sGs + 64;
  float* sEGL = sEG + 64;
  const uint32_t bar0 = sbase + L::oBar;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L::oSlot);

  if (warp == 0) tc::tmem_alloc(smem_u32(tslot), L::kTmemCols);
  if (tid == 32) {
    tc::mbar_init(bar0, 1);
    tc::mbar_init(bar0 + 8, 1);
    tc::fence_mbar_init();
  }

  // per-row gates: beta, lam; scalar decay: in-chunk cumsum by warp 0
  if (tid < kChunk) {
    const size_t ti = (row0 + tid) * H + h;
    sBeta[tid] = (tid < Lr && a.beta) ? __ldg(a.beta + ti) : 0.f;
    sLam[tid] = (tid < Lr && QM) ? __ldg(a.lam + ti) : 0.f;
  }
  if (!CH && warp == 1) {
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
    float* dst = reinterpret_cast<float*>(pkt + P::oGc);
    for (int c = lane; c < DK; c += 32) dst[c] = gc;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tlane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  int fail_at = -1;

  switch (a.flags & 11u) {   // CH | ER | QM select the key-side tiles
#define GDR_PREP(F)                                                                       \
  case F:                                                                                 \
    prep_keys<DK, DV, (F & 1u) != 0, (F & 2u) != 0, (F & 8u) != 0>(                       \
        smem, pkt, a, row0, h, Lr, sBeta, sLam, sEG, sEGL, sPart);                        \
    break;
    GDR_PREP(0) GDR_PREP(1) GDR_PREP(2) GDR_PREP(3)
    GDR_PREP(8) GDR_PREP(9) GDR_PREP(10) GDR_PREP(11)
#undef GDR_PREP
    default: break;
  }
  if (a.flags & 4u)
    prep_z<DK, DV, true>(smem, a, row0, h, Lr, sBeta);
  else
    prep_z<DK, DV, false>(smem, a, row0, h, Lr, sBeta);
  tc::fence_proxy_async();
  __syncthreads();

  // ---- M1: [E_bar; Q'] K_bar^T into columns 0..63 ----
  if (tid == 0) {
    tc::fence_after_sync();
    constexpr uint32_t id = tc::idesc_bf16(128, 64, 0, 0);
    const uint64_t dEQ = tc::smem_desc(sbase + L::oEQ, 16, 1024);
    const uint64_t dKb = tc::smem_desc(sbase + L::oKb, 16, 1024);
#pragma unroll
    for (int k0 = 0; k0 < DK; k0 += 16) {
      const uint32_t ka = (k0 >> 6) * (128 * 128) + (k0 & 63) * 2;
      const uint32_t kb = (k0 >> 6) * (64 * 128) + (k0 & 63) * 2;
      tc::mma_bf16(tmem, dEQ + (ka >> 4), dKb + (kb >> 4), id, k0 > 0);
    }
    tc::commit(bar0);
  }
  if (__syncthreads_or(!tc::mbar_wait(bar0, 0))) {
    fail_at = 4 * n;
  } else {
    tc::fence_after_sync();
    // ---- T (fp32, shared) and A_qk (bf16, packet); lanes 0..63 hold E_bar K_bar^T ----
    {
      const int r = tid & 63;
      const bool isT = tid < 64;
      const int lim = isT ? r : r + 1;       // T strictly lower, A_qk with the diagonal
      const float Gr = CH ? 0.f : sGs[r];
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        float x[32];
        tc::tmem_ld32(tlane + c, x);
        if (CH) {
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = select_f32(c + j < lim, x[j], 0.f);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            x[j] = select_f32(c + j < lim, __expf(fminf(Gr - sGs[c + j], 0.f)) * x[j], 0.f);
        }
        if (isT) {
#pragma unroll
          for (int j = 0; j < 32; ++j) sT[r * 65 + c + j] = x[j];
        } else {
#pragma unroll
          for (int j = 0; j < 32; j += 8) st16(pkt, P::oAqk + tc::tile_off(64, r, c + j), pack8(x + j));
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();

    // ---- A = (I + T)^{-1}, then the bf16 operand tile ----
    invert_unit_lower_64(sT, sAf, sP, warp, lane, [] { __syncthreads(); });
#pragma unroll
    for (int it = tid; it < 64 * 8; it += kThreads) {
      const int r = it >> 3, c0 = (it & 7) * 8;
      float x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = select_f32(c0 + j <= r, sAf[r * 65 + c0 + j], 0.f);
      st16(smem, L::oA + tc::tile_off(64, r, c0), pack8(x));
    }
    tc::fence_proxy_async();
    __syncthreads();

    // ---- M2: Y = A E_abs (columns 0..DK-1), U = A Z (columns DK..DK+DV-1) ----
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t idY = tc::idesc_bf16(64, DK, 0, 1);
      constexpr uint32_t idU = tc::idesc_bf16(64, DV, 0, 1);
      const uint64_t dA = tc::smem_desc(sbase + L::oA, 16, 1024);
      const uint64_t dEa = tc::smem_desc(sbase + L::oEa, 64 * 128, 1024);
      const uint64_t dZ = tc::smem_desc(sbase + L::oZ, 64 * 128, 1024);
#pragma unroll
      for (int k0 = 0; k0 < 64; k0 += 16) {
        const uint32_t kr = ((k0 / 8) * 1024) >> 4;
        tc::mma_bf16(tmem, dA + ((k0 * 2) >> 4), dEa + kr, idY, k0 > 0);
        tc::mma_bf16(tmem + DK, dA + ((k0 * 2) >> 4), dZ + kr, idU, k0 > 0);
      }
      tc::commit(bar0 + 8);
    }
    if (__syncthreads_or(!tc::mbar_wait(bar0 + 8, 0))) {
      fail_at = 4 * n + 1;
    } else {
      tc::fence_after_sync();
      // M=64 accumulators: row 16 w + l in lane l < 16 of warp w
      const int r = warp * 16 + (lane & 15);
#pragma unroll
      for (int c = 0; c < DK; c += 32) {
        float x[32];
        tc::tmem_ld32(tlane + c, x);
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = -x[j];
        if (lane < 16) {
#pragma unroll
          for (int j = 0; j < 32; j += 8)
            st16(pkt, P::oQY + tc::tile_off(128, 64 + r, c + j), pack8(x + j));
        }
      }
#pragma unroll
      for (int c = 0; c < DV; c += 32) {
        float x[32];
        tc::tmem_ld32(tlane + DK + c, x);
        if (lane < 16) {
#pragma unroll
          for (int j = 0; j < 32; j += 8) st16(pkt, P::oU + tc::tile_off(64, r, c + j), pack8(x + j));
        }
      }
    }
  }

  if (fail_at >= 0 && tid == 0 && status) {
    if (atomicCAS(status, 0, 5) == 0) {  // GDR_ERR_TIMEOUT
      status[1] = static_cast<int>((blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x);
      status[2] = fail_at;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, L::kTmemCols);
}

template <int DK, int DV>
cudaError_t launch_prep(const ChunkArgs& a, unsigned char* packets, int* status,
                        cudaStream_t stream) {
  using L = PrepLayout<DK, DV>;
  static_assert(2 * (L::launch_bytes + 1024) <= 233472, "two CTAs per SM");
  auto kern = chunk_prep_kernel<DK, DV>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L::launch_bytes));
  if (err != cudaSuccess) return err;
  const int n_chunks = (a.T + kChunk - 1) / kChunk;
  dim3 grid(n_chunks, a.H, a.B);
  kern<<<grid, kThreads, L::launch_bytes, stream>>>(a, packets, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_prep(const ChunkArgs& a, int dk, unsigned char* packets, int* status,
                              cudaStream_t stream) {
  if (dk == 64 && a.dv == 64) return launch_prep<64, 64>(a, packets, status, stream);
  if (dk == 64 && a.dv == 128) return launch_prep<64, 128>(a, packets, status, stream);
  if (dk == 128 && a.dv == 64) return launch_prep<128, 64>(a, packets, status, stream);
  if (dk == 128 && a.dv == 128) return launch_prep<128, 128>(a, packets, status, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdr
