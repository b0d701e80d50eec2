// Pipelined chunkwise forward for scalar gates (Gated DeltaNet and Q-Delta),
// bf16 inputs, on tcgen05 tensor cores fed by TMA.
//
// Same algorithm as chunk_fwd_tc.cu (Gated DeltaNet-2 notes, key design 2;
// Q-Delta notes, key design 3), rearranged so that Q, K and V go from HBM to
// the tensor cores untouched: with a scalar decay and scalar beta every gate is
// a per-row factor and folds into the small 64x64 matrices:
//
//   T_ri  = beta_r (k_r.k_i + lam_r q_r.k_i) exp(G_r - G_i)   (i < r)
//   A_qk  = s (q_r.k_i) exp(G_r - G_i)                         (i <= r)
//   A     = (I + T)^{-1}
//   Y     = A diag(beta e^G) K + A diag(beta lam e^G) Q        (= A E_abs)
//   U     = A diag(beta) V                                     (= A Z)
//   W     = U - Y S_n
//   O_n   = s diag(e^G) Q S_n + A_qk W                         (= Q_gamma S_n + A_qk W)
//   S_n+1 = e^{G_C} S_n + K^T diag(e^{G_C - G}) W              (= Diag(gamma_C) S_n + K_tail^T W)
//
// Roles (416 threads): warps 0-3 run the state pass of chunk n (S in fp32
// registers, one key channel per thread), warps 4-11 run the intra-chunk work
// of chunk n+1 (T, A_qk, the inverse, Y and U; two warps per tensor-memory lane
// quadrant split the columns), warp 12 streams the next chunks' Q, K, V tiles
// with TMA and their gates with plain loads into a two-stage ring. Groups of
// MMAs are issued from two threads in different warps, since issue, not the
// tensor core, bounds these small products. Hand-offs go through mbarriers; every wait is bounded, and a wait that
// gives up makes all roles leave their loops together, release tensor memory
// and report GDR_ERR_TIMEOUT in the status words.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tri_inverse.cuh"

namespace gdr {
namespace {

constexpr int kThreads = 416;   // 4 scan warps, 8 intra-chunk warps, 1 producer warp
constexpr int kNV = 64;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kScanBar = 1, kIntraBar = 2, kInvBar = 3;
constexpr uint32_t kIntraThreads = 256;

template <int DK>
struct PipeLayout {
  static constexpr uint32_t kKQ = DK * 256;               // K/Q blocks interleaved
  static constexpr uint32_t kStage = kKQ + 8192 + 1024;   // + V + gates (g, beta, lam)
  static constexpr uint32_t oStage = 0;                   // two stages
  static constexpr uint32_t oY = 2 * kStage;              // -Y, 64 x DK (A, K-major)
  static constexpr uint32_t oAqk = oY + DK * 128;         // two 64 x 64 (A, K-major)
  static constexpr uint32_t oRows = oAqk + 2 * 8192;      // two {e^G, e^{G_C-G}, e^{G_C}}
  static constexpr uint32_t oAy = oRows + 2 * 1024;       // A diag(beta e^G)
                                                          // (before the inverse, the three
                                                          // A tiles hold the decay matrix)
  static constexpr uint32_t oAyl = oAy + 8192;            // A diag(beta lam e^G)
  static constexpr uint32_t oAu = oAyl + 8192;            // A diag(beta)
  static constexpr uint32_t oS = oAu + 8192;              // S_n, DK x 64 (B, MN-major)
  static constexpr uint32_t oW = oS + DK * 128;           // W (B, MN-major)
  static constexpr uint32_t oW2 = oW + 8192;              // diag(e^{G_C-G}) W
  static constexpr uint32_t oT = oW2 + 8192;              // fp32 [64][65]
  static constexpr uint32_t oAf = oT + 64 * 65 * 4;       // fp32 [64][65] (also q.k for QMIX)
  static constexpr uint32_t oP = oAf + 64 * 65 * 4;       // fp32 [4][256] per-warp scratch
  static constexpr uint32_t oVec = oP + 4 * 256 * 4;      // intra: G, e^G, beta, lam, e^g [64]
  static constexpr uint32_t oBar = oVec + 5 * 64 * 4;     // mbarriers
  static constexpr int kBars = 15;
  static constexpr uint32_t oSlot = oBar + kBars * 8;
  static constexpr uint32_t oAbort = oSlot + 4;
  static constexpr uint32_t bytes = oAbort + 12;
  static constexpr uint32_t launch_bytes = bytes + 1024;
};

// barrier indices
enum : uint32_t {
  kFull0 = 0, kFree0 = 2, kReady0 = 4, kDuFree0 = 6, kAqkFree0 = 8, kTyFree = 10,
  kM1 = 11, kM2 = 12, kM3 = 13, kM4 = 14
};

template <int DK>
struct PipeTmem {
  static constexpr uint32_t D1 = 0;
  static constexpr uint32_t DY = 64;
  static constexpr uint32_t DU0 = 64 + DK;
  static constexpr uint32_t DQ = DU0 + 2 * kNV;
  static constexpr uint32_t DA = DQ + kNV;
  static constexpr uint32_t DS = DA + kNV;
};

__device__ __forceinline__ uint4 pack8f(const float* x) {
  uint4 u;
  u.x = pack_bf16x2(x[0], x[1]);
  u.y = pack_bf16x2(x[2], x[3]);
  u.z = pack_bf16x2(x[4], x[5]);
  u.w = pack_bf16x2(x[6], x[7]);
  return u;
}

// Bounded mbarrier wait (sleeping between polls) that also gives up early once
// another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t mbar, uint32_t parity,
                                              volatile int* abort_flag) {
  for (uint32_t i = 0; i < tc::kMaxPolls; ++i) {
    if (tc::mbar_try_wait(mbar, parity, tc::kSuspendNs)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

template <int DK>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_fwd_pipe_kernel(const ChunkArgs a, const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, int* status) {
  using L = PipeLayout<DK>;
  using TM = PipeTmem<DK>;
  constexpr uint32_t kStageTx = static_cast<uint32_t>(DK / 64) * 2 * 8192 + 8192;
  extern __shared__ unsigned char smem_raw[];
  // aligned by pointer arithmetic on the shared array, so the compiler keeps
  // every access below in the shared state space
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, bb = blockIdx.z;
  const int col0 = blockIdx.x * kNV;
  const int T = a.T, H = a.H, DV = a.dv;
  const bool QM = a.flags & 8u;
  const int n_chunks = (T + kChunk - 1) / kChunk;
  auto bar = [&](uint32_t i) { return sb + L::oBar + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::oAbort);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L::oSlot);

  if (warp == 0) tc::tmem_alloc(smem_u32(tslot), kTmemCols);
  if (tid == 32) {
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(bar(kFull0 + s), 2);     // expect_tx arrive + gates arrive
      tc::mbar_init(bar(kFree0 + s), 1);
      tc::mbar_init(bar(kReady0 + s), 1);
      tc::mbar_init(bar(kDuFree0 + s), 1);
      tc::mbar_init(bar(kAqkFree0 + s), 1);
    }
    tc::mbar_init(bar(kTyFree), 1);
    tc::mbar_init(bar(kM1), 1);
    for (uint32_t i = kM2; i <= kM4; ++i) tc::mbar_init(bar(i), 2);   // two issuing threads
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tlane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  int fail = -1;

  if (warp == 12) {
    // ------------------------------------------------------------ producer
    int issued = 0;
    for (int n = 0; n < n_chunks; ++n) {
      const int s = n & 1;
      if (n >= 2 && !wait_or_abort(bar(kFree0 + s), ((n - 2) >> 1) & 1, abort_flag)) {
        fail = 4 * n;
        break;
      }
      const uint32_t st = sb + L::oStage + s * L::kStage;
      const int t0 = n * kChunk;
      if (lane == 0) {
        tc::mbar_arrive_expect_tx(bar(kFull0 + s), kStageTx);
#pragma unroll
        for (int blk = 0; blk < DK / 64; ++blk) {
          tc::tma_load_4d(st + (2 * blk) * 8192, &tm_k, blk * 64, h, t0, bb, bar(kFull0 + s));
          tc::tma_load_4d(st + (2 * blk + 1) * 8192, &tm_q, blk * 64, h, t0, bb, bar(kFull0 + s));
        }
        tc::tma_load_4d(st + L::kKQ, &tm_v, col0, h, t0, bb, bar(kFull0 + s));
      }
      issued = n + 1;
      float* gst = reinterpret_cast<float*>(smem + L::oStage + s * L::kStage + L::kKQ + 8192);
      const int Lr = min(kChunk, T - t0);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int r = lane + 32 * half;
        const size_t ti = (size_t(bb) * T + t0 + r) * H + h;
        gst[r] = r < Lr ? __ldg(a.g + ti) : 0.f;
        gst[64 + r] = r < Lr ? __ldg(a.beta + ti) : 0.f;
        gst[128 + r] = (r < Lr && QM) ? __ldg(a.lam + ti) : 0.f;
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar(kFull0 + s));
    }
    // let the loads already issued land before the CTA can exit (a plain
    // bounded wait: an abort elsewhere does not stop a copy in flight)
    for (int n = max(0, issued - 2); n < issued; ++n)
      tc::mbar_wait(bar(kFull0 + (n & 1)), (n >> 1) & 1);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ intra-chunk
    const int it = tid - 128;          // 0 .. 255
    const int half = it >> 7;          // which of the two warps sharing a lane quadrant
    const int w4 = warp & 3;           // lane quadrant of this warp
    float* sT = reinterpret_cast<float*>(smem + L::oT);
    float* sAf = reinterpret_cast<float*>(smem + L::oAf);
    float* sQK = sAf;
    float* sP = reinterpret_cast<float*>(smem + L::oP);
    float* vG = reinterpret_cast<float*>(smem + L::oVec);
    float* vEG = vG + 64;
    float* vBeta = vEG + 64;
    float* vLam = vBeta + 64;
    float* vAl = vLam + 64;     // exp(g_r)
    const float* sD = reinterpret_cast<const float*>(smem + L::oAy);
    auto issue_m1 = [&](uint32_t stage) {   // M1: [K; Q] K^T (M=128, N=64, K=DK), raw tiles
      tc::fence_after_sync();
      constexpr uint32_t id = tc::idesc_bf16(128, 64, 0, 0);
      // descriptors built once per group; K steps advance the address field
      const uint64_t dst = tc::smem_desc(stage, 16, 1024);
#pragma unroll
      for (int k0 = 0; k0 < DK; k0 += 16) {
        const uint32_t kb = (k0 >> 6) * 16384 + (k0 & 63) * 2;
        tc::mma_bf16(tmem + TM::D1, dst + (kb >> 4), dst + (kb >> 4), id, k0 > 0);
      }
      tc::commit(bar(kM1));
    };
    for (int n = 0; n < n_chunks; ++n) {
      const int s = n & 1;
      const uint32_t st = sb + L::oStage + s * L::kStage;
      const float* gst = reinterpret_cast<const float*>(smem + L::oStage + s * L::kStage + L::kKQ + 8192);
      bool ok = wait_or_abort(bar(kFull0 + s), (n >> 1) & 1, abort_flag);
      if (tc::named_any(kIntraBar, kIntraThreads, !ok)) { fail = 4 * n; break; }

      // gates of the chunk: G (in-chunk cumsum), per-row factors. Thread r of
      // the first 64 sums g_0 .. g_r itself from broadcast shared-memory reads
      // (warp shuffles measured far slower here while the tensor memory is busy).
      if (it < 64) {
        const int r = it;
        float G = 0.f, GL = 0.f;
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
          const float4 g4 = *reinterpret_cast<const float4*>(gst + j);
          G += select_f32(j <= r, g4.x, 0.f) + select_f32(j + 1 <= r, g4.y, 0.f) +
               select_f32(j + 2 <= r, g4.z, 0.f) + select_f32(j + 3 <= r, g4.w, 0.f);
          GL += (g4.x + g4.y) + (g4.z + g4.w);
        }
        float* rows = reinterpret_cast<float*>(smem + L::oRows + s * 1024);
        const float e = __expf(G);
        vG[r] = G;
        vEG[r] = e;
        vBeta[r] = gst[64 + r];
        vLam[r] = gst[128 + r];
        vAl[r] = __expf(gst[r]);
        rows[r] = e;
        rows[64 + r] = __expf(GL - G);
        if (r == 0) rows[128] = __expf(GL);
      }
      tc::named_sync(kIntraBar, kIntraThreads);

      // decay matrix D[r][i] = exp(G_r - G_i) for i <= r: thread (i, p) fills
      // column i over rows 16p .. 16p+15 as a running product of exp(g_j),
      // started from exp(G_{16p-1} - G_i) (one exponential per thread)
      {
        float* sDw = reinterpret_cast<float*>(smem + L::oAy);
        const int i = it & 63, p = it >> 6, bi = i >> 4;
        if (p >= bi) {
          float d = p == bi ? 1.f : __expf(vG[max(16 * p - 1, 0)] - vG[i]);
          float al[16];
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            const float4 a4 = *reinterpret_cast<const float4*>(vAl + 16 * p + j);
            al[j] = a4.x; al[j + 1] = a4.y; al[j + 2] = a4.z; al[j + 3] = a4.w;
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            d = select_f32(16 * p + j > i, d * al[j], d);
            sDw[(16 * p + j) * 68 + i] = d;
          }
        }
      }
      // M1 of chunk 0 (later chunks are issued one chunk ahead, below)
      if (n == 0 && it == 0) issue_m1(st);
      ok = wait_or_abort(bar(kM1), n & 1, abort_flag);
      if (tc::named_any(kIntraBar, kIntraThreads, !ok)) { fail = 4 * n + 1; break; }
      tc::fence_after_sync();

      // T (fp32) and A_qk (bf16): rows r of K K^T sit in lanes 0..63,
      // rows r of Q K^T in lanes 64..127
      {
        const int r = it & 63;
        const bool isK = w4 < 2;           // lanes 0..63: K K^T, lanes 64..127: Q K^T
        const int cbeg = 32 * half;        // this warp's half of the 64 columns
        if (!isK) {
          // A_qk[n%2] is free once the state pass of chunk n-2 has used it
          ok = n < 2 || wait_or_abort(bar(kAqkFree0 + s), ((n - 2) >> 1) & 1, abort_flag);
        }
        if (tc::named_any(kIntraBar, kIntraThreads, !ok)) { fail = 4 * n + 2; break; }
        const uint32_t aqk = L::oAqk + s * 8192;
        const float br = vBeta[r], lr = vLam[r];
#pragma unroll
        for (int c = cbeg; c < cbeg + 32; c += 16) {
          float x[16], dr[16], y[16];
#pragma unroll
          for (int j = 0; j < 16; j += 4) {       // decay row first, then the stores
            const float4 d4 = *reinterpret_cast<const float4*>(sD + r * 68 + c + j);
            dr[j] = d4.x; dr[j + 1] = d4.y; dr[j + 2] = d4.z; dr[j + 3] = d4.w;
          }
          tc::tmem_ld16(tlane + TM::D1 + c, x);
          // warp-uniform cases outside the element loop, only selects inside
          if (isK && QM) {
#pragma unroll
            for (int j = 0; j < 16; ++j) y[j] = x[j];
          } else {
            const float f = isK ? br : a.scale;
            const int lim = isK ? r : r + 1;     // T strictly lower, A_qk with diagonal
#pragma unroll
            for (int j = 0; j < 16; ++j) y[j] = select_f32(c + j < lim, f * dr[j] * x[j], 0.f);
          }
          if (isK) {
#pragma unroll
            for (int j = 0; j < 16; ++j) sT[r * 65 + c + j] = y[j];
          } else {
            *reinterpret_cast<uint4*>(smem + aqk + tc::tile_off(64, r, c)) = pack8f(y);
            *reinterpret_cast<uint4*>(smem + aqk + tc::tile_off(64, r, c + 8)) = pack8f(y + 8);
            if (QM) {
#pragma unroll
              for (int j = 0; j < 16; ++j) sQK[r * 65 + c + j] = lr * x[j];
            }
          }
        }
        tc::fence_before_sync();
        if (QM) {
          tc::named_sync(kIntraBar, kIntraThreads);
          if (isK) {
#pragma unroll
            for (int c = cbeg; c < cbeg + 32; c += 16) {
              float t[16], dr[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                t[j] = sT[r * 65 + c + j] + sQK[r * 65 + c + j];
                dr[j] = sD[r * 68 + c + j];
              }
#pragma unroll
              for (int j = 0; j < 16; ++j)
                sT[r * 65 + c + j] = select_f32(c + j < r, br * dr[j] * t[j], 0.f);
            }
          }
        }
      }
      tc::named_sync(kIntraBar, kIntraThreads);
      // A = (I + T)^{-1} on the first four intra warps. Meanwhile one thread of
      // the other four starts M1 of the next chunk (every read of D1 is done),
      // so that its issue and latency hide behind the inverse.
      if (half == 0) {
        invert_unit_lower_64(sT, sAf, sP, w4, lane, [] { tc::named_sync(kInvBar, 128); });
      } else if (it == 128 && n + 1 < n_chunks) {
        const int s1 = (n + 1) & 1;
        ok = wait_or_abort(bar(kFull0 + s1), ((n + 1) >> 1) & 1, abort_flag);
        if (ok) issue_m1(sb + L::oStage + s1 * L::kStage);
      }
      if (tc::named_any(kIntraBar, kIntraThreads, !ok)) { fail = 4 * n + 2; break; }
      // A with the gates folded into its columns, as bf16 operands
#pragma unroll
      for (int rep = 0; rep < 2; ++rep) {
        const int e = it + 256 * rep;
        const int r = e >> 3, c0 = (e & 7) * 8;
        float ay[8], ayl[8], au[8], xa[8], vb[8], ve[8], vl[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          xa[j] = sAf[r * 65 + c0 + j];
          vb[j] = vBeta[c0 + j];
          ve[j] = vEG[c0 + j];
          vl[j] = vLam[c0 + j];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float x = select_f32(c0 + j <= r, xa[j], 0.f);
          au[j] = x * vb[j];
          ay[j] = au[j] * ve[j];
          ayl[j] = ay[j] * vl[j];
        }
        *reinterpret_cast<uint4*>(smem + L::oAy + tc::tile_off(64, r, c0)) = pack8f(ay);
        *reinterpret_cast<uint4*>(smem + L::oAu + tc::tile_off(64, r, c0)) = pack8f(au);
        if (QM) *reinterpret_cast<uint4*>(smem + L::oAyl + tc::tile_off(64, r, c0)) = pack8f(ayl);
      }
      tc::fence_proxy_async();
      tc::named_sync(kIntraBar, kIntraThreads);

      // M2: Y = A_y K (+ A_yl Q) from one thread; U = A_u V into D_U[n%2] from
      // another, once the state pass of chunk n-2 has released D_U[n%2]
      if (it == 0) {
        tc::fence_after_sync();
        constexpr uint32_t idY = tc::idesc_bf16(64, DK, 0, 1);
        const uint64_t dAy = tc::smem_desc(sb + L::oAy, 16, 1024);
        const uint64_t dAyl = tc::smem_desc(sb + L::oAyl, 16, 1024);
        const uint64_t dK = tc::smem_desc(st, 16384, 1024);          // K as MN-major B
        const uint64_t dQ = tc::smem_desc(st + 8192, 16384, 1024);   // Q as MN-major B
#pragma unroll
        for (int k0 = 0; k0 < 64; k0 += 16)
          tc::mma_bf16(tmem + TM::DY, dAy + ((k0 * 2) >> 4), dK + (((k0 / 8) * 1024) >> 4), idY,
                       k0 > 0);
        if (QM) {
#pragma unroll
          for (int k0 = 0; k0 < 64; k0 += 16)
            tc::mma_bf16(tmem + TM::DY, dAyl + ((k0 * 2) >> 4), dQ + (((k0 / 8) * 1024) >> 4),
                         idY, 1);
        }
        tc::commit(bar(kM2));
      } else if (it == 128) {
        ok = n < 2 || wait_or_abort(bar(kDuFree0 + s), ((n - 2) >> 1) & 1, abort_flag);
        if (ok) {
          tc::fence_after_sync();
          constexpr uint32_t idU = tc::idesc_bf16(64, kNV, 0, 1);
          const uint64_t dAu = tc::smem_desc(sb + L::oAu, 16, 1024);
          const uint64_t dV = tc::smem_desc(st + L::kKQ, 8192, 1024);
#pragma unroll
          for (int k0 = 0; k0 < 64; k0 += 16)
            tc::mma_bf16(tmem + TM::DU0 + s * kNV, dAu + ((k0 * 2) >> 4),
                         dV + (((k0 / 8) * 1024) >> 4), idU, k0 > 0);
          tc::commit(bar(kM2));
        }
      }
      if (tc::named_any(kIntraBar, kIntraThreads, !ok)) { fail = 4 * n + 3; break; }
      ok = wait_or_abort(bar(kM2), n & 1, abort_flag);
      // -Y goes to the hand-off tile once the state pass of chunk n-1 has read it
      if (ok && n >= 1) ok = wait_or_abort(bar(kTyFree), (n - 1) & 1, abort_flag);
      if (tc::named_any(kIntraBar, kIntraThreads, !ok)) { fail = 4 * n + 3; break; }
      tc::fence_after_sync();
#pragma unroll
      for (int c = half * (DK / 2); c < (half + 1) * (DK / 2); c += 16) {
        float x[16];
        tc::tmem_ld16(tlane + TM::DY + c, x);
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = -x[j];
        if (lane < 16) {
          const int r = w4 * 16 + lane;
          *reinterpret_cast<uint4*>(smem + L::oY + tc::tile_off(64, r, c)) = pack8f(x);
          *reinterpret_cast<uint4*>(smem + L::oY + tc::tile_off(64, r, c + 8)) = pack8f(x + 8);
        }
      }
      tc::fence_proxy_async();
      tc::fence_before_sync();
      tc::named_sync(kIntraBar, kIntraThreads);
      if (it == 0) tc::mbar_arrive(bar(kReady0 + s));
    }
  } else {
    // ------------------------------------------------------------ state pass
    const bool owner = (DK == 128) || (lane < 16);
    const int srow = (DK == 128) ? tid : warp * 16 + (lane & 15);
    float S[kNV];
    {
      const size_t base = ((size_t(bb) * H + h) * DK + srow) * DV + col0;
#pragma unroll
      for (int j = 0; j < kNV; j += 4) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.h0 && owner) x = *reinterpret_cast<const float4*>(a.h0 + base + j);
        S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
      }
      if (owner) {
#pragma unroll
        for (int j = 0; j < kNV; j += 8)
          *reinterpret_cast<uint4*>(smem + L::oS + tc::tile_off(DK, srow, j)) = pack8f(S + j);
      }
      tc::fence_proxy_async();
      tc::named_sync(kScanBar, 128);
    }
    const int orow = warp * 16 + (lane & 15);   // output row held by this thread
    for (int n = 0; n < n_chunks; ++n) {
      const int s = n & 1;
      const uint32_t st = sb + L::oStage + s * L::kStage;
      const int t0 = n * kChunk;
      const int Lr = min(kChunk, T - t0);
      bool ok = wait_or_abort(bar(kReady0 + s), (n >> 1) & 1, abort_flag);
      if (tc::named_any(kScanBar, 128, !ok)) { fail = 4 * n; break; }
      const float* rows = reinterpret_cast<const float*>(smem + L::oRows + s * 1024);
      const float eg = rows[orow], egl = rows[64 + orow], gc = rows[128];

      // M3: W = U - Y S_n (onto D_U) from thread 0, D_Q = Q S_n from thread 32
      if (tid == 0 || tid == 32) {
        tc::fence_after_sync();
        constexpr uint32_t idN = tc::idesc_bf16(64, kNV, 0, 1);
        const uint64_t dS = tc::smem_desc(sb + L::oS, DK * 128, 1024);
        if (tid == 0) {
          const uint64_t dY = tc::smem_desc(sb + L::oY, 16, 1024);
#pragma unroll
          for (int k0 = 0; k0 < DK; k0 += 16) {
            const uint32_t ky = (k0 >> 6) * 8192 + (k0 & 63) * 2;
            tc::mma_bf16(tmem + TM::DU0 + s * kNV, dY + (ky >> 4), dS + (((k0 / 8) * 1024) >> 4),
                         idN, 1);
          }
        } else {
          const uint64_t dQ = tc::smem_desc(st, 16, 1024);
#pragma unroll
          for (int k0 = 0; k0 < DK; k0 += 16) {
            const uint32_t kq = (k0 >> 6) * 16384 + 8192 + (k0 & 63) * 2;
            tc::mma_bf16(tmem + TM::DQ, dQ + (kq >> 4), dS + (((k0 / 8) * 1024) >> 4), idN,
                         k0 > 0);
          }
        }
        tc::commit(bar(kM3));
      }
      ok = wait_or_abort(bar(kM3), n & 1, abort_flag);
      if (tc::named_any(kScanBar, 128, !ok)) { fail = 4 * n + 1; break; }
      tc::fence_after_sync();
      if (tid == 0) tc::mbar_arrive(bar(kTyFree));

#pragma unroll
      for (int c = 0; c < kNV; c += 16) {
        float x[16];
        tc::tmem_ld16(tlane + TM::DU0 + s * kNV + c, x);
        if (lane < 16) {
          *reinterpret_cast<uint4*>(smem + L::oW + tc::tile_off(64, orow, c)) = pack8f(x);
          *reinterpret_cast<uint4*>(smem + L::oW + tc::tile_off(64, orow, c + 8)) = pack8f(x + 8);
#pragma unroll
          for (int j = 0; j < 16; ++j) x[j] *= egl;
          *reinterpret_cast<uint4*>(smem + L::oW2 + tc::tile_off(64, orow, c)) = pack8f(x);
          *reinterpret_cast<uint4*>(smem + L::oW2 + tc::tile_off(64, orow, c + 8)) = pack8f(x + 8);
        }
      }
      tc::fence_proxy_async();
      tc::fence_before_sync();
      tc::named_sync(kScanBar, 128);

      // M4: D_A = A_qk W from thread 0; D_S = K^T W2 from thread 32
      if (tid == 0) tc::mbar_arrive(bar(kDuFree0 + s));
      if (tid == 0 || tid == 32) {
        tc::fence_after_sync();
        if (tid == 0) {
          constexpr uint32_t idO = tc::idesc_bf16(64, kNV, 0, 1);
          const uint64_t dAqk = tc::smem_desc(sb + L::oAqk + s * 8192, 16, 1024);
          const uint64_t dW = tc::smem_desc(sb + L::oW, 8192, 1024);
#pragma unroll
          for (int k0 = 0; k0 < 64; k0 += 16)
            tc::mma_bf16(tmem + TM::DA, dAqk + ((k0 * 2) >> 4), dW + (((k0 / 8) * 1024) >> 4),
                         idO, k0 > 0);
        } else {
          constexpr uint32_t idS = tc::idesc_bf16(DK, kNV, 1, 1);
          const uint64_t dW2 = tc::smem_desc(sb + L::oW2, 8192, 1024);
          const uint64_t dK = tc::smem_desc(st, 16384, 1024);   // K as MN-major A
#pragma unroll
          for (int k0 = 0; k0 < 64; k0 += 16) {
            const uint32_t kr = ((k0 / 8) * 1024) >> 4;
            tc::mma_bf16(tmem + TM::DS, dK + kr, dW2 + kr, idS, k0 > 0);
          }
        }
        tc::commit(bar(kM4));
      }
      ok = wait_or_abort(bar(kM4), n & 1, abort_flag);
      if (tc::named_any(kScanBar, 128, !ok)) { fail = 4 * n + 2; break; }
      tc::fence_after_sync();
      if (tid == 0) {
        tc::mbar_arrive(bar(kFree0 + s));
        tc::mbar_arrive(bar(kAqkFree0 + s));
      }

      // O_n = s e^{G_r} (Q S_n)_r + (A_qk W)_r
      {
        __nv_bfloat16* op = static_cast<__nv_bfloat16*>(a.o) +
                            ((size_t(bb) * T + t0 + orow) * H + h) * DV + col0;
        const float sq = a.scale * eg;
#pragma unroll
        for (int c = 0; c < kNV; c += 16) {
          float xq[16], xa[16];
          tc::tmem_ld16(tlane + TM::DQ + c, xq);
          tc::tmem_ld16(tlane + TM::DA + c, xa);
#pragma unroll
          for (int j = 0; j < 16; ++j) xq[j] = sq * xq[j] + xa[j];
          if (lane < 16 && orow < Lr) {
            *reinterpret_cast<uint4*>(op + c) = pack8f(xq);
            *reinterpret_cast<uint4*>(op + c + 8) = pack8f(xq + 8);
          }
        }
      }
      // S_{n+1} = e^{G_C} S_n + K^T diag(e^{G_C - G}) W
#pragma unroll
      for (int c = 0; c < kNV; c += 16) {
        float x[16];
        tc::tmem_ld16(tlane + TM::DS + c, x);
#pragma unroll
        for (int j = 0; j < 16; ++j) S[c + j] = gc * S[c + j] + x[j];
        if (owner) {
          *reinterpret_cast<uint4*>(smem + L::oS + tc::tile_off(DK, srow, c)) = pack8f(S + c);
          *reinterpret_cast<uint4*>(smem + L::oS + tc::tile_off(DK, srow, c + 8)) = pack8f(S + c + 8);
        }
      }
      tc::fence_proxy_async();
      tc::fence_before_sync();
      tc::named_sync(kScanBar, 128);
    }
    if (fail < 0 && a.hT && owner) {
      const size_t base = ((size_t(bb) * H + h) * DK + srow) * DV + col0;
#pragma unroll
      for (int j = 0; j < kNV; j += 4)
        *reinterpret_cast<float4*>(a.hT + base + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
  }

  if (fail >= 0 && status && (lane == 0)) {
    if (atomicCAS(status, 0, 5) == 0) {  // GDR_ERR_TIMEOUT
      status[1] = static_cast<int>((blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x);
      status[2] = fail;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

template <int DK>
cudaError_t launch_pipe(const ChunkArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, int* status, cudaStream_t stream) {
  using L = PipeLayout<DK>;
  static_assert(L::launch_bytes <= 232448, "shared memory budget of one CTA");
  auto kern = chunk_fwd_pipe_kernel<DK>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L::launch_bytes));
  if (err != cudaSuccess) return err;
  dim3 grid(a.dv / kNV, a.H, a.B);
  kern<<<grid, kThreads, L::launch_bytes, stream>>>(a, tq, tk, tv, status);
  return cudaGetLastError();
}

}  // namespace

bool chunk_fwd_pipe_supports(unsigned flags) { return (flags & 7u) == 0; }

cudaError_t launch_chunk_fwd_pipe(const ChunkArgs& a, int dk, const CUtensorMap& tq,
                                  const CUtensorMap& tk, const CUtensorMap& tv, int* status,
                                  cudaStream_t stream) {
  if (dk == 64) return launch_pipe<64>(a, tq, tk, tv, status, stream);
  if (dk == 128) return launch_pipe<128>(a, tq, tk, tv, status, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdr
