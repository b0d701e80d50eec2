// Chunk scan kernel, transposed form (bf16 inputs, d_k = d_v = 128, every gate
// variant but the per-value-channel write strength): the cross-chunk state
// pass of the Gated DeltaNet-2 notes, key design 2,
//
//   W_n     = U_n - Y_n S_n
//   O_n     = Q_gamma,n S_n + A_qk,n W_n
//   S_{n+1} = Diag(gamma_C,n) S_n + K_tail,n^T W_n
//
// written for the tensor cores with the state on the A side. One CTA owns one
// (batch, head) and all d_v value columns; tensor-memory lane c holds value
// column c, so the products run transposed, with S^T and W^T read by the MMAs
// straight from tensor memory (bf16, written there by the threads that own
// them) and the packet tiles as the B operands:
//   MMA1  S_n^T [Q_gamma; -Y]^T  -> D1[n%2]   (N=128: columns 0..63 (Q_gamma S_n)^T,
//                                              64..127 (-Y S_n)^T)
//   MMA2  W^T K_tail             -> D_S       (N=d_k, after W^T = U^T + columns 64..127)
//   MMA3  W^T A_qk^T            += D1[n%2]   (N=64: columns 0..63 become O_n^T)
// A tcgen05.mma instruction costs ~70-100 cycles of tensor-pipe time whatever
// its N up to 128, so the chunk takes the fewest instructions (16, K=16 each)
// at the widest N rather than splitting the read-out part of MMA1 off the
// chain (measured slower: 24 instructions per chunk).
// Neither S nor W passes through shared memory: the fp32 state stays in
// registers (one value column and half of the key channels per thread), its
// bf16 copy and W^T go to tensor memory with tcgen05.st. The packets carry U^T
// (d_v rows of 64 tokens; packet.h) for this kernel.
// Roles (384 threads):
//   warps 0-7   the chain, two per tensor-memory lane quadrant (key channels,
//               or tokens of W, split in halves between the two); thread 0
//               issues MMA1 and MMA2
//   warps 8-11  the output: thread 256 issues MMA3 once MMA2 has completed
//               (it then runs while the chain updates S), all four warps move
//               O_n^T from D1[n%2] to o (lane c writes column c of the chunk's
//               64 rows); thread 256 also refills the three-stage packet ring
//               with plain bulk copies
// Every wait is bounded; a wait that gives up makes all roles leave together,
// release tensor memory and report GDR_ERR_TIMEOUT.
//
// With channel decay the packets are rho-folded (chunk_prep.cu, prep_keys_rf):
// they carry Q', -A E_bar and K_bar in place of Q_gamma, -Y and K_tail, plus
// e^{rho} per key channel (rho = G_C / 2), and MMA1 needs diag(e^{rho_n}) S_n.
// The registers therefore hold the scaled state S^_n = diag(e^{rho_n}) S_n,
// whose update needs one factor per key channel: since gamma_C = e^{2 rho},
//   S^_{n+1} = e^{rho_{n+1}} (gamma_C S_n + e^{rho_n} K_bar^T W)
//            = e^{rho_{n+1} + rho_n} (.) (S^_n + K_bar^T W),
// with e^{rho} of the chunk after the last taken as 1, so that the last update
// yields S itself for hT.
//
// Sequence split and time segments (ScanSegments) as in chunk_scan.cu; the
// identity slices of a split are a second CTA per run whose lanes are the d_k
// columns of the run's transition.
#include "common.cuh"
#include "kernels.h"
#include "packet.h"
#include "tc.cuh"
#include "tma.h"

namespace gdr {
namespace {

constexpr int kStages = 3;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kChainBar = 1, kOutBar = 2;
constexpr uint32_t kOutThreads = 128;
// CW chain warps per tensor-memory lane quadrant: 4 CW chain warps, then 4
// output warps
template <int CW>
struct Roles {
  static constexpr int kChainThreads = 128 * CW;
  static constexpr int kOut = kChainThreads;   // first thread of the output role
  static constexpr int kThreads = kChainThreads + kOutThreads;
};
// tensor-memory columns
constexpr uint32_t D10 = 0;        // two accumulators of 128 columns: [O^T | (-Y S)^T]
constexpr uint32_t DS = 256;       // W^T K_tail (d_k columns)
constexpr uint32_t SA = 384;       // S^T as bf16 pairs (d_k / 2 columns): A of MMA1
constexpr uint32_t WA = 448;       // W^T as bf16 pairs (32 columns): A of MMA2 and MMA3

enum : uint32_t {
  kFull0 = 0, kEmpty0 = 3, kBW = 6, kBS = 7, kBO0 = 8, kOFree0 = 10, kZFull0 = 12, kBars = 14
};

template <int DK, bool GATE>
struct TLayout {
  using P = Packet<DK, 128>;
  // the fused epilogue adds a two-slot ring of z tiles and a double-buffered y
  // tile that a TMA store writes out (two packet stages then); the packet
  // stages go back to the ring as soon as MMA3 is done with them
  static constexpr int kNS = GATE ? 2 : kStages;
  static constexpr uint32_t kStage = P::bytes;
  static constexpr uint32_t oZ = kNS * kStage;                    // [2] z tiles
  static constexpr uint32_t oY = oZ + (GATE ? 2 * 16384 : 0);     // [2] y tiles
  static constexpr uint32_t oRed = oY + (GATE ? 2 * 16384 : 0);   // [2][4][64] row sums
  static constexpr uint32_t oM = oRed + (GATE ? 2 * 4 * 64 * 4 : 0);   // RF: update factor
  static constexpr uint32_t oBar = oM + DK * 4;
  static constexpr uint32_t oSlot = oBar + kBars * 8;
  static constexpr uint32_t oAbort = oSlot + 4;
  static constexpr uint32_t bytes = oAbort + 12;
  static constexpr uint32_t launch_bytes = bytes + 1024;
  static_assert(kStage % 1024 == 0 && oZ % 1024 == 0 && oY % 1024 == 0, "tile alignment");
};

__device__ __forceinline__ void unpack8(uint4 u, float* x) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// Polls `mbar` without sleeping for up to `spins` tests first: the chain's
// waits for its own MMAs end within a few hundred cycles, and a sleeping
// waiter wakes up noticeably later than that.
__device__ __forceinline__ bool spin_test(uint32_t mbar, uint32_t parity, int spins) {
  for (int i = 0; i < spins; ++i)
    if (tc::mbar_test(mbar, parity)) return true;
  return false;
}

// tanh by the special-function unit (one instruction, about 2^-11 relative
// error); SiLU below takes sigmoid(z) = (1 + tanh(z / 2)) / 2, one
// special-function operation per element instead of an exponential and a
// reciprocal, which the output role's epilogue is bound by.
__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded mbarrier wait that also gives up once another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t mbar, uint32_t parity,
                                              volatile int* abort_flag) {
  if (tc::mbar_test(mbar, parity)) return true;
  for (uint32_t i = 0; i < tc::kMaxPolls; ++i) {
    if (tc::mbar_try_wait(mbar, parity, tc::kSuspendNs)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

template <int DK, int CW, bool RF, bool GATE>
__global__ void __launch_bounds__(Roles<CW>::kThreads, 1)
    chunk_scan_t_kernel(const ChunkArgs a, const unsigned char* packets, int* status,
                        const ScanSegments sg, const __grid_constant__ CUtensorMap tm_z,
                        const __grid_constant__ CUtensorMap tm_o) {
  constexpr int DV = 128;
  constexpr int KH = DK / CW;      // key channels per chain thread
  constexpr int TW = 64 / CW;      // tokens of W per chain thread
  constexpr int kChainThreads = Roles<CW>::kChainThreads, kOut = Roles<CW>::kOut;
  using L = TLayout<DK, GATE>;
  using P = Packet<DK, DV>;
  constexpr int kStages = L::kNS;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, bb = blockIdx.z / sg.segments, seg = blockIdx.z % sg.segments;
  const int T = a.T, H = a.H;
  const bool hom = blockIdx.x >= 1;   // the identity slice of a split run
  const int SW = hom ? DK : DV;       // width of this CTA's state (= 128 lanes)
  const int n_chunks = (T + kChunk - 1) / kChunk;
  const int c_begin = sg.chunk0 + seg * sg.seg_chunks;
  const int cnt = max(0, min(n_chunks, c_begin + sg.seg_chunks) - c_begin);
  const unsigned char* pk0 = packets + ((size_t(bb) * H + h) * n_chunks + c_begin) * P::bytes;
  const size_t run = (size_t(bb) * H + h) * sg.segments + seg;
  float* const hT = hom ? sg.hT_hom
                        : (sg.hT_per_seg ? a.hT : (seg == sg.segments - 1 ? a.hT : nullptr));
  const size_t hT_idx = (hom || sg.hT_per_seg) ? run : (size_t(bb) * H + h);
  const float* const h0 = hom ? nullptr : (sg.h0_per_seg ? a.h0 : (seg == 0 ? a.h0 : nullptr));
  const size_t h0_idx = sg.h0_per_seg ? run : (size_t(bb) * H + h);
  __nv_bfloat16* const out = hom ? nullptr : static_cast<__nv_bfloat16*>(a.o);
  auto bar = [&](uint32_t i) { return sb + L::oBar + 8 * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::oAbort);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L::oSlot);

  if (warp == 0) tc::tmem_alloc(smem_u32(tslot), kTmemCols);
  if (tid == 32) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(bar(kFull0 + s), 1);
      tc::mbar_init(bar(kEmpty0 + s), 2);   // chain and output each release the stage
    }
    tc::mbar_init(bar(kBW), 1);
    tc::mbar_init(bar(kBS), 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(bar(kBO0 + i), 1);
      tc::mbar_init(bar(kOFree0 + i), 1);
      tc::mbar_init(bar(kZFull0 + i), 1);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  const int q = warp & 3, c = 32 * q + lane;      // lane quadrant; value (state) column
  const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
  int fail = -1;

  auto load_chunk = [&](int n) {   // thread kOut only
    const int s = n % kStages;
    tc::mbar_arrive_expect_tx(bar(kFull0 + s), L::kStage);
    tc::bulk_load(sb + s * L::kStage, pk0 + size_t(n) * P::bytes, P::bytes, bar(kFull0 + s));
  };
  auto load_z = [&](int n) {   // thread kOut only: the chunk's z rows (past T: zeros)
    const int zs = n & 1;
    tc::mbar_arrive_expect_tx(bar(kZFull0 + zs), 16384);
#pragma unroll
    for (int blk = 0; blk < DV / 64; ++blk)
      tc::tma_load_4d(sb + L::oZ + zs * 16384 + blk * 8192, &tm_z, blk * 64, h,
                      (c_begin + n) * kChunk, bb, bar(kZFull0 + zs));
  };
  const bool zring = GATE && out != nullptr;

  if (warp < 4 * CW) {
    // ------------------------------------------------------------ state chain
    const int half = warp >> 2;                    // key channels KH*half.., tokens TW*half..
    float S[KH];                                   // S[KH*half + j][c]
#pragma unroll
    for (int j = 0; j < KH; ++j) {
      const int k = KH * half + j;
      S[j] = h0 ? h0[(h0_idx * DK + k) * SW + c] : 0.f;
      if (hom) S[j] = (k == c) ? 1.f : 0.f;
    }
    // this thread's part of S^T (the scaled state under RF) as bf16 into SA
    constexpr bool rf = RF;
    auto store_sa = [&]() {
#pragma unroll
      for (int p = 0; p < KH / 32; ++p) {
        uint32_t r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = pack_bf16x2(S[32 * p + 2 * i], S[32 * p + 2 * i + 1]);
        tc::tmem_st16(tl + SA + (KH / 2) * half + 16 * p, r);
      }
      tc::tmem_st_wait();
    };
    static_assert(KH % 32 == 0 && (TW == 32 || TW == 16), "chain split");
    // RF: S^_0 = diag(e^{rho_0}) S_0, once chunk 0's packet has landed
    bool ok0 = !rf || cnt == 0 || spin_test(bar(kFull0), 0, 4096) ||
               wait_or_abort(bar(kFull0), 0, abort_flag);
    ok0 = __all_sync(0xffffffffu, ok0);
    if (rf && ok0 && cnt > 0) {
      const float* e0 = reinterpret_cast<const float*>(smem + P::oGc) + DK + KH * half;
#pragma unroll
      for (int j = 0; j < KH; ++j) S[j] *= e0[j];
    }
    if (ok0) store_sa();
    // RF, warp 1: e^{rho} of the chunk after the current one, read from the
    // packets in global memory (complete before this launch) two chunks ahead,
    // so that the update factor never waits for the packet ring
    float rho_next[DK / 32];
    auto load_rho = [&](int m) {   // chunk m of this run, m < cnt
      const float* src = reinterpret_cast<const float*>(pk0 + size_t(m) * P::bytes + P::oGc) + DK;
#pragma unroll
      for (int i = 0; i < DK / 32; ++i) rho_next[i] = __ldg(src + 32 * i + lane);
    };
    if (rf && warp == 1 && cnt > 1) load_rho(1);
    tc::fence_before_sync();
    if (tc::named_any(kChainBar, kChainThreads, !ok0)) fail = 0;
    for (int n = 0; n < (fail < 0 ? cnt : 0); ++n) {
      const int s = n % kStages;
      const uint32_t st = sb + s * L::kStage;
      const unsigned char* sst = smem + s * L::kStage;
      const uint32_t d1 = D10 + (n & 1) * 128;
      bool ok = true;
      if (tid == 0) {
        // MMA1 once the packet has landed and D1[n%2] has been read out (chunk
        // n-2); for n > 0 thread 0 waited for both before the previous barrier
        if (n == 0) ok = wait_or_abort(bar(kFull0), 0, abort_flag);
        if (ok) {
          tc::fence_after_sync();
          constexpr uint32_t id1 = tc::idesc_bf16(128, 128, 0, 0);
          const uint64_t dQY = tc::smem_desc(st + P::oQY, 16, 1024);
#pragma unroll
          for (int k0 = 0; k0 < DK; k0 += 16) {
            const uint32_t kb = (k0 >> 6) * 16384 + (k0 & 63) * 2;
            tc::mma_bf16_ta(tmem + d1, tmem + SA + k0 / 2, dQY + (kb >> 4), id1, k0 > 0);
          }
          tc::commit(bar(kBW));
        } else {
          *abort_flag = 1;   // the waits below give up at once
        }
      }
      __syncwarp();
      // W^T = U^T + (-Y S)^T for tokens 32*half .. +31, once MMA1 has completed
      // and MMA3 of chunk n-1 (which reads the previous W^T) is done
      ok = ok && (spin_test(bar(kBW), n & 1, 4096) || wait_or_abort(bar(kBW), n & 1, abort_flag));
      if (ok && n >= 1)
        ok = wait_or_abort(bar(kBO0 + ((n - 1) & 1)), ((n - 1) >> 1) & 1, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc::fence_after_sync();
        float x[TW];
        if constexpr (TW == 32)
          tc::tmem_ld32(tl + d1 + 64 + TW * half, x);
        else
          tc::tmem_ld16(tl + d1 + 64 + TW * half, x);
        if (!hom) {   // U = 0 for the identity slices: the transition alone
#pragma unroll
          for (int j = 0; j < TW / 8; ++j) {
            float u[8];
            unpack8(*reinterpret_cast<const uint4*>(sst + P::oU +
                                                    tc::tile_off(128, c, TW * half + 8 * j)), u);
#pragma unroll
            for (int i = 0; i < 8; ++i) x[8 * j + i] += u[i];
          }
        }
        uint32_t r[TW / 2];
#pragma unroll
        for (int i = 0; i < TW / 2; ++i) r[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
        if constexpr (TW == 32)
          tc::tmem_st16(tl + WA + (TW / 2) * half, r);
        else
          tc::tmem_st8(tl + WA + (TW / 2) * half, r);
        tc::tmem_st_wait();
      }
      if (rf && warp == 1 && ok) {
        // m = e^{rho_n} e^{rho_{n+1}} per key channel for this chunk's update (the
        // next chunk's factor is 1 after the last chunk); then e^{rho_{n+2}}
        const float* en = reinterpret_cast<const float*>(sst + P::oGc) + DK;
        float mv[DK / 32];
#pragma unroll
        for (int i = 0; i < DK / 32; ++i)
          mv[i] = n + 1 < cnt ? en[32 * i + lane] * rho_next[i] : en[32 * i + lane];
        float* sm = reinterpret_cast<float*>(smem + L::oM);
#pragma unroll
        for (int i = 0; i < DK / 32; ++i) sm[32 * i + lane] = mv[i];
        if (n + 2 < cnt) load_rho(n + 2);
      }
      if (tid == 0 && n + 1 < cnt && ok) {
        // meanwhile: the next chunk's packet and its D1 buffer (read out for chunk n-1)
        ok = wait_or_abort(bar(kFull0 + (n + 1) % kStages), ((n + 1) / kStages) & 1, abort_flag);
        if (ok && n >= 1)
          ok = wait_or_abort(bar(kOFree0 + ((n + 1) & 1)), ((n - 1) >> 1) & 1, abort_flag);
      }
      tc::fence_before_sync();
      if (tc::named_any(kChainBar, kChainThreads, !ok)) { fail = 4 * n + 1; break; }
      // MMA2: W^T K_tail into D_S; MMA3: W^T A_qk^T onto the O part of D1[n%2]
      if (tid == 0) {
        tc::fence_after_sync();
        constexpr uint32_t id2 = tc::idesc_bf16(128, DK, 0, 1);
        const uint64_t dKt = tc::smem_desc(st + P::oKt, 64 * 128, 1024);
#pragma unroll
        for (int k0 = 0; k0 < 64; k0 += 16)
          tc::mma_bf16_ta(tmem + DS, tmem + WA + k0 / 2, dKt + (((k0 / 8) * 1024) >> 4), id2,
                          k0 > 0);
        tc::commit(bar(kBS));
      }
      __syncwarp();
      // S_{n+1} = Diag(gamma_C) S_n + K_tail^T W (MMA2 completing implies that
      // MMA1 ran, so the stage had landed for the gamma_C read)
      ok = spin_test(bar(kBS), n & 1, 4096) || wait_or_abort(bar(kBS), n & 1, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc::fence_after_sync();
        static_assert(KH == 64, "one 64-column load per thread");
        float x[64];
        tc::tmem_ld64(tl + DS + KH * half, x);
        if constexpr (rf) {
          // S^_{n+1} = m (.) (S^_n + K_bar^T W), m = e^{rho_n + rho_{n+1}} from shared memory
          const float4* m4 = reinterpret_cast<const float4*>(smem + L::oM) + (KH / 4) * half;
#pragma unroll
          for (int j = 0; j < 64; j += 4) {
            const float4 m = m4[j / 4];
            S[j] = m.x * (S[j] + x[j]);
            S[j + 1] = m.y * (S[j + 1] + x[j + 1]);
            S[j + 2] = m.z * (S[j + 2] + x[j + 2]);
            S[j + 3] = m.w * (S[j + 3] + x[j + 3]);
          }
        } else {
          const float4* gc4 = reinterpret_cast<const float4*>(sst + P::oGc) + (KH / 4) * half;
#pragma unroll
          for (int j = 0; j < 64; j += 4) {
            const float4 g = gc4[j / 4];
            S[j] = fmaf(g.x, S[j], x[j]);
            S[j + 1] = fmaf(g.y, S[j + 1], x[j + 1]);
            S[j + 2] = fmaf(g.z, S[j + 2], x[j + 2]);
            S[j + 3] = fmaf(g.w, S[j + 3], x[j + 3]);
          }
        }
        if (n + 1 < cnt) store_sa();
      }
      tc::fence_before_sync();
      if (tc::named_any(kChainBar, kChainThreads, !ok)) { fail = 4 * n + 2; break; }
      // the chain is done with chunk n's stage (its MMAs completed with D_S)
      if (tid == 0) tc::mbar_arrive(bar(kEmpty0 + s));
    }
    if (fail < 0 && hT) {
#pragma unroll
      for (int j = 0; j < KH; ++j) hT[(hT_idx * DK + KH * half + j) * SW + c] = S[j];
    }
  } else {
    // ------------------------------------------------------------ output
    int issued = 0, zissued = 0;
    if (tid == kOut) {
      for (int n = 0; n < min(kStages, cnt); ++n) load_chunk(n);
      issued = min(kStages, cnt);
      if (zring) {
        for (int n = 0; n < min(2, cnt); ++n) load_z(n);
        zissued = min(2, cnt);
      }
    }
    for (int n = 0; n < cnt; ++n) {
      const int s = n % kStages;
      bool ok = true;
      if (tid == kOut) {
        // MMA3: W^T A_qk^T onto the O part of D1[n%2] once MMA2 (which reads the
        // same W^T) has completed, so that it runs while the chain updates S
        ok = wait_or_abort(bar(kBS), n & 1, abort_flag);
        if (ok) {
          tc::fence_after_sync();
          constexpr uint32_t id3 = tc::idesc_bf16(128, 64, 0, 0);
          const uint64_t dA = tc::smem_desc(sb + s * L::kStage + P::oAqk, 16, 1024);
#pragma unroll
          for (int k0 = 0; k0 < 64; k0 += 16)
            tc::mma_bf16_ta(tmem + D10 + (n & 1) * 128, tmem + WA + k0 / 2, dA + ((k0 * 2) >> 4),
                            id3, 1);
          tc::commit(bar(kBO0 + (n & 1)));
        }
      }
      if (tc::named_any(kOutBar, kOutThreads, !ok)) { fail = 4 * n + 3; break; }
      ok = wait_or_abort(bar(kBO0 + (n & 1)), (n >> 1) & 1, abort_flag);
      if (tc::named_any(kOutBar, kOutThreads, !ok)) { fail = 4 * n + 3; break; }
      tc::fence_after_sync();
      const int t0 = (c_begin + n) * kChunk;
      const int Lr = min(kChunk, T - t0);
      __syncwarp();
      // O_n^T into registers, then D1[n%2] goes back to the chain before the
      // stores (which then overlap the next chunk)
      float x[64];
      tc::tmem_ld64(tl + D10 + (n & 1) * 128, x);
      tc::fence_before_sync();
      // thread kOut: the stage goes back to the chain's ring once both roles are
      // done with it, and is refilled with chunk n + kStages
      auto release_and_refill = [&]() {
        tc::mbar_arrive(bar(kEmpty0 + s));
        if (n + kStages < cnt) {
          ok = wait_or_abort(bar(kEmpty0 + s), (n / kStages) & 1, abort_flag);
          if (ok) {
            load_chunk(n + kStages);
            issued = n + kStages + 1;
          }
        }
      };
      if (tid == kOut) {
        tc::mbar_arrive(bar(kOFree0 + (n & 1)));
        release_and_refill();   // MMA3 is done with the packet
        if (zring) {
          tc::bulk_wait_read<1>();   // the y tile of chunk n-2 has been read out
          if (ok && !wait_or_abort(bar(kZFull0 + (n & 1)), (n >> 1) & 1, abort_flag)) ok = false;
        }
      }
      if (zring && tc::named_any(kOutBar, kOutThreads, !ok)) { fail = 4 * n + 3; break; }
      if (!zring) tc::named_sync(kOutBar, kOutThreads);
      if constexpr (GATE) {
        if (out) {
          // the output epilogue on the chunk's rows: y = o rsqrt(mean_c o^2 + eps)
          // weight_c silu(z), z from the stage (TMA), y through a shared tile and
          // a TMA store. Each row's sum of squares over the d_v columns is a
          // reduce-scatter over the warp's 32 lanes (lane l ends with token l of
          // the half) and then over the four warps through shared memory.
          const unsigned char* zt = smem + L::oZ + (n & 1) * 16384;
          unsigned char* yt = smem + L::oY + (n & 1) * 16384;
          float* red = reinterpret_cast<float*>(smem + L::oRed) + (n & 1) * 256;
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = x[32 * p + j] * x[32 * p + j];
#pragma unroll
            for (int off = 16, m = 16; off >= 1; off >>= 1, m >>= 1) {
              const bool up = (lane & off) != 0;
#pragma unroll
              for (int i = 0; i < m; ++i) {
                const float send = up ? v[i] : v[i + m];
                const float keep = up ? v[i + m] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
              }
            }
            red[q * 64 + 32 * p + lane] = v[0];
          }
          tc::named_sync(kOutBar, kOutThreads);
          // warp q finishes rows 16 q .. 16 q + 15: rsqrt(mean + eps) into the
          // first 64 floats of this chunk's red buffer (after everyone read the sums)
          float rsv = 0.f;
          if (lane < 16) {
            const int t = 16 * q + lane;
            rsv = rsqrtf((red[t] + red[64 + t] + red[128 + t] + red[192 + t]) * (1.f / DV) +
                         a.geps);
          }
          tc::named_sync(kOutBar, kOutThreads);
          if (lane < 16) red[16 * q + lane] = rsv;
          tc::named_sync(kOutBar, kOutThreads);
          const float wc = a.gw[c];
          const float4* rs4 = reinterpret_cast<const float4*>(red);
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            // all of the quarter's z first: the y stores below could alias the z
            // tile for the compiler, which would otherwise serialise the rows
            float zf[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              zf[j] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
                  zt + tc::tile_off(64, 16 * p + j, c)));
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
              const float4 r4 = rs4[(16 * p + j) / 4];
              const float rr[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float hz = 0.5f * zf[j + i];
                const float silu = fmaf(hz, tanh_fast(hz), hz);   // z sigmoid(z)
                const float y = (x[16 * p + j + i] * rr[i] * wc) * silu;
                *reinterpret_cast<__nv_bfloat16*>(yt + tc::tile_off(64, 16 * p + j + i, c)) =
                    __float2bfloat16_rn(y);
              }
            }
          }
          tc::fence_proxy_async();
          tc::named_sync(kOutBar, kOutThreads);
          if (tid == kOut) {   // rows past T are clipped by the store
#pragma unroll
            for (int blk = 0; blk < DV / 64; ++blk)
              tc::tma_store_4d(&tm_o, blk * 64, h, t0, bb, smem_u32(yt) + blk * 8192);
            tc::bulk_commit();
            if (n + 2 < cnt) {   // this z slot is free again
              load_z(n + 2);
              zissued = n + 3;
            }
          }
        }
      } else if (out) {
        // one column per lane: each warp store covers 32 adjacent columns of a
        // row (64 bytes); fewer instructions than transposing to 16-byte rows,
        // which cost the chain warps more issue slots than they saved
        __nv_bfloat16* op = out + ((size_t(bb) * T + t0) * H + h) * DV + c;
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (j < Lr) op[size_t(j) * H * DV] = __float2bfloat16_rn(x[j]);
      }
      if (tc::named_any(kOutBar, kOutThreads, !ok)) { fail = 4 * n + 3; break; }
    }
    // let the copies already issued land before the CTA can exit (a plain
    // bounded wait: an abort elsewhere does not stop a copy in flight), and
    // the y stores finish
    if (tid == kOut) {
      for (int n = max(0, issued - kStages); n < issued; ++n)
        tc::mbar_wait(bar(kFull0 + n % kStages), (n / kStages) & 1);
      for (int n = max(0, zissued - 2); n < zissued; ++n)
        tc::mbar_wait(bar(kZFull0 + (n & 1)), (n >> 1) & 1);
      if constexpr (GATE) tc::bulk_wait_all<0>();
    }
  }

  if (fail >= 0 && status && lane == 0) {
    if (atomicCAS(status, 0, 5) == 0) {  // GDR_ERR_TIMEOUT
      status[1] = static_cast<int>((blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x);
      status[2] = fail;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

template <int CW, bool RF, bool GATE>
cudaError_t launch_scan_t(const ChunkArgs& a, const unsigned char* packets, int* status,
                          cudaStream_t stream, ScanSegments sg) {
  using L = TLayout<128, GATE>;
  static_assert(L::launch_bytes <= 232448, "shared memory budget of one CTA");
  auto kern = chunk_scan_t_kernel<128, CW, RF, GATE>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L::launch_bytes));
  if (err != cudaSuccess) return err;
  if (sg.segments < 1 || sg.chunk0 < 0) return cudaErrorInvalidValue;
  if (sg.seg_chunks < 1) sg.seg_chunks = (a.T + kChunk - 1) / kChunk - sg.chunk0;
  CUtensorMap tz{}, to{};   // (read only by the fused epilogue)
  if (GATE && (!make_bthd_tmap(&tz, a.gz, a.B, a.T, a.H, 128) ||
               !make_bthd_tmap(&to, a.o, a.B, a.T, a.H, 128)))
    return cudaErrorInvalidValue;
  dim3 grid(sg.hT_hom ? 2 : 1, a.H, static_cast<unsigned>(a.B) * static_cast<unsigned>(sg.segments));
  kern<<<grid, Roles<CW>::kThreads, L::launch_bytes, stream>>>(a, packets, status, sg, tz, to);
  return cudaGetLastError();
}

cudaError_t launch_chunk_scan_t(const ChunkArgs& a, int dk, const unsigned char* packets,
                                int* status, cudaStream_t stream, ScanSegments sg) {
  if (dk != 128 || a.dv != 128 || (a.flags & 16u)) return cudaErrorInvalidValue;
  // channel decay: rho-folded packets; gz: the output epilogue fused
  const bool rf = a.flags & 1u, gate = a.gz != nullptr && a.o != nullptr;
  if (rf)
    return gate ? launch_scan_t<2, true, true>(a, packets, status, stream, sg)
                : launch_scan_t<2, true, false>(a, packets, status, stream, sg);
  return gate ? launch_scan_t<2, false, true>(a, packets, status, stream, sg)
              : launch_scan_t<2, false, false>(a, packets, status, stream, sg);
}

}  // namespace gdr
