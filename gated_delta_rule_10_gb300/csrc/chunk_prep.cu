// Chunk preparation kernel of the two-kernel chunkwise forward (bf16 inputs,
// every gate variant): the intra-chunk half of the WY/UT algorithm of the
// Gated DeltaNet-2 notes, key design 2 (Q-Delta notes, key design 3, for the
// mixed erase input), for all chunks of all (batch, head) pairs at once. Only
// the state pass is sequential in the chunk index, so this half has
// B * H * ceil(T / 64) independent CTAs and fills the GPU even when B * H is
// small.
//
// Persistent CTAs (256 threads; two per SM, three for scalar gates, whose lean
// layout is described at LeanLayout) walk the chunks; per chunk:
//   load    TMA brings the chunk's q, k, v (and b, w) tiles in: the key side as
//           soon as the previous chunk's inverse is done with their shared
//           memory, the value side as soon as its M2 is; the chunk after is
//           prefetched into L2 meanwhile
//   gates   G = in-chunk cumsum of g (per key channel or per row), gamma_C
//   tiles   (scalar gates: see prep_keys_scalar) gated in place: Z = z over v;
//           E_bar = f (.) e, Q' = s f (.) q,
//           K_bar = f^-1 (.) k over b (or a free slot), q and k; E_abs = gamma (.) e
//           over w (after Z has used it); Q_gamma = s gamma (.) q and
//           K_tail = gamma_C / gamma (.) k straight to the packet
//           (channel gates: f = e^{G - rho}, rho = G_C / 2, so every factor stays in range;
//           scalar gates: f = 1 and exp(G_r - G_i) <= 1 multiplies T and A_qk afterwards)
//   M1      D1 = [E_bar; Q'] K_bar^T            (tcgen05, M=128, N=64, K=d_k)
//           T = tril(D1[0:64], -1) (fp32), A_qk = tril(D1[64:128], 0) -> packet
//   UT      A = (I + T)^{-1}                   (blocked forward substitution, 8 warps)
//   M2      [U | Y] = A [Z | E_abs]             (M=64, N=d_v+d_k) -> packet (U, -Y)
// The packet layout is in packet.h. Operands live in shared memory in the
// 128-byte swizzle of tc.cuh (the TMA boxes land in it directly); packet tiles
// go from registers straight to global memory in the same byte layout.
#include "common.cuh"
#include "kernels.h"
#include "packet.h"
#include "tc.cuh"
#include "tma.h"
#include "tri_inverse.cuh"

#include <type_traits>

namespace gdr {
namespace {

constexpr int kThreads = 256;
constexpr uint32_t kInvBar = 1;

constexpr uint32_t align1k(uint32_t x) { return (x + 1023u) & ~1023u; }
constexpr uint32_t cmax(uint32_t a, uint32_t b) { return a > b ? a : b; }

template <int DK, int DV>
struct PrepLayout {
  // region 1: [E; Q] (128 x DK, 16 KB per 64-column block: E rows, then Q rows)
  // and K (64 x DK) until M1 completes, then T and A (fp32 [64][65] each) and
  // the inverse's [32][33] scratch
  static constexpr uint32_t kR1 = align1k(cmax(384 * DK, 2 * 64 * 65 * 4 + 32 * 33 * 4));
  static constexpr uint32_t oEQ = 0;
  static constexpr uint32_t oK = 256 * DK;
  static constexpr uint32_t oT = 0;
  static constexpr uint32_t oAf = 64 * 65 * 4;
  static constexpr uint32_t oX = 2 * 64 * 65 * 4;          // [32][33] inverse scratch
  // v -> Z and w -> E_abs, adjacent: one B operand [Z | E_abs] of N = DV + DK
  static constexpr uint32_t oV = kR1;                       // K=64 x DV (B, MN-major)
  static constexpr uint32_t oEa = oV + 128 * DV;            // K=64 x DK (B, MN-major)
  static constexpr uint32_t oA = oEa + 128 * cmax(DK, DV);  // A 64 x 64 (A, K-major)
  static constexpr uint32_t oP = oA + 8192;                 // [4][256] inverse scratch
  static constexpr uint32_t oPart = oP + 4096;              // per-row-block gate sums
  static constexpr uint32_t oVec = oPart + 8192;            // beta, lam, G, e^G, e^{G_C-G}, e^-G [64]
  static constexpr uint32_t oBar = oVec + 6 * 64 * 4 + 16;  // 4 mbarriers (after a flag word)
  static constexpr uint32_t oSlot = oBar + 32;
  static constexpr uint32_t bytes = oSlot + 16;   // TMEM address, two claimed work items
  static constexpr uint32_t launch_bytes = bytes + 1024;
  static constexpr uint32_t kTmemCols = (DK + DV) > 128 ? 256 : 128;
};

// Scalar gates (the lean variant, three CTAs per SM): the [E; Q] tiles (256 d_k
// bytes) until M1 completes, then inside that region T inverted in place into A
// (fp32 [64][65]), the inverse's scratch and the bf16 A tile; then one slot
// that holds k until M1 completes under QMIX (x = k + lam q takes the E slot)
// and v after it, and E_abs. 128 TMEM columns: M1, then M2 as two groups,
// U = A v and Y = A E_abs, each read out before the next.
template <int DK, int DV>
struct LeanLayout {
  static constexpr uint32_t oEQ = 0;
  static constexpr uint32_t oT = 0;                          // T, then A in place
  static constexpr uint32_t oAf = oT;
  static constexpr uint32_t oP = 64 * 65 * 4;                // [4][128] per-warp scratch
  static constexpr uint32_t oX = oP + 4 * 128 * 4;           // [32][33] inverse scratch
  static constexpr uint32_t oA = align1k(oX + 32 * 33 * 4);  // A 64 x 64 (A, K-major)
  static constexpr uint32_t kR1 = align1k(cmax(256 * DK, oA + 8192));
  // one slot for k (QMIX: the B operand of M1, until M1 completes) and then v
  static constexpr uint32_t oV = kR1;                        // K=64 x DV (B, MN-major)
  static constexpr uint32_t oK = oV;                         // 64 x DK (QMIX only)
  static constexpr uint32_t kKV = 128 * cmax(DK, DV);
  static constexpr uint32_t oEa = oV + kKV;                  // K=64 x DK (B, MN-major)
  static constexpr uint32_t oPart = oP;                      // (channel gates only: not used)
  static constexpr uint32_t oVec = oEa + 128 * DK;
  static constexpr uint32_t oBar = oVec + 6 * 64 * 4 + 16;   // 5 mbarriers (after a flag word)
  static constexpr uint32_t oSlot = oBar + 48;
  static constexpr uint32_t bytes = oSlot + 16;
  static constexpr uint32_t launch_bytes = bytes + 1024;
  static constexpr uint32_t kTmemCols = 128;
  static_assert(oX + 32 * 33 * 4 <= oA && oA + 8192 <= kR1 && 256 * DK <= kR1, "region 1");
  static_assert(oEa + 128 * DK == oVec && oV % 1024 == 0 && oEa % 1024 == 0, "v and E_abs");
  static_assert(oK + 128 * DK <= oEa && oV + 128 * DV <= oEa, "the k / v slot");
};

// Channel decay with d_k = d_v = 128 (the rho-folded variant, see
// prep_keys_rf): the [E_bar; Q'] tiles and K_bar until M1 completes, then T
// inverted in place into A (fp32 [64][65]) with the inverse's scratch over the
// second Q' block and K_bar, while the E_bar rows stay until M2 (Y_bar = A
// E_bar); v (then Z in place) and w; the bf16 A tile; the gate sums.
template <int DK, int DV>
struct RfLayout {
  static constexpr uint32_t oEQ = 0;
  static constexpr uint32_t oK = 256 * DK;
  static constexpr uint32_t kR1 = 384 * DK;
  static constexpr uint32_t oT = 24576;                      // Q' rows of block 1, then K_bar
  static constexpr uint32_t oAf = oT;
  static constexpr uint32_t oX = oT + 64 * 65 * 4;           // [32][33] inverse scratch
  static constexpr uint32_t oP = oX + 32 * 33 * 4;           // [4][128] per-warp scratch
  static constexpr uint32_t oV = kR1;                        // K=64 x DV (B, MN-major)
  static constexpr uint32_t oEa = oV + 128 * DV;             // w (write gate), until Z is formed
  static constexpr uint32_t oA = oEa + 128 * DV;             // A 64 x 64 (K-major)
  static constexpr uint32_t oPart = oA + 8192;               // per-row-block gate sums
  static constexpr uint32_t oVec = oPart + 8192;
  static constexpr uint32_t oBar = oVec + 6 * 64 * 4 + 16;   // 6 mbarriers (after a flag word)
  static constexpr uint32_t oSlot = oBar + 48;
  static constexpr uint32_t bytes = oSlot + 16;
  static constexpr uint32_t launch_bytes = bytes + 1024;
  static constexpr uint32_t kTmemCols = 256;
  static_assert(DK == 128 && DV == 128, "the rho-folded packets are for d_k = d_v = 128");
  static_assert(oP + 4 * 128 * 4 <= kR1, "inverse scratch inside the Q' / K_bar region");
};

// kBarB and kBarW (the erase and write gates loaded on their own) exist in the
// rho-folded variant, which has no second M2 group
enum : uint32_t { kBarV = 0, kBarK = 1, kBarM1 = 2, kBarM2 = 3, kBarM2b = 4, kBarB = 4, kBarW = 5 };

__device__ __forceinline__ uint4 pack8(const float* x) {
  uint4 u;
  u.x = pack_bf16x2(x[0], x[1]);
  u.y = pack_bf16x2(x[2], x[3]);
  u.z = pack_bf16x2(x[4], x[5]);
  u.w = pack_bf16x2(x[6], x[7]);
  return u;
}

__device__ __forceinline__ void unpack8(uint4 u, float* x) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ uint4 ld16(const unsigned char* base, uint32_t off) {
  return *reinterpret_cast<const uint4*>(base + off);
}
__device__ __forceinline__ void st16(unsigned char* base, uint32_t off, uint4 v) {
  *reinterpret_cast<uint4*>(base + off) = v;
}

// The summed log-decay of a chunk below which the factors e^{+-(G - rho)} of
// the channel-gate tiles leave the fp32 range (|G - rho| <= -G_C / 2 < 88 with
// margin); a chunk past it reports GDR_ERR_RANGE into the status words (the
// first report wins): [1] = batch * H + head, [2] = chunk.
constexpr float kDecayFloor = -140.f;

__device__ __forceinline__ void report_range(int* status, int seq, int chunk) {
  if (status && atomicCAS(status, 0, 6) == 0) {   // GDR_ERR_RANGE
    status[1] = seq;
    status[2] = chunk;
  }
}

// Channel gates, first half of the in-chunk cumsum: thread t loads g for the
// RPB consecutive rows from r0 = RPB (t / VK), channels c0 = 8 (t % VK) .. +7
// (rows past the sequence: zeros) and keeps them ...
template <int DK>
__device__ __forceinline__ void load_channel_gate_values(const ChunkArgs& a, size_t row0, int h,
                                                         int Lr,
                                                         float (&gv)[64 * DK / 8 / kThreads][8]) {
  constexpr int VK = DK / 8, RPB = 64 * VK / kThreads;
  const int tid = threadIdx.x, rb = tid / VK, c0 = (tid % VK) * 8, r0 = rb * RPB;
#pragma unroll
  for (int i = 0; i < RPB; ++i) {
    const int r = r0 + i;
    float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
    if (r < Lr) {
      const float4* p = reinterpret_cast<const float4*>(a.g + ((row0 + r) * a.H + h) * DK + c0);
      x0 = __ldg(p);
      x1 = __ldg(p + 1);
    }
    gv[i][0] = x0.x; gv[i][1] = x0.y; gv[i][2] = x0.z; gv[i][3] = x0.w;
    gv[i][4] = x1.x; gv[i][5] = x1.y; gv[i][6] = x1.z; gv[i][7] = x1.w;
  }
}
// ... and writes their sums per row block.
template <int DK>
__device__ __forceinline__ void channel_gate_sums(const float (&gv)[64 * DK / 8 / kThreads][8],
                                                  float* sPart) {
  constexpr int VK = DK / 8, RPB = 64 * VK / kThreads;
  const int tid = threadIdx.x, rb = tid / VK, c0 = (tid % VK) * 8;
  float ps[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) ps[j] = 0.f;
#pragma unroll
  for (int i = 0; i < RPB; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) ps[j] += gv[i][j];
  }
  float4* dst = reinterpret_cast<float4*>(sPart + rb * DK + c0);
  dst[0] = make_float4(ps[0], ps[1], ps[2], ps[3]);
  dst[1] = make_float4(ps[4], ps[5], ps[6], ps[7]);
}

// Key-side tiles, gated in place (same thread-to-element map as the gate loads).
template <int DK, int DV, bool CH, bool ER, bool QM>
__device__ __forceinline__ void prep_keys(unsigned char* smem, unsigned char* pkt,
                                          const ChunkArgs& a, const float* sPart,
                                          const float* sBeta, const float* sLam,
                                          const float* sEG, const float* sEGL,
                                          const float (&gv)[64 * DK / 8 / kThreads][8],
                                          int* status, int seq, int chunk) {
  using L = PrepLayout<DK, DV>;
  using P = Packet<DK, DV>;
  constexpr int VK = DK / 8, RB = kThreads / VK, RPB = 64 / RB;
  const int tid = threadIdx.x, rb = tid / VK, c0 = (tid % VK) * 8, r0 = rb * RPB;

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
      bool low = false;
#pragma unroll
      for (int j = 0; j < 8; ++j) low |= tot[j] < kDecayFloor;
      if (low) report_range(status, seq, chunk);
    }
  }
#pragma unroll
  for (int i = 0; i < RPB; ++i) {
    const int r = r0 + i;
    float qv[8], kv[8], bv[8];
    unpack8(ld16(smem, L::oEQ + tc::tile_off(128, 64 + r, c0)), qv);
    unpack8(ld16(smem, L::oK + tc::tile_off(64, r, c0)), kv);
    if (ER) unpack8(ld16(smem, L::oEQ + tc::tile_off(128, r, c0)), bv);
    const float lam = sLam[r], beta = sBeta[r];
    const float ear = CH ? 0.f : sEG[r], ktr = CH ? 0.f : sEGL[r];
    float Eb[8], Qr[8], Kb[8], Ea[8], Qg[8], Kt[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float x = QM ? kv[j] + lam * qv[j] : kv[j];
      const float e = ER ? bv[j] * x : beta * x;
      float f = 1.f, fi = 1.f, ea = ear, kt = ktr;
      if (CH) {
        G[j] += gv[CH ? i : 0][j];
        f = __expf(G[j] - rho[j]);
        fi = __expf(rho[j] - G[j]);
        ea = f * er[j];
        kt = fi * er[j];
      }
      Eb[j] = f * e;
      Qr[j] = a.scale * f * qv[j];
      Kb[j] = fi * kv[j];
      Ea[j] = ea * e;
      Qg[j] = a.scale * ea * qv[j];
      Kt[j] = kt * kv[j];
    }
    st16(smem, L::oEQ + tc::tile_off(128, r, c0), pack8(Eb));
    st16(smem, L::oEQ + tc::tile_off(128, 64 + r, c0), pack8(Qr));
    st16(smem, L::oK + tc::tile_off(64, r, c0), pack8(Kb));
    st16(smem, L::oEa + tc::tile_off(64, r, c0), pack8(Ea));
    st16(pkt, P::oQY + tc::tile_off(128, r, c0), pack8(Qg));
    st16(pkt, P::oKt + tc::tile_off(64, r, c0), pack8(Kt));
  }
}

// Channel decay, d_k = d_v = 128 (packets for the transposed scan): the decay
// factors e^{+-(G - rho)} with rho = G_C / 2 per key channel form only the
// tiles M1 needs, E_bar = f (.) e, Q' = s f (.) q and K_bar = f^-1 (.) k with
// f = e^{G - rho}; the packet takes Q' (rows 0..63 of its [Q_gamma; -Y] tile),
// K_bar (in K_tail's place), gamma_C and e^{rho}. The factor e^{rho} that
// turns them into Q_gamma = e^{rho} (.) Q', K_tail = e^{rho} (.) K_bar and
// E_abs = e^{rho} (.) E_bar (so Y = A E_bar diag(e^{rho})) is per key
// channel, so the scan applies it to the rows of S instead:
//   [Q_gamma; -Y] S_n = [Q'; -A E_bar] (diag(e^rho) S_n),
//   K_tail^T W = diag(e^rho) K_bar^T W.
template <int DK, int DV, bool ER, bool QM>
__device__ __forceinline__ void prep_keys_rf(unsigned char* smem, unsigned char* pkt,
                                             const ChunkArgs& a, const float* sPart,
                                             const float* sTot, const float* sBeta,
                                             const float* sLam,
                                             const float (&gv)[64 * DK / 8 / kThreads][8],
                                             int* status, int seq, int chunk) {
  using L = RfLayout<DK, DV>;
  using P = Packet<DK, DV>;
  constexpr int VK = DK / 8, RB = kThreads / VK, RPB = 64 / RB;
  const int tid = threadIdx.x, rb = tid / VK, c0 = (tid % VK) * 8, r0 = rb * RPB;
  // sPart: the log-decay summed over the row blocks before this thread's
  // (exclusive prefix per key channel); sTot: over the whole chunk
  float G[8], rho[8], tot[8];
  {
    const float4* pre = reinterpret_cast<const float4*>(sPart + rb * DK + c0);
    const float4* all = reinterpret_cast<const float4*>(sTot + c0);
    const float4 p0 = pre[0], p1 = pre[1], t0 = all[0], t1 = all[1];
    G[0] = p0.x; G[1] = p0.y; G[2] = p0.z; G[3] = p0.w;
    G[4] = p1.x; G[5] = p1.y; G[6] = p1.z; G[7] = p1.w;
    tot[0] = t0.x; tot[1] = t0.y; tot[2] = t0.z; tot[3] = t0.w;
    tot[4] = t1.x; tot[5] = t1.y; tot[6] = t1.z; tot[7] = t1.w;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) rho[j] = 0.5f * tot[j];
  if (rb == 0) {
    bool low = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) low |= tot[j] < kDecayFloor;
    if (low) report_range(status, seq, chunk);
    float gc[8], er[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      gc[j] = __expf(tot[j]);
      er[j] = __expf(rho[j]);
    }
    float4* dst = reinterpret_cast<float4*>(pkt + P::oGc + c0 * 4);
    dst[0] = make_float4(gc[0], gc[1], gc[2], gc[3]);
    dst[1] = make_float4(gc[4], gc[5], gc[6], gc[7]);
    float4* dre = reinterpret_cast<float4*>(pkt + P::oGc + (DK + c0) * 4);
    dre[0] = make_float4(er[0], er[1], er[2], er[3]);
    dre[1] = make_float4(er[4], er[5], er[6], er[7]);
  }
#pragma unroll
  for (int i = 0; i < RPB; ++i) {
    const int r = r0 + i;
    float qv[8], kv[8], bv[8];
    unpack8(ld16(smem, L::oEQ + tc::tile_off(128, 64 + r, c0)), qv);
    unpack8(ld16(smem, L::oK + tc::tile_off(64, r, c0)), kv);
    if (ER) unpack8(ld16(smem, L::oEa + tc::tile_off(64, r, c0)), bv);   // b: the w slot
    const float lam = sLam[r], beta = sBeta[r];
    float Eb[8], Qr[8], Kb[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float x = QM ? kv[j] + lam * qv[j] : kv[j];
      const float e = ER ? bv[j] * x : beta * x;
      G[j] += gv[i][j];
      const float f = __expf(G[j] - rho[j]), fi = __expf(rho[j] - G[j]);
      Eb[j] = f * e;
      Qr[j] = a.scale * f * qv[j];
      Kb[j] = fi * kv[j];
    }
    const uint4 qr = pack8(Qr), kb = pack8(Kb);
    st16(smem, L::oEQ + tc::tile_off(128, r, c0), pack8(Eb));
    st16(smem, L::oEQ + tc::tile_off(128, 64 + r, c0), qr);
    st16(smem, L::oK + tc::tile_off(64, r, c0), kb);
    st16(pkt, P::oQY + tc::tile_off(128, r, c0), qr);
    st16(pkt, P::oKt + tc::tile_off(64, r, c0), kb);
  }
}

// Scalar gates (no channel decay, erase or write gate): beta folds into the rows
// of T and the columns of A, the scale into A_qk, so q, k and v stay as
// loaded and only three tiles are formed per element: E_abs' = e^{G_r} x_r
// (x = k, or k + lam q), Q_gamma and K_tail (packet). k sits in the E slot;
// under QMIX x replaces it there and k moves to the K slot.
template <int DK, int DV, bool QM, typename L = PrepLayout<DK, DV>, bool KINK = false>
__device__ __forceinline__ void prep_keys_scalar(unsigned char* smem, unsigned char* pkt,
                                                 const ChunkArgs& a, const float* sLam,
                                                 const float* sEG, const float* sEGL) {
  // KINK: k was loaded into the K slot (lean layout) and stays there
  static_assert(!QM || KINK || L::oK + 128 * DK <= L::oV, "the K slot exists");
  using P = Packet<DK, DV>;
  constexpr int VK = DK / 8, RB = kThreads / VK, RPB = 64 / RB;
  const int tid = threadIdx.x, rb = tid / VK, c0 = (tid % VK) * 8, r0 = rb * RPB;
#pragma unroll
  for (int i = 0; i < RPB; ++i) {
    const int r = r0 + i;
    float qv[8], kv[8];
    unpack8(ld16(smem, L::oEQ + tc::tile_off(128, 64 + r, c0)), qv);
    const uint4 kraw = ld16(smem, KINK ? L::oK + tc::tile_off(64, r, c0)
                                       : L::oEQ + tc::tile_off(128, r, c0));
    unpack8(kraw, kv);
    const float lam = sLam[r], eg = sEG[r], egl = sEGL[r], sq = a.scale * eg;
    float x[8], Ea[8], Qg[8], Kt[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      x[j] = QM ? kv[j] + lam * qv[j] : kv[j];
      Ea[j] = eg * x[j];
      Qg[j] = sq * qv[j];
      Kt[j] = egl * kv[j];
    }
    if (QM) {
      st16(smem, L::oEQ + tc::tile_off(128, r, c0), pack8(x));
      if (!KINK) st16(smem, L::oK + tc::tile_off(64, r, c0), kraw);
    }
    st16(smem, L::oEa + tc::tile_off(64, r, c0), pack8(Ea));
    st16(pkt, P::oQY + tc::tile_off(128, r, c0), pack8(Qg));
    st16(pkt, P::oKt + tc::tile_off(64, r, c0), pack8(Kt));
  }
}

// Write strength per value channel (PacketVB): Q_gamma = s gamma (.) q and
// K_gamma = gamma (.) k (rows 64..127 of the same packet tile), K_tail =
// gamma_C / gamma (.) k; q and k stay as loaded for M1 (k in the E slot).
template <int DK, int DV>
__device__ __forceinline__ void prep_keys_vb(const unsigned char* smem, unsigned char* pkt,
                                             const ChunkArgs& a, const float* sEG,
                                             const float* sEGL) {
  using L = PrepLayout<DK, DV>;
  using P = PacketVB<DK, DV>;
  constexpr int VK = DK / 8, RB = kThreads / VK, RPB = 64 / RB;
  const int tid = threadIdx.x, rb = tid / VK, c0 = (tid % VK) * 8, r0 = rb * RPB;
#pragma unroll
  for (int i = 0; i < RPB; ++i) {
    const int r = r0 + i;
    float qv[8], kv[8];
    unpack8(ld16(smem, L::oEQ + tc::tile_off(128, 64 + r, c0)), qv);
    unpack8(ld16(smem, L::oEQ + tc::tile_off(128, r, c0)), kv);
    const float eg = sEG[r], egl = sEGL[r], sq = a.scale * eg;
    float Kg[8], Qg[8], Kt[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      Kg[j] = eg * kv[j];
      Qg[j] = sq * qv[j];
      Kt[j] = egl * kv[j];
    }
    st16(pkt, P::oQY + tc::tile_off(128, r, c0), pack8(Qg));
    st16(pkt, P::oQY + tc::tile_off(128, 64 + r, c0), pack8(Kg));
    st16(pkt, P::oKt + tc::tile_off(64, r, c0), pack8(Kt));
  }
}

// Write strength per value channel: V (as loaded, the packet's tile layout) and
// beta (fp32 from memory, bf16 in the tile layout) into the packet.
template <int DK, int DV>
__device__ __forceinline__ void prep_values_vb(const unsigned char* smem, unsigned char* pkt,
                                               const ChunkArgs& a, size_t row0, int h, int Lr) {
  using L = PrepLayout<DK, DV>;
  using P = PacketVB<DK, DV>;
  constexpr int VV = DV / 8, kIter = 64 * VV / kThreads;
  const int tid = threadIdx.x;
#pragma unroll
  for (int u = 0; u < kIter; ++u) {
    const int it = tid + u * kThreads, r = it / VV, c0 = (it % VV) * 8;
    const uint32_t off = tc::tile_off(64, r, c0);
    st16(pkt, P::oU + off, ld16(smem, L::oV + off));
    float bv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (r < Lr) {
      const float4* src = reinterpret_cast<const float4*>(a.beta + ((row0 + r) * a.H + h) * DV + c0);
      const float4 x0 = __ldg(src), x1 = __ldg(src + 1);
      bv[0] = x0.x; bv[1] = x0.y; bv[2] = x0.z; bv[3] = x0.w;
      bv[4] = x1.x; bv[5] = x1.y; bv[6] = x1.z; bv[7] = x1.w;
    }
    st16(pkt, P::oB + off, pack8(bv));
  }
}

// U^T (M=128 accumulator in tensor-memory columns 0..63: lane c = value column,
// column r = token) into the packet's U region as a 128-row tile of 64 tokens:
// warp w reads lane quadrant w % 4, tokens 32 (w / 4) .. +31, and each thread
// writes four 16-byte pieces of its value column's row.
__device__ __forceinline__ void store_ut(unsigned char* pkt, uint32_t tmem, int warp, int lane) {
  using P = Packet<128, 128>;
  const int q = warp & 3, half = warp >> 2, c = 32 * q + lane;
  float x[32];
  tc::tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + 32 * half, x);
#pragma unroll
  for (int j = 0; j < 32; j += 8)
    st16(pkt, P::oU + tc::tile_off(128, c, 32 * half + j), pack8(x + j));
}

// Z = beta v (or w (.) v with the write gate), in place over v.
template <int DK, int DV, bool WR, typename L>
__device__ __forceinline__ void prep_z(unsigned char* smem, const float* sBeta) {
  constexpr int VV = DV / 8, kIter = 64 * VV / kThreads;
  const int tid = threadIdx.x;
  uint4 vr[kIter], wr[WR ? kIter : 1];
#pragma unroll
  for (int u = 0; u < kIter; ++u) {
    const int it = tid + u * kThreads, r = it / VV, c0 = (it % VV) * 8;
    vr[u] = ld16(smem, L::oV + tc::tile_off(64, r, c0));
    if (WR) wr[WR ? u : 0] = ld16(smem, L::oEa + tc::tile_off(64, r, c0));
  }
#pragma unroll
  for (int u = 0; u < kIter; ++u) {
    const int it = tid + u * kThreads, r = it / VV, c0 = (it % VV) * 8;
    float v[8], w[8], z[8];
    unpack8(vr[u], v);
    if (WR) unpack8(wr[WR ? u : 0], w);
    const float beta = sBeta[r];
#pragma unroll
    for (int j = 0; j < 8; ++j) z[j] = WR ? w[j] * v[j] : beta * v[j];
    st16(smem, L::oV + tc::tile_off(64, r, c0), pack8(z));
  }
}

template <int DK, int DV, bool SC, bool VB, bool DYN, bool LEAN, bool RF>
__global__ void __launch_bounds__(kThreads, LEAN ? 3 : 2)
    chunk_prep_kernel(const ChunkArgs a, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_w, unsigned char* packets,
                      int* status, const PrepRange rg) {
  // RF: channel decay with d_k = d_v = 128, rho-folded packets (prep_keys_rf)
  using L = std::conditional_t<LEAN, LeanLayout<DK, DV>,
                               std::conditional_t<RF, RfLayout<DK, DV>, PrepLayout<DK, DV>>>;
  using P = std::conditional_t<VB, PacketVB<DK, DV>, Packet<DK, DV>>;
  static_assert(!VB || SC, "the value-channel packets take the scalar-gate tiles");
  static_assert(!RF || (!SC && !LEAN && !VB && DK == 128 && DV == 128), "rho-folded variant");
  static_assert(!LEAN || (SC && !VB), "the lean variant is for scalar gates");
  // d_k = d_v = 128: the packet carries U^T (d_v rows of 64 tokens) for the
  // transposed scan (chunk_scan_t.cu), produced directly as Z^T A^T
  constexpr bool UT = DK == 128 && DV == 128 && !VB;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, H = a.H, B = a.B;
  const int n_chunks = (T + kChunk - 1) / kChunk;
  // chunks rg.chunk0 .. rg.chunk0 + rc - 1 of every (batch, head)
  const int rc = rg.chunks > 0 ? rg.chunks : n_chunks - rg.chunk0;
  const int total = rc * B * H;
  const bool CH = a.flags & 1u, ER = a.flags & 2u, WR = a.flags & 4u, QM = a.flags & 8u;
  // lean layout under QMIX: k in the shared k / v slot, so a chunk's v is
  // loaded once its M1 has completed and waited for before M2
  const bool vlate = LEAN && QM;

  float* sT = reinterpret_cast<float*>(smem + L::oT);
  float* sAf = reinterpret_cast<float*>(smem + L::oAf);
  float* sP = reinterpret_cast<float*>(smem + L::oP);
  float* sPart = reinterpret_cast<float*>(smem + L::oPart);
  float* sBeta = reinterpret_cast<float*>(smem + L::oVec);
  float* sLam = sBeta + 64;
  float* sGs = sLam + 64;
  float* sEG = sGs + 64;
  float* sEGL = sEG + 64;
  float* sEGn = sEGL + 64;   // scalar gates: exp(-G_r)
  volatile int* sFactor = reinterpret_cast<volatile int*>(sEGn + 64);
  auto bar = [&](uint32_t i) { return sbase + L::oBar + 8 * i; };
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L::oSlot);

  if (warp == 0) tc::tmem_alloc(smem_u32(tslot), L::kTmemCols);
  if (tid == 32) {
    for (uint32_t i = 0; i < (RF ? 6u : LEAN ? 5u : 4u); ++i) tc::mbar_init(bar(i), 1);
    tc::fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;

  // work item w -> (chunk n, batch b, head h), heads fastest so that
  // neighbouring CTAs read neighbouring bytes of each token row
  auto decode = [&](int w, int& n, int& bb, int& h) {
    h = w % H;
    const int rest = w / H;
    bb = rest % B;
    n = rg.chunk0 + rest / B;
  };
  // Work items: a fixed stride over the grid (persistent CTAs), or, with a
  // counter, claimed one at a time by thread 64, at most rg.per_cta per CTA so
  // that CTAs come and go and a concurrent kernel of higher priority gets SMs.
  // A CTA knows its current item, the next, and (from the top of an
  // iteration) the one after, which it publishes in slot iter % 2.
  int* sClaim = reinterpret_cast<int*>(smem + L::oSlot + 4);   // [2]
  auto claim = [&](int k) {   // the CTA's k-th item (thread 64, dynamic mode)
    if (k >= rg.per_cta) return total;
    const int x = atomicAdd(rg.counter, 1);
    return x < total ? x : total;
  };
  // RF with the erase gate: b lands in the w slot (oEa) and has a barrier of
  // its own, issued as soon as the previous chunk's w is consumed (Z formed),
  // and w follows once this chunk's tile pass has read b
  const bool bsep = RF && ER;
  // TMA loads of one chunk's input tiles (thread 64): the value side (v, w) and
  // the key side (q, k, b) each complete one phase of their barrier; the
  // CTA's chunk after that one is prefetched into L2 along with them
  auto load_values = [&](int w, int w_after) {
    int n, bb, h;
    decode(w, n, bb, h);
    const bool lw = WR && !bsep;
    tc::fence_proxy_async();
    tc::mbar_arrive_expect_tx(bar(kBarV), (lw ? 2u : 1u) * 128u * DV);
#pragma unroll
    for (int blk = 0; blk < DV / 64; ++blk) {
      tc::tma_load_4d(sbase + L::oV + blk * 8192, &tm_v, blk * 64, h, n * kChunk, bb, bar(kBarV));
      if (lw)
        tc::tma_load_4d(sbase + L::oEa + blk * 8192, &tm_w, blk * 64, h, n * kChunk, bb, bar(kBarV));
    }
    if (w_after < total) {
      decode(w_after, n, bb, h);
#pragma unroll
      for (int blk = 0; blk < DV / 64; ++blk) {
        tc::tma_prefetch_4d(&tm_v, blk * 64, h, n * kChunk, bb);
        if (WR) tc::tma_prefetch_4d(&tm_w, blk * 64, h, n * kChunk, bb);
      }
    }
  };
  auto load_b = [&](int w) {   // (bsep) b into the w slot
    int n, bb, h;
    decode(w, n, bb, h);
    tc::fence_proxy_async();
    tc::mbar_arrive_expect_tx(bar(kBarB), 128u * DK);
#pragma unroll
    for (int blk = 0; blk < DK / 64; ++blk)
      tc::tma_load_4d(sbase + L::oEa + blk * 8192, &tm_b, blk * 64, h, n * kChunk, bb, bar(kBarB));
  };
  auto load_w = [&](int w) {   // (bsep and the write gate) w into the w slot
    int n, bb, h;
    decode(w, n, bb, h);
    tc::fence_proxy_async();
    tc::mbar_arrive_expect_tx(bar(kBarW), 128u * DV);
#pragma unroll
    for (int blk = 0; blk < DV / 64; ++blk)
      tc::tma_load_4d(sbase + L::oEa + blk * 8192, &tm_w, blk * 64, h, n * kChunk, bb, bar(kBarW));
  };
  auto load_keys = [&](int w, int w_after) {
    int n, bb, h;
    decode(w, n, bb, h);
    tc::fence_proxy_async();
    tc::mbar_arrive_expect_tx(bar(kBarK), ((ER && !bsep) ? 3u : 2u) * 128u * DK);
#pragma unroll
    for (int blk = 0; blk < DK / 64; ++blk) {
      tc::tma_load_4d(sbase + L::oEQ + blk * 16384 + 8192, &tm_q, blk * 64, h, n * kChunk, bb, bar(kBarK));
      if (SC && !vlate)
        tc::tma_load_4d(sbase + L::oEQ + blk * 16384, &tm_k, blk * 64, h, n * kChunk, bb, bar(kBarK));
      else
        tc::tma_load_4d(sbase + L::oK + blk * 8192, &tm_k, blk * 64, h, n * kChunk, bb, bar(kBarK));
      if (ER && !bsep)
        tc::tma_load_4d(sbase + L::oEQ + blk * 16384, &tm_b, blk * 64, h, n * kChunk, bb, bar(kBarK));
    }
    if (w_after < total) {
      decode(w_after, n, bb, h);
#pragma unroll
      for (int blk = 0; blk < DK / 64; ++blk) {
        tc::tma_prefetch_4d(&tm_q, blk * 64, h, n * kChunk, bb);
        tc::tma_prefetch_4d(&tm_k, blk * 64, h, n * kChunk, bb);
        if (ER) tc::tma_prefetch_4d(&tm_b, blk * 64, h, n * kChunk, bb);
      }
    }
  };
  // loads issued and waited for, to drain what is in flight on the way out
  int v_issued = 0, k_issued = 0, v_done = 0, k_done = 0, b_issued = 0, b_done = 0;
  int w_issued = 0, w_done = 0;
  constexpr bool dyn = DYN;   // work claimed from rg.counter
  const int stride = static_cast<int>(gridDim.x);
  int w = static_cast<int>(blockIdx.x), wn = w + stride, wa = wn + stride;   // this, next, after
  if (dyn) {
    if (tid == 64) {
      sClaim[0] = claim(0);
      sClaim[1] = sClaim[0] < total ? claim(1) : total;
    }
    __syncthreads();
    w = sClaim[0];
    wn = sClaim[1];
    wa = total;
    __syncthreads();   // both read before thread 64 writes a slot again
  }
  if (w < total) {
    if (tid == 64) {
      if (!vlate) load_values(w, wn);
      load_keys(w, wn);
      if (bsep) load_b(w);
    }
    v_issued = vlate ? 0 : 1;
    k_issued = 1;
    b_issued = bsep ? 1 : 0;
  }

  // channel gates of the current chunk (RF: the next chunk's are loaded while
  // this chunk's M2 runs, so they are in registers when its gates phase starts)
  float gv[64 * DK / 8 / kThreads][8];
  int fail_at = -1, iter = 0;
  for (; w < total; w = wn, wn = wa, ++iter) {
    // the item after the next one: claimed now (published for the loop step)
    if (dyn) {
      if (tid == 64) {
        wa = wn < total ? claim(iter + 2) : total;
        sClaim[iter & 1] = wa;
      }
    } else {
      wa = wn + stride;
    }
    const uint32_t par = static_cast<uint32_t>(iter & 1);
    int n, bb, h;
    decode(w, n, bb, h);
    const int t0 = n * kChunk, Lr = min(kChunk, T - t0);
    const size_t row0 = size_t(bb) * T + t0;
    unsigned char* pkt = packets + ((size_t(bb) * H + h) * n_chunks + n) * P::bytes;
    int nn = 0, nb = 0, nh = 0;   // this CTA's next chunk
    if (wn < total) decode(wn, nn, nb, nh);

    // gates of the next chunk into L2 (one row each for threads 128..191)
    if (wn < total && tid >= 128 && tid < 128 + kChunk) {
      const int r = tid - 128, nt = nn * kChunk + r;
      if (nt < T) {
        const size_t ti = (size_t(nb) * T + nt) * H + nh;
        if (CH)
          tc::bulk_prefetch(a.g + ti * DK, DK * 4);
        else
          tc::prefetch_l2(a.g + ti);
        if (VB)
          tc::bulk_prefetch(a.beta + ti * DV, DV * 4);
        else if (a.beta)
          tc::prefetch_l2(a.beta + ti);
        if (QM) tc::prefetch_l2(a.lam + ti);
      }
    }

    // per-row gates while the tiles are in flight: beta, lam; scalar decay cumsum
    if (tid < kChunk) {
      const size_t ti = (row0 + tid) * H + h;
      sBeta[tid] = (!VB && tid < Lr && a.beta) ? __ldg(a.beta + ti) : 0.f;
      sLam[tid] = (tid < Lr && QM) ? __ldg(a.lam + ti) : 0.f;
    }
    if (!CH && warp == 3) {
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
      // exp(G_r - G_i) = e^{G_r} e^{-G_i} stays exact in fp32 while G_C >= -80
      sEGn[lane] = __expf(-g0);
      sEGn[lane + 32] = __expf(-g1);
      if (lane == 0) *sFactor = tot >= -80.f ? 1 : 0;
    }
    if (CH) {
      if (!RF || iter == 0) load_channel_gate_values<DK>(a, row0, h, Lr, gv);
      channel_gate_sums<DK>(gv, sPart);
    }
    __syncthreads();
    if constexpr (RF) {
      // per key channel: the row blocks' partial sums become exclusive prefix
      // sums (the same additions, in the same order, as summing them per
      // thread) and the chunk's total G_C goes to sGs (with sEG: the
      // scalar-decay arrays, unused here); the key-side wait below orders
      // these writes before the tile pass reads them
      if (tid < DK) {
        float run = 0.f;
#pragma unroll
        for (int b = 0; b < kThreads / (DK / 8); ++b) {
          const float v = sPart[b * DK + tid];
          sPart[b * DK + tid] = run;
          run += v;
        }
        sGs[tid] = run;
      }
    }

    if (!vlate && !RF) {   // (RF: the value side is waited for after the inverse)
      if (__syncthreads_or(!tc::mbar_wait(bar(kBarV), par))) { fail_at = 4 * n; break; }
      v_done = v_issued;
    }
    if (VB) {
      prep_values_vb<DK, DV>(smem, pkt, a, row0, h, Lr);
      __syncthreads();   // v has been copied out: the next chunk's value tiles may land
      if (wn < total) {
        if (tid == 64) load_values(wn, wa);
        ++v_issued;
      }
    }
    if (!SC && !RF) {
      if (WR)
        prep_z<DK, DV, true, L>(smem, sBeta);
      else
        prep_z<DK, DV, false, L>(smem, sBeta);
      __syncthreads();   // w has been read: its slot takes E_abs below
    }
    if (__syncthreads_or(!tc::mbar_wait(bar(kBarK), par) ||
                         (bsep && !tc::mbar_wait(bar(kBarB), par)))) {
      fail_at = 4 * n;
      break;
    }
    k_done = k_issued;
    b_done = b_issued;
    if (VB) {
      prep_keys_vb<DK, DV>(smem, pkt, a, sEG, sEGL);
    } else if (SC) {
      if constexpr (LEAN) {   // under QMIX k already sits in the K slot
        if (QM)
          prep_keys_scalar<DK, DV, true, L, true>(smem, pkt, a, sLam, sEG, sEGL);
        else
          prep_keys_scalar<DK, DV, false, L>(smem, pkt, a, sLam, sEG, sEGL);
      } else {
        if (QM)
          prep_keys_scalar<DK, DV, true, L>(smem, pkt, a, sLam, sEG, sEGL);
        else
          prep_keys_scalar<DK, DV, false, L>(smem, pkt, a, sLam, sEG, sEGL);
      }
    } else if constexpr (RF) {   // channel decay (launched only with it)
      switch (a.flags & 10u) {
        case 0:
          prep_keys_rf<DK, DV, false, false>(smem, pkt, a, sPart, sGs, sBeta, sLam, gv, status,
                                             bb * H + h, n);
          break;
        case 2:
          prep_keys_rf<DK, DV, true, false>(smem, pkt, a, sPart, sGs, sBeta, sLam, gv, status,
                                            bb * H + h, n);
          break;
        case 8:
          prep_keys_rf<DK, DV, false, true>(smem, pkt, a, sPart, sGs, sBeta, sLam, gv, status,
                                            bb * H + h, n);
          break;
        default:
          prep_keys_rf<DK, DV, true, true>(smem, pkt, a, sPart, sGs, sBeta, sLam, gv, status,
                                           bb * H + h, n);
          break;
      }
    } else switch (a.flags & 11u) {   // CH | ER | QM select the key-side tiles
#define GDR_PREP(F)                                                                       \
  case F:                                                                                 \
    prep_keys<DK, DV, (F & 1u) != 0, (F & 2u) != 0, (F & 8u) != 0>(smem, pkt, a, sPart, sBeta, \
                                                                   sLam, sEG, sEGL, gv,   \
                                                                   status, bb * H + h, n); \
    break;
      GDR_PREP(0) GDR_PREP(1) GDR_PREP(2) GDR_PREP(3)
      GDR_PREP(8) GDR_PREP(9) GDR_PREP(10) GDR_PREP(11)
#undef GDR_PREP
      default: break;
    }
    tc::fence_proxy_async();
    __syncthreads();
    if (bsep) {   // b is read: the w slot takes this chunk's w, or (no write gate) the next b
      if (WR) {
        if (tid == 64) load_w(w);
        ++w_issued;
      } else if (wn < total) {
        if (tid == 64) load_b(wn);
        ++b_issued;
      }
    }

    // ---- M1: [E_bar; Q'] K_bar^T into columns 0..63 ----
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t id = tc::idesc_bf16(128, 64, 0, 0);
      const uint64_t dEQ = tc::smem_desc(sbase + L::oEQ, 16, 1024);
      // K_bar: the K slot, or for scalar gates without QMIX k itself in the E slot
      const bool kInE = SC && !QM;
      const uint64_t dKb = tc::smem_desc(sbase + (kInE ? L::oEQ : L::oK), 16, 1024);
      const uint32_t kBlk = kInE ? 16384u : 8192u;
#pragma unroll
      for (int k0 = 0; k0 < DK; k0 += 16) {
        const uint32_t ka = (k0 >> 6) * 16384 + (k0 & 63) * 2;
        const uint32_t kb = (k0 >> 6) * kBlk + (k0 & 63) * 2;
        tc::mma_bf16(tmem, dEQ + (ka >> 4), dKb + (kb >> 4), id, k0 > 0);
      }
      tc::commit(bar(kBarM1));
    }
    if (__syncthreads_or(!tc::mbar_wait(bar(kBarM1), par))) { fail_at = 4 * n + 1; break; }
    tc::fence_after_sync();
    if (vlate) {   // M1 has read k: this chunk's v may take the slot
      if (tid == 64) load_values(w, wn);
      ++v_issued;
    }
    // ---- T (fp32, shared) and A_qk (bf16, packet): warp w reads lane quadrant
    // w % 4 (quadrants 0-1: E_bar K_bar^T rows, 2-3: Q' K_bar^T rows), columns
    // 32 (w / 4) .. +31 ----
    {
      const int q = warp & 3, c = 32 * (warp >> 2);
      const int r = (32 * q + lane) & 63;
      const bool isT = q < 2;
      const int lim = isT ? r : r + 1;       // T strictly lower, A_qk with the diagonal
      float x[32];
      tc::tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + c, x);
      if (SC) {   // the row factors the scalar-gate tiles left out: beta_r (T), s (A_qk)
        const float f = isT ? (VB ? 1.f : sBeta[r]) : a.scale;
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] *= f;
      }
      if (CH) {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = select_f32(c + j < lim, x[j], 0.f);
      } else if (*sFactor) {
        const float er = sEG[r];
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = select_f32(c + j < lim, er * sEGn[c + j] * x[j], 0.f);
      } else {
        const float Gr = sGs[r];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          x[j] = select_f32(c + j < lim, __expf(fminf(Gr - sGs[c + j], 0.f)) * x[j], 0.f);
      }
      if (isT && VB) {   // L to the packet, fp32 row-major
        float4* dst = reinterpret_cast<float4*>(pkt + PacketVB<DK, DV>::oL + (r * 64 + c) * 4);
#pragma unroll
        for (int j = 0; j < 32; j += 4) dst[j / 4] = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
      } else if (isT) {
#pragma unroll
        for (int j = 0; j < 32; ++j) sT[r * 65 + c + j] = x[j];
      } else {
#pragma unroll
        for (int j = 0; j < 32; j += 8) st16(pkt, P::oAqk + tc::tile_off(64, r, c + j), pack8(x + j));
      }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (VB) {
      // no inverse and no M2: the key-side tiles are consumed, the chunk is done
      if (wn < total) {
        if (tid == 64) load_keys(wn, wa);
        ++k_issued;
      }
      tc::fence_after_sync();
      if (dyn) wa = sClaim[iter & 1];
      continue;
    }

    // ---- A = (I + T)^{-1} (all 8 warps), then the bf16 operand tile ----
    if constexpr (LEAN || RF)
      invert_unit_lower_64_w8_inplace(sT, sP, reinterpret_cast<float*>(smem + L::oX), warp, lane,
                                      [] { tc::named_sync(kInvBar, 128); },
                                      [] { __syncthreads(); });
    else
      invert_unit_lower_64_w8(sT, sAf, sP, reinterpret_cast<float*>(smem + L::oX), warp, lane,
                              [] { tc::named_sync(kInvBar, 128); }, [] { __syncthreads(); });
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int it = tid + u * kThreads, r = it >> 3, c0 = (it & 7) * 8;
      float x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = select_f32(c0 + j <= r, sAf[r * 65 + c0 + j], 0.f);
      if (SC) {   // A diag(beta): U = A diag(beta) V, Y = A diag(beta) (e^G x)
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] *= sBeta[c0 + j];
      }
      st16(smem, L::oA + tc::tile_off(64, r, c0), pack8(x));
    }
    tc::fence_proxy_async();
    __syncthreads();
    // T and A are consumed: the key-side tiles of the next chunk may land now
    // (lean variant: the A tile sits in their region, so after M2)
    if (!LEAN && wn < total) {
      if (tid == 64) load_keys(wn, wa);
      ++k_issued;
    }

    if constexpr (LEAN && UT) {
      // ---- M2 as one group within 128 TMEM columns, both products M = 128,
      // N = 64 with the A tile as the K-major B: U^T = Z^T A^T into columns
      // 0..63 and Y^T = E_abs^T A^T into 64..127 (Z and E_abs as MN-major A) ----
      const uint64_t dA = tc::smem_desc(sbase + L::oA, 16, 1024);
      if (vlate) {
        if (__syncthreads_or(!tc::mbar_wait(bar(kBarV), par))) { fail_at = 4 * n + 2; break; }
        v_done = v_issued;
      }
      if (tid == 0) {
        tc::fence_after_sync();
        const uint64_t dZ = tc::smem_desc(sbase + L::oV, 64 * 128, 1024);
        const uint64_t dE = tc::smem_desc(sbase + L::oEa, 64 * 128, 1024);
        constexpr uint32_t idu = tc::idesc_bf16(128, 64, 1, 0);
#pragma unroll
        for (int k0 = 0; k0 < 64; k0 += 16)
          tc::mma_bf16(tmem, dZ + (((k0 / 8) * 1024) >> 4), dA + ((k0 * 2) >> 4), idu, k0 > 0);
#pragma unroll
        for (int k0 = 0; k0 < 64; k0 += 16)
          tc::mma_bf16(tmem + 64, dE + (((k0 / 8) * 1024) >> 4), dA + ((k0 * 2) >> 4), idu,
                       k0 > 0);
        tc::commit(bar(kBarM2));
      }
      if (__syncthreads_or(!tc::mbar_wait(bar(kBarM2), par))) { fail_at = 4 * n + 2; break; }
      tc::fence_after_sync();
      // v, the A tile and E_abs are consumed: the next chunk's value side
      // (under QMIX after its M1) and its key side may land now
      if (!vlate && wn < total) {
        if (tid == 64) load_values(wn, wa);
        ++v_issued;
      }
      if (wn < total) {
        if (tid == 64) load_keys(wn, wa);
        ++k_issued;
      }
      store_ut(pkt, tmem, warp, lane);
      {
        // -Y into rows 64..127 of the packet's [Q_gamma; -Y] tile: lane c of
        // quadrant w % 4 holds key channel c, tokens 32 (w / 4) .. +31; a warp's
        // store covers 32 adjacent channels of one row (64 bytes)
        const int q = warp & 3, half = warp >> 2, c = 32 * q + lane;
#pragma unroll
        for (int p16 = 0; p16 < 2; ++p16) {
          const int t0 = 32 * half + 16 * p16;
          float x[16];
          tc::tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + 64 + t0, x);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            *reinterpret_cast<__nv_bfloat16*>(pkt + P::oQY + tc::tile_off(128, 64 + t0 + j, c)) =
                __float2bfloat16_rn(-x[j]);
        }
      }
    } else if constexpr (LEAN) {
      // ---- M2 in two groups within 128 TMEM columns: U = A Z (N = DV), read
      // out, then Y = A E_abs (N = DK), read out ----
      const uint64_t dA = tc::smem_desc(sbase + L::oA, 16, 1024);
      // M=64 accumulators: row 16 q + l in lane l < 16 of quadrant q; warp w
      // takes quadrant w % 4 and half w / 4 of the columns
      const int q = warp & 3, half = warp >> 2;
      const int r = 16 * q + (lane & 15);
      const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
      if (vlate) {
        if (__syncthreads_or(!tc::mbar_wait(bar(kBarV), par))) { fail_at = 4 * n + 2; break; }
        v_done = v_issued;
      }
      if (tid == 0) {
        tc::fence_after_sync();
        const uint64_t dZ = tc::smem_desc(sbase + L::oV, 64 * 128, 1024);
        if constexpr (UT) {   // U^T = Z^T A^T: Z as the MN-major A, the A tile as a K-major B
          constexpr uint32_t idu = tc::idesc_bf16(128, 64, 1, 0);
#pragma unroll
          for (int k0 = 0; k0 < 64; k0 += 16)
            tc::mma_bf16(tmem, dZ + (((k0 / 8) * 1024) >> 4), dA + ((k0 * 2) >> 4), idu, k0 > 0);
        } else {
          constexpr uint32_t idu = tc::idesc_bf16(64, DV, 0, 1);
#pragma unroll
          for (int k0 = 0; k0 < 64; k0 += 16)
            tc::mma_bf16(tmem, dA + ((k0 * 2) >> 4), dZ + (((k0 / 8) * 1024) >> 4), idu, k0 > 0);
        }
        tc::commit(bar(kBarM2));
      }
      if (__syncthreads_or(!tc::mbar_wait(bar(kBarM2), par))) { fail_at = 4 * n + 2; break; }
      tc::fence_after_sync();
      // v is consumed: the value-side tiles of the next chunk may land now
      // (under QMIX after the next chunk's M1)
      if (!vlate && wn < total) {
        if (tid == 64) load_values(wn, wa);
        ++v_issued;
      }
      if constexpr (UT) {
        store_ut(pkt, tmem, warp, lane);
      } else {
#pragma unroll
        for (int c = half * (DV / 2); c < (half + 1) * (DV / 2); c += 32) {
          float x[32];
          tc::tmem_ld32(tl + c, x);
          if (lane < 16) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) st16(pkt, P::oU + tc::tile_off(64, r, c + j), pack8(x + j));
          }
        }
      }
      tc::fence_before_sync();
      __syncthreads();   // U is read out: the columns take Y
      if (tid == 0) {
        tc::fence_after_sync();
        constexpr uint32_t idy = tc::idesc_bf16(64, DK, 0, 1);
        const uint64_t dE = RF ? tc::smem_desc(sbase + L::oEQ, 128 * 128, 1024)
                               : tc::smem_desc(sbase + L::oEa, 64 * 128, 1024);
#pragma unroll
        for (int k0 = 0; k0 < 64; k0 += 16)
          tc::mma_bf16(tmem, dA + ((k0 * 2) >> 4), dE + (((k0 / 8) * 1024) >> 4), idy, k0 > 0);
        tc::commit(bar(kBarM2b));
      }
      if (__syncthreads_or(!tc::mbar_wait(bar(kBarM2b), par))) { fail_at = 4 * n + 3; break; }
      tc::fence_after_sync();
      // the A tile and E_abs are consumed: the key-side tiles of the next chunk may land now
      if (wn < total) {
        if (tid == 64) load_keys(wn, wa);
        ++k_issued;
      }
#pragma unroll
      for (int c = half * (DK / 2); c < (half + 1) * (DK / 2); c += 32) {
        float x[32];
        tc::tmem_ld32(tl + c, x);
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = -x[j];
        if (lane < 16) {
#pragma unroll
          for (int j = 0; j < 32; j += 8)
            st16(pkt, P::oQY + tc::tile_off(128, 64 + r, c + j), pack8(x + j));
        }
      }
    } else {
    // ---- M2: [U | Y] = A [Z | E_abs] (N = DV + DK): U in columns 0..DV-1,
    // Y in columns DV..DV+DK-1 ----
    if constexpr (RF) {
      // the value side, loaded since the start of the chunk (w since the tile
      // pass when b came first): Z = w (.) v or beta v
      if (__syncthreads_or(!tc::mbar_wait(bar(kBarV), par) ||
                           (bsep && WR && !tc::mbar_wait(bar(kBarW), par)))) {
        fail_at = 4 * n + 2;
        break;
      }
      v_done = v_issued;
      w_done = w_issued;
      if (WR)
        prep_z<DK, DV, true, L>(smem, sBeta);
      else
        prep_z<DK, DV, false, L>(smem, sBeta);
      tc::fence_proxy_async();
      __syncthreads();
      if (bsep && WR && wn < total) {   // w is consumed: the next chunk's b
        if (tid == 64) load_b(wn);
        ++b_issued;
      }
    }
    // (U^T case: U^T = Z^T A^T in columns 0..63, Y in columns 64..64+DK-1;
    // RF: Y_bar = A E_bar from the E_bar rows of the [E_bar; Q'] tile)
    constexpr uint32_t kYcol = UT ? 64 : DV;
    if (tid == 0) {
      tc::fence_after_sync();
      const uint64_t dA = tc::smem_desc(sbase + L::oA, 16, 1024);
      const uint64_t dZE = tc::smem_desc(sbase + L::oV, 64 * 128, 1024);
      if constexpr (UT) {
        constexpr uint32_t idu = tc::idesc_bf16(128, 64, 1, 0);
        constexpr uint32_t idy = tc::idesc_bf16(64, DK, 0, 1);
        const uint64_t dE = RF ? tc::smem_desc(sbase + L::oEQ, 128 * 128, 1024)
                               : tc::smem_desc(sbase + L::oEa, 64 * 128, 1024);
#pragma unroll
        for (int k0 = 0; k0 < 64; k0 += 16)
          tc::mma_bf16(tmem, dZE + (((k0 / 8) * 1024) >> 4), dA + ((k0 * 2) >> 4), idu, k0 > 0);
#pragma unroll
        for (int k0 = 0; k0 < 64; k0 += 16)
          tc::mma_bf16(tmem + kYcol, dA + ((k0 * 2) >> 4), dE + (((k0 / 8) * 1024) >> 4), idy,
                       k0 > 0);
      } else {
        constexpr uint32_t id2 = tc::idesc_bf16(64, DV + DK, 0, 1);
#pragma unroll
        for (int k0 = 0; k0 < 64; k0 += 16)
          tc::mma_bf16(tmem, dA + ((k0 * 2) >> 4), dZE + (((k0 / 8) * 1024) >> 4), id2, k0 > 0);
      }
      tc::commit(bar(kBarM2));
    }
    if (RF && wn < total) {   // the next chunk's channel gates, in flight during M2
      const int t0n = nn * kChunk;
      load_channel_gate_values<DK>(a, size_t(nb) * T + t0n, nh, min(kChunk, T - t0n), gv);
    }
    if (__syncthreads_or(!tc::mbar_wait(bar(kBarM2), par))) { fail_at = 4 * n + 2; break; }
    tc::fence_after_sync();
    // Z and E_abs are consumed: the value-side tiles of the next chunk may land now
    // (RF: and the key side, E_bar being consumed too)
    if (wn < total) {
      if (tid == 64) load_values(wn, wa);
      ++v_issued;
    }
    {
      // M=64 accumulators: row 16 q + l in lane l < 16 of quadrant q; warp w
      // takes quadrant w % 4 and half w / 4 of the columns
      const int q = warp & 3, half = warp >> 2;
      const int r = 16 * q + (lane & 15);
      const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
#pragma unroll
      for (int c = half * (DK / 2); c < (half + 1) * (DK / 2); c += 32) {
        float x[32];
        tc::tmem_ld32(tl + kYcol + c, x);
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = -x[j];
        if (lane < 16) {
#pragma unroll
          for (int j = 0; j < 32; j += 8)
            st16(pkt, P::oQY + tc::tile_off(128, 64 + r, c + j), pack8(x + j));
        }
      }
      if constexpr (UT) {
        store_ut(pkt, tmem, warp, lane);
      } else {
#pragma unroll
        for (int c = half * (DV / 2); c < (half + 1) * (DV / 2); c += 32) {
          float x[32];
          tc::tmem_ld32(tl + c, x);
          if (lane < 16) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) st16(pkt, P::oU + tc::tile_off(64, r, c + j), pack8(x + j));
          }
        }
      }
    }
    }   // !LEAN
    // the next chunk reuses every shared tile and the tensor memory
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (dyn) wa = sClaim[iter & 1];
  }

  if (fail_at >= 0) {
    // no TMA copy may still be writing this CTA's shared memory when it exits
    if (tid == 64) {
      if (v_issued > v_done) tc::mbar_wait(bar(kBarV), static_cast<uint32_t>((v_issued - 1) & 1));
      if (k_issued > k_done) tc::mbar_wait(bar(kBarK), static_cast<uint32_t>((k_issued - 1) & 1));
      if (b_issued > b_done) tc::mbar_wait(bar(kBarB), static_cast<uint32_t>((b_issued - 1) & 1));
      if (w_issued > w_done) tc::mbar_wait(bar(kBarW), static_cast<uint32_t>((w_issued - 1) & 1));
    }
    if (tid == 0 && status && atomicCAS(status, 0, 5) == 0) {  // GDR_ERR_TIMEOUT
      status[1] = static_cast<int>(blockIdx.x);
      status[2] = fail_at;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, L::kTmemCols);
}

template <int DK, int DV, bool SC, bool VB, bool DYN, bool LEAN = false, bool RF = false>
cudaError_t launch_prep_kernel(const ChunkArgs& a, unsigned char* packets, int* status,
                               const PrepRange& rg, cudaStream_t stream) {
  using L = std::conditional_t<LEAN, LeanLayout<DK, DV>,
                               std::conditional_t<RF, RfLayout<DK, DV>, PrepLayout<DK, DV>>>;
  constexpr int kPerSm = LEAN ? 3 : 2;
  static_assert(kPerSm * (L::launch_bytes + 1024) <= 233472, "CTAs per SM");
  CUtensorMap tq, tk, tv, tb, tw;
  if (!make_bthd_tmap(&tq, a.q, a.B, a.T, a.H, DK) || !make_bthd_tmap(&tk, a.k, a.B, a.T, a.H, DK) ||
      !make_bthd_tmap(&tv, a.v, a.B, a.T, a.H, DV))
    return cudaErrorInvalidValue;
  tb = tq;   // placeholders, read only under the matching flag
  tw = tq;
  if ((a.flags & 2u) && !make_bthd_tmap(&tb, a.b, a.B, a.T, a.H, DK)) return cudaErrorInvalidValue;
  if ((a.flags & 4u) && !make_bthd_tmap(&tw, a.w, a.B, a.T, a.H, DV)) return cudaErrorInvalidValue;
  auto kern = chunk_prep_kernel<DK, DV, SC, VB, DYN, LEAN, RF>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L::launch_bytes));
  if (err != cudaSuccess) return err;
  if (LEAN &&   // three CTAs' shared memory needs the largest carve-out
      (err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  static_cast<int>(cudaSharedmemCarveoutMaxShared))) != cudaSuccess)
    return err;
  // persistent: two CTAs per SM (three for the lean layout) walk the B * H * ceil(T / 64)
  // chunks
  int dev = 0, sms = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return err;
  const int n_chunks = (a.T + kChunk - 1) / kChunk;
  const int rc = rg.chunks > 0 ? rg.chunks : n_chunks - rg.chunk0;
  if (rg.chunk0 < 0 || rc < 1 || rg.chunk0 + rc > n_chunks) return cudaErrorInvalidValue;
  const long long total = static_cast<long long>(rc) * a.B * a.H;
  long long grid = total < 1LL * kPerSm * sms ? total : 1LL * kPerSm * sms;
  if (DYN != (rg.counter != nullptr)) return cudaErrorInvalidValue;
  if (DYN) {   // claimed work: enough CTAs of at most per_cta items each
    if (rg.per_cta < 1) return cudaErrorInvalidValue;
    grid = (total + rg.per_cta - 1) / rg.per_cta;
  }
  kern<<<static_cast<unsigned>(grid), kThreads, L::launch_bytes, stream>>>(a, tq, tk, tv, tb, tw,
                                                                          packets, status, rg);
  return cudaGetLastError();
}

template <int DK, int DV, bool DYN>
cudaError_t launch_prep(const ChunkArgs& a, unsigned char* packets, int* status,
                        const PrepRange& rg, cudaStream_t stream) {
  if (a.flags & 16u)
    return launch_prep_kernel<DK, DV, true, true, DYN>(a, packets, status, rg, stream);
  if ((a.flags & 7u) == 0)   // scalar gates: three CTAs per SM
    return launch_prep_kernel<DK, DV, true, false, DYN, true>(a, packets, status, rg, stream);
  if constexpr (DK == 128 && DV == 128) {   // channel decay: rho-folded packets
    if (a.flags & 1u)
      return launch_prep_kernel<DK, DV, false, false, DYN, false, true>(a, packets, status, rg,
                                                                        stream);
  }
  return launch_prep_kernel<DK, DV, false, false, DYN>(a, packets, status, rg, stream);
}

template <bool DYN>
cudaError_t launch_prep_dims(const ChunkArgs& a, int dk, unsigned char* packets, int* status,
                             cudaStream_t stream, const PrepRange& rg) {
  if (dk == 64 && a.dv == 64) return launch_prep<64, 64, DYN>(a, packets, status, rg, stream);
  if (dk == 64 && a.dv == 128) return launch_prep<64, 128, DYN>(a, packets, status, rg, stream);
  if (dk == 128 && a.dv == 64) return launch_prep<128, 64, DYN>(a, packets, status, rg, stream);
  if (dk == 128 && a.dv == 128) return launch_prep<128, 128, DYN>(a, packets, status, rg, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

// The kernel is compiled twice: with a fixed persistent stride here, and with
// claimed work items in chunk_prep_claimed.cu (which defines
// GDR_PREP_CLAIMED and includes this file), so that the stride variant carries
// no code of the other and the two build in parallel.
#ifndef GDR_PREP_CLAIMED
cudaError_t launch_chunk_prep(const ChunkArgs& a, int dk, unsigned char* packets, int* status,
                              cudaStream_t stream, const PrepRange& rg) {
  if (rg.counter) return launch_chunk_prep_claimed(a, dk, packets, status, stream, rg);
  return launch_prep_dims<false>(a, dk, packets, status, stream, rg);
}
#else
cudaError_t launch_chunk_prep_claimed(const ChunkArgs& a, int dk, unsigned char* packets,
                                      int* status, cudaStream_t stream, const PrepRange& rg) {
  if (!rg.counter) return cudaErrorInvalidValue;
  return launch_prep_dims<true>(a, dk, packets, status, stream, rg);
}
#endif

}  // namespace gdr
