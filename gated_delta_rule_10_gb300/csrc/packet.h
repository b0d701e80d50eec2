// Per-chunk packet written by the chunk preparation kernel and read by the
// chunk scan kernel of the two-kernel chunkwise forward (bf16 inputs).
//
// A packet holds everything the state pass needs from one chunk of C = 64
// tokens of one (batch, head), in the order of the Gated DeltaNet-2 notes, key
// design 2 (S_{n+1} = Diag(gamma_C) S_n + K_tail^T (U - Y S_n),
// O_n = Q_gamma S_n + A_qk (U - Y S_n)):
//
//   Q_gamma  64 x d_k  bf16, s gamma_r (.) q_r           (A operand, K-major)
//   -Y       64 x d_k  bf16, -(A E_abs)                  (A operand, K-major)
//   K_tail   64 x d_k  bf16, (gamma_C / gamma_r) (.) k_r  (A operand, MN-major)
//   A_qk     64 x 64   bf16, tril(Q_gamma K_bar^T)       (A operand, K-major)
//   gamma_C  d_k fp32 (padded to 1 KB)
//   U        64 x d_v  bf16, A Z                         (64-column blocks)
//
// Tiles are stored as byte images of the 128-byte-swizzled shared-memory
// layout (tc::tile_off), so one plain bulk copy to a 1024-aligned shared
// address yields MMA-ready operands. The part before U is loaded whole by every
// value slice; U is loaded one 64-column block (8 KB) per slice.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace gdr {

template <int DK, int DV>
struct Packet {
  static constexpr uint32_t oQg = 0;
  static constexpr uint32_t oY = oQg + 128 * DK;
  static constexpr uint32_t oKt = oY + 128 * DK;
  static constexpr uint32_t oAqk = oKt + 128 * DK;
  static constexpr uint32_t oGc = oAqk + 8192;
  static constexpr uint32_t kCommon = oGc + 1024;   // Q_gamma .. gamma_C
  static constexpr uint32_t oU = kCommon;
  static constexpr uint32_t kUSlice = 8192;         // one 64-column block of U
  static constexpr uint32_t bytes = oU + 128 * DV;
  static_assert(bytes % 1024 == 0, "packets stay 1024-byte multiples");
};

inline size_t packet_bytes(int dk, int dv) {
  return static_cast<size_t>(3 * 128 * dk + 8192 + 1024 + 128 * dv);
}

}  // namespace gdr
