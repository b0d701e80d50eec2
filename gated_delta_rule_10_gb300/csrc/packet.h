// Per-chunk packet written by the chunk preparation kernel and read by the
// chunk scan kernel of the two-kernel chunkwise forward (bf16 inputs).
//
// A packet holds everything the state pass needs from one chunk of C = 64
// tokens of one (batch, head), in the order of the Gated DeltaNet-2 notes, key
// design 2 (S_{n+1} = Diag(gamma_C) S_n + K_tail^T (U - Y S_n),
// O_n = Q_gamma S_n + A_qk (U - Y S_n)):
//
//   [Q_gamma; -Y]  128 x d_k bf16: rows 0..63 s gamma_r (.) q_r, rows 64..127
//                  -(A E_abs); one M=128 A operand (K-major), so a single MMA
//                  group gives Q_gamma S_n and -Y S_n
//   K_tail   64 x d_k  bf16, (gamma_C / gamma_r) (.) k_r  (A operand, MN-major)
//   gamma_C  d_k fp32 (padded to 1 KB)
//   A_qk     64 x 64   bf16, tril(Q_gamma K_bar^T)       (A operand, K-major)
//   U        64 x d_v  bf16, A Z                         (64-column blocks)
// U follows A_qk directly (also in the scan's shared-memory stage), so an M=128
// operand starting at A_qk reads finite bf16 values in its lower half.
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
  static constexpr uint32_t oQY = 0;                 // [Q_gamma; -Y], 128 rows
  static constexpr uint32_t oKt = oQY + 256 * DK;
  static constexpr uint32_t oGc = oKt + 128 * DK;
  static constexpr uint32_t oAqk = oGc + 1024;
  static constexpr uint32_t kCommon = oAqk + 8192;  // [Q_gamma; -Y] .. A_qk
  static constexpr uint32_t oU = kCommon;
  static constexpr uint32_t kUSlice = 8192;         // one 64-column block of U
  static constexpr uint32_t bytes = oU + 128 * DV;
  static_assert(bytes % 1024 == 0, "packets stay 1024-byte multiples");
};

inline size_t packet_bytes(int dk, int dv) {
  return static_cast<size_t>(3 * 128 * dk + 8192 + 1024 + 128 * dv);
}

// Packet of the write strength per value channel (one scalar decay per head,
// beta per value channel; LLMs from scratch ch. 11, section 11.3). Each value
// column c has its own transition, so there is no shared (I + T)^{-1}; the
// packet carries what the scan needs to solve per column
//   (I + diag(beta_c) L) W_c = diag(beta_c) (V_c - K_gamma S_n)_c
// by substitution, with L = tril(decay (.) K K^T, -1) shared by the columns:
//   [Q_gamma; K_gamma] 128 x d_k bf16: rows 64..127 hold +gamma_r k_r
//   K_tail, gamma_C, A_qk              as in Packet
//   V        64 x d_v bf16 in U's place (64-column blocks, right after A_qk)
//   L        64 x 64 fp32, row-major, zero on and above the diagonal
//   beta     64 x d_v bf16, 64-column blocks in the tile layout
template <int DK, int DV>
struct PacketVB {
  static constexpr uint32_t oQY = 0;
  static constexpr uint32_t oKt = oQY + 256 * DK;
  static constexpr uint32_t oGc = oKt + 128 * DK;
  static constexpr uint32_t oAqk = oGc + 1024;
  static constexpr uint32_t kCommon = oAqk + 8192;
  static constexpr uint32_t oU = kCommon;           // V
  static constexpr uint32_t kUSlice = 8192;
  static constexpr uint32_t oL = oU + 128 * DV;
  static constexpr uint32_t kL = 64 * 64 * 4;
  static constexpr uint32_t oB = oL + kL;            // beta
  static constexpr uint32_t kBSlice = 8192;
  static constexpr uint32_t bytes = oB + 128 * DV;
  static_assert(bytes % 1024 == 0, "packets stay 1024-byte multiples");
};

inline size_t packet_vb_bytes(int dk, int dv) {
  return static_cast<size_t>(3 * 128 * dk + 8192 + 1024 + 256 * dv + 64 * 64 * 4);
}

}  // namespace gdr
