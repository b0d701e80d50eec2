// (I + T)^{-1} for a strictly lower-triangular 64x64 fp32 matrix T, by one
// warpgroup (4 warps), used by the tensor-core chunk kernels.
//
// This is the forward substitution of the Gated DeltaNet-2 notes, key design 2
// (A = (I + T)^{-1}), organised in blocks: each warp inverts one 16x16
// diagonal block by substitution in fp32 (lane c owns column c); the
// off-diagonal blocks follow from
//   A_IJ = -Dinv_I T_IJ Dinv_J                         (16-row blocks (1,0), (3,2))
//   A[32:64, 0:32] = -A2 T[32:64, 0:32] A1             (A1, A2 the 32x32 diagonal blocks)
// with the products on warp-level MMA, each fp32 operand split into bf16
// hi + lo (hi*hi + hi*lo + lo*hi keeps ~2^-16 relative accuracy).
#pragma once

#include "common.cuh"

namespace gdr {

// fp32 pair -> bf16 pair hi + lo (x ~= hi + lo to ~2^-17 relative)
__device__ __forceinline__ void split2(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x - hf.x, y - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// One 16x8 tile C += M[r0.., mk0..mk0+15] * N[nk0..nk0+15, n0..n0+7] from
// row-major fp32 shared matrices, with both operands split into bf16 hi + lo
// and the products hi*hi + hi*lo + lo*hi (warp-level MMA, fp32 accumulation).
__device__ __forceinline__ void mma16x8x16_f32(float (&c)[4], const float* M, int ldm, int r0,
                                               int mk0, const float* N, int ldn, int nk0, int n0) {
  const int l = threadIdx.x & 31;
  const int r = r0 + (l >> 2), kc = mk0 + 2 * (l & 3), n = n0 + (l >> 2), kr = nk0 + 2 * (l & 3);
  uint32_t ah[4], al[4], bh0, bl0, bh1, bl1;
  split2(M[r * ldm + kc], M[r * ldm + kc + 1], ah[0], al[0]);
  split2(M[(r + 8) * ldm + kc], M[(r + 8) * ldm + kc + 1], ah[1], al[1]);
  split2(M[r * ldm + kc + 8], M[r * ldm + kc + 9], ah[2], al[2]);
  split2(M[(r + 8) * ldm + kc + 8], M[(r + 8) * ldm + kc + 9], ah[3], al[3]);
  split2(N[kr * ldn + n], N[(kr + 1) * ldn + n], bh0, bl0);
  split2(N[(kr + 8) * ldn + n], N[(kr + 9) * ldn + n], bh1, bl1);
  mma_bf16_16816(c, ah, bh0, bh1);
  mma_bf16_16816(c, ah, bl0, bl1);
  mma_bf16_16816(c, al, bh0, bh1);
}

// Stores sign * C of a 16x8 accumulator tile at (r0, n0) of a row-major fp32
// matrix.
__device__ __forceinline__ void store_tile(float* D, int ld, int r0, int n0, const float (&c)[4],
                                           float sign) {
  const int l = threadIdx.x & 31;
  const int r = r0 + (l >> 2), n = n0 + 2 * (l & 3);
  D[r * ld + n] = sign * c[0];
  D[r * ld + n + 1] = sign * c[1];
  D[(r + 8) * ld + n] = sign * c[2];
  D[(r + 8) * ld + n + 1] = sign * c[3];
}

// Column `lane` (< 16) of the inverse of the unit lower-triangular diagonal
// block I + T[base.., base..] (16 x 16, T strictly lower in a [..][65] fp32
// array) by forward substitution, right-looking: once col[j] is known it is
// folded into the running sums of every later row, so each row's sum takes its
// terms in the same order (j = 0, 1, ...) as a row-by-row dot product, and the
// result is the same to the bit, but a row waits only for the one update that
// its predecessor adds, not for a whole dot product.
__device__ __forceinline__ void diag_block_column(const float* sT, int base, int lane,
                                                  float (&col)[16]) {
  float acc[16];
#pragma unroll
  for (int r = 0; r < 16; ++r) acc[r] = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    col[j] = (j == lane ? 1.f : 0.f) - acc[j];
#pragma unroll
    for (int r = j + 1; r < 16; ++r) acc[r] = fmaf(sT[(base + r) * 65 + base + j], col[j], acc[r]);
  }
}

// T: [64][65] fp32 (zeros on and above the diagonal); A: [64][65] fp32 out
// (blocks above the diagonal are left undefined); scratch: 4 x 256 floats.
// `w` is the warp index within the warpgroup, `sync` a barrier over it.
template <typename Sync>
__device__ __forceinline__ void invert_unit_lower_64(const float* sT, float* sAf, float* sP,
                                                     int w, int lane, Sync sync) {
  if (lane < 16) {
    const int base = w * 16;
    float col[16];
    diag_block_column(sT, base, lane, col);
#pragma unroll
    for (int r = 0; r < 16; ++r) sAf[(base + r) * 65 + base + lane] = col[r];
  }
  sync();
  // 16-row blocks (1,0) and (3,2): A_IJ = -Dinv_I T_IJ Dinv_J. Warp w takes
  // block (1,0) for w < 2, else (3,2), value columns 8 (w & 1) .. +7.
  {
    float* sX = sP + w * 256;                     // per-warp 32 x 8 scratch
    const int I = w < 2 ? 1 : 3, J = I - 1, n0 = 16 * J + 8 * (w & 1);
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    mma16x8x16_f32(c, sT, 65, 16 * I, 16 * J, sAf, 65, 16 * J, n0);
    store_tile(sX, 8, 0, 0, c, -1.f);              // X = -T_IJ Dinv_J (16 x 8)
    __syncwarp();
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    mma16x8x16_f32(d, sAf, 65, 16 * I, 16 * I, sX, 8, 0, 0);
    store_tile(sAf, 65, 16 * I, n0, d, 1.f);       // A_IJ = Dinv_I X
  }
  sync();
  // 32-row blocks: A[32:64, 0:32] = -A2 T[32:64, 0:32] A1 with
  // A1 = A[0:32, 0:32], A2 = A[32:64, 32:64]; warp w: columns 8w .. 8w+7.
  {
    float* sX = sP + w * 256;
    const int n0 = 8 * w;
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    if (n0 < 16) {                                  // A1 rows 0..15 vanish past column 15
      mma16x8x16_f32(c0, sT, 65, 32, 0, sAf, 65, 0, n0);
      mma16x8x16_f32(c1, sT, 65, 48, 0, sAf, 65, 0, n0);
    }
    mma16x8x16_f32(c0, sT, 65, 32, 16, sAf, 65, 16, n0);
    mma16x8x16_f32(c1, sT, 65, 48, 16, sAf, 65, 16, n0);
    store_tile(sX, 8, 0, 0, c0, -1.f);             // X = -T[32:64, 0:32] A1 (32 x 8)
    store_tile(sX, 8, 16, 0, c1, -1.f);
    __syncwarp();
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
    mma16x8x16_f32(d0, sAf, 65, 32, 32, sX, 8, 0, 0);    // A2 rows 0..15 vanish past col 15
    mma16x8x16_f32(d1, sAf, 65, 48, 32, sX, 8, 0, 0);
    mma16x8x16_f32(d1, sAf, 65, 48, 48, sX, 8, 16, 0);
    store_tile(sAf, 65, 32, n0, d0, 1.f);
    store_tile(sAf, 65, 48, n0, d1, 1.f);
  }
  sync();
}

// The same inverse on two warpgroups (8 warps, `w` = 0..7): the diagonal
// blocks and the 16-row level as above on warps 0-3 (warps 4-7 wait), the
// 32-row level split over all 8 warps, one 16 x 8 output tile each:
//   X = -T[32:64, 0:32] A1          (warp w: rows 32 + 16 (w >> 2), columns 8 (w & 3))
//   A[32:64, 0:32] = A2 X           (same tile), after a barrier over the 8 warps.
// `sync4` is a barrier over warps 0-3, `sync8` over all 8. X goes to sX
// ([32][33] fp32, shared).
template <typename Sync4, typename Sync8>
__device__ __forceinline__ void invert_unit_lower_64_w8(const float* sT, float* sAf, float* sP,
                                                        float* sX, int w, int lane, Sync4 sync4,
                                                        Sync8 sync8) {
  if (w < 4) {
    if (lane < 16) {
      const int base = w * 16;
      float col[16];
      diag_block_column(sT, base, lane, col);
#pragma unroll
      for (int r = 0; r < 16; ++r) sAf[(base + r) * 65 + base + lane] = col[r];
    }
    sync4();
    float* sY = sP + w * 256;                      // per-warp 16 x 8 scratch
    const int I = w < 2 ? 1 : 3, J = I - 1, n0 = 16 * J + 8 * (w & 1);
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    mma16x8x16_f32(c, sT, 65, 16 * I, 16 * J, sAf, 65, 16 * J, n0);
    store_tile(sY, 8, 0, 0, c, -1.f);              // -T_IJ Dinv_J
    __syncwarp();
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    mma16x8x16_f32(d, sAf, 65, 16 * I, 16 * I, sY, 8, 0, 0);
    store_tile(sAf, 65, 16 * I, n0, d, 1.f);       // A_IJ
  }
  sync8();
  const int r0 = 32 + 16 * (w >> 2), n0 = 8 * (w & 3);
  {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    if (n0 < 16) mma16x8x16_f32(c, sT, 65, r0, 0, sAf, 65, 0, n0);   // A1 rows 0..15 vanish past column 15
    mma16x8x16_f32(c, sT, 65, r0, 16, sAf, 65, 16, n0);
    store_tile(sX, 33, r0 - 32, n0, c, -1.f);
  }
  sync8();
  {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    mma16x8x16_f32(d, sAf, 65, r0, 32, sX, 33, 0, n0);                // A2 columns 32..47
    if (r0 == 48) mma16x8x16_f32(d, sAf, 65, r0, 48, sX, 33, 16, n0);  // rows 48.. also see 48..63
    store_tile(sAf, 65, r0, n0, d, 1.f);
  }
  sync8();
}

// invert_unit_lower_64_w8 in place: sA ([64][65] fp32, shared) holds T on
// entry and A on exit. A block of A overwrites the block of T at its place only
// once every read of that T block is done: within the warp for the diagonal
// blocks, over warps 0-3 for the 16-row level; the 32-row level writes after the
// barrier that ends its reads of T. sP: per-warp 16 x 8 scratch (4 x 128
// floats); sX: [32][33] floats.
template <typename Sync4, typename Sync8>
__device__ __forceinline__ void invert_unit_lower_64_w8_inplace(float* sA, float* sP, float* sX,
                                                                int w, int lane, Sync4 sync4,
                                                                Sync8 sync8) {
  if (w < 4) {
    if (lane < 16) {
      const int base = w * 16;
      float col[16];
      diag_block_column(sA, base, lane, col);
      __syncwarp(0x0000ffffu);                     // every lane has read its rows of T_JJ
#pragma unroll
      for (int r = 0; r < 16; ++r) sA[(base + r) * 65 + base + lane] = col[r];
    }
    sync4();
    float* sY = sP + w * 128;
    const int I = w < 2 ? 1 : 3, J = I - 1, n0 = 16 * J + 8 * (w & 1);
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    mma16x8x16_f32(c, sA, 65, 16 * I, 16 * J, sA, 65, 16 * J, n0);
    store_tile(sY, 8, 0, 0, c, -1.f);              // -T_IJ Dinv_J
    __syncwarp();
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    mma16x8x16_f32(d, sA, 65, 16 * I, 16 * I, sY, 8, 0, 0);
    sync4();                                       // both warps of block (I, J) have read T_IJ
    store_tile(sA, 65, 16 * I, n0, d, 1.f);        // A_IJ
  }
  sync8();
  const int r0 = 32 + 16 * (w >> 2), n0 = 8 * (w & 3);
  {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    if (n0 < 16) mma16x8x16_f32(c, sA, 65, r0, 0, sA, 65, 0, n0);
    mma16x8x16_f32(c, sA, 65, r0, 16, sA, 65, 16, n0);
    store_tile(sX, 33, r0 - 32, n0, c, -1.f);
  }
  sync8();
  {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    mma16x8x16_f32(d, sA, 65, r0, 32, sX, 33, 0, n0);
    if (r0 == 48) mma16x8x16_f32(d, sA, 65, r0, 48, sX, 33, 16, n0);
    store_tile(sA, 65, r0, n0, d, 1.f);
  }
  sync8();
}

}  // namespace gdr
