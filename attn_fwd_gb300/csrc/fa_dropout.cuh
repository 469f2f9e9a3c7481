// fa_dropout.cuh -- regenerated dropout masks for the attention kernels.
//
// The forward keeps only O(N) statistics and the backward regenerates the
// random dropout mask instead of reading a stored one ("Как работает
// FlashAttention математически", section 5; "FlashAttention" notes,
// "Backward Pass of flashattention").  Generator: Philox4x32-10, the
// counter-based generator of Salmon, Moraes, Dror and Shaw, "Parallel random
// numbers: as easy as 1, 2, 3" (SC'11), with key = the 64-bit seed and counter
// (key j / 4, query i / 4, head h, batch b): one call gives a 4 x 4 block of
// bytes, byte j % 4 of word i % 4 belonging to (i, j).  A pair is kept iff its
// byte is >= t = round(256 p); kept values are scaled by 256 / (256 - t).
//
// Lanes whose index differs only in its two low bits own four consecutive
// query rows (forward) or key rows (backward), so the four lanes of a quad
// compute four different blocks and exchange words: each call yields 16 used
// decisions on both sides.
#pragma once

#include <cstdint>

namespace fa {

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;                 // Weyl increments of the key
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// x[k] of a runtime index k in 0..3 (selects, no local memory).
__device__ __forceinline__ uint32_t pick4(const uint32_t (&x)[4], uint32_t k) {
  const uint32_t a = (k & 1u) ? x[1] : x[0];
  const uint32_t b = (k & 1u) ? x[3] : x[2];
  return (k & 2u) ? b : a;
}

// Across the four lanes of a quad (u = lane & 3): y[t] = x of lane t, word u.
__device__ __forceinline__ void quad_transpose(const uint32_t (&x)[4], uint32_t u, uint32_t (&y)[4]) {
  uint32_t r[4];
  r[0] = pick4(x, u);
  r[1] = __shfl_xor_sync(0xffffffffu, pick4(x, u ^ 1u), 1);   // = word u of lane u ^ 1
  r[2] = __shfl_xor_sync(0xffffffffu, pick4(x, u ^ 2u), 2);
  r[3] = __shfl_xor_sync(0xffffffffu, pick4(x, u ^ 3u), 3);
#pragma unroll
  for (uint32_t t = 0; t < 4; ++t) y[t] = pick4(r, t ^ u);
}

// 4 x 4 byte transpose within a thread: y[t] = (byte t of w[0], w[1], w[2], w[3]).
__device__ __forceinline__ void byte_transpose(const uint32_t (&w)[4], uint32_t (&y)[4]) {
  const uint32_t a0 = __byte_perm(w[0], w[1], 0x5140), a1 = __byte_perm(w[0], w[1], 0x7362);
  const uint32_t a2 = __byte_perm(w[2], w[3], 0x5140), a3 = __byte_perm(w[2], w[3], 0x7362);
  y[0] = __byte_perm(a0, a2, 0x5410);
  y[1] = __byte_perm(a0, a2, 0x7632);
  y[2] = __byte_perm(a1, a3, 0x5410);
  y[3] = __byte_perm(a1, a3, 0x7632);
}

// Keep decisions of 16 bytes (byte v of y[t], kept iff >= t_drop) as bits:
// byte v of y[t] -> bit 16 (v >> 1) + 2 t + (v & 1).  `add` = (256 - t_drop)
// in both 16-bit halves: a byte plus add carries into bit 8 iff byte >= t_drop.
__device__ __forceinline__ uint32_t keep_bits16(const uint32_t (&y)[4], uint32_t add) {
  uint32_t acc = 0;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t e = (y[t] & 0x00FF00FFu) + add;          // bytes 0, 2
    const uint32_t o = ((y[t] >> 8) & 0x00FF00FFu) + add;   // bytes 1, 3
    acc |= ((e >> 8) & 0x00010001u) << (2 * t);
    acc |= ((o >> 8) & 0x00010001u) << (2 * t + 1);
  }
  return acc;
}

// Bit of column c (0..31) in a word built from two 16-column groups g = c / 16
// (the second shifted left by 8): column 16 g + 4 t + v.
__host__ __device__ constexpr int keep_bit(int c) {
  return 8 * ((c >> 4) & 1) + 16 * ((c & 3) >> 1) + 2 * ((c >> 2) & 3) + (c & 1);
}

// Forward: keep bits of 32 key columns kc0 .. kc0 + 31 (kc0 a multiple of 32)
// for this lane's query row i.
__device__ __forceinline__ uint32_t keep_bits_row(int i, int kc0, uint32_t h, uint32_t b, uint32_t seed_lo,
                                                  uint32_t seed_hi, uint32_t add, uint32_t u) {
  uint32_t bits = 0;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const uint4 w4 = philox4x32_10(
        make_uint4(static_cast<uint32_t>(kc0 / 4 + 4 * g) + u, static_cast<uint32_t>(i) >> 2, h, b), seed_lo,
        seed_hi);
    const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
    uint32_t y[4];
    quad_transpose(w, u, y);
    bits |= keep_bits16(y, add) << (8 * g);
  }
  return bits;
}

// Backward: keep bits of 32 query columns qc0 .. qc0 + 31 (qc0 a multiple of
// 4) for this lane's key row j.
__device__ __forceinline__ uint32_t keep_bits_col(int j, int qc0, uint32_t h, uint32_t b, uint32_t seed_lo,
                                                  uint32_t seed_hi, uint32_t add, uint32_t u) {
  uint32_t bits = 0;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const uint4 w4 = philox4x32_10(
        make_uint4(static_cast<uint32_t>(j) >> 2, static_cast<uint32_t>(qc0 / 4 + 4 * g) + u, h, b), seed_lo,
        seed_hi);
    const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
    uint32_t t4[4], y[4];
    byte_transpose(w, t4);
    quad_transpose(t4, u, y);
    bits |= keep_bits16(y, add) << (8 * g);
  }
  return bits;
}

}  // namespace fa
