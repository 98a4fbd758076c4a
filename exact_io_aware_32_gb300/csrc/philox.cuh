// Dropout masks from Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel
// random numbers: as easy as 1, 2, 3", SC 2011), a counter-based generator, so
// that the backward makes the forward's mask again from the seed alone, as
// chapter 09 of "FlashAttention and GPU Memory" describes (the mask is never
// stored).
//
// One call covers a block of 4 queries by 4 keys of one head: counter
// (j / 4, i / 4, bh, offset), key = the 64-bit seed; word i mod 4, byte
// j mod 4 of the output is element (i, j)'s random byte, and the element is
// kept iff that byte >= p256 (dropout probability p256 / 256).
//
// The four lanes of a quad (lanes 4m .. 4m + 3) hold four consecutive rows
// (queries in the forward and dQ kernels, keys in the dK/dV kernel), so each
// lane computes a quarter of the quad's calls and the quad exchanges words.
#pragma once

#include <cstdint>

namespace fa {
namespace philox {

constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;  // round multipliers
constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;  // key increments

// Round keys (k0 + r W0, k1 + r W1), r = 0 .. 9, of a 64-bit seed, as rk[2r], rk[2r + 1].
__host__ __device__ inline void round_keys(unsigned long long seed, uint32_t (&rk)[20]) {
  uint32_t k0 = (uint32_t)(seed & 0xFFFFFFFFull), k1 = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    rk[2 * r] = k0;
    rk[2 * r + 1] = k1;
    k0 += kW0;
    k1 += kW1;
  }
}

// Philox4x32-10 of counter (c0, c1, c2, c3) with precomputed round keys.
__device__ __forceinline__ void philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                              const uint32_t* rk, uint32_t (&x)[4]) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(kM0, c0), lo0 = kM0 * c0;
    const uint32_t hi1 = __umulhi(kM1, c2), lo1 = kM1 * c2;
    c0 = hi1 ^ c1 ^ rk[2 * r];
    c1 = lo1;
    c2 = hi0 ^ c3 ^ rk[2 * r + 1];
    c3 = lo0;
  }
  x[0] = c0;
  x[1] = c1;
  x[2] = c2;
  x[3] = c3;
}

// 4 x 4 transpose of words across the lanes of a quad: lane a ends with
// x[s] = (lane s's x)[a]. Two exchanges, with lanes a ^ 2 and a ^ 1; every
// lane of the warp must take part.
__device__ __forceinline__ void quad_transpose(uint32_t (&x)[4]) {
  const int a = threadIdx.x & 3;
  const bool b1 = (a & 2) != 0;
  uint32_t s0 = b1 ? x[0] : x[2], s1 = b1 ? x[1] : x[3];
  uint32_t r0 = __shfl_xor_sync(0xffffffffu, s0, 2), r1 = __shfl_xor_sync(0xffffffffu, s1, 2);
  if (b1) {
    x[0] = r0;
    x[1] = r1;
  } else {
    x[2] = r0;
    x[3] = r1;
  }
  const bool b0 = (a & 1) != 0;
  s0 = b0 ? x[0] : x[1];
  s1 = b0 ? x[2] : x[3];
  r0 = __shfl_xor_sync(0xffffffffu, s0, 1);
  r1 = __shfl_xor_sync(0xffffffffu, s1, 1);
  if (b0) {
    x[0] = r0;
    x[2] = r1;
  } else {
    x[1] = r0;
    x[3] = r1;
  }
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// 4 x 4 transpose of the bytes of four words: byte b of x[w] moves to byte w of x[b].
__device__ __forceinline__ void byte_transpose(uint32_t (&x)[4]) {
  const uint32_t t01l = prmt(x[0], x[1], 0x5140u), t01h = prmt(x[0], x[1], 0x7362u);
  const uint32_t t23l = prmt(x[2], x[3], 0x5140u), t23h = prmt(x[2], x[3], 0x7362u);
  x[0] = prmt(t01l, t23l, 0x5410u);
  x[1] = prmt(t01l, t23l, 0x7632u);
  x[2] = prmt(t01h, t23h, 0x5410u);
  x[3] = prmt(t01h, t23h, 0x7632u);
}

// Per byte: 0xFF where the byte is >= the threshold (kept), else 0.
__device__ __forceinline__ uint32_t keep_bytes(uint32_t x, uint32_t thr4) { return __vcmpgeu4(x, thr4); }

// The 16-bit masks of a bf16 pair from two bytes of a keep word: bytes (0, 1) or (2, 3).
__device__ __forceinline__ uint32_t pair_mask_lo(uint32_t keep) { return prmt(keep, 0u, 0x1100u); }
__device__ __forceinline__ uint32_t pair_mask_hi(uint32_t keep) { return prmt(keep, 0u, 0x3322u); }

// Drop factor of byte b of a keep word: f (the scale 256 / (256 - p256)) if kept, else 0.
__device__ __forceinline__ float keep_factor(uint32_t keep, int b, float f) {
  return ((keep >> (8 * b)) & 1u) ? f : 0.f;
}

}  // namespace philox
}  // namespace fa
