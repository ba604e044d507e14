// Device-side dropout generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
// "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11, section 4.2),
// written from the paper's definition.
//
// The WGSL backward page multiplies by dropout_scale(p, seed, bh, qi, kj)
// whose hash is not published; this library fixes it as:
//   key = (seed lo32, seed hi32), counter = (qi >> 2, kj, bh, 0),
//   word = output (qi & 3), keep iff word >= T, T = min(floor(p 2^32), 2^32-1),
//   M = keep ? 1/(1-p) : 0.
// One call therefore serves four consecutive queries of one key, which is how
// the dK/dV kernel walks its score tile (one key per thread, queries along
// the thread's registers).
#pragma once
#include <cstdint>

namespace attnbwd {

struct Philox4 {
  uint32_t w[4];
};

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2,
                                                 uint32_t c3, uint32_t k0, uint32_t k1) {
  // round multipliers and Weyl key increments of Philox4x32 (SC'11)
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(M0, c0), lo0 = M0 * c0;
    const uint32_t hi1 = __umulhi(M1, c2), lo1 = M1 * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0;
    const uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += W0;
    k1 += W1;
  }
  Philox4 out;
  out.w[0] = c0;
  out.w[1] = c1;
  out.w[2] = c2;
  out.w[3] = c3;
  return out;
}

}  // namespace attnbwd
