// Dropout keep bits drawn from Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC 2011), shared by the
// layer's dropout kernels and the attention core's probabilities kernel.
// Element e of a site with seed and stream takes the 16-bit field 16 (e mod 2)
// of output word (e mod 8) / 2 at counter (e / 8 as two words, low first, then
// stream as two words) under key (seed as two words), and is kept iff the
// field is >= the threshold floor(p 2^16).
#pragma once

#include <stdint.h>

namespace tp {

__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(M0, c0), lo0 = M0 * c0;
    const uint32_t hi1 = __umulhi(M1, c2), lo1 = M1 * c2;
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
    k0 += W0;
    k1 += W1;
  }
  return make_uint4(c0, c1, c2, c3);
}

// Keep bits of the 8 elements of generator block `blk` (bit f = element 8 blk + f).
__device__ __forceinline__ uint32_t keep8(uint64_t blk, uint64_t seed, uint64_t stream, uint32_t thr) {
  const uint4 w = philox4x32_10(static_cast<uint32_t>(blk), static_cast<uint32_t>(blk >> 32),
                                static_cast<uint32_t>(stream), static_cast<uint32_t>(stream >> 32),
                                static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  uint32_t bits = 0;
#pragma unroll
  for (int f = 0; f < 8; ++f) {
    const uint32_t field = (ws[f >> 1] >> (16 * (f & 1))) & 0xFFFFu;
    bits |= (field >= thr ? 1u : 0u) << f;
  }
  return bits;
}

// Keep bits of the 16 elements 16 b .. 16 b + 15 (bit f = element 16 b + f).
__device__ __forceinline__ uint32_t keep16(uint64_t b, uint64_t seed, uint64_t stream, uint32_t thr) {
  return keep8(2 * b, seed, stream, thr) | (keep8(2 * b + 1, seed, stream, thr) << 8);
}

}  // namespace tp
