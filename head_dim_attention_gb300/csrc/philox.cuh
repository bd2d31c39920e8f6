// Dropout keep masks from the counter-based generator Philox4x32-10 (Salmon,
// Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC 2011: four 32-bit words, ten rounds).
//
// The dropout contract (the pages name no generator): for query row i and key
// j of query head h in batch b, the generator runs on counter
// (j / 8, i, b * Hq + h, offset) with key (seed lo, seed hi); score (i, j)
// reads the 16-bit field j mod 2 of output word (j mod 8) / 2 and is kept when
// that value is at least the threshold t = round(p * 65536) (at most 65535).
// One generator call serves eight consecutive keys of one query row.
#pragma once

#include <cstdint>

namespace ffpa {

struct DropKey {
  uint32_t k0, k1;  // the 64-bit seed
  uint32_t bh;      // b * Hq + h of the query head
  uint32_t off;     // stream offset
  uint32_t t;       // keep threshold
};

// Ten Philox rounds on counter c with key (k0, k1).  Each round takes the
// 64-bit products of the round multipliers with words 0 and 2 and mixes their
// halves with words 1 and 3 and the key; the key advances by the Weyl
// increments between rounds.
__device__ __forceinline__ void philox4x32_10(uint32_t (&c)[4], uint32_t k0, uint32_t k1) {
  constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
  constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint64_t p0 = static_cast<uint64_t>(kM0) * c[0];
    const uint64_t p1 = static_cast<uint64_t>(kM1) * c[2];
    const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ c[1] ^ k0;
    const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = static_cast<uint32_t>(p1);
    c[2] = n2;
    c[3] = static_cast<uint32_t>(p0);
  }
}

// Keep bits of keys 8 jb .. 8 jb + 7 of query row i: bit v for key 8 jb + v.
__device__ __forceinline__ uint32_t keep8(const DropKey& dk, uint32_t jb, uint32_t i) {
  uint32_t c[4] = {jb, i, dk.bh, dk.off};
  philox4x32_10(c, dk.k0, dk.k1);
  uint32_t m = 0;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    m |= ((c[w] & 0xFFFFu) >= dk.t ? 1u : 0u) << (2 * w);
    m |= ((c[w] >> 16) >= dk.t ? 1u : 0u) << (2 * w + 1);
  }
  return m;
}

// Keep bits of keys j0 .. j0 + 63 of query row i (j0 a multiple of 8): bit e
// of lo (e < 32) or hi (e >= 32) for key j0 + e.  The eight generator calls
// run in a loop that is not unrolled: eight inlined copies of the ten rounds
// overflowed the instruction cache of the kernels that call this.
__device__ __forceinline__ void keep64_row(const DropKey& dk, int j0, int i, uint32_t& lo, uint32_t& hi) {
  uint64_t bits = 0;
#pragma unroll 1
  for (int g = 0; g < 8; ++g)
    bits |= static_cast<uint64_t>(keep8(dk, static_cast<uint32_t>(j0 / 8 + g), static_cast<uint32_t>(i))) << (8 * g);
  lo = static_cast<uint32_t>(bits);
  hi = static_cast<uint32_t>(bits >> 32);
}

// The transposed layout: lane l of a warp holds key j0 + l (j0 a multiple of
// 32) and needs the keep bits of query rows i0 .. i0 + 63 for it: bit e of lo
// (e < 32) or hi (e >= 32) for query row i0 + e.  Each lane runs the
// generator for one (query row, 8-key block) pair per group of eight query
// rows (row i0 + 8 g + (l mod 8), keys of lanes 8 (l / 8) .. 8 (l / 8) + 7),
// and the bits go to the lanes that need them by warp shuffles.  All 32 lanes
// must call it together.
__device__ __forceinline__ void keep64_col(const DropKey& dk, int j0, int i0, int lane, uint32_t& lo,
                                           uint32_t& hi) {
  // byte g of m: the bits of this lane's generator call for group g (a loop
  // that is not unrolled, as in keep64_row)
  uint64_t m = 0;
  const uint32_t jb = static_cast<uint32_t>(j0 / 8 + (lane >> 3));
#pragma unroll 1
  for (int g = 0; g < 8; ++g)
    m |= static_cast<uint64_t>(keep8(dk, jb, static_cast<uint32_t>(i0 + 8 * g + (lane & 7)))) << (8 * g);
  const uint32_t m_lo = static_cast<uint32_t>(m), m_hi = static_cast<uint32_t>(m >> 32);
  lo = 0;
  hi = 0;
  const int sh = lane & 7;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    // lane (l & ~7) | k ran the calls of query rows i0 + 8 g + k; bit (l & 7) of
    // each byte is this lane's key
    const int src = (lane & ~7) | k;
    const uint32_t a = __shfl_sync(0xffffffffu, m_lo, src);
    const uint32_t b = __shfl_sync(0xffffffffu, m_hi, src);
    lo |= ((a >> sh) & 0x01010101u) << k;
    hi |= ((b >> sh) & 0x01010101u) << k;
  }
}

}  // namespace ffpa
