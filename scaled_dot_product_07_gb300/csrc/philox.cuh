// Counter-based dropout RNG of the attention kernels.
//
// Philox-4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11): per round, counter words 0 and 2 are
// multiplied by two fixed constants; the high halves of the products are
// XORed with the other counter words and the round key, the low halves move
// into the odd words; the key advances by two Weyl constants.
//
// The counter is a function of the absolute element index only ("REDO of
// dropout support for mem eff #102038", pytorch PR 103704, Summary: the RNG
// uses the absolute index, and (seed, offset) travel from forward to
// backward), so the forward and backward kernels regenerate the same mask
// whatever their tiling:
//   n   = ((b*H + h)*Sq + i)*Sk + j
//   ctr = (lo32(n>>2), hi32(n>>2), lo32(offset), hi32(offset)), key = (lo32 seed, hi32 seed)
//   u   = Philox(ctr, key)[n & 3];  keep <=> u >= threshold = floor(p * 2^32)
#pragma once

#include <cstdint>

namespace sdpa {

struct PhiloxKey {
  uint32_t k0, k1;    // seed
  uint32_t off_lo, off_hi;  // offset (counter words 2, 3)
};

__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo_a = 0xD2511F53u * c0;
    const uint32_t hi_a = __umulhi(0xD2511F53u, c0);
    const uint32_t lo_b = 0xCD9E8D57u * c2;
    const uint32_t hi_b = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi_b ^ c1 ^ k0;
    const uint32_t n2 = hi_a ^ c3 ^ k1;
    c0 = n0;
    c1 = lo_b;
    c2 = n2;
    c3 = lo_a;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return make_uint4(c0, c1, c2, c3);
}

// The four draws of group g = n >> 2 (elements n = 4g .. 4g+3).
__device__ __forceinline__ uint4 philox_group(uint64_t g, const PhiloxKey& pk) {
  return philox4x32_10(static_cast<uint32_t>(g), static_cast<uint32_t>(g >> 32), pk.off_lo,
                       pk.off_hi, pk.k0, pk.k1);
}

// Keep bits of the 32*W consecutive absolute indices n0 .. n0+32W-1:
// bit e of bits[e/32] is 1 iff element n0+e is kept.
template <int W>
__device__ __forceinline__ void keep_bits(uint64_t n0, uint32_t threshold, const PhiloxKey& pk,
                                          uint32_t (&bits)[W]) {
  const uint64_t g0 = n0 >> 2;
  const uint32_t a = static_cast<uint32_t>(n0 & 3u);
  // 8W+1 groups cover the range for any alignment a; stream bit 4t+w holds
  // the decision of n = 4(g0+t)+w, i.e. of element e = 4t+w-a.
  uint32_t s[W + 1];
#pragma unroll
  for (int i = 0; i <= W; ++i) s[i] = 0u;
#pragma unroll
  for (int t = 0; t < 8 * W + 1; ++t) {
    const uint4 u = philox_group(g0 + t, pk);
    const uint32_t nib = (u.x >= threshold ? 1u : 0u) | (u.y >= threshold ? 2u : 0u) |
                         (u.z >= threshold ? 4u : 0u) | (u.w >= threshold ? 8u : 0u);
    s[(4 * t) / 32] |= nib << ((4 * t) % 32);
  }
#pragma unroll
  for (int i = 0; i < W; ++i) bits[i] = __funnelshift_r(s[i], s[i + 1], a);
}

// The key of one launch: the one passed in the kernel parameters, or, when
// the caller handed over a device pointer to {seed, offset} (so that a
// captured graph can be replayed with fresh values), the one read from it.
__device__ __forceinline__ PhiloxKey launch_key(const PhiloxKey& pk, const uint64_t* rng_dev) {
  if (rng_dev == nullptr) return pk;
  const uint64_t seed = rng_dev[0], off = rng_dev[1];
  PhiloxKey k;
  k.k0 = static_cast<uint32_t>(seed);
  k.k1 = static_cast<uint32_t>(seed >> 32);
  k.off_lo = static_cast<uint32_t>(off);
  k.off_hi = static_cast<uint32_t>(off >> 32);
  return k;
}

// Flat (batch, head) index of the counter: b*H + h over the whole problem,
// so a launch that holds a slice of the batches and heads (b0, h0 its first
// ones, H_total the problem's heads per batch) draws the slice of the whole
// problem's mask.
__device__ __forceinline__ uint64_t counter_bh(int b, int h, int b0, int h0, int H_total) {
  return static_cast<uint64_t>(b0 + b) * static_cast<uint64_t>(H_total) +
         static_cast<uint64_t>(h0 + h);
}

// Keep bit of one absolute index.
__device__ __forceinline__ bool keep_one(uint64_t n, uint32_t threshold, const PhiloxKey& pk) {
  const uint4 u = philox_group(n >> 2, pk);
  const uint32_t w = static_cast<uint32_t>(n & 3u);
  const uint32_t v = w == 0 ? u.x : (w == 1 ? u.y : (w == 2 ? u.z : u.w));
  return v >= threshold;
}

}  // namespace sdpa
