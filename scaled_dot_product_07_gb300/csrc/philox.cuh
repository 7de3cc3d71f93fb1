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
    // one 32x32 -> 64-bit product gives both halves
    const uint64_t pa = static_cast<uint64_t>(0xD2511F53u) * c0;
    const uint64_t pb = static_cast<uint64_t>(0xCD9E8D57u) * c2;
    const uint32_t n0 = static_cast<uint32_t>(pb >> 32) ^ c1 ^ k0;
    const uint32_t n2 = static_cast<uint32_t>(pa >> 32) ^ c3 ^ k1;
    c0 = n0;
    c1 = static_cast<uint32_t>(pb);
    c2 = n2;
    c3 = static_cast<uint32_t>(pa);
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

// The ten round keys of a key (seed): words 2r and 2r+1 are the key of round r.
struct PhiloxRoundKeys {
  uint32_t w[20];
};

__host__ __device__ inline PhiloxRoundKeys philox_round_keys(const PhiloxKey& pk) {
  PhiloxRoundKeys rk;
  uint32_t k0 = pk.k0, k1 = pk.k1;
  for (int r = 0; r < 10; ++r) {
    rk.w[2 * r] = k0;
    rk.w[2 * r + 1] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return rk;
}

// Group g drawn with round keys that the host formed and passed in the
// kernel parameters: each round reads its key as a constant operand, so the
// key schedule costs no registers and no additions (the same draws as
// philox_group with the key the round keys came from).
__device__ __forceinline__ uint4 philox_group_rk(uint64_t g, uint32_t off_lo, uint32_t off_hi,
                                                 const PhiloxRoundKeys& rk) {
  uint32_t c0 = static_cast<uint32_t>(g), c1 = static_cast<uint32_t>(g >> 32);
  uint32_t c2 = off_lo, c3 = off_hi;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t pa = static_cast<uint64_t>(0xD2511F53u) * c0;
    const uint64_t pb = static_cast<uint64_t>(0xCD9E8D57u) * c2;
    const uint32_t n0 = static_cast<uint32_t>(pb >> 32) ^ c1 ^ rk.w[2 * r];
    const uint32_t n2 = static_cast<uint32_t>(pa >> 32) ^ c3 ^ rk.w[2 * r + 1];
    c0 = n0;
    c1 = static_cast<uint32_t>(pb);
    c2 = n2;
    c3 = static_cast<uint32_t>(pa);
  }
  return make_uint4(c0, c1, c2, c3);
}

// 32 x 32 bit transpose across a warp: lane l passes row l (bit c = column
// c) and gets column l back (bit r = row r). Five butterfly stages; in the
// stage of distance s each lane keeps its own half of every 2s-bit block
// and takes the matching half from lane l ^ s. All 32 lanes must call it.
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x, int lane) {
  const uint32_t masks[5] = {0x0000ffffu, 0x00ff00ffu, 0x0f0f0f0fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    const int s = 16 >> i;
    const uint32_t m = masks[i];
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, s);
    x = (lane & s) ? ((x & ~m) | ((y & ~m) >> s)) : ((x & m) | ((y & m) << s));
  }
  return x;
}

// Keep bits of the 16 groups g0 .. g0+15 (elements 4 g0 .. 4 g0 + 63): bit
// 4t + w of words[t / 8] (t mod 8 in place of t) is 1 iff element
// 4(g0 + t) + w is kept. RK: the round keys the host formed (rk); else
// formed from pk.
template <bool RK>
__device__ __forceinline__ void keep_words_aligned(uint64_t g0, uint32_t threshold,
                                                   const PhiloxKey& pk, const PhiloxRoundKeys& rk,
                                                   uint32_t (&words)[2]) {
  words[0] = words[1] = 0u;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const uint4 u = RK ? philox_group_rk(g0 + t, pk.off_lo, pk.off_hi, rk) : philox_group(g0 + t, pk);
    const uint32_t nib = (u.x >= threshold ? 1u : 0u) | (u.y >= threshold ? 2u : 0u) |
                         (u.z >= threshold ? 4u : 0u) | (u.w >= threshold ? 8u : 0u);
    words[t >> 3] |= nib << (4 * (t & 7));
  }
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

// Keep bits of one key column: the 32*W elements (i0 + c, kj), c < 32W, whose
// absolute indices are n_base + c*Sk (n_base the index of (i0, kj)). For Sk a
// multiple of 4 the four lanes of a quad (lanes 4m .. 4m+3 of a warp, holding
// keys 4u .. 4u+3 in that order, all with the same i0) need the same groups:
// group (n_base + c*Sk) >> 2 holds the quad's four keys at row i0 + c. Lane
// q = lane & 3 draws the groups of rows c = 4t + q and the quad swaps the
// keep nibbles, so each group is drawn once instead of four times. Bit c of
// kb[c / 32] is 1 iff element (i0 + c, kj) is kept. All 32 lanes of the warp
// must call it together.
template <int W>
__device__ __forceinline__ void keep_bits_quad(uint64_t n_base, uint64_t Sk, uint32_t threshold,
                                               const PhiloxKey& pk, uint32_t (&kb)[W]) {
  const uint32_t q = threadIdx.x & 3u;
  const uint32_t quad = threadIdx.x & 28u;  // lane of the quad's first key
  const uint64_t g0 = n_base >> 2;
  const uint64_t gs = Sk >> 2;
#pragma unroll
  for (int m = 0; m < W; ++m) {
    // nibble t: keep bits of the quad's keys 0..3 at row 32m + 4t + q
    uint32_t own = 0u;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint4 u = philox_group(g0 + static_cast<uint64_t>(32 * m + 4 * t + q) * gs, pk);
      const uint32_t nib = (u.x >= threshold ? 1u : 0u) | (u.y >= threshold ? 2u : 0u) |
                           (u.z >= threshold ? 4u : 0u) | (u.w >= threshold ? 8u : 0u);
      own |= nib << (4 * t);
    }
    // row 32m + 4t + o comes from lane o of the quad, bit q of its nibble t
    uint32_t bits = 0u;
#pragma unroll
    for (int o = 0; o < 4; ++o) {
      const uint32_t wo = __shfl_sync(0xffffffffu, own, quad | static_cast<uint32_t>(o));
      bits |= ((wo >> q) & 0x11111111u) << o;
    }
    kb[m] = bits;
  }
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
