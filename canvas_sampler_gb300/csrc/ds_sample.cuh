// Counter-based random draws and the Gumbel-max race of the sampler step (device code used by
// the row kernels in ds_rows.cu).
#pragma once

#include "ds_common.cuh"

namespace ds {

// ----------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
// SC'11): ten rounds of two 32x32->64-bit products mixed with the key, key bumped by Weyl
// constants between rounds.
// ----------------------------------------------------------------------------------------
struct u32x4 {
  uint32_t x, y, z, w;
};

DS_DEV u32x4 philox4x32_10(u32x4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = u32x4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
  }
  return c;
}

// N independent blocks under the same key, round by round, so their multiply chains overlap.
template <int N>
DS_DEV void philox4x32_10_n(u32x4 (&c)[N], uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
#pragma unroll
    for (int q = 0; q < N; ++q) {
      const uint32_t hi0 = __umulhi(0xD2511F53u, c[q].x), lo0 = 0xD2511F53u * c[q].x;
      const uint32_t hi1 = __umulhi(0xCD9E8D57u, c[q].z), lo1 = 0xCD9E8D57u * c[q].z;
      c[q] = u32x4{hi1 ^ c[q].y ^ k0, lo1, hi0 ^ c[q].w ^ k1, lo0};
    }
  }
}

DS_DEV uint32_t word_of(const u32x4& v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

// Streams of the sampler's draws (the low two bits of counter word 3).
constexpr uint32_t kGumbelStream = 0, kRenoiseStream = 1;

// u in (0, 1) from a word: (2 (r >> 9) + 1) / 2^24, exact in fp32.
DS_DEV float word_to_uniform(uint32_t r) {
  return (float)(((r >> 9) << 1) | 1u) * 5.9604644775390625e-8f;
}

// Gumbel noise g = -ln(-ln u).
DS_DEV float gumbel_from_word(uint32_t r) { return -logf(-logf(word_to_uniform(r))); }

// Uniform token in [0, V): (r * V) >> 32.
DS_DEV int32_t token_from_word(uint32_t r, uint32_t V) {
  return (int32_t)(((uint64_t)r * (uint64_t)V) >> 32);
}

// Counter word 2 of a sequence's draws: b + 2^16 block, where blk points at the block index of a
// block-autoregressive run (nullptr or 0 for a single canvas).
DS_DEV uint32_t stream_id(uint32_t b, const int32_t* blk) {
  return b + ((blk ? (uint32_t)*blk : 0u) << 16);
}

// The Gumbel counter of token block j>>2 at position i of sequence b.
DS_DEV u32x4 gumbel_block(uint32_t jblk, uint32_t i, uint32_t b, uint32_t step, uint64_t seed) {
  return philox4x32_10(u32x4{jblk, i, b, (step << 2) | kGumbelStream}, (uint32_t)seed,
                       (uint32_t)(seed >> 32));
}

// A token more than this below the row maximum cannot win the Gumbel-max: the largest Gumbel
// draw is -ln(-ln(1 - 2^-24)) = 16.64, the smallest -ln(-ln 2^-24) = -2.81, and
// 19.6 > 16.64 + 2.81 leaves margin for fp32 rounding.
constexpr float kGumbelReach = 19.6f;

// One token's entry in the exponential race: p_j > 0 its probability (relative to the row
// maximum), r the Philox word of its Gumbel draw. f = 1 + (r >> 9) 2^-23 from the mantissa bits;
// u = (2 (r >> 9) + 1) / 2^24 = (f - 1) + 2^-24 and 1 - u = (2 - f) - 2^-24, both exact in fp32
// (24 significant bits), without an integer-to-float conversion. 1 - u > kc p_j proves
// E_j / p_j > kc without the logarithm (-ln u >= 1 - u; the factor 1 - 2^-20 covers the rounding
// of the computed key), so the token cannot beat a key kc that is already known.
DS_DEV void gumbel_token(float pe, uint32_t r, int32_t j, float kc, float& kbest, int32_t& bj,
                         float& bp) {
  const float f = __uint_as_float(0x3F800000u | (r >> 9));
  const float omu = (2.0f - f) - 5.9604644775390625e-8f;
  if (omu * (1.0f - 9.5367431640625e-7f) > kc * pe) return;
  const float key = -logf((f - 1.0f) + 5.9604644775390625e-8f) / pe;
  if (key < kbest) {
    kbest = key;
    bj = j;
    bp = pe;
  }
}

// p of the 8 tokens of a bf16 hi / lo group (two tokens per word, the lower token in the low
// half), times the group's scale.
DS_DEV void unpack_p8(const uint4& hi, const uint4& lo, float sc, float (&p)[8]) {
  const uint32_t hw[4] = {hi.x, hi.y, hi.z, hi.w};
  const uint32_t lw[4] = {lo.x, lo.y, lo.z, lo.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    p[2 * e] = (__uint_as_float(hw[e] << 16) + __uint_as_float(lw[e] << 16)) * sc;
    p[2 * e + 1] = (__uint_as_float(hw[e] & 0xFFFF0000u) + __uint_as_float(lw[e] & 0xFFFF0000u)) * sc;
  }
}

// The Gumbel-max exponential race over 16 consecutive tokens j .. j + 15 of position i of
// sequence b: with E_j = -ln u_j (u_j from the Gumbel stream of Philox) and p_j = exp(y_j - m)
// (m the row maximum), argmax_j (y_j - ln E_j) = argmin_j E_j / p_j. p_j arrives as bf16 hi + lo
// in two groups of eight with scales sa, sb. Tokens are tested against kc = min(kbest, cut),
// cut being a key some token has already reached (the warp's best so far): a group of four is
// skipped without its draw when even the smallest E (> 2^-24) over its largest p cannot beat kc,
// and a token without its logarithm when 1 - u_j proves it cannot; both skips need a strict
// inequality, so a token tying the best is never skipped. The four draws are computed together.
// Tokens arrive in increasing j, so a strict comparison keeps the lowest token on ties. With
// SKIP4 the first four tokens are left out (already raced by gumbel_seed4).
template <bool SKIP4 = false>
DS_DEV void gumbel_race16(const uint4& hia, const uint4& loa, float sa, const uint4& hib,
                          const uint4& lob, float sb, int64_t j, uint32_t i, uint32_t b,
                          uint32_t step, uint64_t seed, float cut, float& kbest, int32_t& bj,
                          float& bp) {
  float p[16];
  {
    float pa[8], pb[8];
    unpack_p8(hia, loa, sa, pa);
    unpack_p8(hib, lob, sb, pb);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      p[e] = pa[e];
      p[8 + e] = pb[e];
    }
  }
  bool need[4];
  bool any = false;
  const float kc0 = fminf(kbest, cut);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float pm = fmaxf(fmaxf(p[4 * q], p[4 * q + 1]), fmaxf(p[4 * q + 2], p[4 * q + 3]));
    need[q] = !(SKIP4 && q == 0) && !(5.9604645e-8f >= kc0 * pm);
    any |= need[q];
  }
  if (!any) return;
  u32x4 w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q)
    w[q] = u32x4{(uint32_t)((j + 4 * q) >> 2), i, b, (step << 2) | kGumbelStream};
  philox4x32_10_n<4>(w, (uint32_t)seed, (uint32_t)(seed >> 32));
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (!need[q]) continue;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float pe = p[4 * q + e];
      if (!(pe > 0.f)) continue;
      gumbel_token(pe, word_of(w[q], e), (int32_t)(j + 4 * q + e), fminf(kbest, cut), kbest, bj,
                   bp);
    }
  }
}

// The race over the first four tokens j .. j + 3 of a group (words hi.x, hi.y) without any
// cutoff, for every lane of a warp at once: its result seeds the warp's cutoff before the lanes
// race their other tokens, so that the logarithm is taken on few tokens (and few lanes).
DS_DEV void gumbel_seed4(const uint4& hi, const uint4& lo, float sc, int64_t j, uint32_t i,
                         uint32_t b, uint32_t step, uint64_t seed, float& kbest, int32_t& bj,
                         float& bp) {
  float p[8];
  unpack_p8(hi, lo, sc, p);
  u32x4 w[1] = {u32x4{(uint32_t)(j >> 2), i, b, (step << 2) | kGumbelStream}};
  philox4x32_10_n<1>(w, (uint32_t)seed, (uint32_t)(seed >> 32));
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (p[e] > 0.f) gumbel_token(p[e], word_of(w[0], e), (int32_t)(j + e), INFINITY, kbest, bj, bp);
}

}  // namespace ds
