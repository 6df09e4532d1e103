// Counter-based random draws and the Gumbel-max race of the sampler step (device code used by
// the row kernels in ds_rows.cu and by the self-conditioning kernel, which runs the race on
// warps beside its GEMM).
#pragma once

#include <climits>

#include "ds_internal.h"

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
    const uint64_t p0 = (uint64_t)0xD2511F53u * c.x, p1 = (uint64_t)0xCD9E8D57u * c.z;
    c = u32x4{(uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k1,
              (uint32_t)p0};
  }
  return c;
}

// N independent blocks under the same key, round by round, so their multiply chains overlap.
// Each product is one 32 x 32 -> 64-bit multiply (high and low words from the same product;
// measured 3-8% faster in the race than separate high and low multiplies).
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
      const uint64_t p0 = (uint64_t)0xD2511F53u * c[q].x, p1 = (uint64_t)0xCD9E8D57u * c[q].z;
      c[q] = u32x4{(uint32_t)(p1 >> 32) ^ c[q].y ^ k0, (uint32_t)p1,
                   (uint32_t)(p0 >> 32) ^ c[q].w ^ k1, (uint32_t)p0};
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

// Token e (0..7) of a group of eight bf16 values (two per word, the lower token in the low half)
// as fp32; e is a constant after unrolling.
DS_DEV float bf16_at(const uint4& g, int e) {
  const uint32_t w = e < 2 ? g.x : (e < 4 ? g.y : (e < 6 ? g.z : g.w));
  return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

// hi is p rounded to bf16, so |lo| <= 2^-8 hi and hi sc (1 + 2^-7), rounded twice, is above
// (hi + lo) sc rounded: an upper bound of p from the hi half alone.
constexpr float kHiBound = 1.0078125f;
// kc (1 + 2^-19), rounded, exceeds kc / (1 - 2^-20): with it the pre-test of gumbel_race16 skips
// only tokens that gumbel_token would skip.
constexpr float kCutBound = 1.0000019073486328f;

// The Gumbel-max exponential race over 16 consecutive tokens j .. j + 15 of position i of
// sequence b: with E_j = -ln u_j (u_j from the Gumbel stream of Philox) and p_j = exp(y_j - m)
// (m the row maximum), argmax_j (y_j - ln E_j) = argmin_j E_j / p_j. p_j arrives as bf16 hi + lo
// in two groups of eight with scales sa, sb. Tokens are tested against kc = min(kbest, cut),
// cut being a key some token has already reached (the warp's best so far): a group of four is
// skipped without its draw when even the smallest E (> 2^-24) over its largest p cannot beat kc,
// and a token without its logarithm when 1 - u_j proves it cannot. Both tests first use the
// upper bound of p from the hi half (kHiBound); the exact p = (hi + lo) sc is formed only for the
// tokens that pass, and gumbel_token then decides with it exactly as without the pre-test. Every
// skip needs a strict inequality, so a token tying the best is never skipped. The four draws are
// computed together. Tokens arrive in increasing j, so a strict comparison keeps the lowest token
// on ties. With SKIP4 the first four tokens are left out (already raced by gumbel_seed4).
template <bool SKIP4 = false>
DS_DEV void gumbel_race16(const uint4& hia, const uint4& loa, float sa, const uint4& hib,
                          const uint4& lob, float sb, int64_t j, uint32_t i, uint32_t b,
                          uint32_t step, uint64_t seed, float cut, float& kbest, int32_t& bj,
                          float& bp) {
  // the upper bound of p of each group of four from its largest hi half: hi is a non-negative
  // bf16 (the sign bit clear), so the integer order of the 16-bit patterns is the value order,
  // and fp32 multiplication by the positive scale is monotone, so this is exactly the largest
  // of the four tokens' bounds hi sc (1 + 2^-7)
  const float sau = sa * kHiBound, sbu = sb * kHiBound;
  auto group_bound = [](uint32_t w0, uint32_t w1, float scale) {
    const uint32_t m2 = __vmaxu2(w0, w1);
    return __uint_as_float(max(m2 & 0xFFFFu, m2 >> 16) << 16) * scale;
  };
  float pmq[4];
  pmq[0] = group_bound(hia.x, hia.y, sau);
  pmq[1] = group_bound(hia.z, hia.w, sau);
  pmq[2] = group_bound(hib.x, hib.y, sbu);
  pmq[3] = group_bound(hib.z, hib.w, sbu);
  bool need[4];
  bool any = false;
  const float kc0 = fminf(kbest, cut);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    need[q] = !(SKIP4 && q == 0) && !(5.9604645e-8f >= kc0 * pmq[q]);
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
    const float kcs = fminf(kbest, cut) * kCutBound;
    {
      // 1 - u is smallest for the largest word and kcs p is largest for the group's largest
      // bound: if even that pair fails the token test, every token of the group fails it (same
      // fp32 operations, monotone), so the four tests are skipped. Same box, B = 1: the race as
      // its own launch 0.074-0.077 -> 0.065-0.066 ms.
      const uint32_t rmax = max(max(w[q].x, w[q].y), max(w[q].z, w[q].w));
      const float fmx = __uint_as_float(0x3F800000u | (rmax >> 9));
      if ((2.0f - fmx) - 5.9604644775390625e-8f > kcs * pmq[q]) continue;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int t = 4 * q + e;
      const uint32_t r = word_of(w[q], e);
      const float f = __uint_as_float(0x3F800000u | (r >> 9));
      const float pu = t < 8 ? bf16_at(hia, t) * sau : bf16_at(hib, t - 8) * sbu;
      if ((2.0f - f) - 5.9604644775390625e-8f > kcs * pu) continue;
      const float pe = t < 8 ? (bf16_at(hia, t) + bf16_at(loa, t)) * sa
                             : (bf16_at(hib, t - 8) + bf16_at(lob, t - 8)) * sb;
      if (!(pe > 0.f)) continue;
      gumbel_token(pe, r, (int32_t)(j + t), fminf(kbest, cut), kbest, bj, bp);
    }
  }
}

// The race over the first four tokens j .. j + 3 of a group (words hi.x, hi.y) without any
// cutoff, for every lane of a warp at once: its result seeds the warp's cutoff before the lanes
// race their other tokens, so that the logarithm is taken on few tokens (and few lanes).
DS_DEV void gumbel_seed4(const uint4& hi, const uint4& lo, float sc, int64_t j, uint32_t i,
                         uint32_t b, uint32_t step, uint64_t seed, float& kbest, int32_t& bj,
                         float& bp) {
  u32x4 w[1] = {u32x4{(uint32_t)(j >> 2), i, b, (step << 2) | kGumbelStream}};
  philox4x32_10_n<1>(w, (uint32_t)seed, (uint32_t)(seed >> 32));
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float pe = (bf16_at(hi, e) + bf16_at(lo, e)) * sc;
    if (pe > 0.f) gumbel_token(pe, word_of(w[0], e), (int32_t)(j + e), INFINITY, kbest, bj, bp);
  }
}

// ----------------------------------------------------------------------------------------
// The race over one (row, 8192-token chunk) by one warp
// ----------------------------------------------------------------------------------------
// Sixteen consecutive tokens of one lane: two groups of eight (bf16 hi and lo) with the scale of
// their segment (0: nothing to race, nothing loaded).
struct Slab16 {
  uint4 h0, h1, l0, l1;
  float sc;
};

DS_DEV void slab_load(Slab16& t, const uint16_t* ph, const uint16_t* pl, float sc) {
  t.sc = sc;
  if (sc > 0.f) {
    t.h0 = __ldcs(reinterpret_cast<const uint4*>(ph));
    t.h1 = __ldcs(reinterpret_cast<const uint4*>(ph + 8));
    t.l0 = __ldcs(reinterpret_cast<const uint4*>(pl));
    t.l1 = __ldcs(reinterpret_cast<const uint4*>(pl + 8));
  } else {
    t.h0 = t.h1 = t.l0 = t.l1 = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Position of the n-th set bit (from 0) of m, n < popc(m): halving search on population counts.
DS_DEV int nth_set_bit(uint32_t m, int n) {
  int pos = 0;
#pragma unroll
  for (int w = 16; w; w >>= 1) {
    const int c = __popc(m & ((1u << w) - 1u));
    if (n >= c) {
      n -= c;
      m >>= w;
      pos += w;
    }
  }
  return pos;
}

// The exponential race over segments u0 .. u1 - 1 (u1 - u0 <= 64) of chunk c of row r by one
// warp, p_j = (P_hi + P_lo)[j] exp(m_ref - m) with m the row maximum and m_ref the maximum the
// probabilities were taken against: of token j's 128-token segment, or with tile_ref of its
// 256-token tile (the larger of the two segment maxima). Leaves in each lane its best key
// E_j / p_j, token and p (lowest token on equal keys within the lane); skipped segments and
// skipped draws are exactly those that cannot win. Segments more than kGumbelReach below m are
// not read; the others are raced four at a time in token order (lane l takes tokens
// 16 (l % 8) .. 16 (l % 8) + 15 of the (4 k + l / 8)-th segment in reach in round k), the next
// round loaded while the current one is raced. The lanes race the first round's first four
// tokens in full, and the warp's best key then cuts the rest. With shared_cut (a key as its bit
// pattern, in shared memory) several warps racing parts of the same chunk exchange their best
// keys after every round: any key a token of the chunk has reached is a valid cutoff for the
// chunk's winner (keys are >= 0, so their bit patterns order like the values).
DS_DEV void gumbel_race_segments(const GumbelWork& g, int64_t V, int r, int c, int u0, int u1,
                                 float& kbest, int32_t& bj, float& bp,
                                 unsigned* shared_cut = nullptr) {
  constexpr int kSegTok = 128;
  const int lane = threadIdx.x & 31;
  const int b = r / g.L, i = r % g.L;
  // from L2: in the queue the record may have been written in this launch, after another
  // record of the same line was read here
  const float m = __ldcg(&g.rs[r].m);
  const int64_t j0 = (int64_t)c * kChunk;
  const ChunkStat* sg = g.seg + (size_t)r * (V / kSegTok) + j0 / kSegTok;
  kbest = INFINITY;
  bp = 1.f;
  bj = INT_MAX;
  // segment scales: lane l holds segments u0 + l and u0 + l + 32
  float sc[2];
  uint32_t in[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int u = u0 + lane + 32 * h;
    float v = 0.f;
    if (u < u1) {
      const float mg = sg[u].m;
      // chunks start at multiples of 256 tokens, so segment pairs (2w, 2w + 1) are tiles
      if (mg >= m - kGumbelReach) v = expf((g.tile_ref ? fmaxf(mg, sg[u ^ 1].m) : mg) - m);
    }
    sc[h] = v;
    in[h] = __ballot_sync(0xffffffffu, v > 0.f);
  }
  const int n0 = __popc(in[0]), n_in = n0 + __popc(in[1]);
  if (n_in == 0) return;  // no token of these segments can win
  // this lane's 16 tokens in round k (offset in the chunk) and their scale (0: none)
  auto locate = [&](int k, float& s) -> int {
    const int n = 4 * k + (lane >> 3);
    int t = 0;
    if (n < n_in) t = n < n0 ? nth_set_bit(in[0], n) : 32 + nth_set_bit(in[1], n - n0);
    const float a0 = __shfl_sync(0xffffffffu, sc[0], t & 31);
    const float a1 = __shfl_sync(0xffffffffu, sc[1], t & 31);
    s = n < n_in ? (t < 32 ? a0 : a1) : 0.f;
    return kSegTok * (u0 + t) + 16 * (lane & 7);
  };
  const uint32_t st = (uint32_t)g.step[b];
  const uint32_t sid = stream_id((uint32_t)b, g.blk);
  const uint16_t* ph = g.Phi + (size_t)r * V + j0;
  const uint16_t* pl = g.Plo + (size_t)r * V + j0;
  const int rounds = (n_in + 3) / 4;
  float cut, s;
  Slab16 cur, nxt;
  int off = locate(0, s);
  slab_load(cur, ph + off, pl + off, s);
  for (int k = 0; k < rounds; ++k) {
    int off_n = 0;
    if (k + 1 < rounds) {
      off_n = locate(k + 1, s);
      slab_load(nxt, ph + off_n, pl + off_n, s);
    }
    const int64_t j = g.j_offset + j0 + off;  // global token index (draws and winners)
    if (k == 0) {
      if (cur.sc > 0.f)
        gumbel_seed4(cur.h0, cur.l0, cur.sc, j, (uint32_t)i, sid, st, g.seed, kbest, bj, bp);
      cut = warp_min(kbest);
      if (cur.sc > 0.f)
        gumbel_race16<true>(cur.h0, cur.l0, cur.sc, cur.h1, cur.l1, cur.sc, j, (uint32_t)i, sid,
                            st, g.seed, cut, kbest, bj, bp);
    } else if (cur.sc > 0.f) {
      gumbel_race16(cur.h0, cur.l0, cur.sc, cur.h1, cur.l1, cur.sc, j, (uint32_t)i, sid, st,
                    g.seed, cut, kbest, bj, bp);
    }
    cut = warp_min(fminf(cut, kbest));
    if (shared_cut) {
      if (lane == 0) atomicMin(shared_cut, __float_as_uint(cut));
      __syncwarp();
      cut = fminf(cut, __uint_as_float(*(volatile unsigned*)shared_cut));
    }
    cur = nxt;
    off = off_n;
  }
}

// Winner of the exponential race over chunk c of row r (all its segments) by one warp, written
// to best[r, c] as a Best record (v = -key, rel = 1, y = ln p of the winner): largest -key, then
// lowest token.
DS_DEV void gumbel_chunk_warp(const GumbelWork& g, int64_t V, int r, int c) {
  const int64_t j0 = (int64_t)c * kChunk, j1 = min(V, j0 + kChunk);
  const int nseg = (int)((j1 - j0) / 128);  // whole segments: V is a multiple of 256
  float kbest, bp;
  int32_t bj;
  gumbel_race_segments(g, V, r, c, 0, nseg, kbest, bj, bp);
  float v = -kbest;
  int32_t jw = bj;
  warp_best(v, jw);
  // the winner's p comes from the lane that holds it (every lane when there is none: p = 1)
  const uint32_t owner = __ballot_sync(0xffffffffu, bj == jw);
  const float pw = __shfl_sync(0xffffffffu, bp, __ffs(owner) - 1);
  if ((threadIdx.x & 31) == 0) g.best[(size_t)r * g.n_chunks + c] = Best{v, jw, logf(pw), 1};
}

// The row statistics of k_row_merge computed by one warp, bit for bit: lane l stands for the
// eight threads l + 32 j (j = 0 .. 7) of that kernel's 256-thread CTA, each taking the segments
// q = base + t + 256 k in the same order, with the same fp32 Kahan sums per thread, the same
// shuffle tree per warp of eight and the same fp64 sum over the eight warps: m and argmax
// (lowest token on equal maxima), l = sum_g l_g e^{m_g - m}, a = sum_g (a_g + l_g (m_g - m))
// e^{m_g - m}, entropy ln l - a / l. Valid in lane 0.
DS_DEV RowStat row_merge_warp(const ChunkStat* __restrict__ c, int n) {
  constexpr int kT = 256, kPer = 16, kJ = kT / 32;
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  int32_t arg = INT_MAX;
  for (int base = 0; base < n; base += kT * kPer)
    for (int k = 0; k < kPer; ++k) {
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        const int q = base + lane + 32 * j + kT * k;
        if (q < n) {
          const ChunkStat t = c[q];
          if (better(t.m, t.arg, m, arg)) {
            m = t.m;
            arg = t.arg;
          }
        }
      }
    }
  warp_best(m, arg);  // the maximum and its lowest token do not depend on the order
  float l[kJ], a[kJ], cl[kJ], ca[kJ];
#pragma unroll
  for (int j = 0; j < kJ; ++j) l[j] = a[j] = cl[j] = ca[j] = 0.f;
  auto kahan = [](float& sum, float& comp, float x) {
    const float y = x - comp;
    const float t = sum + y;
    comp = (t - sum) - y;
    sum = t;
  };
  for (int base = 0; base < n; base += kT * kPer)
    for (int k = 0; k < kPer; ++k) {
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        const int q = base + lane + 32 * j + kT * k;
        if (q < n) {
          const ChunkStat t = c[q];
          if (t.arg == INT_MAX) continue;
          const float dm = t.m - m;
          const float sc = expf(dm);
          kahan(l[j], cl[j], __fmul_rn(t.l, sc));
          kahan(a[j], ca[j], __fmul_rn(fmaf(t.l, dm, t.a), sc));
        }
      }
    }
  double tl = 0.0, ta = 0.0;
#pragma unroll
  for (int j = 0; j < kJ; ++j) {
    float lj = l[j] - cl[j], aj = a[j] - ca[j];
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      lj += __shfl_xor_sync(0xffffffffu, lj, o);
      aj += __shfl_xor_sync(0xffffffffu, aj, o);
    }
    tl += (double)lj;
    ta += (double)aj;
  }
  return RowStat{m, (float)tl, (float)(log(tl) - ta / tl), arg};
}

// One warp's share of the queue: items are taken one at a time until the queue is empty;
// finished sequences' items are skipped (their records are not written). With g.rs_out the first
// R items are row merges, and a race item first waits (bounded) for its row's merge.
DS_DEV void gumbel_queue_warp(const GumbelWork& g, int64_t V) {
  const int lane = threadIdx.x & 31;
  const bool merge = g.rs_out != nullptr;
  const uint32_t n_merge = merge ? (uint32_t)g.R : 0u;
  const uint32_t n_items = n_merge + (uint32_t)g.R * (uint32_t)g.n_chunks;
  const uint32_t gen = merge ? *(volatile const uint32_t*)(g.ctr + 2) + 1u : 0u;
  const int n_seg = (int)(V / 128);
  for (;;) {
    uint32_t it = 0;
    if (lane == 0) it = atomicAdd(g.ctr, 1u);
    it = __shfl_sync(0xffffffffu, it, 0);
    if (it >= n_items) return;
    if (it < n_merge) {
      const int r = (int)it;
      if (g.done && g.done[r / g.L]) continue;
      const RowStat st = row_merge_warp(g.seg + (size_t)r * n_seg, n_seg);
      if (lane == 0) {
        g.rs_out[r] = st;
        __threadfence();
        st_release_gpu(g.row_flags + r, gen);
      }
      continue;
    }
    it -= n_merge;
    const int r = (int)(it / (uint32_t)g.n_chunks), c = (int)(it % (uint32_t)g.n_chunks);
    if (g.done && g.done[r / g.L]) continue;
    if (merge) {
      int ok = 1;
      if (lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(g.row_flags + r) != gen) {
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(g.err, kErrTimeout);
            ok = 0;
            break;
          }
          __nanosleep(64);
        }
      }
      // the other lanes read the row's record after lane 0's acquire
      __syncwarp();
      if (!__shfl_sync(0xffffffffu, ok, 0)) continue;
    }
    gumbel_chunk_warp(g, V, r, c);
  }
}

// After every warp of the CTA has left gumbel_queue_warp (a __syncthreads in between), one
// thread of each CTA: the last CTA of the grid returns the queue counters to zero and advances
// the generation.
DS_DEV void gumbel_queue_release(const GumbelWork& g) {
  __threadfence();
  if (atomicAdd(g.ctr + 1, 1u) == gridDim.x - 1) {
    atomicExch(g.ctr, 0u);
    atomicExch(g.ctr + 1, 0u);
    atomicAdd(g.ctr + 2, 1u);  // the next launch's row flags
  }
}

}  // namespace ds
