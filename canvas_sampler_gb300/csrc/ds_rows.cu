// Row-level kernels of the sampler step: softmax statistics over the vocabulary, the
// bf16 hi/lo split of exp(y - m) that feeds the self-conditioning GEMM, Gumbel-max sampling
// (optionally restricted to the top-k logits), the final reduction of s, and the
// lock / re-noise / stop kernel.
//
// Definitions: DiffusionGemma Technical Report, section 6 "Sampling" (full-precision softmax
// over the vocabulary, self-conditioning matmul), section 6 "Multi-user throughput" (top-k
// truncation of the sampling step); "DiffusionGemma: Google's open diffusion LLM", section "A
// diffusion language model refines 256 tokens in 12 steps" (accept confident tokens,
// re-noise the rest uniformly, at most 48 steps).
#include <algorithm>
#include <cfloat>
#include <climits>

#include "ds_internal.h"
#include "ds_sample.cuh"

namespace ds {

namespace {

constexpr int kThreads = 256;
constexpr int kPer = kChunk / kThreads;   // 32 values per thread
constexpr int kGroups = kPer / 4;         // float4 groups per thread

__device__ float block_sum(float v, float* sh) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, ln = threadIdx.x & 31;
  __syncthreads();
  if (ln == 0) sh[w] = v;
  __syncthreads();
  v = ln < (int)(blockDim.x >> 5) ? sh[ln] : 0.f;
  return warp_sum(v);
}

// Best (v, j) over the block, then the y carried by the winner; every thread gets the result.
__device__ void block_best(float& v, int32_t& j, float& y, float* shv, int32_t* shj, float* shy) {
  float bv = v;
  int32_t bj = j;
  warp_best(bv, bj);
  const int w = threadIdx.x >> 5, ln = threadIdx.x & 31;
  __syncthreads();
  if (ln == 0) {
    shv[w] = bv;
    shj[w] = bj;
  }
  __syncthreads();
  bv = ln < (int)(blockDim.x >> 5) ? shv[ln] : -INFINITY;
  bj = ln < (int)(blockDim.x >> 5) ? shj[ln] : INT_MAX;
  warp_best(bv, bj);
  __syncthreads();
  if (j == bj && v == bv && bj != INT_MAX) *shy = y;
  __syncthreads();
  v = bv;
  j = bj;
  y = (bj != INT_MAX) ? *shy : 0.f;
}

// Inclusive/exclusive scan of one int per thread over the block (256 threads).
__device__ int block_exclusive_scan(int x, int* sh, int* total) {
  const int w = threadIdx.x >> 5, ln = threadIdx.x & 31;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (ln >= o) incl += t;
  }
  __syncthreads();
  if (ln == 31) sh[w] = incl;
  __syncthreads();
  if (w == 0) {
    int v = ln < (int)(blockDim.x >> 5) ? sh[ln] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, v, o);
      if (ln >= o) v += t;
    }
    if (ln < (int)(blockDim.x >> 5)) sh[ln] = v;  // inclusive warp totals
  }
  __syncthreads();
  const int warp_off = w > 0 ? sh[w - 1] : 0;
  *total = sh[(blockDim.x >> 5) - 1];
  return warp_off + incl - x;
}

// Select the k largest keys held by the block (NPER per thread, element order (q, thread)),
// ties at the k-th key broken toward earlier elements. Calls emit(q, slot) for each selected
// element with slot in [0, k) following element order. Radix select on 8-bit digits.
template <int NPER, class Emit>
__device__ void block_select_topk(const uint32_t (&key)[NPER], const bool (&valid)[NPER], int k,
                                  int* hist, int* scan_sh, Emit emit) {
  uint32_t prefix = 0, mask = 0;
  int need = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int t = threadIdx.x; t < 256; t += blockDim.x) hist[t] = 0;
    __syncthreads();
#pragma unroll
    for (int q = 0; q < NPER; ++q)
      if (valid[q] && (key[q] & mask) == prefix) atomicAdd(&hist[(key[q] >> shift) & 255u], 1);
    __syncthreads();
    __shared__ int sel_bin, sel_need;
    if (threadIdx.x == 0) {
      int cum = 0, bin = 0;
      for (bin = 255; bin >= 0; --bin) {
        if (cum + hist[bin] >= need) break;
        cum += hist[bin];
      }
      if (bin < 0) bin = 0;  // fewer valid elements than k: take everything
      sel_bin = bin;
      sel_need = need - cum;
    }
    __syncthreads();
    prefix |= (uint32_t)sel_bin << shift;
    mask |= 255u << shift;
    need = sel_need;
    __syncthreads();
  }
  // `prefix` is the k-th largest key; take all larger ones and the first `need` equal ones.
  int base = 0;
#pragma unroll
  for (int q = 0; q < NPER; ++q) {
    const bool gt = valid[q] && key[q] > prefix;
    const bool eq = valid[q] && key[q] == prefix;
    int total_eq = 0;
    const int eq_rank = block_exclusive_scan(eq ? 1 : 0, scan_sh, &total_eq);
    int dummy = 0;
    const bool take = gt || (eq && eq_rank < need);
    const int slot = block_exclusive_scan(take ? 1 : 0, scan_sh, &dummy);
    if (take) emit(q, base + slot);
    base += dummy;
    need -= min(need, total_eq);
  }
}

// ----------------------------------------------------------------------------------------

__global__ void __launch_bounds__(kThreads) k_chunk_stats(const float* __restrict__ Y, int64_t V,
                                                          int L, const uint8_t* __restrict__ done,
                                                          ChunkStat* __restrict__ cs,
                                                          int n_chunks) {
  __shared__ float shf[32];
  __shared__ float shv[32], shy;
  __shared__ int32_t shj[32];
  const int c = blockIdx.x, r = blockIdx.y;
  if (done && done[r / L]) return;
  const float* y = Y + (size_t)r * V;
  const int64_t j0 = (int64_t)c * kChunk, j1 = min(V, j0 + kChunk);
  float v[kPer];
  float m = -INFINITY;
  int32_t arg = INT_MAX;
#pragma unroll
  for (int g = 0; g < kGroups; ++g) {
    const int64_t j = j0 + 4 * (threadIdx.x + kThreads * g);
    if (j < j1) {
      const float4 t = *reinterpret_cast<const float4*>(y + j);
      v[4 * g] = t.x;
      v[4 * g + 1] = t.y;
      v[4 * g + 2] = t.z;
      v[4 * g + 3] = t.w;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (better(v[4 * g + e], (int32_t)(j + e), m, arg)) {
          m = v[4 * g + e];
          arg = (int32_t)(j + e);
        }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[4 * g + e] = -INFINITY;
    }
  }
  float dummy_y = 0.f;
  block_best(m, arg, dummy_y, shv, shj, &shy);
  float l = 0.f, a = 0.f;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    if (v[q] != -INFINITY) {
      const float t = v[q] - m;
      const float e = expf(t);
      l += e;
      a = fmaf(e, t, a);
    }
  }
  l = block_sum(l, shf);
  a = block_sum(a, shf);
  if (threadIdx.x == 0) cs[(size_t)r * n_chunks + c] = ChunkStat{m, l, a, arg};
}

// One CTA per row: merge of the chunk statistics (max and lowest argmax, then the rescaled
// sums in fp64; the rescale factors exp(m_c - m) <= 1 are taken in fp32, relative error ~1e-7,
// because GB300's fp64 units are slow). Each thread takes every 256th chunk; all its loads
// are issued before any arithmetic.
__global__ void __launch_bounds__(kThreads) k_row_merge(const ChunkStat* __restrict__ cs,
                                                        int n_chunks, int L,
                                                        const uint8_t* __restrict__ done,
                                                        RowStat* __restrict__ rs) {
  constexpr int kPer = 16;  // chunks per thread per batch (one batch up to 4096 chunks)
  __shared__ float shv[32], shy;
  __shared__ int32_t shj[32];
  __shared__ double shd[2][32];
  pdl_wait();
  const int r = blockIdx.x;
  if (done && done[r / L]) return;
  const ChunkStat* c = cs + (size_t)r * n_chunks;
  auto load_batch = [&](int base, ChunkStat (&mine)[kPer]) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int q = base + threadIdx.x + kThreads * k;
      mine[k] = q < n_chunks ? c[q] : ChunkStat{-INFINITY, 0.f, 0.f, INT_MAX};
    }
  };
  float m = -INFINITY, dummy_y = 0.f;
  int32_t arg = INT_MAX;
  ChunkStat mine[kPer];
  for (int base = 0; base < n_chunks; base += kThreads * kPer) {
    load_batch(base, mine);
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if (better(mine[k].m, mine[k].arg, m, arg)) {
        m = mine[k].m;
        arg = mine[k].arg;
      }
  }
  block_best(m, arg, dummy_y, shv, shj, &shy);
  // l = sum_g l_g e^{m_g - m} and a = sum_g (a_g + l_g (m_g - m)) e^{m_g - m}: every term has one
  // sign (l_g > 0, a_g <= 0, m_g <= m), so there is no cancellation; each thread sums its terms
  // in fp32 with a compensation term (Kahan), the warps by a shuffle tree and the block's eight
  // warp sums in fp64, a relative error of a few fp32 units. The products are rounded on their
  // own (no contraction into the compensated sum), so row_merge_warp (ds_sample.cuh) reproduces
  // this kernel bit for bit
  float l = 0.f, a = 0.f, cl = 0.f, ca = 0.f;
  auto kahan = [](float& sum, float& comp, float x) {
    const float y = x - comp;
    const float t = sum + y;
    comp = (t - sum) - y;
    sum = t;
  };
  for (int base = 0; base < n_chunks; base += kThreads * kPer) {
    if (base > 0 || n_chunks > kThreads * kPer) load_batch(base, mine);
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      if (mine[k].arg == INT_MAX) continue;
      const float dm = mine[k].m - m;
      const float sc = expf(dm);
      kahan(l, cl, __fmul_rn(mine[k].l, sc));
      kahan(a, ca, __fmul_rn(fmaf(mine[k].l, dm, mine[k].a), sc));
    }
  }
  l -= cl;
  a -= ca;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    l += __shfl_xor_sync(0xffffffffu, l, o);
    a += __shfl_xor_sync(0xffffffffu, a, o);
  }
  const int w = threadIdx.x >> 5, ln = threadIdx.x & 31;
  if (ln == 0) {
    shd[0][w] = (double)l;
    shd[1][w] = (double)a;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double tl = 0.0, ta = 0.0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
      tl += shd[0][i];
      ta += shd[1][i];
    }
    rs[r] = RowStat{m, (float)tl, (float)(log(tl) - ta / tl), arg};
  }
}

// exp(y - m) as bf16 hi + lo (the A operand of the self-conditioning GEMM) and, when `gumbel`
// is set, the chunk's Gumbel-max winner.
//
// Gumbel-max in its exponential-race form: with E_j = -ln u_j and p_j = exp(y_j - m),
//   argmax_j (y_j - ln(-ln u_j)) = argmin_j E_j / p_j,
// because ln(E_j / p_j) = m - (y_j + g_j) is decreasing in the perturbed logit. p_j is already
// at hand for the split, and the logarithm is only needed for a token that can beat the
// thread's best key so far: -ln u >= 1 - u, so 1 - u > key_best * p_j proves E_j / p_j >
// key_best without it. A whole group of four is skipped when even the smallest possible
// E (2^-24 < -ln(1 - 2^-24)) over its largest p_j cannot beat key_best, or when all four logits
// are more than kGumbelReach below the row maximum. The chunk's winner is written as
// v = -key (larger is better), comparable across the chunks of a row.
__global__ void __launch_bounds__(kThreads, 4) k_convert(const float* __restrict__ Y,
                                                      const RowStat* __restrict__ rs, int64_t V,
                                                      int L, const uint8_t* __restrict__ done,
                                                      const int32_t* __restrict__ step,
                                                      uint64_t seed, const int32_t* blk,
                                                      int gumbel, uint16_t* __restrict__ Phi,
                                                      uint16_t* __restrict__ Plo,
                                                      Best* __restrict__ best, int n_chunks) {
  __shared__ float shv[32], shy;
  __shared__ int32_t shj[32];
  const int c = blockIdx.x, r = blockIdx.y;
  const int b = r / L, i = r % L;
  const uint32_t sid = stream_id((uint32_t)b, blk);
  if (done && done[b]) return;
  const float m = rs[r].m;
  const uint32_t st = gumbel ? (uint32_t)step[b] : 0u;
  const float* y = Y + (size_t)r * V;
  uint16_t* ph = Phi + (size_t)r * V;
  uint16_t* pl = Plo + (size_t)r * V;
  const int64_t j0 = (int64_t)c * kChunk, j1 = min(V, j0 + kChunk);
  const float floor_y = m - kGumbelReach;
  float kbest = INFINITY, by = 0.f;
  int32_t bj = INT_MAX;
  // loads in two batches of four 16-byte loads: the second batch is in flight while the
  // first is processed (four CTAs per SM overlap the rest)
  constexpr int kBatch = kGroups / 2;
  float4 ld[kBatch];
  auto load_batch = [&](int g0) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t j = j0 + 4 * (threadIdx.x + kThreads * (g0 + u));
      ld[u] = j < j1 ? __ldcs(reinterpret_cast<const float4*>(y + j))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  load_batch(0);
#pragma unroll
  for (int g = 0; g < kGroups; ++g) {
    const int64_t j = j0 + 4 * (threadIdx.x + kThreads * g);
    const float4 cur = ld[g % kBatch];
    if (g + 1 == kBatch) load_batch(kBatch);
    if (j >= j1) continue;
    const float yy[4] = {cur.x, cur.y, cur.z, cur.w};
    // p = exp(y - m) = 2^((y - m) log2 e): the argument carries a relative rounding error of
    // ~2^-23 and ex2.approx ~2^-22, so p is within ~3e-6 relative for y - m > -30 (smaller
    // terms do not matter at that precision); p of the row maximum is exactly 1.
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = exp2_approx((yy[e] - m) * 1.4426950408889634f);
    uint2 hi, lo;
    split_bf16x2(p[0], p[1], hi.x, lo.x);
    split_bf16x2(p[2], p[3], hi.y, lo.y);
    *reinterpret_cast<uint2*>(ph + j) = hi;
    *reinterpret_cast<uint2*>(pl + j) = lo;
    if (!gumbel) continue;
    const float pmax = fmaxf(fmaxf(p[0], p[1]), fmaxf(p[2], p[3]));
    const float ymax = fmaxf(fmaxf(yy[0], yy[1]), fmaxf(yy[2], yy[3]));
    if (ymax < floor_y || !(pmax > 0.f) || 5.9604645e-8f >= kbest * pmax) continue;
    const u32x4 w = gumbel_block((uint32_t)(j >> 2), (uint32_t)i, sid, st, seed);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (!(p[e] > 0.f)) continue;
      const uint32_t q = word_of(w, e) >> 9;
      // 1 - u for u = (2q + 1) / 2^24, exact in fp32
      const float one_minus_u = __uint2float_rn(0xFFFFFFu - 2u * q) * 5.9604644775390625e-8f;
      if (one_minus_u * (1.0f - 9.5367431640625e-7f) > kbest * p[e]) continue;
      const float key = -logf(word_to_uniform(word_of(w, e))) / p[e];
      const int32_t jj = (int32_t)(j + e);
      if (key < kbest || (key == kbest && jj < bj)) {
        kbest = key;
        bj = jj;
        by = yy[e];
      }
    }
  }
  if (gumbel) {
    float v = -kbest;
    block_best(v, bj, by, shv, shj, &shy);
    if (threadIdx.x == 0) best[(size_t)r * n_chunks + c] = Best{v, bj, by, 0};
  }
}

// Gumbel-max over stored probabilities as a launch of its own (the fused vocabulary pass, and
// shapes where the self-conditioning launch does not carry the race): (row, 8192-token chunk)
// items, each raced by wpi warps (1, 2, 4 or 8; more when there are few items to fill the GPU)
// over consecutive parts of the chunk's segments (gumbel_race_segments, ds_sample.cuh), sharing
// their best key through shared memory; the item's record is the best of its warps' bests
// (largest -key, then lowest token), with ln p of the winner.
__global__ void __launch_bounds__(kThreads, 2) k_gumbel_items(const __grid_constant__ GumbelWork g,
                                                           int64_t V, int wpi) {
  constexpr int kWarps = kThreads / 32;
  __shared__ unsigned sh_cut[kWarps];
  __shared__ float sh_v[kWarps], sh_y[kWarps];
  __shared__ int32_t sh_j[kWarps];
  pdl_wait();
  const int w = (int)(threadIdx.x >> 5), lane = (int)(threadIdx.x & 31);
  const int slot = w / wpi, part = w % wpi;
  const int64_t item = (int64_t)blockIdx.x * (kWarps / wpi) + slot;
  if (lane == 0 && part == 0) sh_cut[slot] = 0x7F800000u;  // +inf
  __syncthreads();
  bool active = item < (int64_t)g.R * g.n_chunks;
  int r = 0, c = 0;
  if (active) {
    r = (int)(item / g.n_chunks);
    c = (int)(item % g.n_chunks);
    active = !(g.done && g.done[r / g.L]);
  }
  float kbest = INFINITY, bp = 1.f;
  int32_t bj = INT_MAX;
  if (active) {
    const int64_t j0 = (int64_t)c * kChunk, j1 = min(V, j0 + kChunk);
    const int nseg = (int)((j1 - j0) / 128);
    gumbel_race_segments(g, V, r, c, nseg * part / wpi, nseg * (part + 1) / wpi, kbest, bj, bp,
                         wpi > 1 ? &sh_cut[slot] : nullptr);
  }
  float v = -kbest;
  int32_t jw = bj;
  warp_best(v, jw);
  const uint32_t owner = __ballot_sync(0xffffffffu, bj == jw);
  const float pw = __shfl_sync(0xffffffffu, bp, __ffs(owner) - 1);
  if (lane == 0) {
    sh_v[w] = v;
    sh_j[w] = jw;
    sh_y[w] = logf(pw);
  }
  __syncthreads();
  if (active && part == 0 && lane == 0) {
    float bv = sh_v[w], by = sh_y[w];
    int32_t bjj = sh_j[w];
    for (int q = 1; q < wpi; ++q)
      if (better(sh_v[w + q], sh_j[w + q], bv, bjj)) {
        bv = sh_v[w + q];
        bjj = sh_j[w + q];
        by = sh_y[w + q];
      }
    g.best[(size_t)r * g.n_chunks + c] = Best{bv, bjj, bjj == INT_MAX ? 0.f : by, 1};
  }
}

// The k largest logits of a chunk (ties toward lower tokens), written in token order.
// Element q of thread t is token j0 + t + 256 q, so the selection's (q, thread) order is
// token order.
__global__ void __launch_bounds__(kThreads) k_topk_chunk(const float* __restrict__ Y, int64_t V,
                                                         int L, const uint8_t* __restrict__ done,
                                                         int k, Cand* __restrict__ cand,
                                                         int n_chunks) {
  __shared__ int hist[256];
  __shared__ int scan_sh[32];
  const int c = blockIdx.x, r = blockIdx.y;
  if (done && done[r / L]) return;
  const float* y = Y + (size_t)r * V;
  const int64_t j0 = (int64_t)c * kChunk, j1 = min(V, j0 + kChunk);
  uint32_t key[kPer];
  bool valid[kPer];
  float val[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int64_t j = j0 + threadIdx.x + (int64_t)kThreads * q;
    valid[q] = j < j1;
    val[q] = valid[q] ? y[j] : -INFINITY;
    key[q] = float_key(val[q]);
  }
  Cand* out = cand + ((size_t)r * n_chunks + c) * k;
  for (int t = threadIdx.x; t < k; t += kThreads) out[t] = Cand{-INFINITY, INT_MAX};
  __syncthreads();
  block_select_topk<kPer>(key, valid, k, hist, scan_sh, [&](int q, int slot) {
    out[slot] = Cand{val[q], (int32_t)(j0 + threadIdx.x + (int64_t)kThreads * q)};
  });
}

// Top-k of a row from the stored probabilities, one CTA (8 warps) per row. The k largest
// segment maxima are k distinct tokens, so the row's k-th largest logit is at least the k-th
// largest segment maximum theta, and only segments whose maximum reaches theta can hold a top-k
// token (about k of them: every segment when the logits are all equal). The selection is a
// radix select (8-bit digits from the top) over float keys, first of the segment maxima, then
// of p_j = P e^{m_t - m} (the same order as y, up to the ~17 significant bits of hi + lo) over
// the tokens of those segments, re-read from P on each pass; histogram updates are aggregated per
// warp (lanes with the same digit add once). Of the tokens whose key equals the k-th, the lowest
// are taken (a second select over their indices when not all of them fit). The k selected are
// written with y = m + ln p in a fixed order (warp by warp, each warp's segments in list order):
// finalize does not depend on the order of its candidates, only on their set.
namespace {

constexpr int kTkWarps = kThreads / 32;
// Candidate segments listed in shared memory (more, e.g. when every logit is equal, are found by
// scanning the segment maxima on every pass instead).
constexpr int kTkListCap = 2048;

// Warp-aggregated histogram increment of digit `bin` for the lanes with `mine`; called by all
// lanes of the warp together.
DS_DEV void tk_hist_add(int* hist, bool mine, uint32_t bin) {
  const unsigned act = __ballot_sync(0xffffffffu, mine);
  if (mine) {
    const unsigned peers = __match_any_sync(act, bin);
    if ((int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
  }
}

// One radix select over the keys a functor enumerates: each_key(f) calls f(valid, key) for
// every key of this thread, in the same order on every call and with all lanes of a warp
// together. Returns the k-th largest key and, in *need, how many keys equal to it are taken.
template <class EachKey>
DS_DEV uint32_t tk_select(EachKey each_key, int k, int* hist, int* sel, int* need_out) {
  uint32_t prefix = 0, mask = 0;
  int need = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int t = threadIdx.x; t < 256; t += blockDim.x) hist[t] = 0;
    __syncthreads();
    each_key([&](bool valid, uint32_t key) {
      tk_hist_add(hist, valid && (key & mask) == prefix, (key >> shift) & 255u);
    });
    __syncthreads();
    if (threadIdx.x == 0) {
      int cum = 0, bin = 255;
      for (; bin >= 0; --bin) {
        if (cum + hist[bin] >= need) break;
        cum += hist[bin];
      }
      if (bin < 0) bin = 0;  // fewer valid keys than k: all of them are taken
      sel[0] = bin;
      sel[1] = need - cum;
    }
    __syncthreads();
    prefix |= (uint32_t)sel[0] << shift;
    mask |= 255u << shift;
    need = sel[1];
    __syncthreads();
  }
  *need_out = need;
  return prefix;
}

}  // namespace

__global__ void __launch_bounds__(kThreads) k_topk_row(const uint16_t* __restrict__ Phi,
                                                       const uint16_t* __restrict__ Plo,
                                                       const ChunkStat* __restrict__ seg,
                                                       const float* __restrict__ mtile_t,
                                                       const RowStat* __restrict__ rs, int R,
                                                       int64_t V, int L,
                                                       const uint8_t* __restrict__ done, int k,
                                                       Cand* __restrict__ cand,
                                                       int64_t j_offset) {
  __shared__ int hist[256];
  __shared__ int sel[2];
  __shared__ int sh_cnt[2][kTkWarps];
  __shared__ int scan_sh[32];
  __shared__ int sh_list[kTkListCap];
  pdl_wait();
  const int r = blockIdx.x;
  if (done && done[r / L]) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float m = rs[r].m;
  const int nseg = (int)(V / 128);
  const ChunkStat* sg = seg + (size_t)r * nseg;
  const uint16_t* ph = Phi + (size_t)r * V;
  const uint16_t* pl = Plo + (size_t)r * V;
  Cand* out = cand + (size_t)r * k;
  for (int t = threadIdx.x; t < k; t += kThreads) out[t] = Cand{-INFINITY, INT_MAX};

  // theta: the min(k, nseg)-th largest segment maximum
  int dummy = 0;
  const int n_it = (nseg + kThreads - 1) / kThreads;
  const uint32_t theta = tk_select(
      [&](auto f) {
        for (int it = 0; it < n_it; ++it) {
          const int g = threadIdx.x + kThreads * it;
          f(g < nseg, g < nseg ? float_key(sg[g].m) : 0u);
        }
      },
      min(k, nseg), hist, sel, &dummy);

  // the segments whose maximum reaches theta, listed once (thread t's segments t, t + 256, ...
  // in turn, threads in order)
  int n_cand = 0;
  {
    int mine = 0;
    for (int it = 0; it < n_it; ++it) {
      const int g = threadIdx.x + kThreads * it;
      mine += (g < nseg && float_key(sg[g].m) >= theta) ? 1 : 0;
    }
    const int base = block_exclusive_scan(mine, scan_sh, &n_cand);
    if (n_cand <= kTkListCap) {
      int o = base;
      for (int it = 0; it < n_it; ++it) {
        const int g = threadIdx.x + kThreads * it;
        if (g < nseg && float_key(sg[g].m) >= theta) sh_list[o++] = g;
      }
    }
    __syncthreads();
  }
  const bool listed = n_cand <= kTkListCap;
  // the tokens of those segments, warp w taking the w-th, (w + 8)-th, ... of them; lane l takes
  // tokens 4 l .. 4 l + 3 of a segment
  auto each_token = [&](auto f) {
    const int n_walk = listed ? n_cand : nseg;
    for (int e = warp; e < n_walk; e += kTkWarps) {
      const int g = listed ? sh_list[e] : e;
      if (!listed && float_key(sg[g].m) < theta) continue;  // the whole warp skips it
      const float scale = expf(mtile_t[(size_t)(g >> 1) * R + r] - m);
      const int64_t j = (int64_t)g * 128 + 4 * lane;
      const uint2 h = *reinterpret_cast<const uint2*>(ph + j);
      const uint2 lo = *reinterpret_cast<const uint2*>(pl + j);
      const uint32_t hw[2] = {h.x, h.y}, lw[2] = {lo.x, lo.y};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t hb = (e & 1) ? (hw[e >> 1] & 0xFFFF0000u) : (hw[e >> 1] << 16);
        const uint32_t lb = (e & 1) ? (lw[e >> 1] & 0xFFFF0000u) : (lw[e >> 1] << 16);
        const float p = (__uint_as_float(hb) + __uint_as_float(lb)) * scale;
        f(j + e, p, float_key(p));
      }
    }
  };
  int need = 0;
  const uint32_t kth = tk_select(
      [&](auto f) { each_token([&](int64_t, float, uint32_t key) { f(true, key); }); }, k, hist,
      sel, &need);

  // per warp: keys above the k-th, and keys equal to it
  int gt = 0, eq = 0;
  each_token([&](int64_t, float, uint32_t key) {
    gt += __popc(__ballot_sync(0xffffffffu, key > kth));
    eq += __popc(__ballot_sync(0xffffffffu, key == kth));
  });
  if (lane == 0) {
    sh_cnt[0][warp] = gt;
    sh_cnt[1][warp] = eq;
  }
  __syncthreads();
  int eq_total = 0;
  for (int w = 0; w < kTkWarps; ++w) eq_total += sh_cnt[1][w];
  // Keys equal to the k-th are taken lowest tokens first: when only `need` of them fit, a second
  // select over their token indices (key ~j, larger for lower tokens) finds the need-th lowest.
  uint32_t jcut = 0;  // tie tokens with ~j >= jcut are taken
  if (need < eq_total) {
    int dummy2 = 0;
    jcut = tk_select(
        [&](auto f) {
          each_token([&](int64_t j, float, uint32_t key) { f(key == kth, ~(uint32_t)j); });
        },
        need, hist, sel, &dummy2);
  }
  auto take_tie = [&](int64_t j, uint32_t key) {
    return key == kth && (need >= eq_total || ~(uint32_t)j >= jcut);
  };
  int eq_take = 0;
  if (need < eq_total) {
    each_token([&](int64_t j, float, uint32_t key) {
      eq_take += __popc(__ballot_sync(0xffffffffu, take_tie(j, key)));
    });
  } else {
    eq_take = eq;
  }
  __syncthreads();  // every warp has read the tie counts before they are replaced
  if (lane == 0) sh_cnt[1][warp] = eq_take;
  __syncthreads();
  int take_before = 0;
  for (int w = 0; w < warp; ++w) take_before += sh_cnt[0][w] + sh_cnt[1][w];
  int taken = 0;
  const unsigned below = (1u << lane) - 1u;
  each_token([&](int64_t j, float p, uint32_t key) {
    const bool take = key > kth || take_tie(j, key);
    const unsigned tk_b = __ballot_sync(0xffffffffu, take);
    if (take) {
      const int slot = take_before + taken + __popc(tk_b & below);
      if (slot < k) out[slot] = Cand{p > 0.f ? m + logf(p) : -INFINITY, (int32_t)(j + j_offset)};
    }
    taken += __popc(tk_b);
  });
}

// Per row: the sampled token, its confidence, the entropy and the argmax.
// With Opart set, it also writes s for the row: the sum of the vocabulary-split partials in
// split order, divided by the softmax normaliser.
// POOL: the top-k selection over a pool of several chunks' candidates (the CUDA-core and
// no-allocation top-k paths), whose per-thread arrays set the kernel's register count; without
// it the kernel needs far fewer registers and more CTAs fit on an SM. NB: split partials a
// thread requests at once — 16 where the rows fit in one wave anyway (the 13 splits of a canvas
// in one round trip: latency decides), 8 where they take several (fewer registers, more CTAs:
// occupancy decides). Same sums in the same order either way. Same box, finalize per step:
// B = 1 0.0148–0.0156 against 0.0141–0.0145 ms with one kernel for every path (two CTAs an SM),
// B = 2 0.020 against 0.041, B = 4 0.021 against 0.047, B = 8 0.039 against 0.096–0.099.
template <bool POOL, int NB>
__global__ void __launch_bounds__(kThreads) k_finalize(
    const RowStat* __restrict__ rs, const Best* __restrict__ best, const Cand* __restrict__ cand,
    int n_chunks, int k, int L, const uint8_t* __restrict__ done, const int32_t* __restrict__ step,
    uint64_t seed, const int32_t* blk, int32_t* __restrict__ sampled, float* __restrict__ conf,
    float* __restrict__ entropy, int32_t* __restrict__ argmax, const float* __restrict__ Opart,
    int S, int R, int d, float* __restrict__ s_out, const float* __restrict__ mref) {
  __shared__ float shv[32], shy, shf[32];
  __shared__ float sh_sc[kMaxSplits];
  __shared__ int32_t shj[32];
  __shared__ int hist[256];
  __shared__ int scan_sh[32];
  __shared__ float sel_y[kMaxTopK];
  __shared__ int32_t sel_j[kMaxTopK];
  pdl_wait();
  const int r = blockIdx.x;
  const int b = r / L, i = r % L;
  if (done && done[b]) return;
  const RowStat st = rs[r];
  if (Opart) {
    // partial sp is relative to exp(mref[sp] - m) (1 for the unfused splits); summed in split
    // order
    for (int sp = threadIdx.x; sp < S; sp += kThreads)
      sh_sc[sp] = mref ? expf(mref[(size_t)sp * R + r] - st.m) : 1.f;
    __syncthreads();
    const int64_t plane = (int64_t)R * d;
    const float4* src = reinterpret_cast<const float4*>(Opart + (size_t)r * d);
    float4* dst = reinterpret_cast<float4*>(s_out + (size_t)r * d);
    for (int q = threadIdx.x; q < d / 4; q += kThreads) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      // the split partials are loaded NB at a time before they are summed (in split order), so
      // that a thread's loads are in flight together
      int sp = 0;
      for (; sp + NB <= S; sp += NB) {
        float4 t[NB];
#pragma unroll
        for (int u = 0; u < NB; ++u) t[u] = src[(sp + u) * plane / 4 + q];
#pragma unroll
        for (int u = 0; u < NB; ++u) {
          const float c = sh_sc[sp + u];
          acc.x = fmaf(t[u].x, c, acc.x);
          acc.y = fmaf(t[u].y, c, acc.y);
          acc.z = fmaf(t[u].z, c, acc.z);
          acc.w = fmaf(t[u].w, c, acc.w);
        }
      }
      float4 t[NB];
#pragma unroll
      for (int u = 0; u < NB; ++u)
        if (sp + u < S) t[u] = src[(sp + u) * plane / 4 + q];
#pragma unroll
      for (int u = 0; u < NB; ++u)
        if (sp + u < S) {
          const float c = sh_sc[sp + u];
          acc.x = fmaf(t[u].x, c, acc.x);
          acc.y = fmaf(t[u].y, c, acc.y);
          acc.z = fmaf(t[u].z, c, acc.z);
          acc.w = fmaf(t[u].w, c, acc.w);
        }
      dst[q] = make_float4(acc.x / st.l, acc.y / st.l, acc.z / st.l, acc.w / st.l);
    }
  }
  float bv = -INFINITY, by = 0.f;
  int32_t bj = INT_MAX;
  float cval = 0.f;
  if (k == 0) {
    // Best::y is y at the winner, or y - m where Best::rel is 1
    for (int q = threadIdx.x; q < n_chunks; q += kThreads) {
      const Best t = best[(size_t)r * n_chunks + q];
      if (better(t.v, t.j, bv, bj)) {
        bv = t.v;
        bj = t.j;
        by = t.rel ? t.y : t.y - st.m;
      }
    }
    block_best(bv, bj, by, shv, shj, &shy);
    cval = expf(by) / st.l;
  } else if (n_chunks == 1) {
    // the pool is the row's k candidates already (one per slot, unused slots with token
    // INT_MAX): Gumbel-max over them and the truncated normaliser, no selection
    float e_sum = 0.f;
    for (int t = threadIdx.x; t < k; t += kThreads) {
      const Cand c = cand[(size_t)r * k + t];
      if (c.j == INT_MAX) continue;
      const u32x4 w = gumbel_block((uint32_t)(c.j >> 2), (uint32_t)i, stream_id((uint32_t)b, blk),
                                   (uint32_t)step[b], seed);
      const float v = c.y + gumbel_from_word(word_of(w, c.j & 3));
      if (better(v, c.j, bv, bj)) {
        bv = v;
        bj = c.j;
        by = c.y;
      }
      e_sum += expf(c.y - st.m);
    }
    e_sum = block_sum(e_sum, shf);
    block_best(bv, bj, by, shv, shj, &shy);
    cval = expf(by - st.m) / e_sum;
  } else if constexpr (POOL) {
    // The pool holds each chunk's candidates in token order, chunks in order, so pool order
    // is token order; element q of thread t is pool entry t + 256 q.
    constexpr int NP = kMaxTopKPool / kThreads;
    const int pool = n_chunks * k;
    uint32_t key[NP];
    bool valid[NP];
    float val[NP];
    int32_t tok[NP];
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      const int idx = threadIdx.x + kThreads * q;
      const Cand t = idx < pool ? cand[(size_t)r * pool + idx] : Cand{-INFINITY, INT_MAX};
      valid[q] = t.j != INT_MAX;
      val[q] = t.y;
      tok[q] = t.j;
      key[q] = float_key(t.y);
    }
    for (int t = threadIdx.x; t < kMaxTopK; t += kThreads) sel_j[t] = INT_MAX;
    __syncthreads();
    block_select_topk<NP>(key, valid, k, hist, scan_sh, [&](int q, int slot) {
      sel_y[slot] = val[q];
      sel_j[slot] = tok[q];
    });
    __syncthreads();
    // Gumbel-max over the selected set and the truncated normaliser (fixed-order sum).
    float e_sum = 0.f;
    for (int t = threadIdx.x; t < k; t += kThreads) {
      const int32_t j = sel_j[t];
      if (j == INT_MAX) continue;
      const float yy = sel_y[t];
      const u32x4 w = gumbel_block((uint32_t)(j >> 2), (uint32_t)i, stream_id((uint32_t)b, blk),
                                   (uint32_t)step[b], seed);
      const float v = yy + gumbel_from_word(word_of(w, j & 3));
      if (better(v, j, bv, bj)) {
        bv = v;
        bj = j;
        by = yy;
      }
      e_sum += expf(yy - st.m);
    }
    e_sum = block_sum(e_sum, shf);
    block_best(bv, bj, by, shv, shj, &shy);
    cval = expf(by - st.m) / e_sum;
  }
  if (threadIdx.x == 0) {
    sampled[r] = bj;
    conf[r] = cval;
    entropy[r] = st.ent;
    argmax[r] = st.arg;
  }
}

__global__ void k_reduce_s(const float* __restrict__ Opart, int S, int R, int d, int L,
                           const uint8_t* __restrict__ done, const RowStat* __restrict__ rs,
                           float* __restrict__ s) {
  const int64_t n4 = (int64_t)R * d / 4;
  const int64_t plane = (int64_t)R * d;
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < n4;
       q += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)((q * 4) / d);
    if (done && done[r / L]) continue;
    float4 acc = *reinterpret_cast<const float4*>(Opart + q * 4);
    for (int sp = 1; sp < S; ++sp) {
      const float4 t = *reinterpret_cast<const float4*>(Opart + sp * plane + q * 4);
      acc.x += t.x;
      acc.y += t.y;
      acc.z += t.z;
      acc.w += t.w;
    }
    const float l = rs[r].l;
    acc.x /= l;
    acc.y /= l;
    acc.z /= l;
    acc.w /= l;
    *reinterpret_cast<float4*>(s + q * 4) = acc;
  }
}

// Lock / re-noise / stop for one sequence per CTA (blockDim = L).
__global__ void k_lock(int L, uint32_t V, int max_steps, uint64_t seed, const int32_t* blk,
                       const float* __restrict__ tau, const int32_t* __restrict__ sampled,
                       const float* __restrict__ conf, int32_t* __restrict__ step,
                       int32_t* __restrict__ canvas, uint8_t* __restrict__ lock,
                       uint8_t* __restrict__ done) {
  __shared__ float shv[32];
  __shared__ int32_t shj[32];
  pdl_wait();
  const int b = blockIdx.x, i = threadIdx.x;
  if (done[b]) return;
  const int st = step[b];
  const bool final_step = st + 1 >= max_steps;
  const size_t at = (size_t)b * L + i;
  const bool locked = lock[at] != 0;
  const float c = conf[at];
  const bool pass = !locked && (final_step || c >= tau[b]);
  const int any_pass = __syncthreads_or(pass);
  const int any_open = __syncthreads_or(!locked);
  bool forced = false;
  if (!any_pass && any_open) {
    float v = locked ? -INFINITY : c;
    int32_t j = locked ? INT_MAX : i;
    warp_best(v, j);
    const int w = i >> 5, ln = i & 31;
    if (ln == 0) {
      shv[w] = v;
      shj[w] = j;
    }
    __syncthreads();
    if (w == 0) {
      v = ln < (int)(blockDim.x >> 5) ? shv[ln] : -INFINITY;
      j = ln < (int)(blockDim.x >> 5) ? shj[ln] : INT_MAX;
      warp_best(v, j);
      if (ln == 0) shj[0] = j;
    }
    __syncthreads();
    forced = (i == shj[0]);
  }
  const bool newly = pass || forced;
  if (newly) {
    canvas[at] = sampled[at];
    lock[at] = 1;
  } else if (!locked) {
    const u32x4 w = philox4x32_10(u32x4{(uint32_t)(i >> 2), 0u, stream_id((uint32_t)b, blk),
                                        ((uint32_t)st << 2) | kRenoiseStream},
                                  (uint32_t)seed, (uint32_t)(seed >> 32));
    canvas[at] = token_from_word(word_of(w, i & 3), V);
  }
  const int all_locked = __syncthreads_and(locked || newly);
  if (i == 0) {
    step[b] = st + 1;
    done[b] = all_locked ? 1 : 0;
  }
}

__global__ void k_philox(const uint32_t* __restrict__ ctr, uint64_t seed, uint32_t* __restrict__ out,
                         int64_t n) {
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < n;
       q += (int64_t)gridDim.x * blockDim.x) {
    const uint4 c = reinterpret_cast<const uint4*>(ctr)[q];
    const u32x4 v = philox4x32_10(u32x4{c.x, c.y, c.z, c.w}, (uint32_t)seed, (uint32_t)(seed >> 32));
    reinterpret_cast<uint4*>(out)[q] = make_uint4(v.x, v.y, v.z, v.w);
  }
}

__global__ void k_loop_begin(const uint8_t* __restrict__ done, int B, int32_t* iter, int max_iters,
                             cudaGraphConditionalHandle h) {
  int open = 0;
  for (int b = threadIdx.x; b < B; b += 32) open |= (done[b] == 0);
  open = __any_sync(0xffffffffu, open);
  if (threadIdx.x == 0) {
    *iter = 0;
    cudaGraphSetConditional(h, (open && max_iters > 0) ? 1u : 0u);
  }
}

__global__ void k_loop_end(const uint8_t* __restrict__ done, int B, int32_t* iter, int max_iters,
                           cudaGraphConditionalHandle h) {
  int open = 0;
  for (int b = threadIdx.x; b < B; b += 32) open |= (done[b] == 0);
  open = __any_sync(0xffffffffu, open);
  if (threadIdx.x == 0) {
    const int it = *iter + 1;
    *iter = it;
    cudaGraphSetConditional(h, (open && it < max_iters) ? 1u : 0u);
  }
}

// Per-sequence temperature of the linear schedule at each sequence's step.
__global__ void k_temperature(const int32_t* __restrict__ step, int B, float t_start, float t_end,
                              int max_steps, float* __restrict__ T) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  T[b] = max_steps > 1
             ? t_start + (t_end - t_start) * ((float)step[b] / (float)(max_steps - 1))
             : t_start;
}

// The pages' default sampler for one sequence per CTA (blockDim = L): accept positions from the
// lowest to the highest entropy (ties in position order) until the budget is spent, at least
// one; re-noise the others; stop on a confident (mean entropy < stop_entropy) and stable (argmax
// unchanged) canvas, or at the last step, with the canvas set to the argmax. Entropies below zero
// (rounding) count as zero. Sort: bitonic over the next power of two; the running sum is a
// Hillis-Steele scan in a fixed order, so the result is deterministic.
__global__ void __launch_bounds__(1024) k_lock_entropy(
    int L, uint32_t V, int max_steps, uint64_t seed, const int32_t* blk, float budget,
    float stop_entropy,
    const int32_t* __restrict__ sampled, const float* __restrict__ entropy,
    const int32_t* __restrict__ argmax, int32_t* __restrict__ prev_argmax,
    int32_t* __restrict__ step, int32_t* __restrict__ canvas, uint8_t* __restrict__ lock,
    uint8_t* __restrict__ done) {
  __shared__ float key[1024];
  __shared__ int32_t idx[1024];
  __shared__ int32_t rank_of[1024];
  __shared__ float shf[32];
  const int b = blockIdx.x, i = threadIdx.x;
  if (done[b]) return;
  const size_t at = (size_t)b * L + i;
  const int st = step[b];
  const float h = fmaxf(entropy[at], 0.f);
  const int32_t am = argmax[at];
  const int same = __syncthreads_and(am == prev_argmax[at]);
  const float mean = block_sum(h, shf) / (float)L;
  const bool stop = st > 0 && same && mean < stop_entropy;
  if (stop || st + 1 >= max_steps) {
    canvas[at] = am;
    lock[at] = 1;
    prev_argmax[at] = am;
    if (i == 0) {
      step[b] = st + 1;
      done[b] = 1;
    }
    return;
  }
  int P = 1;
  while (P < L) P <<= 1;
  for (int t = i; t < P; t += blockDim.x) {  // t < L only for t == i
    key[t] = t < L ? h : INFINITY;
    idx[t] = t;
  }
  __syncthreads();
  for (int kk = 2; kk <= P; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int t = i; t < P / 2; t += blockDim.x) {
        const int i1 = 2 * j * (t / j) + (t % j), i2 = i1 + j;
        const bool up = (i1 & kk) == 0;
        const bool gt = key[i1] > key[i2] || (key[i1] == key[i2] && idx[i1] > idx[i2]);
        if (gt == up) {
          const float tk = key[i1];
          key[i1] = key[i2];
          key[i2] = tk;
          const int32_t ti = idx[i1];
          idx[i1] = idx[i2];
          idx[i2] = ti;
        }
      }
      __syncthreads();
    }
  }
  // inclusive running sum of the sorted entropies, thread r holding rank r
  float v = key[i];
  rank_of[idx[i]] = i;
  __syncthreads();
  for (int off = 1; off < L; off <<= 1) {
    const float t = i >= off ? key[i - off] : 0.f;
    __syncthreads();
    v += t;
    key[i] = v;
    __syncthreads();
  }
  const int n_acc = max(1, __syncthreads_count(v <= budget));
  const bool accepted = rank_of[i] < n_acc;
  if (accepted) {
    canvas[at] = sampled[at];
  } else {
    const u32x4 w = philox4x32_10(u32x4{(uint32_t)(i >> 2), 0u, stream_id((uint32_t)b, blk),
                                        ((uint32_t)st << 2) | kRenoiseStream},
                                  (uint32_t)seed, (uint32_t)(seed >> 32));
    canvas[at] = token_from_word(word_of(w, i & 3), V);
  }
  lock[at] = accepted ? 1 : 0;
  prev_argmax[at] = am;
  if (i == 0) step[b] = st + 1;
}

// A wait that nothing will satisfy: one mbarrier expecting one arrival that never comes.
__global__ void k_wait_selftest(uint64_t limit_ns, uint32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(b, 0)) {
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(err, kErrTimeout);
      return;
    }
  }
}

}  // namespace

// ---- block-autoregressive driver (see launch_block_start / check / rollover) ----

// Block first_block from init_canvas[0] with fresh state: no locks, step 0, not done, no
// previous argmax, s = 0 (the stand-in's s_prev of the first step).
__global__ void k_block_start(int32_t* ctl, int first_block, const int32_t* __restrict__ init0,
                              BlockState bs, int B, int L, int d) {
  const int64_t BL = (int64_t)B * L, n = BL * d;
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < n;
       q += (int64_t)gridDim.x * blockDim.x) {
    if (q < BL) {
      bs.canvas[q] = init0[q];
      bs.lock[q] = 0;
      if (bs.prev_argmax) bs.prev_argmax[q] = -1;
    }
    if (q < B) {
      bs.step[q] = 0;
      bs.done[q] = 0;
    }
    bs.s[q] = 0.f;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    ctl[0] = first_block;
    ctl[1] = 0;
    ctl[2] = 0;
    ctl[3] = 0;
  }
}

// After every step of the run (one warp): when no sequence of the current block is open, the
// block is to be committed (ctl[2] = its local index) and, if blocks remain, the block index
// advances so that the next step already draws for the next block; ctl[1] records the action.
__global__ void k_block_check(int32_t* ctl, const uint8_t* __restrict__ done, int B,
                              int first_block, int n_blocks, int max_iters, int use_cond,
                              cudaGraphConditionalHandle h) {
  int open = 0;
  for (int b = threadIdx.x; b < B; b += 32) open |= (done[b] == 0);
  open = __any_sync(0xffffffffu, open);
  if (threadIdx.x == 0) {
    const int blk = ctl[0];
    int action = 0;
    if (!open) {
      action = blk + 1 < first_block + n_blocks ? 1 : 2;
      ctl[2] = blk - first_block;
      if (action == 1) ctl[0] = blk + 1;
    }
    ctl[1] = action;
    const int it = ctl[3] + 1;
    ctl[3] = it;
    if (use_cond) cudaGraphSetConditional(h, (action != 2 && it < max_iters) ? 1u : 0u);
  }
}

// Commit the finished block (tokens and step counts) and, for action 1, load the next block's
// initial canvas with fresh state. Each element is read and written by one thread only.
__global__ void k_block_rollover(const int32_t* __restrict__ ctl,
                                 const int32_t* __restrict__ init_canvas,
                                 int32_t* __restrict__ out_canvas, int32_t* __restrict__ out_steps,
                                 BlockState bs, int B, int L, int d) {
  const int action = ctl[1];
  if (action == 0) return;
  const int64_t k = ctl[2];
  const int64_t BL = (int64_t)B * L, n = action == 1 ? BL * d : BL;
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < n;
       q += (int64_t)gridDim.x * blockDim.x) {
    if (q < BL) {
      out_canvas[k * BL + q] = bs.canvas[q];
      if (action == 1) {
        bs.canvas[q] = init_canvas[(k + 1) * BL + q];
        bs.lock[q] = 0;
        if (bs.prev_argmax) bs.prev_argmax[q] = -1;
      }
    }
    if (q < B) {
      out_steps[k * B + q] = bs.step[q];
      if (action == 1) {
        bs.step[q] = 0;
        bs.done[q] = 0;
      }
    }
    if (action == 1) bs.s[q] = 0.f;
  }
}

void launch_block_start(int32_t* ctl, int first_block, const int32_t* init_canvas, BlockState bs,
                        int B, int L, int d, cudaStream_t st) {
  k_block_start<<<2 * 152, 256, 0, st>>>(ctl, first_block, init_canvas, bs, B, L, d);
}

void launch_block_check(int32_t* ctl, const uint8_t* done, int B, int first_block, int n_blocks,
                        int max_iters, bool use_cond, cudaGraphConditionalHandle h,
                        cudaStream_t st) {
  k_block_check<<<1, 32, 0, st>>>(ctl, done, B, first_block, n_blocks, max_iters,
                                  use_cond ? 1 : 0, h);
}

void launch_block_rollover(const int32_t* ctl, const int32_t* init_canvas, int32_t* out_canvas,
                           int32_t* out_steps, BlockState bs, int B, int L, int d,
                           cudaStream_t st) {
  k_block_rollover<<<2 * 152, 256, 0, st>>>(ctl, init_canvas, out_canvas, out_steps, bs, B, L, d);
}

void launch_temperature(const int32_t* step, int B, float t_start, float t_end, int max_steps,
                        float* T, cudaStream_t st) {
  k_temperature<<<(B + 127) / 128, 128, 0, st>>>(step, B, t_start, t_end, max_steps, T);
}

void launch_lock_entropy(int B, int L, int64_t V, int max_steps, uint64_t seed,
                         const int32_t* blk, float budget, float stop_entropy,
                         const int32_t* sampled, const float* entropy, const int32_t* argmax,
                         int32_t* prev_argmax, int32_t* step, int32_t* canvas, uint8_t* lock,
                         uint8_t* done, cudaStream_t st) {
  k_lock_entropy<<<B, L, 0, st>>>(L, (uint32_t)V, max_steps, seed, blk, budget, stop_entropy,
                                  sampled, entropy, argmax, prev_argmax, step, canvas, lock, done);
}

void launch_wait_selftest(uint64_t limit_ns, uint32_t* err, cudaStream_t st) {
  k_wait_selftest<<<1, 32, 0, st>>>(limit_ns, err);
}

void launch_chunk_stats(const float* Y, int R, int64_t V, int L, const uint8_t* done,
                        ChunkStat* cs, cudaStream_t st) {
  const int nc = n_chunks_of(V);
  k_chunk_stats<<<dim3(nc, R), kThreads, 0, st>>>(Y, V, L, done, cs, nc);
}

void launch_row_merge(const ChunkStat* cs, int n_chunks, int R, int L, const uint8_t* done,
                      RowStat* rs, cudaStream_t st) {
  launch_k(k_row_merge, dim3(R), dim3(kThreads), 0, st, cs, n_chunks, L, done, rs);
}

void launch_convert(const float* Y, const RowStat* rs, int R, int64_t V, int L,
                    const uint8_t* done, const int32_t* step, uint64_t seed, const int32_t* blk,
                    bool gumbel, uint16_t* Phi, uint16_t* Plo, Best* best, cudaStream_t st) {
  const int nc = n_chunks_of(V);
  k_convert<<<dim3(nc, R), kThreads, 0, st>>>(Y, rs, V, L, done, step, seed, blk, gumbel ? 1 : 0,
                                              Phi, Plo, best, nc);

}

void launch_topk_chunk(const float* Y, int R, int64_t V, int L, const uint8_t* done, int k,
                       Cand* cand, cudaStream_t st) {
  const int nc = n_chunks_of(V);
  k_topk_chunk<<<dim3(nc, R), kThreads, 0, st>>>(Y, V, L, done, k, cand, nc);
}

void launch_topk_row(const uint16_t* Phi, const uint16_t* Plo, const ChunkStat* seg,
                     const float* mtile_t, const RowStat* rs, int R, int64_t V, int L,
                     const uint8_t* done, int k, Cand* cand, cudaStream_t st,
                     int64_t j_offset) {
  launch_k(k_topk_row, dim3(R), dim3(kThreads), 0, st, Phi, Plo, seg, mtile_t, rs, R, V, L, done,
           k, cand, j_offset);
}

void launch_finalize(const RowStat* rs, const Best* best, const Cand* cand, int n_chunks, int k,
                     int R, int L, const uint8_t* done, const int32_t* step, uint64_t seed,
                     const int32_t* blk, int32_t* sampled, float* conf, float* entropy,
                     int32_t* argmax, cudaStream_t st) {
  launch_finalize_with_s(rs, best, cand, n_chunks, k, R, L, done, step, seed, blk, sampled, conf,
                         entropy, argmax, nullptr, 0, 0, nullptr, nullptr, st);
}

void launch_finalize_with_s(const RowStat* rs, const Best* best, const Cand* cand, int n_chunks,
                            int k, int R, int L, const uint8_t* done, const int32_t* step,
                            uint64_t seed, const int32_t* blk, int32_t* sampled, float* conf,
                            float* entropy, int32_t* argmax, const float* Opart, int S, int d,
                            float* s, const float* mref, cudaStream_t st) {
  // rows in one wave at two CTAs an SM: the per-row latency decides, so all of a canvas's split
  // partials are requested at once; more rows: occupancy decides (same sums in the same order)
  const bool one_wave = R <= 2 * std::max(1, tc_num_sms());
  if (k > 0 && n_chunks > 1)
    launch_k(k_finalize<true, 8>, dim3(R), dim3(kThreads), 0, st, rs, best, cand, n_chunks, k, L,
             done, step, seed, blk, sampled, conf, entropy, argmax, Opart, S, R, d, s, mref);
  else if (one_wave)
    launch_k(k_finalize<false, 16>, dim3(R), dim3(kThreads), 0, st, rs, best, cand, n_chunks, k,
             L, done, step, seed, blk, sampled, conf, entropy, argmax, Opart, S, R, d, s, mref);
  else
    launch_k(k_finalize<false, 8>, dim3(R), dim3(kThreads), 0, st, rs, best, cand, n_chunks, k, L,
             done, step, seed, blk, sampled, conf, entropy, argmax, Opart, S, R, d, s, mref);
}

void launch_gumbel_items(const uint16_t* Phi, const uint16_t* Plo, const ChunkStat* seg,
                       const RowStat* rs, int R, int64_t V, int L, const uint8_t* done,
                       const int32_t* step, uint64_t seed, const int32_t* blk, bool tile_ref,
                       Best* best, cudaStream_t st, int64_t j_offset) {
  const int nc = n_chunks_of(V);
  const GumbelWork g{Phi, Plo, seg,     rs, done,    step, blk, seed, best, nullptr, R, L, nc,
                     tile_ref ? 1 : 0, nullptr, nullptr, nullptr, j_offset};
  // warps per item: doubled while the items' warps would not fill the warps every SM holds
  // (two CTAs of 8). Race time measured against the rule at 1024 / 2048 / 4096 items:
  // 0.024 / 0.031 / 0.118 ms (4, 2, 1 warps), 0.025 / 0.039 / 0.118 with half as many warps,
  // 0.028 / 0.035 / 0.118 with twice as many.
  const int64_t items = (int64_t)R * nc;
  const int64_t resident = (int64_t)std::max(1, tc_num_sms()) * 16;
  int wpi = 1;
  while (wpi < kThreads / 32 && items * wpi < resident) wpi *= 2;
  const int per_cta = kThreads / 32 / wpi;
  launch_k(k_gumbel_items, dim3((unsigned)((items + per_cta - 1) / per_cta)), dim3(kThreads), 0, st,
           g, V, wpi);
}

void launch_reduce_s(const float* Opart, int S, int R, int d, int L, const uint8_t* done,
                     const RowStat* rs, float* s, cudaStream_t st) {
  const int64_t n4 = (int64_t)R * d / 4;
  const int blocks = (int)std::min<int64_t>((n4 + 255) / 256, 4096);
  k_reduce_s<<<blocks, 256, 0, st>>>(Opart, S, R, d, L, done, rs, s);
}

void launch_lock(int B, int L, int64_t V, int max_steps, uint64_t seed, const int32_t* blk,
                 const float* tau, const int32_t* sampled, const float* conf, int32_t* step,
                 int32_t* canvas, uint8_t* lock, uint8_t* done, cudaStream_t st) {
  launch_k(k_lock, dim3(B), dim3(L), 0, st, L, (uint32_t)V, max_steps, seed, blk, tau, sampled,
           conf, step, canvas, lock, done);
}

void launch_philox(const uint32_t* ctr, uint64_t seed, uint32_t* out, int64_t n, cudaStream_t st) {
  const int blocks = (int)std::min<int64_t>((n + 255) / 256, 4096);
  if (n > 0) k_philox<<<blocks, 256, 0, st>>>(ctr, seed, out, n);
}

void launch_loop_begin(const uint8_t* done, int B, int32_t* iter, int max_iters,
                       cudaGraphConditionalHandle h, cudaStream_t st) {
  k_loop_begin<<<1, 32, 0, st>>>(done, B, iter, max_iters, h);
}

void launch_loop_end(const uint8_t* done, int B, int32_t* iter, int max_iters,
                     cudaGraphConditionalHandle h, cudaStream_t st) {
  k_loop_end<<<1, 32, 0, st>>>(done, B, iter, max_iters, h);
}

// ------------------------------------------------------------------------------------------
// vocabulary shards: one step's partial record over a token range, and the merge of the records
// of every range (DiffusionGemma Technical Report, section 6 "Multi-user throughput": scaling
// the sampler; the softmax, its entropy and s decompose over any partition of the vocabulary)
// ------------------------------------------------------------------------------------------

// Per row of a shard's step: the row statistics with the global argmax token, the shard's race
// winner (best of its chunk records: score -key and ln p relative to the shard's maximum m_r),
// the un-normalised self-conditioning sum O_r = sum_split exp(mref - m_r) O_split (split order)
// and, with top-k, the row's k candidates.
__global__ void __launch_bounds__(kThreads) k_shard_export(
    const RowStat* __restrict__ rs, const Best* __restrict__ best, int n_chunks,
    const Cand* __restrict__ cand, int k, int L, const uint8_t* __restrict__ done,
    const float* __restrict__ Opart, int S, int R, int d, const float* __restrict__ mref,
    int64_t j_offset, RowStat* __restrict__ rows_out, Best* __restrict__ best_out,
    float* __restrict__ O_out, Cand* __restrict__ cand_out) {
  __shared__ float shv[32], shy;
  __shared__ int32_t shj[32];
  __shared__ float sh_sc[kMaxSplits];
  pdl_wait();
  const int r = blockIdx.x;
  if (done && done[r / L]) return;
  const RowStat st = rs[r];
  for (int sp = threadIdx.x; sp < S; sp += kThreads)
    sh_sc[sp] = mref ? expf(mref[(size_t)sp * R + r] - st.m) : 1.f;
  __syncthreads();
  const int64_t plane = (int64_t)R * d;
  const float4* src = reinterpret_cast<const float4*>(Opart + (size_t)r * d);
  float4* dst = reinterpret_cast<float4*>(O_out + (size_t)r * d);
  for (int q = threadIdx.x; q < d / 4; q += kThreads) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp = 0; sp < S; ++sp) {
      const float4 t = src[sp * plane / 4 + q];
      const float c = sh_sc[sp];
      acc.x = fmaf(t.x, c, acc.x);
      acc.y = fmaf(t.y, c, acc.y);
      acc.z = fmaf(t.z, c, acc.z);
      acc.w = fmaf(t.w, c, acc.w);
    }
    dst[q] = acc;
  }
  if (k == 0) {
    float bv = -INFINITY, by = 0.f;
    int32_t bj = INT_MAX;
    for (int q = threadIdx.x; q < n_chunks; q += kThreads) {
      const Best t = best[(size_t)r * n_chunks + q];
      if (better(t.v, t.j, bv, bj)) {
        bv = t.v;
        bj = t.j;
        by = t.y;
      }
    }
    block_best(bv, bj, by, shv, shj, &shy);
    if (threadIdx.x == 0) best_out[r] = Best{bv, bj, bj == INT_MAX ? 0.f : by, 1};
  } else {
    for (int t = threadIdx.x; t < k; t += kThreads) cand_out[(size_t)r * k + t] = cand[(size_t)r * k + t];
  }
  if (threadIdx.x == 0)
    rows_out[r] = RowStat{st.m, st.l, st.ent, (int32_t)(st.arg + j_offset)};
}

// Per row, the records of n shards (shard-major arrays, shards in increasing token order):
// m = max m_q; l = sum_q l_q e^{m_q - m}; entropy by the mixture identity H = sum_q w_q H_q -
// sum_q w_q ln w_q with w_q = l_q e^{m_q - m} / l (fp64); argmax the largest m_q, lowest token
// on ties; s = sum_q e^{m_q - m} O_q / l (shard order). Without top-k each shard's race winner
// becomes a record comparable across shards: key_q is relative to m_q, and relative to m it is
// key_q e^{m - m_q}, so its score is (m_q - m) - ln key_q and its ln p is lnp_q + (m_q - m);
// with top-k each shard's candidates go to the row's pool in token order.
__global__ void __launch_bounds__(kThreads) k_shard_merge(
    int n, const RowStat* __restrict__ rows, const Best* __restrict__ best,
    const float* __restrict__ O, const Cand* __restrict__ cand, int k, int R, int d, int L,
    const uint8_t* __restrict__ done, RowStat* __restrict__ rs_out, Best* __restrict__ best_out,
    Cand* __restrict__ pool_out, float* __restrict__ s_out) {
  __shared__ float sh_sc[kMaxShards];
  __shared__ float sh_l;
  pdl_wait();
  const int r = blockIdx.x;
  if (done && done[r / L]) return;
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    int32_t arg = INT_MAX;
    for (int q = 0; q < n; ++q) {
      const RowStat t = rows[(size_t)q * R + r];
      if (better(t.m, t.arg, m, arg)) {
        m = t.m;
        arg = t.arg;
      }
    }
    double l = 0.0;
    for (int q = 0; q < n; ++q) {
      const RowStat t = rows[(size_t)q * R + r];
      const double wq = (double)t.l * exp((double)t.m - (double)m);
      sh_sc[q] = expf(t.m - m);
      l += wq;
    }
    double h = 0.0;
    for (int q = 0; q < n; ++q) {
      const RowStat t = rows[(size_t)q * R + r];
      const double wq = (double)t.l * exp((double)t.m - (double)m) / l;
      if (wq > 0.0) h += wq * ((double)t.ent - log(wq));
    }
    rs_out[r] = RowStat{m, (float)l, (float)h, arg};
    sh_l = (float)l;
    if (k == 0) {
      for (int q = 0; q < n; ++q) {
        const Best b = best[(size_t)q * R + r];
        const float dm = rows[(size_t)q * R + r].m - m;
        const bool has = b.j != INT_MAX && b.v > -INFINITY;
        best_out[(size_t)r * n + q] =
            Best{has ? dm - logf(-b.v) : -INFINITY, b.j, has ? b.y + dm : 0.f, 1};
      }
    }
  }
  if (k > 0) {
    // each shard's k candidates (distinct tokens, or unused slots with token INT_MAX) placed in
    // token order: candidate t goes to the slot of its rank among the shard's tokens
    for (int e = threadIdx.x; e < n * k; e += kThreads) {
      const int q = e / k;
      const Cand c = cand[((size_t)q * R + r) * k + e % k];
      int rank = 0;
      for (int u = 0; u < k; ++u) {
        const int32_t ju = cand[((size_t)q * R + r) * k + u].j;
        rank += (ju < c.j || (ju == c.j && u < e % k)) ? 1 : 0;
      }
      pool_out[(size_t)r * n * k + (size_t)q * k + rank] = c;
    }
  }
  __syncthreads();
  const float l = sh_l;
  const int64_t plane = (int64_t)R * d;
  const float4* src = reinterpret_cast<const float4*>(O + (size_t)r * d);
  float4* dst = reinterpret_cast<float4*>(s_out + (size_t)r * d);
  for (int c4 = threadIdx.x; c4 < d / 4; c4 += kThreads) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < n; ++q) {
      const float4 t = src[q * plane / 4 + c4];
      const float c = sh_sc[q];
      acc.x = fmaf(t.x, c, acc.x);
      acc.y = fmaf(t.y, c, acc.y);
      acc.z = fmaf(t.z, c, acc.z);
      acc.w = fmaf(t.w, c, acc.w);
    }
    dst[c4] = make_float4(acc.x / l, acc.y / l, acc.z / l, acc.w / l);
  }
}

void launch_shard_export(const RowStat* rs, const Best* best, int n_chunks, const Cand* cand,
                         int k, int R, int L, const uint8_t* done, const float* Opart, int S,
                         int d, const float* mref, int64_t j_offset, RowStat* rows_out,
                         Best* best_out, float* O_out, Cand* cand_out, cudaStream_t st) {
  launch_k(k_shard_export, dim3(R), dim3(kThreads), 0, st, rs, best, n_chunks, cand, k, L, done,
           Opart, S, R, d, mref, j_offset, rows_out, best_out, O_out, cand_out);
}

void launch_shard_merge(int n, const RowStat* rows, const Best* best, const float* O,
                        const Cand* cand, int k, int R, int d, int L, const uint8_t* done,
                        RowStat* rs_out, Best* best_out, Cand* pool_out, float* s_out,
                        cudaStream_t st) {
  launch_k(k_shard_merge, dim3(R), dim3(kThreads), 0, st, n, rows, best, O, cand, k, R, d, L,
           done, rs_out, best_out, pool_out, s_out);
}

}  // namespace ds
