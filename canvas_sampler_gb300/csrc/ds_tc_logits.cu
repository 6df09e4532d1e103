// Tensor-core logits of the sampler step on sm_103a, with the softmax statistics of every
// 128-token segment of each row fused into the epilogue:
//   y[r, j] = (sum_k H[r, k] E[j, k]) / T_b        bf16 x bf16 -> fp32 (H [B*L, d], E [V, d])
//   for each row and segment g: max m_g, lowest argmax, sum exp(y - m_g), sum exp(y - m_g)(y - m_g)
// and, by output mode, either y itself (kOutY, the top-k path) or the probabilities relative to
// the row's maximum over the 256-token tile, P = exp(y - m_t) as bf16 hi + lo, with m_t stored
// tile-major (kOutP: y never reaches memory).
// Definitions: DiffusionGemma Technical Report, section 6 "Sampling" (softmax over the full
// vocabulary in full precision). Pipeline structure: ds_tc_common.cuh.
#include <algorithm>
#include <cstdlib>

#include "ds_tc_common.cuh"

namespace ds {
namespace {

using namespace tcpipe;

// ------------------------------------------------------------------------------------------
// logits (+ softmax statistics of each 128-token segment of a row)
// ------------------------------------------------------------------------------------------
// LG_CHUNK_KB: k-blocks (of 4 MMAs) accumulated into one TMEM chunk before the epilogue adds it
// to its fp32 registers. Longer chains carry more of the accumulator's round-toward-zero error
// but leave the epilogue's round trip (drain, release, next issue) and the output of each tile
// more time to hide behind the MMAs. Measured against the fp64 oracle at V = 262144, d = 2816
// (49 positions) and V = 32768, d = 1024 (256 positions), largest relative errors of s /
// entropy: 2 k-blocks 2.4e-6 / 1.9e-6, 4: 3.6e-6 / 3.2e-6, 6: 3.6e-6 / 4.3e-6, 8: 5.5e-6 /
// 7.2e-6, with the logits kernel at 0.393, 0.350, 0.335 and 0.327 ms.
constexpr int LG_BM = 128, LG_BN = 256, LG_BK = 64, LG_STAGES = 4, LG_CHUNK_KB = 6;
// The first chunk of each tile is longer: while the epilogue writes a tile's output the MMAs
// of the next tile can only fill the two TMEM buffers, so a longer first chunk hides more of
// that output phase behind MMAs. Same-box A/B at 2070 MHz (logits kernel per step, 6 stages):
// first chunk 6 / 12 / 18 / 24 k-blocks at B = 1: 0.323 (5 stages) / 0.312 / 0.310 / 0.309 ms;
// B = 4: 1.117 (5 stages) / 1.060 / 1.045 / 1.033 ms; B = 8: 2.21 (5 stages) / 2.11 / 2.05 / 2.00
// ms. Largest relative errors against the oracle (s / entropy / confidence; V = 262144, d = 2816,
// 98 positions, and V = 32768, d = 1024, all 256 positions): 12 k-blocks 5.8e-6 / 8.4e-6 /
// 6.8e-6, 16: 1.0e-5 / 1.4e-5 / 1.6e-5 (at d = 1024 that is the whole K in one chain), 24: 1.1e-5
// / 1.4e-5 / 1.6e-5: 12 keeps a 2.4x margin to the 2e-5 tolerance.
constexpr int LG_FIRST_KB = 12;
constexpr int LG_COLS = LG_BN / 2;
constexpr uint32_t LG_A_BYTES = LG_BM * LG_BK * 2;
constexpr uint32_t LG_B_BYTES = LG_BN * LG_BK * 2;
constexpr uint32_t LG_STAGE_BYTES = LG_A_BYTES + LG_B_BYTES;
// The output leaves through 4 KB staging boxes, written by one epilogue warp and stored by TMA
// (full lines in global memory): one 32 x 32 fp32 box of y, or a 32 x 32 bf16 box each of the
// hi and lo parts of P.
constexpr uint32_t LG_STG_BYTES = 32 * 32 * 4;
// CTA pair: each CTA stages its 128 rows of H and 128 of the tile's 256 rows of E (32 KB a
// stage), so an SM takes in 2/3 of the bytes per MAC of a one-CTA tile. Measured at the bench
// size (logits kernel per step), first chunks of 6 k-blocks: 5 stages with one staging box per
// warp 0.323 ms, with two boxes used in turn (a warp writes the next box while the store of the
// previous one still reads it) 0.328 ms, 6 stages with one box 0.327 ms, 4 stages with two 0.344
// ms; with first chunks of 12 k-blocks (same box, same day): 5 stages 0.320, 6 stages 0.312 ms
// at B = 1, 1.066 / 1.060 ms at B = 4, 2.126 / 2.112 ms at B = 8. 6 stages and one box per warp
// use 225 KB of the 227 KB of shared memory a CTA may have.
#ifndef DS_LG2_STAGES
#define DS_LG2_STAGES 6
#endif
#ifndef DS_LG2_STG_BOXES
#define DS_LG2_STG_BOXES 1
#endif
constexpr int LG2_STAGES = DS_LG2_STAGES, LG2_STG_BOXES = DS_LG2_STG_BOXES;
constexpr uint32_t LG2_STAGE_BYTES = LG_A_BYTES + LG_B_BYTES / 2;
static_assert(LG2_STAGES <= tcpipe::kMaxStages && LG_STAGES <= tcpipe::kMaxStages, "stages");
constexpr size_t LG_SMEM =
    (size_t)LG_STAGES * LG_STAGE_BYTES + (size_t)kEpiWarps * LG_STG_BYTES + 1024;
constexpr size_t LG2_SMEM = (size_t)LG2_STAGES * LG2_STAGE_BYTES +
                            (size_t)kEpiWarps * LG2_STG_BOXES * LG_STG_BYTES + 1024;

// kStandin: the same GEMM with A = U [R, 2d] (bf16(s_prev) | E[canvas]), B = W [d, 2d] and the
// epilogue H = bf16(tanh(acc)) instead of y and the statistics (V plays N = d, d plays K = 2d).
enum { kOutY = 0, kOutP = 1, kStandin = 2 };

// PAIR: launched in clusters of two CTAs; a work item is a 256-row x 256-token tile computed by
// M = 256 MMAs that the even CTA issues for both, each CTA holding the accumulator of its own
// 128 rows (its epilogue is the one-CTA epilogue of that 128 x 256 tile). Needs R % 256 == 0.
template <int MODE, bool PAIR>
__global__ void __launch_bounds__(kThreadsTC, 1)
    k_logits_tc(const __grid_constant__ CUtensorMap mapH, const __grid_constant__ CUtensorMap mapE,
                const __grid_constant__ CUtensorMap mapY, const __grid_constant__ CUtensorMap mapPlo,
                int R, int64_t V, int d, int L, const float* __restrict__ T,
                const uint8_t* __restrict__ done, ChunkStat* __restrict__ seg_stats,
                float* __restrict__ mseg_t, uint16_t* __restrict__ Hout, uint32_t* err,
                int first_kb) {
  constexpr bool STANDIN = MODE == kStandin;
  constexpr int STAGES = PAIR ? LG2_STAGES : LG_STAGES;
  constexpr uint32_t STAGE_BYTES = PAIR ? LG2_STAGE_BYTES : LG_STAGE_BYTES;
  constexpr int ROWS = PAIR ? 2 * LG_BM : LG_BM;  // rows of a work item
  constexpr int NSTG = PAIR ? LG2_STG_BOXES : 1;  // staging boxes per epilogue warp
  extern __shared__ uint8_t dyn_smem[];
  __shared__ Ctl ctl;
  // kOutP: the two column halves' segment maxima of each row, and per TMEM lane quadrant a
  // barrier of its two epilogue warps (bounded), passed twice an item: after the maxima are
  // written and after they are read
  __shared__ float xmax[2][LG_BM];
  __shared__ uint64_t xbar[4];
  uint8_t* smem = align1024(dyn_smem);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int n_units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int n_it = R / ROWS;  // row items
  const int n_ct = (int)(V / LG_BN);
  const int n_tiles = n_it * n_ct;
  const int nk = d / LG_BK;
  // chunk 0 of a tile takes first_kb k-blocks, the others LG_CHUNK_KB: a longer first chunk
  // lets the MMAs of a tile run further ahead while the epilogue writes the previous tile's
  // output (one longer accumulation chain per tile)
  const int fkb = min(max(first_kb, 1), nk);
  const int n_ch = 1 + (nk - fkb + LG_CHUNK_KB - 1) / LG_CHUNK_KB;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&xbar[i]), 2);
    // pair: one arrival per epilogue warp of both CTAs releases a TMEM buffer of the pair
    ctl_init(ctl, STAGES, PAIR ? 2 * kEpiWarps : 32 * kEpiWarps);  // ends with the init fence
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapH);
    tma_prefetch_desc(&mapE);
    if (!STANDIN) tma_prefetch_desc(&mapY);
    if (MODE == kOutP) tma_prefetch_desc(&mapPlo);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(&ctl.tmem_base), 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&ctl.tmem_base), 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // both CTAs' barriers initialised before any remote use
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* abort_flag = &ctl.abort;
  // the setup above is local; H, T and done may still be being written by the kernel before
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_E = policy_evict_first(), pol_H = policy_evict_last();
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = unit; tile < n_tiles && ok; tile += n_units) {
        const int it = tile % n_it, ct = tile / n_it;
        if (rows_done(done, it * ROWS, ROWS, L)) continue;
        const int rt = PAIR ? 2 * it + (int)rank : it;
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait(smem_u32(&ctl.empty[stage]), phase ^ 1, abort_flag, err)) {
            ok = false;
            break;
          }
          const uint32_t sa = sbase + stage * STAGE_BYTES, sb = sa + LG_A_BYTES;
          const uint32_t fb = smem_u32(&ctl.full[stage]);
          if constexpr (PAIR) {
            // both CTAs' copies complete on the even CTA's barrier, which expects all of them
            if (rank == 0) mbar_arrive_expect_tx(fb, 2 * STAGE_BYTES);
            const uint32_t fb0 = mapa_shared(fb, 0);
            tma_load_2d_pair(sa, &mapH, fb0, kc * LG_BK, rt * LG_BM, pol_H);
            tma_load_2d_pair(sb, &mapE, fb0, kc * LG_BK, ct * LG_BN + (int)rank * (LG_BN / 2),
                             pol_E);
          } else {
            mbar_arrive_expect_tx(fb, STAGE_BYTES);
            tma_load_2d(sa, &mapH, fb, kc * LG_BK, rt * LG_BM, pol_H);
            tma_load_2d(sb, &mapE, fb, kc * LG_BK, ct * LG_BN, pol_E);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // (pair: the odd CTA's copies complete on the even CTA's barriers, which its own
      // producer drains)
      if (!ok && rank == 0) producer_drain(ctl, issued, STAGES);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(ROWS, LG_BN, false, false);
      int stage = 0, cc = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = unit; tile < n_tiles && ok; tile += n_units) {
        const int it = tile % n_it;
        if (rows_done(done, it * ROWS, ROWS, L)) continue;
        for (int ch = 0; ch < n_ch && ok; ++ch, ++cc) {
          const int buf = cc & 1;
          const uint32_t par = (uint32_t)((cc >> 1) & 1);
          if (!mbar_wait(smem_u32(&ctl.tempty[buf]), par ^ 1, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dt = tmem + (uint32_t)(buf * LG_BN);
          const int kc0 = ch == 0 ? 0 : fkb + (ch - 1) * LG_CHUNK_KB;
          const int kc1 = ch == 0 ? fkb : min(nk, kc0 + LG_CHUNK_KB);
          for (int kc = kc0; kc < kc1; ++kc) {
            if (!mbar_wait(smem_u32(&ctl.full[stage]), phase, abort_flag, err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            *(volatile int*)&ctl.consumed = ctl.consumed + 1;
            const uint32_t sa = sbase + stage * STAGE_BYTES, sb = sa + LG_A_BYTES;
#pragma unroll
            for (int k = 0; k < LG_BK / 16; ++k) {
              const uint64_t ad = sdesc_sw128(sa + 32 * k, 16, 1024);
              const uint64_t bd = sdesc_sw128(sb + 32 * k, 16, 1024);
              const uint32_t acc_in = (kc != kc0 || k) ? 1u : 0u;
              if constexpr (PAIR) umma_bf16_pair(dt, ad, bd, idesc, acc_in);
              else umma_bf16(dt, ad, bd, idesc, acc_in);
            }
            if constexpr (PAIR) umma_commit_pair(smem_u32(&ctl.empty[stage]), 0x3);
            else umma_commit(smem_u32(&ctl.empty[stage]));
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          if constexpr (PAIR) umma_commit_pair(smem_u32(&ctl.tfull[buf]), 0x3);
          else umma_commit(smem_u32(&ctl.tfull[buf]));
        }
      }
      if constexpr (PAIR) umma_commit_pair(smem_u32(&ctl.mma_done), 0x1);
      else umma_commit(smem_u32(&ctl.mma_done));
      mbar_wait_quiet(smem_u32(&ctl.mma_done), 0);
    }
  } else {
    const int q = warp & 3;              // TMEM lane quadrant this warp may access
    const int half = (warp - 2) >> 2;    // column half of the tile
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    // pair: the TMEM buffers are released on the even CTA's barriers, once per warp
    const uint32_t tempty0 = PAIR ? mapa_shared(smem_u32(&ctl.tempty[0]), 0) : 0u;
    const uint32_t tempty1 = PAIR ? mapa_shared(smem_u32(&ctl.tempty[1]), 0) : 0u;
    int cc = 0, items = 0;
    bool ok = true;
    for (int tile = unit; tile < n_tiles && ok; tile += n_units) {
      const int it = tile % n_it, ct = tile / n_it;
      if (rows_done(done, it * ROWS, ROWS, L)) continue;
      const int rt = PAIR ? 2 * it + (int)rank : it;
      const int b = (rt * LG_BM) / L;
      float acc[LG_COLS];
#pragma unroll
      for (int i = 0; i < LG_COLS; ++i) acc[i] = 0.f;
      for (int ch = 0; ch < n_ch; ++ch, ++cc) {
        const int buf = cc & 1;
        const uint32_t par = (uint32_t)((cc >> 1) & 1);
        if (!mbar_wait(smem_u32(&ctl.tfull[buf]), par, abort_flag, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_accumulate<LG_COLS>(tmem + (uint32_t)(buf * LG_BN + half * LG_COLS) + lane_base, acc);
        tc_fence_before();
        if constexpr (PAIR) {
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(buf ? tempty1 : tempty0);
        } else {
          mbar_arrive(smem_u32(&ctl.tempty[buf]));
        }
      }
      if (!ok) break;
      if constexpr (STANDIN) {
        const int64_t n0 = (int64_t)ct * LG_BN + half * LG_COLS;
        uint16_t* hrow = Hout + (size_t)(rt * LG_BM + q * 32 + lane) * V + n0;
#pragma unroll
        for (int v = 0; v < LG_COLS / 8; ++v) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 h2 =
                __floats2bfloat162_rn(tanhf(acc[8 * v + 2 * e]), tanhf(acc[8 * v + 2 * e + 1]));
            w4[e] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          *reinterpret_cast<uint4*>(hrow + 8 * v) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        continue;
      }
      // y = z / T (as z * (1/T), rounded once: no fused multiply-add with the subtraction, so
      // y - m is exactly 0 at the maximum); the segment's max, argmax (lowest token), sum of
      // exp(y - m) and sum of exp(y - m) (y - m). x * invT is monotone in x for invT > 0, so the
      // max of the scaled values is the scaled max, at the same lowest index.
      const float invT = 1.0f / T[b];
      const int row0 = rt * LG_BM + q * 32;
      const int64_t j0 = (int64_t)ct * LG_BN + half * LG_COLS;
      float zmax = -INFINITY;
      int arg = 0;
#pragma unroll
      for (int i = 0; i < LG_COLS; ++i) {
        if (acc[i] > zmax) {
          zmax = acc[i];
          arg = i;
        }
      }
      const float m = __fmul_rn(zmax, invT);
      // kOutP: P is relative to the maximum of the row over the whole 256-token tile (both
      // column halves), so that one TMEM chunk of the self-conditioning GEMM covers a tile;
      // the statistics stay relative to the segment's own maximum m
      float ptile = 1.f;  // exp(m - m_tile)
      float m_tile = m;
      if constexpr (MODE == kOutP) {
        xmax[half][q * 32 + lane] = m;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&xbar[q]));
        if (!mbar_wait(smem_u32(&xbar[q]), (uint32_t)(items & 1), abort_flag, err)) {
          ok = false;
          break;
        }
        ++items;
        m_tile = fmaxf(m, xmax[half ^ 1][q * 32 + lane]);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&xbar[q]));
        if (!mbar_wait(smem_u32(&xbar[q]), (uint32_t)(items & 1), abort_flag, err)) {
          ok = false;
          break;
        }
        ++items;
        ptile = exp2_approx((m - m_tile) * 1.4426950408889634f);
      }
      float l = 0.f, a = 0.f;
      const uint32_t stg0 =
          sbase + STAGES * STAGE_BYTES + (uint32_t)((warp - 2) * NSTG) * LG_STG_BYTES;
#pragma unroll
      for (int bx = 0; bx < LG_COLS / 32; ++bx) {
        const uint32_t stg = stg0 + (uint32_t)(bx % NSTG) * LG_STG_BYTES;
        // the store issued from this box NSTG boxes ago has read it
        if (lane == 0) {
          if constexpr (NSTG == 2) bulk_wait_read_le1();
          else bulk_wait_read_all();
        }
        __syncwarp();
        if constexpr (MODE == kOutY) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            float y4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              y4[e] = __fmul_rn(acc[bx * 32 + c * 4 + e], invT);
              const float t = y4[e] - m;
              const float x = __expf(t);
              l += x;
              a = fmaf(x, t, a);
            }
            // row `lane` of the box, 16-byte chunk c at its 128-byte-swizzled position
            st_shared_f4(stg + lane * 128 + ((c ^ (lane & 7)) << 4), y4[0], y4[1], y4[2], y4[3]);
          }
        } else {
          // exp(y - m) = 2^((y - m) log2 e) (within ~3e-6 relative for y - m > -30; 1 at the
          // maximum); P = exp(y - m) exp(m - m_tile) as bf16 hi = RN(P) and lo = RN(P - hi);
          // one 32 x 32 box each for hi and lo, rows of 64 bytes in the 64-byte swizzle
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float p[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float t = __fmul_rn(acc[bx * 32 + c * 8 + e], invT) - m;
              p[e] = exp2_approx(t * 1.4426950408889634f);
              l += p[e];
              a = fmaf(p[e], t, a);
              p[e] *= ptile;
            }
            uint32_t h[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) split_bf16x2(p[2 * e], p[2 * e + 1], h[e], lo[e]);
            const uint32_t off = lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4);
            st_shared_u4(stg + off, h[0], h[1], h[2], h[3]);
            st_shared_u4(stg + 2048 + off, lo[0], lo[1], lo[2], lo[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&mapY, stg, (int32_t)(j0 + bx * 32), row0);
          if constexpr (MODE == kOutP) tma_store_2d(&mapPlo, stg + 2048, (int32_t)(j0 + bx * 32), row0);
          bulk_commit();
        }
      }
      const int seg = (int)(j0 / LG_COLS);
      seg_stats[(size_t)(row0 + lane) * (V / LG_COLS) + seg] =
          ChunkStat{m, l, a, (int32_t)(j0 + arg)};
      if constexpr (MODE == kOutP)
        if (half == 0) mseg_t[(size_t)ct * R + row0 + lane] = m_tile;
    }
    if (!STANDIN && lane == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  // pair: neither CTA frees its TMEM or exits while the other may still use its barriers,
  // shared memory or TMEM
  if constexpr (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, 512);
    else tmem_dealloc(tmem, 512);
  }
}

}  // namespace

// Clusters of the pair kernel that can be resident at once (a TPC with an SM unavailable holds
// none), so that no pair starts its items after the others have finished theirs.
static int g_pairs_resident = 1;

void tc_prepare_logits() {
  const int smem = (int)LG_SMEM;
  cudaFuncSetAttribute(k_logits_tc<kOutY, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaFuncSetAttribute(k_logits_tc<kOutP, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaFuncSetAttribute(k_logits_tc<kStandin, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       smem);
  cudaFuncSetAttribute(k_logits_tc<kOutY, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)LG2_SMEM);
  cudaFuncSetAttribute(k_logits_tc<kOutP, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)LG2_SMEM);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::max(2, sms - sms % 2));
  cfg.blockDim = dim3(kThreadsTC);
  cfg.dynamicSmemBytes = LG2_SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_logits_tc<kOutP, true>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = std::max(1, sms / 2);
  }
  g_pairs_resident = n;
}

// k-blocks of the first TMEM chunk of each logits tile (LG_FIRST_KB, or DS_LOGITS_FIRST_KB in
// the environment for measurements).
int logits_first_kb() {
  static const int v = [] {
    const char* e = getenv("DS_LOGITS_FIRST_KB");
    const int x = e ? atoi(e) : LG_FIRST_KB;
    return x >= 1 ? x : LG_FIRST_KB;
  }();
  return v;
}

bool logits_pair_enabled(int R) {
  static const bool on = [] {
    const char* e = getenv("DS_LOGITS_PAIR");
    return !(e && e[0] == '0');
  }();
  return on && R % (2 * LG_BM) == 0 && tc_num_sms() >= 2;
}

namespace {

// One launch of the logits GEMM in mode MODE: one CTA per SM, or (pair) one cluster of two CTAs
// per two SMs.
template <int MODE>
cudaError_t launch_logits_mode(const CUtensorMap& mH, const CUtensorMap& mE1,
                               const CUtensorMap& mE2, const CUtensorMap& mOut,
                               const CUtensorMap& mOut2, int R, int64_t V, int d, int L,
                               const float* T, const uint8_t* done, ChunkStat* seg_stats,
                               float* mseg_t, uint32_t* err, cudaStream_t st) {
  const int n_ct = (int)(V / LG_BN);
  if (logits_pair_enabled(R)) {
    const int n_items = (R / (2 * LG_BM)) * n_ct;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreadsTC);
    cfg.dynamicSmemBytes = LG2_SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    const int pairs = std::max(1, std::min(n_items, g_pairs_resident));
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    return cudaLaunchKernelEx(&cfg, k_logits_tc<MODE, true>, mH, mE2, mOut, mOut2, R, V, d, L, T,
                              done, seg_stats, mseg_t, (uint16_t*)nullptr, err, logits_first_kb());
  }
  const int n_tiles = (R / LG_BM) * n_ct;
  const int grid = std::max(1, std::min(n_tiles, tc_num_sms()));
  return launch_k(k_logits_tc<MODE, false>, dim3(grid), dim3(kThreadsTC), LG_SMEM, st, mH, mE1,
                  mOut, mOut2, R, V, d, L, T, done, seg_stats, mseg_t, (uint16_t*)nullptr, err,
                  logits_first_kb());
}

}  // namespace

cudaError_t launch_logits_tc(const uint16_t* H, const uint16_t* E, int R, int64_t V, int d, int L,
                             const float* T, const uint8_t* done, float* Y, ChunkStat* seg_stats,
                             uint32_t* err, cudaStream_t st) {
  if (!tc_available()) return cudaErrorNotSupported;
  CUtensorMap mH, mE, mE2, mY;
  if (!tc_make_map_bf16(&mH, H, (uint64_t)R, (uint64_t)d, LG_BM, LG_BK) ||
      !tc_make_map_bf16(&mE, E, (uint64_t)V, (uint64_t)d, LG_BN, LG_BK) ||
      !tc_make_map_bf16(&mE2, E, (uint64_t)V, (uint64_t)d, LG_BN / 2, LG_BK) ||
      !tc_make_map_f32(&mY, Y, (uint64_t)R, (uint64_t)V, 32, 32))
    return cudaErrorInvalidValue;
  return launch_logits_mode<kOutY>(mH, mE, mE2, mY, mY, R, V, d, L, T, done, seg_stats, nullptr,
                                   err, st);
}

cudaError_t launch_logits_p_tc(const uint16_t* H, const uint16_t* E, int R, int64_t V, int d,
                               int L, const float* T, const uint8_t* done, uint16_t* Phi,
                               uint16_t* Plo, ChunkStat* seg_stats, float* mseg_t, uint32_t* err,
                               cudaStream_t st) {
  if (!tc_available()) return cudaErrorNotSupported;
  CUtensorMap mH, mE, mE2, mPh, mPl;
  if (!tc_make_map_bf16(&mH, H, (uint64_t)R, (uint64_t)d, LG_BM, LG_BK) ||
      !tc_make_map_bf16(&mE, E, (uint64_t)V, (uint64_t)d, LG_BN, LG_BK) ||
      !tc_make_map_bf16(&mE2, E, (uint64_t)V, (uint64_t)d, LG_BN / 2, LG_BK) ||
      !tc_make_map_bf16_sw64(&mPh, Phi, (uint64_t)R, (uint64_t)V, 32, 32) ||
      !tc_make_map_bf16_sw64(&mPl, Plo, (uint64_t)R, (uint64_t)V, 32, 32))
    return cudaErrorInvalidValue;
  return launch_logits_mode<kOutP>(mH, mE, mE2, mPh, mPl, R, V, d, L, T, done, seg_stats, mseg_t,
                                   err, st);
}

cudaError_t launch_standin_tc(const uint16_t* U, const uint16_t* W, int R, int d, int L,
                              const uint8_t* done, uint16_t* H_out, uint32_t* err,
                              cudaStream_t st) {
  if (!tc_available()) return cudaErrorNotSupported;
  if (d % LG_BN) return cudaErrorInvalidValue;
  CUtensorMap mU, mW;
  if (!tc_make_map_bf16(&mU, U, (uint64_t)R, (uint64_t)(2 * d), LG_BM, LG_BK) ||
      !tc_make_map_bf16(&mW, W, (uint64_t)d, (uint64_t)(2 * d), LG_BN, LG_BK))
    return cudaErrorInvalidValue;
  const int n_tiles = (R / LG_BM) * (d / LG_BN);
  const int grid = std::max(1, std::min(n_tiles, tc_num_sms()));
  k_logits_tc<kStandin, false><<<grid, kThreadsTC, LG_SMEM, st>>>(mU, mW, mU, mU, R, (int64_t)d, 2 * d,
                                                            L, nullptr, done, nullptr, nullptr,
                                                            H_out, err, LG_CHUNK_KB);
  return cudaGetLastError();
}

}  // namespace ds
