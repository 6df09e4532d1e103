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

#include "ds_tc_common.cuh"

namespace ds {
namespace {

using namespace tcpipe;

// ------------------------------------------------------------------------------------------
// logits (+ softmax statistics of each 128-token segment of a row)
// ------------------------------------------------------------------------------------------
constexpr int LG_BM = 128, LG_BN = 256, LG_BK = 64, LG_STAGES = 4, LG_CHUNK_KB = 2;
constexpr int LG_COLS = LG_BN / 2;
constexpr uint32_t LG_A_BYTES = LG_BM * LG_BK * 2;
constexpr uint32_t LG_B_BYTES = LG_BN * LG_BK * 2;
constexpr uint32_t LG_STAGE_BYTES = LG_A_BYTES + LG_B_BYTES;
// y leaves through one 32 x 32 fp32 staging box per epilogue warp (128-byte swizzle, written
// by the warp, stored by one TMA bulk store), so the global stores are full lines.
constexpr uint32_t LG_STG_BYTES = 32 * 32 * 4;
constexpr size_t LG_SMEM =
    (size_t)LG_STAGES * LG_STAGE_BYTES + (size_t)kEpiWarps * LG_STG_BYTES + 1024;

// kStandin: the same GEMM with A = U [R, 2d] (bf16(s_prev) | E[canvas]), B = W [d, 2d] and the
// epilogue H = bf16(tanh(acc)) instead of y and the statistics (V plays N = d, d plays K = 2d).
enum { kOutY = 0, kOutP = 1, kStandin = 2 };

template <int MODE>
__global__ void __launch_bounds__(kThreadsTC, 1)
    k_logits_tc(const __grid_constant__ CUtensorMap mapH, const __grid_constant__ CUtensorMap mapE,
                const __grid_constant__ CUtensorMap mapY, const __grid_constant__ CUtensorMap mapPlo,
                int R, int64_t V, int d, int L, const float* __restrict__ T,
                const uint8_t* __restrict__ done, ChunkStat* __restrict__ seg_stats,
                float* __restrict__ mseg_t, uint16_t* __restrict__ Hout, uint32_t* err) {
  constexpr bool STANDIN = MODE == kStandin;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ Ctl ctl;
  // kOutP: the two column halves' segment maxima of each row, and a barrier of all epilogue
  // warps (bounded), passed twice an item: after the maxima are written and after they are read
  __shared__ float xmax[2][LG_BM];
  __shared__ uint64_t xbar;
  uint8_t* smem = align1024(dyn_smem);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_rt = R / LG_BM;
  const int n_ct = (int)(V / LG_BN);
  const int n_tiles = n_rt * n_ct;
  const int nk = d / LG_BK;
  const int n_ch = (nk + LG_CHUNK_KB - 1) / LG_CHUNK_KB;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&xbar), kEpiWarps);
    ctl_init(ctl, LG_STAGES);  // ends with the mbarrier-init fence
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapH);
    tma_prefetch_desc(&mapE);
    if (!STANDIN) tma_prefetch_desc(&mapY);
    if (MODE == kOutP) tma_prefetch_desc(&mapPlo);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* abort_flag = &ctl.abort;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_E = policy_evict_first(), pol_H = policy_evict_last();
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int rt = tile % n_rt, ct = tile / n_rt;
        if (done && done[(rt * LG_BM) / L]) continue;
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait(smem_u32(&ctl.empty[stage]), phase ^ 1, abort_flag, err)) {
            ok = false;
            break;
          }
          const uint32_t sa = sbase + stage * LG_STAGE_BYTES, sb = sa + LG_A_BYTES;
          const uint32_t fb = smem_u32(&ctl.full[stage]);
          mbar_arrive_expect_tx(fb, LG_STAGE_BYTES);
          tma_load_2d(sa, &mapH, fb, kc * LG_BK, rt * LG_BM, pol_H);
          tma_load_2d(sb, &mapE, fb, kc * LG_BK, ct * LG_BN, pol_E);
          ++issued;
          if (++stage == LG_STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) producer_drain(ctl, issued, LG_STAGES);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(LG_BM, LG_BN, false, false);
      int stage = 0, cc = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int rt = tile % n_rt;
        if (done && done[(rt * LG_BM) / L]) continue;
        for (int ch = 0; ch < n_ch && ok; ++ch, ++cc) {
          const int buf = cc & 1;
          const uint32_t par = (uint32_t)((cc >> 1) & 1);
          if (!mbar_wait(smem_u32(&ctl.tempty[buf]), par ^ 1, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dt = tmem + (uint32_t)(buf * LG_BN);
          const int kc0 = ch * LG_CHUNK_KB, kc1 = min(nk, kc0 + LG_CHUNK_KB);
          for (int kc = kc0; kc < kc1; ++kc) {
            if (!mbar_wait(smem_u32(&ctl.full[stage]), phase, abort_flag, err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            *(volatile int*)&ctl.consumed = ctl.consumed + 1;
            const uint32_t sa = sbase + stage * LG_STAGE_BYTES, sb = sa + LG_A_BYTES;
#pragma unroll
            for (int k = 0; k < LG_BK / 16; ++k)
              umma_bf16(dt, sdesc_sw128(sa + 32 * k, 16, 1024),
                        sdesc_sw128(sb + 32 * k, 16, 1024), idesc, (kc != kc0 || k) ? 1u : 0u);
            umma_commit(smem_u32(&ctl.empty[stage]));
            if (++stage == LG_STAGES) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          umma_commit(smem_u32(&ctl.tfull[buf]));
        }
      }
      umma_commit(smem_u32(&ctl.mma_done));
      mbar_wait_quiet(smem_u32(&ctl.mma_done), 0);
    }
  } else {
    const int q = warp & 3;              // TMEM lane quadrant this warp may access
    const int half = (warp - 2) >> 2;    // column half of the tile
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int cc = 0, items = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      const int rt = tile % n_rt, ct = tile / n_rt;
      const int b = (rt * LG_BM) / L;
      if (done && done[b]) continue;
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
        mbar_arrive(smem_u32(&ctl.tempty[buf]));
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
        if (lane == 0) mbar_arrive(smem_u32(&xbar));
        if (!mbar_wait(smem_u32(&xbar), (uint32_t)(items & 1), abort_flag, err)) {
          ok = false;
          break;
        }
        ++items;
        m_tile = fmaxf(m, xmax[half ^ 1][q * 32 + lane]);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&xbar));
        if (!mbar_wait(smem_u32(&xbar), (uint32_t)(items & 1), abort_flag, err)) {
          ok = false;
          break;
        }
        ++items;
        ptile = exp2_approx((m - m_tile) * 1.4426950408889634f);
      }
      float l = 0.f, a = 0.f;
      const uint32_t stg = sbase + LG_STAGES * LG_STAGE_BYTES + (uint32_t)(warp - 2) * LG_STG_BYTES;
#pragma unroll
      for (int bx = 0; bx < LG_COLS / 32; ++bx) {
        if (lane == 0) bulk_wait_read_all();  // the previous store has read the staging box
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
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

void tc_prepare_logits() {
  cudaFuncSetAttribute(k_logits_tc<kOutY>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)LG_SMEM);
  cudaFuncSetAttribute(k_logits_tc<kOutP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)LG_SMEM);
  cudaFuncSetAttribute(k_logits_tc<kStandin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)LG_SMEM);
}

cudaError_t launch_logits_tc(const uint16_t* H, const uint16_t* E, int R, int64_t V, int d, int L,
                             const float* T, const uint8_t* done, float* Y, ChunkStat* seg_stats,
                             uint32_t* err, cudaStream_t st) {
  if (!tc_available()) return cudaErrorNotSupported;
  CUtensorMap mH, mE, mY;
  if (!tc_make_map_bf16(&mH, H, (uint64_t)R, (uint64_t)d, LG_BM, LG_BK) ||
      !tc_make_map_bf16(&mE, E, (uint64_t)V, (uint64_t)d, LG_BN, LG_BK) ||
      !tc_make_map_f32(&mY, Y, (uint64_t)R, (uint64_t)V, 32, 32))
    return cudaErrorInvalidValue;
  const int n_tiles = (R / LG_BM) * (int)(V / LG_BN);
  const int grid = std::max(1, std::min(n_tiles, tc_num_sms()));
  k_logits_tc<kOutY><<<grid, kThreadsTC, LG_SMEM, st>>>(mH, mE, mY, mY, R, V, d, L, T, done,
                                                         seg_stats, nullptr, nullptr, err);
  return cudaGetLastError();
}

cudaError_t launch_logits_p_tc(const uint16_t* H, const uint16_t* E, int R, int64_t V, int d,
                               int L, const float* T, const uint8_t* done, uint16_t* Phi,
                               uint16_t* Plo, ChunkStat* seg_stats, float* mseg_t, uint32_t* err,
                               cudaStream_t st) {
  if (!tc_available()) return cudaErrorNotSupported;
  CUtensorMap mH, mE, mPh, mPl;
  if (!tc_make_map_bf16(&mH, H, (uint64_t)R, (uint64_t)d, LG_BM, LG_BK) ||
      !tc_make_map_bf16(&mE, E, (uint64_t)V, (uint64_t)d, LG_BN, LG_BK) ||
      !tc_make_map_bf16_sw64(&mPh, Phi, (uint64_t)R, (uint64_t)V, 32, 32) ||
      !tc_make_map_bf16_sw64(&mPl, Plo, (uint64_t)R, (uint64_t)V, 32, 32))
    return cudaErrorInvalidValue;
  const int n_tiles = (R / LG_BM) * (int)(V / LG_BN);
  const int grid = std::max(1, std::min(n_tiles, tc_num_sms()));
  k_logits_tc<kOutP><<<grid, kThreadsTC, LG_SMEM, st>>>(mH, mE, mPh, mPl, R, V, d, L, T, done,
                                                         seg_stats, mseg_t, nullptr, err);
  return cudaGetLastError();
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
  k_logits_tc<kStandin><<<grid, kThreadsTC, LG_SMEM, st>>>(mU, mW, mU, mU, R, (int64_t)d, 2 * d,
                                                            L, nullptr, done, nullptr, nullptr,
                                                            H_out, err);
  return cudaGetLastError();
}

}  // namespace ds
