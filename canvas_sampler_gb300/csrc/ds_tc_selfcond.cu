// Tensor-core self-conditioning partials of the sampler step on sm_103a:
//   O_s[r, n] = sum_{j in split s} (P_hi + P_lo)[r, j] E[j, n]
// where P_hi + P_lo = exp(y - m) split into two bf16 terms, so the product keeps ~16
// significant bits of the probabilities (a single bf16 keeps 8); the splits over the vocabulary
// are summed and divided by the softmax normaliser afterwards.
// SCALED: P is relative to the row's maximum m_t over each 256-token tile t (the logits kernel's
// kOutP output); each tile is one TMEM chunk, promoted into registers scaled by exp(m_t - M_s)
// with M_s the running maximum of the split (the registers are rescaled when it grows), and M_s
// is stored beside the partial, O_s = sum_t exp(m_t - M_s) sum_{j in t} P_t[r, j] E[j, n].
// Definitions: DiffusionGemma Technical Report, section 6 "Sampling" (the self-conditioning
// embedding matmul, in full precision). Pipeline structure: ds_tc_common.cuh.
// With Gumbel work the kernel also runs the step's Gumbel-max race (ds_sample.cuh): the GEMM is
// bound by the tensor pipe and leaves the SM's issue slots mostly idle, so two warps of its own
// race (row, chunk) items from a queue from the start, and every other warp joins the queue once
// its part of the GEMM is done (all warps of a CTA without a GEMM item race from the start).
#include <algorithm>

#include "ds_sample.cuh"
#include "ds_tc_common.cuh"

namespace ds {
namespace {

using namespace tcpipe;

// ------------------------------------------------------------------------------------------
// self-conditioning partials
// ------------------------------------------------------------------------------------------
constexpr int SC_BM = 128, SC_BK = 64, SC_STAGES = 3, SC_BN_MAX = 256, SC_CHUNK_KB = 4;
constexpr uint32_t SC_A_BYTES = SC_BM * SC_BK * 2;        // one of hi / lo
constexpr uint32_t SC_BOX_BYTES = 64 * SC_BK * 2;          // 64 d-columns x 64 tokens
constexpr uint32_t SC_STAGE_BYTES = 2 * SC_A_BYTES + (SC_BN_MAX / 64) * SC_BOX_BYTES;
constexpr size_t SC_SMEM = (size_t)SC_STAGES * SC_STAGE_BYTES + 1024;
// the pipeline's warps (producer, MMA, 8 epilogue) and two racing warps
constexpr int SC_THREADS = kThreadsTC + 64;

template <int BN, bool SCALED>
__global__ void __launch_bounds__(SC_THREADS, 1)
    k_selfcond_tc(const __grid_constant__ CUtensorMap mapPhi,
                  const __grid_constant__ CUtensorMap mapPlo,
                  const __grid_constant__ CUtensorMap mapE, int R, int64_t V, int d, int L,
                  int S, int kb_per_split, const uint8_t* __restrict__ done,
                  float* __restrict__ Opart, const float* __restrict__ mtile_t,
                  float* __restrict__ mref, uint32_t* err, const __grid_constant__ GumbelWork gw) {
  constexpr int COLS = BN / 2;
  constexpr int CHUNK_KB = SC_CHUNK_KB;  // 4 K blocks = one 256-token tile
  static_assert(CHUNK_KB * SC_BK == 256, "a chunk is one tile of the P reference maxima");
  extern __shared__ uint8_t dyn_smem[];
  __shared__ Ctl ctl;
  uint8_t* smem = align1024(dyn_smem);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_rt = R / SC_BM, n_dt = d / BN;
  const int n_tiles = n_rt * n_dt;
  const int n_items = n_tiles * S;
  const int nkb = (int)(V / SC_BK);
  constexpr uint32_t stage_tx = 2 * SC_A_BYTES + (BN / 64) * SC_BOX_BYTES;
  if (threadIdx.x == 0) ctl_init(ctl, SC_STAGES);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapPhi);
    tma_prefetch_desc(&mapPlo);
    tma_prefetch_desc(&mapE);
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
  // the setup above is local; P, the tile maxima and done come from the kernels before
  pdl_wait();

  auto item_coords = [&](int w, int& split, int& rt, int& dt, int& kb0, int& kb1) {
    split = w / n_tiles;
    const int tile = w % n_tiles;
    rt = tile % n_rt;
    dt = tile / n_rt;
    kb0 = split * kb_per_split;
    kb1 = min(nkb, kb0 + kb_per_split);
  };

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_E = policy_evict_last(), pol_P = policy_evict_first();
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
        int split, rt, dt, kb0, kb1;
        item_coords(w, split, rt, dt, kb0, kb1);
        if (done && done[(rt * SC_BM) / L]) continue;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(smem_u32(&ctl.empty[stage]), phase ^ 1, abort_flag, err)) {
            ok = false;
            break;
          }
          const uint32_t sa = sbase + stage * SC_STAGE_BYTES;
          const uint32_t fb = smem_u32(&ctl.full[stage]);
          mbar_arrive_expect_tx(fb, stage_tx);
          tma_load_2d(sa, &mapPhi, fb, kb * SC_BK, rt * SC_BM, pol_P);
          tma_load_2d(sa + SC_A_BYTES, &mapPlo, fb, kb * SC_BK, rt * SC_BM, pol_P);
#pragma unroll
          for (int bx = 0; bx < BN / 64; ++bx)
            tma_load_2d(sa + 2 * SC_A_BYTES + bx * SC_BOX_BYTES, &mapE, fb, dt * BN + bx * 64,
                        kb * SC_BK, pol_E);
          ++issued;
          if (++stage == SC_STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) producer_drain(ctl, issued, SC_STAGES);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(SC_BM, BN, false, true);
      int stage = 0, cc = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
        int split, rt, dt, kb0, kb1;
        item_coords(w, split, rt, dt, kb0, kb1);
        if (done && done[(rt * SC_BM) / L]) continue;
        for (int c0 = kb0; c0 < kb1 && ok; c0 += CHUNK_KB, ++cc) {
          const int buf = cc & 1;
          const uint32_t par = (uint32_t)((cc >> 1) & 1);
          if (!mbar_wait(smem_u32(&ctl.tempty[buf]), par ^ 1, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dtm = tmem + (uint32_t)(buf * BN);
          const int c1 = min(kb1, c0 + CHUNK_KB);
          for (int kb = c0; kb < c1; ++kb) {
            if (!mbar_wait(smem_u32(&ctl.full[stage]), phase, abort_flag, err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            *(volatile int*)&ctl.consumed = ctl.consumed + 1;
            const uint32_t sa = sbase + stage * SC_STAGE_BYTES;
            const uint32_t sb = sa + 2 * SC_A_BYTES;
#pragma unroll
            for (int k = 0; k < SC_BK / 16; ++k) {
              // B = E tile, tokens x d-columns with d contiguous: MN-major, 64-column boxes
              // SC_BOX_BYTES apart (leading offset), 8-token groups 1024 B apart (stride offset).
              const uint64_t bdesc = sdesc_sw128(sb + k * 16 * 128, SC_BOX_BYTES, 1024);
              umma_bf16(dtm, sdesc_sw128(sa + 32 * k, 16, 1024), bdesc, idesc,
                        (kb != c0 || k != 0) ? 1u : 0u);
              umma_bf16(dtm, sdesc_sw128(sa + SC_A_BYTES + 32 * k, 16, 1024), bdesc, idesc, 1u);
            }
            umma_commit(smem_u32(&ctl.empty[stage]));
            if (++stage == SC_STAGES) {
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
  } else if (warp < 2 + kEpiWarps) {
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int cc = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      int split, rt, dt, kb0, kb1;
      item_coords(w, split, rt, dt, kb0, kb1);
      if (done && done[(rt * SC_BM) / L]) continue;
      float acc[COLS];
#pragma unroll
      for (int i = 0; i < COLS; ++i) acc[i] = 0.f;
      const int row = rt * SC_BM + q * 32 + lane;
      float mrun = -INFINITY, mnext = 0.f;
      if constexpr (SCALED) mnext = mtile_t[(size_t)(kb0 / CHUNK_KB) * R + row];
      for (int c0 = kb0; c0 < kb1; c0 += CHUNK_KB, ++cc) {
        float beta = 1.f;
        if constexpr (SCALED) {
          const float mg = mnext;
          // the next tile's maximum is loaded while this chunk is waited for
          if (c0 + CHUNK_KB < kb1) mnext = mtile_t[(size_t)(c0 / CHUNK_KB + 1) * R + row];
          if (mg > mrun) {
            const float alpha = expf(mrun - mg);
#pragma unroll
            for (int i = 0; i < COLS; ++i) acc[i] *= alpha;
            mrun = mg;
          }
          beta = expf(mg - mrun);
        }
        const int buf = cc & 1;
        const uint32_t par = (uint32_t)((cc >> 1) & 1);
        if (!mbar_wait(smem_u32(&ctl.tfull[buf]), par, abort_flag, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if constexpr (SCALED)
          tmem_accumulate_scaled<COLS>(tmem + (uint32_t)(buf * BN + half * COLS) + lane_base,
                                       acc, beta);
        else
          tmem_accumulate<COLS>(tmem + (uint32_t)(buf * BN + half * COLS) + lane_base, acc);
        tc_fence_before();
        mbar_arrive(smem_u32(&ctl.tempty[buf]));
      }
      if (!ok) break;
      if constexpr (SCALED)
        if (dt == 0 && half == 0) mref[(size_t)split * R + row] = mrun;
      float* orow = Opart + ((size_t)split * R + row) * d + (size_t)dt * BN + half * COLS;
#pragma unroll
      for (int v = 0; v < COLS / 4; ++v)
        *reinterpret_cast<float4*>(orow + 4 * v) =
            make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
    }
  }
  if (gw.best) gumbel_queue_warp(gw, V);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (gw.best && threadIdx.x == 0) gumbel_queue_release(gw);
}

int selfcond_bn(int d) { return d % 256 == 0 ? 256 : (d % 128 == 0 ? 128 : 64); }

}  // namespace

void tc_prepare_selfcond() {
  cudaFuncSetAttribute(k_selfcond_tc<256, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)SC_SMEM);
  cudaFuncSetAttribute(k_selfcond_tc<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)SC_SMEM);
  cudaFuncSetAttribute(k_selfcond_tc<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)SC_SMEM);
  cudaFuncSetAttribute(k_selfcond_tc<256, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)SC_SMEM);
  cudaFuncSetAttribute(k_selfcond_tc<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)SC_SMEM);
  cudaFuncSetAttribute(k_selfcond_tc<64, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)SC_SMEM);
}

int selfcond_tc_splits(int R, int64_t V, int d, int num_sms) {
  const int n_tiles = (R / SC_BM) * (d / selfcond_bn(d));
  const int nkb = (int)(V / SC_BK);
  int best_S = 1;
  double best_score = -1.0;
  for (int S = 1; S <= 64 && S <= nkb; ++S) {
    const int per = (nkb + S - 1) / S;
    if ((S - 1) * per >= nkb) continue;  // would leave an empty split
    if (per < 8 && S > 1) break;
    const long items = (long)n_tiles * S;
    const long waves = (items + num_sms - 1) / num_sms;
    const double eff = (double)items / (double)(waves * num_sms);
    const double score = eff - 0.004 * S;
    if (score > best_score + 1e-12) {
      best_score = score;
      best_S = S;
    }
  }
  return best_S;
}

cudaError_t launch_selfcond_tc(const uint16_t* Phi, const uint16_t* Plo, const uint16_t* E, int R,
                               int64_t V, int d, int L, const uint8_t* done, int S, float* Opart,
                               const float* mtile_t, float* mref, uint32_t* err,
                               const GumbelWork* gw, cudaStream_t st) {
  if (!tc_available()) return cudaErrorNotSupported;
  const int bn = selfcond_bn(d);
  CUtensorMap mPh, mPl, mE;
  if (!tc_make_map_bf16(&mPh, Phi, (uint64_t)R, (uint64_t)V, SC_BM, SC_BK) ||
      !tc_make_map_bf16(&mPl, Plo, (uint64_t)R, (uint64_t)V, SC_BM, SC_BK) ||
      !tc_make_map_bf16(&mE, E, (uint64_t)V, (uint64_t)d, SC_BK, 64))
    return cudaErrorInvalidValue;
  const int nkb = (int)(V / SC_BK);
  const bool scaled = mtile_t != nullptr;
  int per = (nkb + S - 1) / S;
  if (scaled) per = (per + SC_CHUNK_KB - 1) / SC_CHUNK_KB * SC_CHUNK_KB;  // splits start on a tile
  const int n_items = (R / SC_BM) * (d / bn) * S;
  // with the race every SM takes part (CTAs beyond the GEMM items only race)
  const int grid = gw ? tc_num_sms() : std::max(1, std::min(n_items, tc_num_sms()));
  GumbelWork g{};
  if (gw) g = *gw;
  cudaError_t e = cudaSuccess;
#define DS_SELFCOND_LAUNCH(BN, SC)                                                             \
  e = launch_k(k_selfcond_tc<BN, SC>, dim3(grid), dim3(SC_THREADS), SC_SMEM, st, mPh, mPl, mE, \
               R, V, d, L, S, per, done, Opart, mtile_t, mref, err, g)
  if (scaled) {
    if (bn == 256)
      DS_SELFCOND_LAUNCH(256, true);
    else if (bn == 128)
      DS_SELFCOND_LAUNCH(128, true);
    else
      DS_SELFCOND_LAUNCH(64, true);
  } else {
    if (bn == 256)
      DS_SELFCOND_LAUNCH(256, false);
    else if (bn == 128)
      DS_SELFCOND_LAUNCH(128, false);
    else
      DS_SELFCOND_LAUNCH(64, false);
  }
#undef DS_SELFCOND_LAUNCH
  return e;
}

}  // namespace ds
