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
#include <cstdlib>

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
// CTA pair (BN = 256): each CTA stages its 128 rows of P hi and lo and 128 of the tile's 256
// d-columns of E (48 KB a stage instead of 64), so an SM takes in 3/4 of the operand bytes per
// MAC of a one-CTA tile and holds four stages in the same shared memory. The one-CTA kernel
// measured bound by that operand stream as much as by its MMAs (same box, B = 1, V = 262144,
// d = 2816, the GEMM alone: 452 us; its MMAs on operands already in shared memory 395 us; all
// operands loaded but half the MMAs 393 us; 48 KB a k-block loaded instead of 64, 432 us).
constexpr int SC2_STAGES = 4;
constexpr uint32_t SC2_STAGE_BYTES = 2 * SC_A_BYTES + (SC_BN_MAX / 128) * SC_BOX_BYTES;
constexpr size_t SC2_SMEM = (size_t)SC2_STAGES * SC2_STAGE_BYTES + 1024;
static_assert(SC2_STAGES <= kMaxStages && SC_STAGES <= kMaxStages, "stages");
// the pipeline's warps (producer, MMA, 8 epilogue) and two racing warps
constexpr int SC_THREADS = kThreadsTC + 64;

// PAIR: launched in clusters of two CTAs; a work item is 256 rows (the CTAs' row tiles 2i and
// 2i + 1) x BN = 256 d-columns x one vocabulary split, computed by M = 256 MMAs that the even CTA
// issues for both, each CTA holding the accumulator of its own 128 rows (its epilogue is the
// one-CTA epilogue). Needs R % 256 == 0 and BN == 256.
template <int BN, bool SCALED, bool PAIR>
__global__ void __launch_bounds__(SC_THREADS, 1)
    k_selfcond_tc(const __grid_constant__ CUtensorMap mapPhi,
                  const __grid_constant__ CUtensorMap mapPlo,
                  const __grid_constant__ CUtensorMap mapE, int R, int64_t V, int d, int L,
                  int S, int kb_per_split, const uint8_t* __restrict__ done,
                  float* __restrict__ Opart, const float* __restrict__ mtile_t,
                  float* __restrict__ mref, uint32_t* err, const __grid_constant__ GumbelWork gw) {
  static_assert(!PAIR || BN == 256, "pair tiles are 256 d-columns wide");
  constexpr int COLS = BN / 2;
  constexpr int CHUNK_KB = SC_CHUNK_KB;  // 4 K blocks = one 256-token tile
  static_assert(CHUNK_KB * SC_BK == 256, "a chunk is one tile of the P reference maxima");
  constexpr int STAGES = PAIR ? SC2_STAGES : SC_STAGES;
  constexpr uint32_t STAGE_BYTES = PAIR ? SC2_STAGE_BYTES : SC_STAGE_BYTES;
  constexpr int ROWS = PAIR ? 2 * SC_BM : SC_BM;  // rows of a work item
  constexpr int EBOX = PAIR ? BN / 128 : BN / 64;  // 64-column boxes of E a CTA stages
  extern __shared__ uint8_t dyn_smem[];
  __shared__ Ctl ctl;
  uint8_t* smem = align1024(dyn_smem);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int n_units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int n_it = R / ROWS, n_dt = d / BN;
  const int n_tiles = n_it * n_dt;
  const int n_items = n_tiles * S;
  const int nkb = (int)(V / SC_BK);
  constexpr uint32_t stage_tx = 2 * SC_A_BYTES + EBOX * SC_BOX_BYTES;
  if (threadIdx.x == 0)  // pair: one arrival per epilogue warp of both CTAs releases a buffer
    ctl_init(ctl, STAGES, PAIR ? 2 * kEpiWarps : 32 * kEpiWarps);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapPhi);
    tma_prefetch_desc(&mapPlo);
    tma_prefetch_desc(&mapE);
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
  // the setup above is local; P, the tile maxima and done come from the kernels before
  pdl_wait();

  // splits in reverse vocabulary order: the logits kernel has just written the end of P, so
  // the first wave finds part of it in L2
  auto item_coords = [&](int w, int& split, int& it, int& dt, int& kb0, int& kb1) {
    split = (S - 1) - w / n_tiles;
    const int tile = w % n_tiles;
    it = tile % n_it;
    dt = tile / n_it;
    kb0 = split * kb_per_split;
    kb1 = min(nkb, kb0 + kb_per_split);
  };
  // (pair: both CTAs skip exactly the same items)
  auto skip = [&](int it) { return rows_done(done, it * ROWS, ROWS, L); };

  if (warp == 0) {
    if (lane == 0) {
      // P tiles are read by every d-tile item of their split (items of one split run side by
      // side) and kept in L2; an E tile is read once (pair) or twice, in the same wave. Same box,
      // B = 1: E evict-last / P evict-first 0.501 ms (with the race), E evict-first / P
      // evict-last 0.472 ms.
      const uint64_t pol_E = policy_evict_first(), pol_P = policy_evict_last();
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int w = unit; w < n_items && ok; w += n_units) {
        int split, it, dt, kb0, kb1;
        item_coords(w, split, it, dt, kb0, kb1);
        if (skip(it)) continue;
        const int rt = PAIR ? 2 * it + (int)rank : it;
        const int e_col = dt * BN + (PAIR ? (int)rank * (BN / 2) : 0);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(smem_u32(&ctl.empty[stage]), phase ^ 1, abort_flag, err)) {
            ok = false;
            break;
          }
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint32_t fb = smem_u32(&ctl.full[stage]);
          if constexpr (PAIR) {
            // both CTAs' copies complete on the even CTA's barrier, which expects all of them
            if (rank == 0) mbar_arrive_expect_tx(fb, 2 * stage_tx);
            const uint32_t fb0 = mapa_shared(fb, 0);
            tma_load_2d_pair(sa, &mapPhi, fb0, kb * SC_BK, rt * SC_BM, pol_P);
            tma_load_2d_pair(sa + SC_A_BYTES, &mapPlo, fb0, kb * SC_BK, rt * SC_BM, pol_P);
#pragma unroll
            for (int bx = 0; bx < EBOX; ++bx)
              tma_load_2d_pair(sa + 2 * SC_A_BYTES + bx * SC_BOX_BYTES, &mapE, fb0,
                               e_col + bx * 64, kb * SC_BK, pol_E);
          } else {
            mbar_arrive_expect_tx(fb, stage_tx);
            tma_load_2d(sa, &mapPhi, fb, kb * SC_BK, rt * SC_BM, pol_P);
            tma_load_2d(sa + SC_A_BYTES, &mapPlo, fb, kb * SC_BK, rt * SC_BM, pol_P);
#pragma unroll
            for (int bx = 0; bx < EBOX; ++bx)
              tma_load_2d(sa + 2 * SC_A_BYTES + bx * SC_BOX_BYTES, &mapE, fb, e_col + bx * 64,
                          kb * SC_BK, pol_E);
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
      constexpr uint32_t idesc = idesc_bf16_f32(ROWS, BN, false, true);
      int stage = 0, cc = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int w = unit; w < n_items && ok; w += n_units) {
        int split, it, dt, kb0, kb1;
        item_coords(w, split, it, dt, kb0, kb1);
        if (skip(it)) continue;
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
            const uint32_t sa = sbase + stage * STAGE_BYTES;
            const uint32_t sb = sa + 2 * SC_A_BYTES;
#pragma unroll
            for (int k = 0; k < SC_BK / 16; ++k) {
              // B = E tile, tokens x d-columns with d contiguous: MN-major, 64-column boxes
              // SC_BOX_BYTES apart (leading offset), 8-token groups 1024 B apart (stride
              // offset); pair: each CTA holds its half of the tile's columns this way
              const uint64_t bdesc = sdesc_sw128(sb + k * 16 * 128, SC_BOX_BYTES, 1024);
              const uint64_t ahi = sdesc_sw128(sa + 32 * k, 16, 1024);
              const uint64_t alo = sdesc_sw128(sa + SC_A_BYTES + 32 * k, 16, 1024);
              const uint32_t acc_in = (kb != c0 || k != 0) ? 1u : 0u;
              if constexpr (PAIR) {
                umma_bf16_pair(dtm, ahi, bdesc, idesc, acc_in);
                umma_bf16_pair(dtm, alo, bdesc, idesc, 1u);
              } else {
                umma_bf16(dtm, ahi, bdesc, idesc, acc_in);
                umma_bf16(dtm, alo, bdesc, idesc, 1u);
              }
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
  } else if (warp < 2 + kEpiWarps) {
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    // pair: the TMEM buffers are released on the even CTA's barriers, once per warp
    const uint32_t tempty0 = PAIR ? mapa_shared(smem_u32(&ctl.tempty[0]), 0) : 0u;
    const uint32_t tempty1 = PAIR ? mapa_shared(smem_u32(&ctl.tempty[1]), 0) : 0u;
    int cc = 0;
    bool ok = true;
    for (int w = unit; w < n_items && ok; w += n_units) {
      int split, it, dt, kb0, kb1;
      item_coords(w, split, it, dt, kb0, kb1);
      if (skip(it)) continue;
      const int rt = PAIR ? 2 * it + (int)rank : it;
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
        if constexpr (PAIR) {
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(buf ? tempty1 : tempty0);
        } else {
          mbar_arrive(smem_u32(&ctl.tempty[buf]));
        }
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
  // pair: neither CTA frees its TMEM or exits while the other may still use its barriers,
  // shared memory or TMEM
  if constexpr (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, 512);
    else tmem_dealloc(tmem, 512);
  }
  if (gw.best && threadIdx.x == 0) gumbel_queue_release(gw);
}

int selfcond_bn(int d) { return d % 256 == 0 ? 256 : (d % 128 == 0 ? 128 : 64); }

}  // namespace

// Clusters of the pair kernel that can be resident at once (a TPC with an SM unavailable holds
// none).
static int g_sc_pairs_resident = 1;

void tc_prepare_selfcond() {
#define DS_SELFCOND_ATTR(BN, SC, PR)                                                          \
  cudaFuncSetAttribute(k_selfcond_tc<BN, SC, PR>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                       (int)(PR ? SC2_SMEM : SC_SMEM))
  DS_SELFCOND_ATTR(256, false, false);
  DS_SELFCOND_ATTR(128, false, false);
  DS_SELFCOND_ATTR(64, false, false);
  DS_SELFCOND_ATTR(256, true, false);
  DS_SELFCOND_ATTR(128, true, false);
  DS_SELFCOND_ATTR(64, true, false);
  DS_SELFCOND_ATTR(256, false, true);
  DS_SELFCOND_ATTR(256, true, true);
#undef DS_SELFCOND_ATTR
  // (runs inside the one-time setup that tc_num_sms waits for, so it asks the device itself)
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::max(2, sms - sms % 2));
  cfg.blockDim = dim3(SC_THREADS);
  cfg.dynamicSmemBytes = SC2_SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_selfcond_tc<256, true, true>, &cfg) != cudaSuccess ||
      n < 1) {
    cudaGetLastError();
    n = std::max(1, sms / 2);
  }
  g_sc_pairs_resident = n;
}

// The pair kernel serves tiles of 256 d-columns over row pairs (DS_SELFCOND_PAIR=0 in the
// environment keeps the one-CTA kernel, for measurements).
static bool selfcond_pair(int R, int d) {
  static const bool on = [] {
    const char* e = getenv("DS_SELFCOND_PAIR");
    return !(e && e[0] == '0');
  }();
  return on && R % (2 * SC_BM) == 0 && d % 256 == 0 && tc_num_sms() >= 2;
}

int selfcond_tc_splits(int R, int64_t V, int d, int num_sms) {
  const int n_tiles = (R / SC_BM) * (d / selfcond_bn(d));
  // (pair: items of two row tiles on two CTAs, so the same count per CTA)
  if (selfcond_pair(R, d)) num_sms = std::min(num_sms, 2 * g_sc_pairs_resident);
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
  GumbelWork g{};
  if (gw) g = *gw;
  if (selfcond_pair(R, d)) {
    // with the race every resident pair takes part (pairs beyond the GEMM items only race)
    const int n_items = (R / (2 * SC_BM)) * (d / 256) * S;
    const int pairs = gw ? g_sc_pairs_resident : std::max(1, std::min(n_items, g_sc_pairs_resident));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(SC_THREADS);
    cfg.dynamicSmemBytes = SC2_SMEM;
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
    if (scaled)
      return cudaLaunchKernelEx(&cfg, k_selfcond_tc<256, true, true>, mPh, mPl, mE, R, V, d, L, S,
                                per, done, Opart, mtile_t, mref, err, g);
    return cudaLaunchKernelEx(&cfg, k_selfcond_tc<256, false, true>, mPh, mPl, mE, R, V, d, L, S,
                              per, done, Opart, mtile_t, mref, err, g);
  }
  const int n_items = (R / SC_BM) * (d / bn) * S;
  // with the race every SM takes part (CTAs beyond the GEMM items only race)
  const int grid = gw ? tc_num_sms() : std::max(1, std::min(n_items, tc_num_sms()));
  cudaError_t e = cudaSuccess;
#define DS_SELFCOND_LAUNCH(BN, SC)                                                    \
  e = launch_k(k_selfcond_tc<BN, SC, false>, dim3(grid), dim3(SC_THREADS), SC_SMEM, st, mPh, \
               mPl, mE, R, V, d, L, S, per, done, Opart, mtile_t, mref, err, g)
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
