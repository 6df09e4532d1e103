// Tensor-core (tcgen05 / TMEM / TMA) GEMMs of the sampler step on sm_103a.
//
//   logits:          Y[r, j] = (sum_k H[r, k] E[j, k]) / T_b    bf16 x bf16 -> fp32
//   self-condition:  O_s[r, n] = sum_{j in split s} (P_hi + P_lo)[r, j] E[j, n]
//                    where P_hi + P_lo = exp(y - m) split into two bf16 terms, so the product
//                    keeps ~16 significant bits of the probabilities (a single bf16 keeps 8).
//
// Definitions: DiffusionGemma Technical Report, section 6 "Sampling" (logits and softmax over
// the full vocabulary in full precision; the self-conditioning embedding matmul).
//
// Structure (both kernels): one persistent CTA per SM, 10 warps.
//   warp 0  one thread issues TMA copies of the operand tiles into a ring of shared-memory
//           stages (128-byte swizzle), completion counted on "full" mbarriers;
//   warp 1  allocates 512 TMEM columns; one thread issues tcgen05.mma into one of two TMEM
//           accumulators and commits "empty" (stage reusable) and "tmem full" barriers;
//   warps 2-9 drain the other accumulator (tcgen05.ld, lane = row) into fp32 registers while
//           the next chunk's MMAs run, then arrive on "tmem empty".
// Every wait is bounded; on a time-out the CTA raises an abort flag, records the device error
// word, waits (bounded) for its copies and MMAs in flight, frees TMEM and exits.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "ds_internal.h"

namespace ds {
namespace {

constexpr uint64_t kDrainLimitNs = 200000000ull;
constexpr int kEpiWarps = 8;
constexpr int kThreadsTC = 64 + 32 * kEpiWarps;

struct Ctl {
  uint64_t full[4];
  uint64_t empty[4];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  int consumed;
};

DS_DEV uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Bounded wait that ignores the abort flag (used while draining after an abort).
DS_DEV bool mbar_wait_quiet(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > kDrainLimitNs) return false;
  return true;
}

DS_DEV void ctl_init(Ctl& c, int stages) {
  for (int s = 0; s < stages; ++s) {
    mbar_init(smem_u32(&c.full[s]), 1);
    mbar_init(smem_u32(&c.empty[s]), 1);
  }
  for (int b = 0; b < 2; ++b) {
    mbar_init(smem_u32(&c.tfull[b]), 1);
    mbar_init(smem_u32(&c.tempty[b]), 32 * kEpiWarps);
  }
  mbar_init(smem_u32(&c.mma_done), 1);
  c.abort = 0;
  c.consumed = 0;
  fence_mbar_init();
}

// After an abort: wait for the copies issued but not consumed by the MMA thread.
DS_DEV void producer_drain(Ctl& c, int issued, int stages) {
  const int consumed = *(volatile int*)&c.consumed;
  for (int q = consumed; q < issued; ++q)
    mbar_wait_quiet(smem_u32(&c.full[q % stages]), (uint32_t)((q / stages) & 1));
}

// ------------------------------------------------------------------------------------------
// Two-level accumulation. The tensor core's fp32 accumulator rounds toward zero, so its error
// grows linearly with the number of MMAs accumulated into it. Each tile is therefore
// accumulated in short chunks: the MMA thread accumulates one chunk into one of two TMEM
// buffers while the epilogue warps add the other buffer into fp32 registers (round to nearest),
// so no TMEM accumulation chain is longer than one chunk.
// Epilogue warps: warp w >= 2 reads TMEM lane quadrant (w % 4) and column half (w - 2) / 4.
// ------------------------------------------------------------------------------------------

// Add COLS fp32 TMEM columns starting at taddr (this warp's 32 lanes) to acc[0..COLS).
// Loads go 16 columns at a time to keep register pressure low next to the accumulator
// (registers are charged per group of four warps, so a 10-warp CTA gets at most 168 each).
template <int COLS>
DS_DEV void tmem_accumulate(uint32_t taddr, float (&acc)[COLS]) {
#pragma unroll
  for (int c = 0; c < COLS / 16; ++c) {
    uint32_t r[16];
    tmem_ld_16cols(taddr + (uint32_t)(c * 16), r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[c * 16 + i] += __uint_as_float(r[i]);
  }
}

// ------------------------------------------------------------------------------------------
// logits (+ softmax statistics of each 128-token segment of a row)
// ------------------------------------------------------------------------------------------
constexpr int LG_BM = 128, LG_BN = 256, LG_BK = 64, LG_STAGES = 4, LG_CHUNK_KB = 2;
constexpr int LG_COLS = LG_BN / 2;
constexpr uint32_t LG_A_BYTES = LG_BM * LG_BK * 2;
constexpr uint32_t LG_B_BYTES = LG_BN * LG_BK * 2;
constexpr uint32_t LG_STAGE_BYTES = LG_A_BYTES + LG_B_BYTES;
constexpr size_t LG_SMEM = (size_t)LG_STAGES * LG_STAGE_BYTES + 1024;

__global__ void __launch_bounds__(kThreadsTC, 1)
    k_logits_tc(const __grid_constant__ CUtensorMap mapH, const __grid_constant__ CUtensorMap mapE,
                int R, int64_t V, int d, int L, const float* __restrict__ T,
                const uint8_t* __restrict__ done, float* __restrict__ Y,
                ChunkStat* __restrict__ seg_stats, uint32_t* err) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ Ctl ctl;
  uint8_t* smem = align1024(dyn_smem);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_rt = R / LG_BM;
  const int n_ct = (int)(V / LG_BN);
  const int n_tiles = n_rt * n_ct;
  const int nk = d / LG_BK;
  const int n_ch = (nk + LG_CHUNK_KB - 1) / LG_CHUNK_KB;
  if (threadIdx.x == 0) ctl_init(ctl, LG_STAGES);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapH);
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
    int cc = 0;
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
      // y = z / T (as z * (1/T)); the segment's max, argmax (lowest token), sum of exp(y - m)
      // and sum of exp(y - m) (y - m)
      const float invT = 1.0f / T[b];
      const int row = rt * LG_BM + q * 32 + lane;
      const int64_t j0 = (int64_t)ct * LG_BN + half * LG_COLS;
      // (x * invT is monotone in x for invT > 0, so the max of the scaled values is the
      // scaled max, at the same lowest index)
      float zmax = -INFINITY;
      int arg = 0;
#pragma unroll
      for (int i = 0; i < LG_COLS; ++i) {
        if (acc[i] > zmax) {
          zmax = acc[i];
          arg = i;
        }
      }
      const float m = zmax * invT;
      float l = 0.f, a = 0.f;
      float* yrow = Y + (size_t)row * V + j0;
#pragma unroll
      for (int v = 0; v < LG_COLS / 4; ++v) {
        float y4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          y4[e] = acc[4 * v + e] * invT;
          const float t = y4[e] - m;
          const float x = expf(t);
          l += x;
          a = fmaf(x, t, a);
        }
        *reinterpret_cast<float4*>(yrow + 4 * v) = make_float4(y4[0], y4[1], y4[2], y4[3]);
      }
      seg_stats[(size_t)row * (V / LG_COLS) + (j0 / LG_COLS)] =
          ChunkStat{m, l, a, (int32_t)(j0 + arg)};
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------------------------------
// self-conditioning partials
// ------------------------------------------------------------------------------------------
constexpr int SC_BM = 128, SC_BK = 64, SC_STAGES = 3, SC_BN_MAX = 256, SC_CHUNK_KB = 4;
constexpr uint32_t SC_A_BYTES = SC_BM * SC_BK * 2;        // one of hi / lo
constexpr uint32_t SC_BOX_BYTES = 64 * SC_BK * 2;          // 64 d-columns x 64 tokens
constexpr uint32_t SC_STAGE_BYTES = 2 * SC_A_BYTES + (SC_BN_MAX / 64) * SC_BOX_BYTES;
constexpr size_t SC_SMEM = (size_t)SC_STAGES * SC_STAGE_BYTES + 1024;

template <int BN>
__global__ void __launch_bounds__(kThreadsTC, 1)
    k_selfcond_tc(const __grid_constant__ CUtensorMap mapPhi,
                  const __grid_constant__ CUtensorMap mapPlo,
                  const __grid_constant__ CUtensorMap mapE, int R, int64_t V, int d, int L,
                  int S, int kb_per_split, const uint8_t* __restrict__ done,
                  float* __restrict__ Opart, uint32_t* err) {
  constexpr int COLS = BN / 2;
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
        for (int c0 = kb0; c0 < kb1 && ok; c0 += SC_CHUNK_KB, ++cc) {
          const int buf = cc & 1;
          const uint32_t par = (uint32_t)((cc >> 1) & 1);
          if (!mbar_wait(smem_u32(&ctl.tempty[buf]), par ^ 1, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dtm = tmem + (uint32_t)(buf * BN);
          const int c1 = min(kb1, c0 + SC_CHUNK_KB);
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
  } else {
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
      for (int c0 = kb0; c0 < kb1; c0 += SC_CHUNK_KB, ++cc) {
        const int buf = cc & 1;
        const uint32_t par = (uint32_t)((cc >> 1) & 1);
        if (!mbar_wait(smem_u32(&ctl.tfull[buf]), par, abort_flag, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_accumulate<COLS>(tmem + (uint32_t)(buf * BN + half * COLS) + lane_base, acc);
        tc_fence_before();
        mbar_arrive(smem_u32(&ctl.tempty[buf]));
      }
      if (!ok) break;
      const int row = rt * SC_BM + q * 32 + lane;
      float* orow = Opart + ((size_t)split * R + row) * d + (size_t)dt * BN + half * COLS;
#pragma unroll
      for (int v = 0; v < COLS / 4; ++v)
        *reinterpret_cast<float4*>(orow + 4 * v) =
            make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
int g_sms = 0;

void resolve() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
  cudaFuncSetAttribute(k_logits_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LG_SMEM);
  cudaFuncSetAttribute(k_selfcond_tc<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)SC_SMEM);
  cudaFuncSetAttribute(k_selfcond_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)SC_SMEM);
  cudaFuncSetAttribute(k_selfcond_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)SC_SMEM);
}

// 2-D bf16 tensor map over a row-major [rows, cols] array, box [box_rows, box_cols], 128 B swizzle.
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
              uint32_t box_cols) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int selfcond_bn(int d) { return d % 256 == 0 ? 256 : (d % 128 == 0 ? 128 : 64); }

}  // namespace

bool tc_available() {
  std::call_once(g_once, resolve);
  return g_encode != nullptr;
}

int tc_num_sms() {
  std::call_once(g_once, resolve);
  return g_sms;
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

cudaError_t launch_logits_tc(const uint16_t* H, const uint16_t* E, int R, int64_t V, int d, int L,
                             const float* T, const uint8_t* done, float* Y, ChunkStat* seg_stats,
                             uint32_t* err, cudaStream_t st) {
  if (!tc_available()) return cudaErrorNotSupported;
  CUtensorMap mH, mE;
  if (!make_map(&mH, H, (uint64_t)R, (uint64_t)d, LG_BM, LG_BK) ||
      !make_map(&mE, E, (uint64_t)V, (uint64_t)d, LG_BN, LG_BK))
    return cudaErrorInvalidValue;
  const int n_tiles = (R / LG_BM) * (int)(V / LG_BN);
  const int grid = std::max(1, std::min(n_tiles, g_sms));
  k_logits_tc<<<grid, kThreadsTC, LG_SMEM, st>>>(mH, mE, R, V, d, L, T, done, Y, seg_stats, err);
  return cudaGetLastError();
}

cudaError_t launch_selfcond_tc(const uint16_t* Phi, const uint16_t* Plo, const uint16_t* E, int R,
                               int64_t V, int d, int L, const uint8_t* done, int S, float* Opart,
                               uint32_t* err, cudaStream_t st) {
  if (!tc_available()) return cudaErrorNotSupported;
  const int bn = selfcond_bn(d);
  CUtensorMap mPh, mPl, mE;
  if (!make_map(&mPh, Phi, (uint64_t)R, (uint64_t)V, SC_BM, SC_BK) ||
      !make_map(&mPl, Plo, (uint64_t)R, (uint64_t)V, SC_BM, SC_BK) ||
      !make_map(&mE, E, (uint64_t)V, (uint64_t)d, SC_BK, 64))
    return cudaErrorInvalidValue;
  const int nkb = (int)(V / SC_BK);
  const int per = (nkb + S - 1) / S;
  const int n_items = (R / SC_BM) * (d / bn) * S;
  const int grid = std::max(1, std::min(n_items, g_sms));
  if (bn == 256)
    k_selfcond_tc<256><<<grid, kThreadsTC, SC_SMEM, st>>>(mPh, mPl, mE, R, V, d, L, S, per, done,
                                                          Opart, err);
  else if (bn == 128)
    k_selfcond_tc<128><<<grid, kThreadsTC, SC_SMEM, st>>>(mPh, mPl, mE, R, V, d, L, S, per, done,
                                                          Opart, err);
  else
    k_selfcond_tc<64><<<grid, kThreadsTC, SC_SMEM, st>>>(mPh, mPl, mE, R, V, d, L, S, per, done,
                                                         Opart, err);
  return cudaGetLastError();
}

}  // namespace ds
