// Fused tensor-core vocabulary pass of the sampler step on sm_103a: the logits GEMM, the softmax
// statistics, the bf16 hi/lo split of the probabilities and the self-conditioning GEMM in one
// persistent kernel, so that the HBM-bound logits work of some SMs runs under the tensor-bound
// self-conditioning work of the others.
//
// One CTA per SM, launched cooperatively (every CTA is resident, so the waits between CTAs end),
// 10 warps with the roles of ds_tc_common.cuh. After a producer item's last chunk the epilogue
// parks its fp32 sums in that chunk's TMEM buffer and reads them back 32 columns at a time, so
// the output phase runs with few registers. Work items come from two global queues:
//
//   producer item (row tile rt of 128 rows, vocabulary tile vt of 256 tokens):
//     z = H E^T over d (two-level accumulation), y = z / T_b. For each row and each of the
//     tile's two 128-token segments g: m_g = max y, l_g = sum exp(y - m_g),
//     a_g = sum exp(y - m_g)(y - m_g) and the lowest argmax; P_g = exp(y - m_g) as bf16 hi + lo
//     goes to global memory. Then the ready flag of (rt, vt) is released.
//   consumer item (range q of kvt vocabulary tiles, row tile rt, d tile dt of 256 columns):
//     acquires the ready flags of its tiles and accumulates
//       O_q[r, n] = sum_g exp(m_g - M_q) sum_{j in g} (P_hi + P_lo)[r, j] E[j, n]
//     (each segment is one TMEM chunk, promoted into registers scaled by exp(m_g - M), where M
//     is the running maximum; the registers are rescaled when M grows), then stores O_q and
//     M_q. The ranges' partials are summed, rescaled to the row maximum, in range order
//     afterwards (k_finalize), so s does not depend on timing.
// CTAs with blockIdx.x < producers start on the producer queue and move to the consumer queue
// when it runs dry. The Gumbel-max sample is drawn afterwards from the stored probabilities
// (k_gumbel_items, ds_rows.cu).
//
// Definitions: DiffusionGemma Technical Report, section 6 "Sampling" (full-precision softmax
// over the vocabulary and the self-conditioning embedding matmul).
#include <algorithm>
#include <climits>

#include "ds_tc_common.cuh"

namespace ds {
namespace {

using namespace tcpipe;

constexpr int VP_BM = 128, VP_BN = 256, VP_BK = 64;
constexpr int VP_COLS = VP_BN / 2;  // columns of one epilogue warp = one 128-token segment
constexpr int VP_CHUNK_KB = 2;      // K blocks per TMEM chunk (logits: 8 MMAs; s: 16 MMAs)
constexpr uint32_t VP_A_BYTES = VP_BM * VP_BK * 2;  // 16 KB
constexpr uint32_t VP_B_BYTES = VP_BN * VP_BK * 2;  // 32 KB
constexpr uint32_t VP_EBOX_BYTES = 64 * VP_BK * 2;  // 64 tokens x 64 d-columns
// Two rings over the same 192 KB: producer items stream H and E through four 48 KB stages
// (A = H, then B = E), consumer items P_hi, P_lo and E through three 64 KB stages. A CTA
// switches from the first to the second once, after every producer stage has been consumed.
constexpr int VP_PSTAGES = 4, VP_CSTAGES = 3;
constexpr uint32_t VP_PSTAGE_BYTES = VP_A_BYTES + VP_B_BYTES;
constexpr uint32_t VP_CSTAGE_BYTES = 2 * VP_A_BYTES + VP_B_BYTES;
constexpr uint32_t VP_RING_BYTES = VP_CSTAGES * VP_CSTAGE_BYTES;
static_assert(VP_PSTAGES * VP_PSTAGE_BYTES <= VP_RING_BYTES, "producer ring too large");
constexpr int VP_RING = 2;   // published work items
constexpr int VP_MRING = 4;  // segment maxima of consumer vocabulary tiles in flight
constexpr uint32_t VP_MRING_OFF = VP_RING_BYTES;
constexpr uint32_t VP_MSLOT_BYTES = 2 * VP_BM * 4;
constexpr size_t VP_SMEM = (size_t)VP_MRING_OFF + VP_MRING * VP_MSLOT_BYTES + 1024;
constexpr int kEnd = -1;
// control block: [0] producer queue, [1] consumer queue, [2] abort, [3] unused,
// then ready flags [n_rt * n_vt]
constexpr int kSyncHeader = 4;

struct VpArgs {
  int R, L, d, nk;
  int n_rt, n_vt, n_dt, n_seg;
  int kvt;
  int n_prod_items, n_cons_items, producers;
  int64_t V;
  const float* T;
  const uint8_t* done;
  const int32_t* step;
  uint64_t seed;
  uint16_t* Phi;   // [R, V]
  uint16_t* Plo;   // [R, V]
  ChunkStat* seg;  // [R, n_seg]
  float* mseg_t;   // [n_seg, R]
  float* Opart;    // [n_ranges, R, d]
  float* mref;     // [n_ranges, R]
  uint32_t* sync;
  uint32_t* err;
};

struct VpCtl {
  uint64_t pfull[VP_PSTAGES], pempty[VP_PSTAGES];
  uint64_t cfull[VP_CSTAGES], cempty[VP_CSTAGES];
  uint64_t tfull[2], tempty[2];
  uint64_t item_full[VP_RING], item_empty[VP_RING];
  uint64_t mfull[VP_MRING], mempty[VP_MRING];
  uint64_t epi;  // end of an item's output by all epilogue warps (bounded, unlike bar.sync)
  uint64_t mma_done;
  int items[VP_RING];
  uint32_t tmem_base;
  int abort;
  int consumed_p, consumed_c;  // stages consumed by the MMA thread (for the abort drain)
};

// Wait until *flag >= target (acquire). Gives up on the CTA's or the grid's abort flag, or
// after kWaitLimitNs (then raises both and sets the error word).
DS_DEV bool wait_at_least(const uint32_t* flag, uint32_t target, uint32_t* gabort,
                          volatile int* abort_flag, uint32_t* err) {
  if (ld_acquire_gpu(flag) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i) {
      __nanosleep(64);
      if (ld_acquire_gpu(flag) >= target) return true;
    }
    if (*abort_flag || *(volatile uint32_t*)gabort) {
      *abort_flag = 1;
      return false;
    }
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicExch(gabort, 1u);
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}

// After an abort: wait (bounded) for the copies issued into a ring but not consumed.
DS_DEV void drain_ring(uint64_t* full, int stages, int consumed, int issued) {
  for (int q = consumed; q < issued; ++q)
    mbar_wait_quiet(smem_u32(&full[q % stages]), (uint32_t)((q / stages) & 1));
}

struct ConsumerItem {
  int q, rt, dt, vt0, vt1;
};

DS_DEV ConsumerItem decode_consumer(const VpArgs& A, int c) {
  ConsumerItem it;
  const int tiles = A.n_rt * A.n_dt;
  it.q = c / tiles;
  const int t = c % tiles;
  it.rt = t % A.n_rt;
  it.dt = t / A.n_rt;
  it.vt0 = it.q * A.kvt;
  it.vt1 = min(A.n_vt, it.vt0 + A.kvt);
  return it;
}

// acc[OFF .. OFF + 32) -> 32 TMEM columns at taddr (this warp's lanes)
template <int OFF>
DS_DEV void park32(uint32_t taddr, const float (&acc)[VP_COLS]) {
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = acc[OFF + i];
  tmem_st_32cols(taddr + OFF, v);
}

__global__ void __launch_bounds__(kThreadsTC, 1)
    k_vocab_pass(const __grid_constant__ CUtensorMap mapH, const __grid_constant__ CUtensorMap mapEk,
                 const __grid_constant__ CUtensorMap mapEmn,
                 const __grid_constant__ CUtensorMap mapPhi,
                 const __grid_constant__ CUtensorMap mapPlo, const VpArgs A) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ VpCtl vc;
  uint8_t* smem = align1024(dyn_smem);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* const gabort = A.sync + 2;
  uint32_t* const ready = A.sync + kSyncHeader;

  if (threadIdx.x == 0) {
    for (int s = 0; s < VP_PSTAGES; ++s) {
      mbar_init(smem_u32(&vc.pfull[s]), 1);
      mbar_init(smem_u32(&vc.pempty[s]), 1);
    }
    for (int s = 0; s < VP_CSTAGES; ++s) {
      mbar_init(smem_u32(&vc.cfull[s]), 1);
      mbar_init(smem_u32(&vc.cempty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&vc.tfull[b]), 1);
      mbar_init(smem_u32(&vc.tempty[b]), 32 * kEpiWarps);
    }
    for (int s = 0; s < VP_RING; ++s) {
      mbar_init(smem_u32(&vc.item_full[s]), 1);
      mbar_init(smem_u32(&vc.item_empty[s]), 1 + kEpiWarps);
    }
    for (int s = 0; s < VP_MRING; ++s) {
      mbar_init(smem_u32(&vc.mfull[s]), 1);
      mbar_init(smem_u32(&vc.mempty[s]), kEpiWarps);
    }
    mbar_init(smem_u32(&vc.epi), kEpiWarps);
    mbar_init(smem_u32(&vc.mma_done), 1);
    vc.abort = 0;
    vc.consumed_p = 0;
    vc.consumed_c = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapH);
    tma_prefetch_desc(&mapEk);
    tma_prefetch_desc(&mapEmn);
    tma_prefetch_desc(&mapPhi);
    tma_prefetch_desc(&mapPlo);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&vc.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = vc.tmem_base;
  volatile int* abort_flag = &vc.abort;

  if (warp == 0) {
    // ---------------- scheduler + TMA producer (one thread) ----------------
    if (lane == 0) {
      const uint64_t pol_keep = policy_evict_last(), pol_once = policy_evict_first();
      int pstage = 0, cstage = 0, issued_p = 0, issued_c = 0, slot = 0, ms = 0;
      uint32_t pphase = 0, cphase = 0, rphase = 0, mphase = 0;
      bool producing = (int)blockIdx.x < A.producers, switched = false, ok = true;
      // next work item (kEnd when both queues are exhausted); items of done sequences skipped
      auto fetch = [&]() -> int {
        while (ok) {
          if (*(volatile uint32_t*)gabort) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          if (producing) {
            const int p = (int)atomicAdd(&A.sync[0], 1u);
            if (p >= A.n_prod_items) {
              producing = false;
              continue;
            }
            if (A.done && A.done[((p % A.n_rt) * VP_BM) / A.L]) continue;
            return p;
          }
          const int c = (int)atomicAdd(&A.sync[1], 1u);
          if (c >= A.n_cons_items) break;
          if (A.done && A.done[(decode_consumer(A, c).rt * VP_BM) / A.L]) continue;
          return A.n_prod_items + c;
        }
        return kEnd;
      };
      int next = fetch();
      for (;;) {
        if (!ok) break;
        const int code = next;
        if (!mbar_wait(smem_u32(&vc.item_empty[slot]), rphase ^ 1, abort_flag, A.err)) {
          ok = false;
          break;
        }
        vc.items[slot] = code;
        mbar_arrive(smem_u32(&vc.item_full[slot]));
        if (++slot == VP_RING) {
          slot = 0;
          rphase ^= 1;
        }
        if (code == kEnd) break;
        if (code < A.n_prod_items) {
          // claim the next item now and start pulling its E tile into L2, so that its loads
          // find it there
          next = fetch();
          if (next >= 0 && next < A.n_prod_items)
            for (int kc = 0; kc < A.nk; ++kc)
              tma_prefetch_l2_2d(&mapEk, kc * VP_BK, (next / A.n_rt) * VP_BN);
        }
        if (code < A.n_prod_items) {
          const int vt = code / A.n_rt, rt = code % A.n_rt;
          for (int kc = 0; kc < A.nk; ++kc) {
            if (!mbar_wait(smem_u32(&vc.pempty[pstage]), pphase ^ 1, abort_flag, A.err)) {
              ok = false;
              break;
            }
            const uint32_t sa = sbase + pstage * VP_PSTAGE_BYTES;
            const uint32_t fb = smem_u32(&vc.pfull[pstage]);
            mbar_arrive_expect_tx(fb, VP_PSTAGE_BYTES);
            tma_load_2d(sa, &mapH, fb, kc * VP_BK, rt * VP_BM, pol_keep);
            tma_load_2d(sa + VP_A_BYTES, &mapEk, fb, kc * VP_BK, vt * VP_BN, pol_keep);
            ++issued_p;
            if (++pstage == VP_PSTAGES) {
              pstage = 0;
              pphase ^= 1;
            }
          }
        } else {
          if (!switched) {
            // the consumer ring overlays the producer ring: every producer stage must have
            // been read by its MMAs first (use u of a stage completes phase u of its empty)
            for (int u = max(0, issued_p - VP_PSTAGES); u < issued_p && ok; ++u)
              ok = mbar_wait(smem_u32(&vc.pempty[u % VP_PSTAGES]),
                             (uint32_t)((u / VP_PSTAGES) & 1), abort_flag, A.err);
            if (!ok) break;
            switched = true;
          }
          const ConsumerItem it = decode_consumer(A, code - A.n_prod_items);
          for (int vt = it.vt0; vt < it.vt1 && ok; ++vt) {
            if (!wait_at_least(ready + it.rt * A.n_vt + vt, 1u, gabort, abort_flag, A.err)) {
              ok = false;
              break;
            }
            fence_proxy_async_global();
            // the two segment maxima of this tile for the 128 rows
            if (!mbar_wait(smem_u32(&vc.mempty[ms]), mphase ^ 1, abort_flag, A.err)) {
              ok = false;
              break;
            }
            const uint32_t mb = smem_u32(&vc.mfull[ms]);
            const uint32_t md = sbase + VP_MRING_OFF + ms * VP_MSLOT_BYTES;
            mbar_arrive_expect_tx(mb, VP_MSLOT_BYTES);
            bulk_load_1d(md, A.mseg_t + (size_t)(2 * vt) * A.R + it.rt * VP_BM, VP_BM * 4, mb);
            bulk_load_1d(md + VP_BM * 4, A.mseg_t + (size_t)(2 * vt + 1) * A.R + it.rt * VP_BM,
                         VP_BM * 4, mb);
            if (++ms == VP_MRING) {
              ms = 0;
              mphase ^= 1;
            }
            for (int kb = 4 * vt; kb < 4 * vt + 4; ++kb) {
              if (!mbar_wait(smem_u32(&vc.cempty[cstage]), cphase ^ 1, abort_flag, A.err)) {
                ok = false;
                break;
              }
              const uint32_t sa = sbase + cstage * VP_CSTAGE_BYTES;
              const uint32_t fb = smem_u32(&vc.cfull[cstage]);
              mbar_arrive_expect_tx(fb, VP_CSTAGE_BYTES);
              tma_load_2d(sa, &mapPhi, fb, kb * VP_BK, it.rt * VP_BM, pol_once);
              tma_load_2d(sa + VP_A_BYTES, &mapPlo, fb, kb * VP_BK, it.rt * VP_BM, pol_once);
#pragma unroll
              for (int bx = 0; bx < VP_BN / 64; ++bx)
                tma_load_2d(sa + 2 * VP_A_BYTES + bx * VP_EBOX_BYTES, &mapEmn, fb,
                            it.dt * VP_BN + bx * 64, kb * VP_BK, pol_keep);
              ++issued_c;
              if (++cstage == VP_CSTAGES) {
                cstage = 0;
                cphase ^= 1;
              }
            }
          }
          if (ok) next = fetch();
        }
        if (!ok) break;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicExch(gabort, 1u);
        drain_ring(vc.pfull, VP_PSTAGES, *(volatile int*)&vc.consumed_p, issued_p);
        drain_ring(vc.cfull, VP_CSTAGES, *(volatile int*)&vc.consumed_c, issued_c);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (one thread) ----------------
    if (lane == 0) {
      constexpr uint32_t idesc_lg = idesc_bf16_f32(VP_BM, VP_BN, false, false);
      constexpr uint32_t idesc_sc = idesc_bf16_f32(VP_BM, VP_BN, false, true);
      int pstage = 0, cstage = 0, cc = 0, slot = 0;
      uint32_t pphase = 0, cphase = 0, rphase = 0;
      bool ok = true;
      for (;;) {
        if (!mbar_wait(smem_u32(&vc.item_full[slot]), rphase, abort_flag, A.err)) break;
        const int code = vc.items[slot];
        mbar_arrive(smem_u32(&vc.item_empty[slot]));
        if (++slot == VP_RING) {
          slot = 0;
          rphase ^= 1;
        }
        if (code == kEnd) break;
        const bool prod = code < A.n_prod_items;
        int nkb;
        if (prod) {
          nkb = A.nk;
        } else {
          const ConsumerItem it = decode_consumer(A, code - A.n_prod_items);
          nkb = 4 * (it.vt1 - it.vt0);
        }
        for (int kb0 = 0; kb0 < nkb && ok; kb0 += VP_CHUNK_KB, ++cc) {
          const int buf = cc & 1;
          const uint32_t par = (uint32_t)((cc >> 1) & 1);
          if (!mbar_wait(smem_u32(&vc.tempty[buf]), par ^ 1, abort_flag, A.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dtm = tmem + (uint32_t)(buf * VP_BN);
          const int kb1 = min(nkb, kb0 + VP_CHUNK_KB);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (prod) {
              if (!mbar_wait(smem_u32(&vc.pfull[pstage]), pphase, abort_flag, A.err)) {
                ok = false;
                break;
              }
              tc_fence_after();
              *(volatile int*)&vc.consumed_p = vc.consumed_p + 1;
              const uint32_t sa = sbase + pstage * VP_PSTAGE_BYTES, sb = sa + VP_A_BYTES;
#pragma unroll
              for (int k = 0; k < VP_BK / 16; ++k)
                umma_bf16(dtm, sdesc_sw128(sa + 32 * k, 16, 1024),
                          sdesc_sw128(sb + 32 * k, 16, 1024), idesc_lg,
                          (kb != kb0 || k) ? 1u : 0u);
              umma_commit(smem_u32(&vc.pempty[pstage]));
              if (++pstage == VP_PSTAGES) {
                pstage = 0;
                pphase ^= 1;
              }
            } else {
              if (!mbar_wait(smem_u32(&vc.cfull[cstage]), cphase, abort_flag, A.err)) {
                ok = false;
                break;
              }
              tc_fence_after();
              *(volatile int*)&vc.consumed_c = vc.consumed_c + 1;
              const uint32_t sa = sbase + cstage * VP_CSTAGE_BYTES, sb = sa + 2 * VP_A_BYTES;
#pragma unroll
              for (int k = 0; k < VP_BK / 16; ++k) {
                // B = E tile, tokens x d-columns with d contiguous: MN-major, 64-column boxes
                // VP_EBOX_BYTES apart (leading offset), 8-token groups 1024 B apart (stride).
                const uint64_t bdesc = sdesc_sw128(sb + k * 16 * 128, VP_EBOX_BYTES, 1024);
                umma_bf16(dtm, sdesc_sw128(sa + 32 * k, 16, 1024), bdesc, idesc_sc,
                          (kb != kb0 || k) ? 1u : 0u);
                umma_bf16(dtm, sdesc_sw128(sa + VP_A_BYTES + 32 * k, 16, 1024), bdesc,
                          idesc_sc, 1u);
              }
              umma_commit(smem_u32(&vc.cempty[cstage]));
              if (++cstage == VP_CSTAGES) {
                cstage = 0;
                cphase ^= 1;
              }
            }
          }
          if (!ok) break;
          umma_commit(smem_u32(&vc.tfull[buf]));
        }
        if (!ok) break;
      }
      umma_commit(smem_u32(&vc.mma_done));
      mbar_wait_quiet(smem_u32(&vc.mma_done), 0);
    }
  } else {
    // ---------------- epilogue warps ----------------
    const int ew = warp - 2;
    const int q4 = warp & 3;    // TMEM lane quadrant this warp may access
    const int half = ew >> 2;   // column half of the tile
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const int rloc = q4 * 32 + lane;
    int cc = 0, slot = 0, ms = 0;
    uint32_t rphase = 0, mphase = 0, ephase = 0;
    bool ok = true;
    // all epilogue warps have passed this point of the current item (their global writes,
    // fenced before, are then ordered before whatever the caller publishes next)
    auto epi_barrier = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&vc.epi));
      const bool r = mbar_wait(smem_u32(&vc.epi), ephase, abort_flag, A.err);
      ephase ^= 1;
      return r;
    };
    for (;;) {
      if (!mbar_wait(smem_u32(&vc.item_full[slot]), rphase, abort_flag, A.err)) {
        ok = false;
        break;
      }
      const int code = vc.items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&vc.item_empty[slot]));
      if (++slot == VP_RING) {
        slot = 0;
        rphase ^= 1;
      }
      if (code == kEnd) break;
      float acc[VP_COLS];
#pragma unroll
      for (int i = 0; i < VP_COLS; ++i) acc[i] = 0.f;
      int held = 0;  // TMEM buffer of the item's last chunk, kept until its output is done
      if (code < A.n_prod_items) {
        // ---- producer item: logits, segment statistics, Gumbel race, P hi/lo ----
        const int vt = code / A.n_rt, rt = code % A.n_rt;
        const int n_ch = (A.nk + VP_CHUNK_KB - 1) / VP_CHUNK_KB;
        for (int ch = 0; ch < n_ch; ++ch, ++cc) {
          const int buf = cc & 1;
          const uint32_t par = (uint32_t)((cc >> 1) & 1);
          if (!mbar_wait(smem_u32(&vc.tfull[buf]), par, abort_flag, A.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          tmem_accumulate<VP_COLS>(tmem + (uint32_t)(buf * VP_BN + half * VP_COLS) + lane_base,
                                   acc);
          if (ch + 1 < n_ch) {
            tc_fence_before();
            mbar_arrive(smem_u32(&vc.tempty[buf]));
          } else {
            held = buf;
          }
        }
        if (!ok) break;
        const int row = rt * VP_BM + rloc;
        const int b = row / A.L;
        const float invT = 1.0f / A.T[b];
        const int64_t j0 = (int64_t)vt * VP_BN + half * VP_COLS;
        const int seg = (int)(j0 / VP_COLS);
        // y = z * (1/T) is monotone in z, so the max of y is the scaled max of z, at the same
        // lowest index.
        float zmax = -INFINITY;
        int arg = 0;
#pragma unroll
        for (int k = 0; k < VP_COLS; ++k) {
          if (acc[k] > zmax) {
            zmax = acc[k];
            arg = k;
          }
        }
        // y = z * (1/T) rounded once, as a value of its own (no fused multiply-add with the
        // subtraction below), so y - m is exactly 0 at the maximum
        const float m = __fmul_rn(zmax, invT);
        // park the fp32 sums in the held TMEM buffer and work through them 32 columns at a
        // time, so the output phase needs few registers
        const uint32_t tacc = tmem + (uint32_t)(held * VP_BN + half * VP_COLS) + lane_base;
        park32<0>(tacc, acc);
        park32<32>(tacc, acc);
        park32<64>(tacc, acc);
        park32<96>(tacc, acc);
        tmem_st_wait();
        float l = 0.f, a = 0.f;
        uint16_t* const phi = A.Phi + (size_t)row * A.V + j0;
        uint16_t* const plo = A.Plo + (size_t)row * A.V + j0;
#pragma unroll 1
        for (int bx = 0; bx < VP_COLS / 32; ++bx) {
          uint32_t zr[32];
          tmem_ld_32cols(tacc + (uint32_t)(bx * 32), zr);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float p[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float t = __fmul_rn(__uint_as_float(zr[c * 8 + e]), invT) - m;
              // exp(t) = 2^(t log2 e): within ~3e-6 relative for t > -30; 1 at the maximum
              p[e] = exp2_approx(t * 1.4426950408889634f);
              l += p[e];
              a = fmaf(p[e], t, a);
            }
            uint4 h, lo;
            split_bf16x2(p[0], p[1], h.x, lo.x);
            split_bf16x2(p[2], p[3], h.y, lo.y);
            split_bf16x2(p[4], p[5], h.z, lo.z);
            split_bf16x2(p[6], p[7], h.w, lo.w);
            *reinterpret_cast<uint4*>(phi + bx * 32 + c * 8) = h;
            *reinterpret_cast<uint4*>(plo + bx * 32 + c * 8) = lo;
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&vc.tempty[held]));
        A.seg[(size_t)row * A.n_seg + seg] = ChunkStat{m, l, a, (int32_t)(j0 + arg)};
        A.mseg_t[(size_t)seg * A.R + row] = m;
        __threadfence();
        if (!epi_barrier()) {
          ok = false;
          break;
        }
        if (ew == 0 && lane == 0) st_release_gpu(ready + rt * A.n_vt + vt, 1u);
      } else {
        // ---- consumer item: scaled self-conditioning partial, ordered add into O ----
        const ConsumerItem it = decode_consumer(A, code - A.n_prod_items);
        float mrun = -INFINITY, m0 = 0.f, m1 = 0.f;
        for (int g = 2 * it.vt0; g < 2 * it.vt1; ++g, ++cc) {
          if ((g & 1) == 0) {
            if (!mbar_wait(smem_u32(&vc.mfull[ms]), mphase, abort_flag, A.err)) {
              ok = false;
              break;
            }
            const float* mr = reinterpret_cast<const float*>(smem + VP_MRING_OFF +
                                                             ms * VP_MSLOT_BYTES);
            m0 = mr[rloc];
            m1 = mr[VP_BM + rloc];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&vc.mempty[ms]));
            if (++ms == VP_MRING) {
              ms = 0;
              mphase ^= 1;
            }
          }
          const float mg = (g & 1) ? m1 : m0;
          if (mg > mrun) {
            const float alpha = expf(mrun - mg);
#pragma unroll
            for (int k = 0; k < VP_COLS; ++k) acc[k] *= alpha;
            mrun = mg;
          }
          const float beta = expf(mg - mrun);
          const int buf = cc & 1;
          const uint32_t par = (uint32_t)((cc >> 1) & 1);
          if (!mbar_wait(smem_u32(&vc.tfull[buf]), par, abort_flag, A.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          tmem_accumulate_scaled<VP_COLS>(
              tmem + (uint32_t)(buf * VP_BN + half * VP_COLS) + lane_base, acc, beta);
          tc_fence_before();
          mbar_arrive(smem_u32(&vc.tempty[buf]));
        }
        if (!ok) break;
        const int row = it.rt * VP_BM + rloc;
        float4* orow = reinterpret_cast<float4*>(A.Opart + ((size_t)it.q * A.R + row) * A.d +
                                                 it.dt * VP_BN + half * VP_COLS);
#pragma unroll
        for (int v = 0; v < VP_COLS / 4; ++v)
          orow[v] = make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
        if (it.dt == 0 && half == 0) A.mref[(size_t)it.q * A.R + row] = mrun;
      }
    }
    if (!ok) {
      *abort_flag = 1;
      atomicExch(gabort, 1u);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int g_blocks_per_sm = 0;

}  // namespace

void tc_prepare_vocab_pass() {
  if (cudaFuncSetAttribute(k_vocab_pass, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)VP_SMEM) != cudaSuccess) {
    cudaGetLastError();
    g_blocks_per_sm = 0;
    return;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_vocab_pass, kThreadsTC, VP_SMEM) !=
      cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  g_blocks_per_sm = n;
}

VocabPassShape vocab_pass_shape(int R, int64_t V, int d, int num_sms, int producers) {
  VocabPassShape s{};
  if (!tc_available() || g_blocks_per_sm < 1 || d % VP_BN || R % VP_BM || V % VP_BN ||
      num_sms < 2)
    return s;
  s.n_rt = R / VP_BM;
  s.n_vt = (int)(V / VP_BN);
  s.n_dt = d / VP_BN;
  s.grid = num_sms;
  // consumer ranges: about nine consumer items per CTA
  const double tiles = (double)s.n_rt * s.n_dt;
  long kvt = std::lround((double)s.n_vt * tiles / (9.0 * s.grid));
  kvt = std::max(1L, std::min(kvt, (long)s.n_vt));
  // the finalize kernel combines at most kMaxSplits range partials
  kvt = std::max(kvt, (long)((s.n_vt + kMaxSplits - 1) / kMaxSplits));
  s.kvt = (int)kvt;
  s.n_ranges = (s.n_vt + s.kvt - 1) / s.kvt;
  if (producers <= 0) {
    // split in proportion to the work: a consumer token-column costs two MMA passes (hi, lo),
    // a producer one pass plus the Gumbel/split epilogue (about a third more)
    const double wp = 1.35 * d;
    const double wc = 2.0 * VP_BN * s.n_dt;
    producers = (int)std::lround(s.grid * wp / (wp + wc));
  }
  s.producers = std::max(1, std::min(producers, s.grid - 1));
  return s;
}

size_t vocab_pass_sync_words(const VocabPassShape& sh) {
  return (size_t)kSyncHeader + (size_t)sh.n_rt * sh.n_vt;
}

cudaError_t launch_vocab_pass_tc(const VocabPassShape& sh, const uint16_t* H, const uint16_t* E,
                                 int R, int64_t V, int d, int L, const float* T,
                                 const uint8_t* done, const int32_t* step, uint64_t seed,
                                 uint16_t* Phi, uint16_t* Plo, ChunkStat* seg, float* mseg_t,
                                 float* Opart, float* mref, uint32_t* sync, uint32_t* err,
                                 cudaStream_t st) {
  if (!tc_available() || sh.grid < 2) return cudaErrorNotSupported;
  CUtensorMap mH, mEk, mEmn, mPh, mPl;
  if (!tc_make_map_bf16(&mH, H, (uint64_t)R, (uint64_t)d, VP_BM, VP_BK) ||
      !tc_make_map_bf16(&mEk, E, (uint64_t)V, (uint64_t)d, VP_BN, VP_BK) ||
      !tc_make_map_bf16(&mEmn, E, (uint64_t)V, (uint64_t)d, VP_BK, 64) ||
      !tc_make_map_bf16(&mPh, Phi, (uint64_t)R, (uint64_t)V, VP_BM, VP_BK) ||
      !tc_make_map_bf16(&mPl, Plo, (uint64_t)R, (uint64_t)V, VP_BM, VP_BK))
    return cudaErrorInvalidValue;
  VpArgs a{};
  a.R = R;
  a.L = L;
  a.d = d;
  a.nk = d / VP_BK;
  a.n_rt = sh.n_rt;
  a.n_vt = sh.n_vt;
  a.n_dt = sh.n_dt;
  a.n_seg = (int)(V / kVpSegment);
  a.kvt = sh.kvt;
  a.n_prod_items = sh.n_rt * sh.n_vt;
  a.n_cons_items = sh.n_ranges * sh.n_rt * sh.n_dt;
  a.producers = sh.producers;
  a.V = V;
  a.T = T;
  a.done = done;
  a.step = step;
  a.seed = seed;
  a.Phi = Phi;
  a.Plo = Plo;
  a.seg = seg;
  a.mseg_t = mseg_t;
  a.Opart = Opart;
  a.mref = mref;
  a.sync = sync;
  a.err = err;
  cudaError_t e = cudaMemsetAsync(sync, 0, vocab_pass_sync_words(sh) * sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)sh.grid);
  cfg.blockDim = dim3(kThreadsTC);
  cfg.dynamicSmemBytes = VP_SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_vocab_pass, mH, mEk, mEmn, mPh, mPl, a);
}

}  // namespace ds
