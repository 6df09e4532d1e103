// Shared pieces of the tensor-core (tcgen05 / TMEM / TMA) kernels of the sampler step:
// the control block of the warp-specialised pipeline, bounded waits used while draining, and
// the promotion of short TMEM accumulation chains into fp32 registers.
//
// Structure of both kernels: one persistent CTA per SM, 10 warps (the self-conditioning kernel
// adds two that run the Gumbel-max race beside its GEMM).
//   warp 0  one thread issues TMA copies of the operand tiles into a ring of shared-memory
//           stages (128-byte swizzle), completion counted on "full" mbarriers;
//   warp 1  allocates 512 TMEM columns; one thread issues tcgen05.mma into one of two TMEM
//           accumulators and commits "empty" (stage reusable) and "tmem full" barriers;
//   warps 2-9 drain the other accumulator (tcgen05.ld, lane = row) into fp32 registers while
//           the next chunk's MMAs run, then arrive on "tmem empty".
// Every wait is bounded; on a time-out the CTA raises an abort flag, records the device error
// word, waits (bounded) for its copies and MMAs in flight, frees TMEM and exits.
//
// Two-level accumulation. The tensor core's fp32 accumulator rounds toward zero, so its error
// grows linearly with the number of MMAs accumulated into it. Each tile is therefore
// accumulated in short chunks: the MMA thread accumulates one chunk into one of two TMEM
// buffers while the epilogue warps add the other buffer into fp32 registers (round to nearest),
// so no TMEM accumulation chain is longer than one chunk.
// Epilogue warps: warp w >= 2 reads TMEM lane quadrant (w % 4) and column half (w - 2) / 4.
#pragma once

#include "ds_internal.h"

namespace ds {
namespace tcpipe {

constexpr uint64_t kDrainLimitNs = 200000000ull;
constexpr int kEpiWarps = 8;
constexpr int kThreadsTC = 64 + 32 * kEpiWarps;

constexpr int kMaxStages = 6;

struct Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
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

// tempty_count: arrivals that release a TMEM buffer (every epilogue thread by default).
DS_DEV void ctl_init(Ctl& c, int stages, uint32_t tempty_count = 32 * kEpiWarps) {
  for (int s = 0; s < stages; ++s) {
    mbar_init(smem_u32(&c.full[s]), 1);
    mbar_init(smem_u32(&c.empty[s]), 1);
  }
  for (int b = 0; b < 2; ++b) {
    mbar_init(smem_u32(&c.tfull[b]), 1);
    mbar_init(smem_u32(&c.tempty[b]), tempty_count);
  }
  mbar_init(smem_u32(&c.mma_done), 1);
  c.abort = 0;
  c.consumed = 0;
  fence_mbar_init();
}

// True when every sequence with a row in [r0, r0 + n) is finished.
DS_DEV bool rows_done(const uint8_t* done, int r0, int n, int L) {
  if (!done) return false;
  for (int b = r0 / L; b <= (r0 + n - 1) / L; ++b)
    if (!done[b]) return false;
  return true;
}

// After an abort: wait for the copies issued but not consumed by the MMA thread.
DS_DEV void producer_drain(Ctl& c, int issued, int stages) {
  const int consumed = *(volatile int*)&c.consumed;
  for (int q = consumed; q < issued; ++q)
    mbar_wait_quiet(smem_u32(&c.full[q % stages]), (uint32_t)((q / stages) & 1));
}


// Add COLS fp32 TMEM columns starting at taddr (this warp's 32 lanes) to acc[0..COLS), two
// 16-column loads per wait to keep register pressure low next to the accumulator (registers
// are charged per group of four warps, so a 10-warp CTA gets at most 168 each).
template <int COLS>
DS_DEV void tmem_accumulate(uint32_t taddr, float (&acc)[COLS]) {
#pragma unroll
  for (int c = 0; c < COLS / 32; ++c) {
    uint32_t r0[16], r1[16];
    tmem_ld_16cols(taddr + (uint32_t)(c * 32), r0);
    tmem_ld_16cols(taddr + (uint32_t)(c * 32 + 16), r1);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      acc[c * 32 + i] += __uint_as_float(r0[i]);
      acc[c * 32 + 16 + i] += __uint_as_float(r1[i]);
    }
  }
}

// acc[i] += scale * TMEM column i, for COLS columns starting at taddr (this warp's 32 lanes).
template <int COLS>
DS_DEV void tmem_accumulate_scaled(uint32_t taddr, float (&acc)[COLS], float scale) {
#pragma unroll
  for (int c = 0; c < COLS / 32; ++c) {
    uint32_t r0[16], r1[16];
    tmem_ld_16cols(taddr + (uint32_t)(c * 32), r0);
    tmem_ld_16cols(taddr + (uint32_t)(c * 32 + 16), r1);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      acc[c * 32 + i] = fmaf(__uint_as_float(r0[i]), scale, acc[c * 32 + i]);
      acc[c * 32 + 16 + i] = fmaf(__uint_as_float(r1[i]), scale, acc[c * 32 + 16 + i]);
    }
  }
}

}  // namespace tcpipe
}  // namespace ds
