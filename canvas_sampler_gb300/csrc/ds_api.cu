// C ABI of the canvas sampler (include/ds_sampler.h): argument validation, the workspace, the
// order of kernel launches in a step, the host-buffer variant and the CUDA-graph denoising loop.
//
// A step enqueues, on the caller's stream, with the tensor cores and top_k = 0:
//   fused vocabulary pass (ds_tc_fused.cu)    -> segment statistics and Gumbel winners, O
//   row merge                                 -> m, l, entropy, argmax, sample per row
//   finalize (s = O / l, confidence)
//   lock / re-noise / stop
// otherwise (top-k, or the CUDA-core path for fp32 inputs):
//   logits GEMM (tensor cores or CUDA cores)  -> y [B*L, V] fp32
//   chunk statistics, row merge               -> m, l, entropy, argmax per row
//   [top-k candidates per chunk]
//   exp(y - m) as bf16 hi/lo + chunk Gumbel-max
//   self-conditioning GEMM over vocabulary splits -> O partials
//   reduction s = sum(O) / l; finalize (sample, confidence)
//   lock / re-noise / stop
// The loop (report section 6, "Eliminating CPU-GPU synchronization") is one graph launch: a
// while node whose condition the last kernel of each iteration sets from the done flags.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/ds_sampler.h"
#include "ds_internal.h"

using namespace ds;

namespace {
// A named range on the host timeline for each entry point that enqueues work (NVTX: shown by
// profilers that record it, a no-op otherwise).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};
}  // namespace

namespace {

struct LoopGraph {
  ds_loop_args key;
  int batch;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

struct BlockGraph {
  ds_block_args key;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

}  // namespace

struct ds_sampler {
  ds_sampler_config cfg{};
  int device = 0;
  int impl = DS_IMPL_SIMT;
  bool fused = false;     // tensor cores, top_k = 0: the fused vocabulary pass
  int vp_producers = 0;   // CTAs that start as producers in the fused pass (0: default)
  int num_sms = 1;
  int n_chunks = 1;
  size_t ws_bytes = 0;
  float* Y = nullptr;
  uint16_t* Phi = nullptr;
  uint16_t* Plo = nullptr;
  ChunkStat* cs = nullptr;
  RowStat* rs = nullptr;
  Best* best = nullptr;
  Cand* cand = nullptr;
  float* Opart = nullptr;
  size_t opart_floats = 0;
  uint16_t* U = nullptr;  // stand-in operand [B*L, 2d] (tensor-core path)
  float* Teff = nullptr;  // scheduled temperatures [B]
  ChunkStat* seg = nullptr;  // fused pass: segment statistics [B*L, V/128]
  float* mseg_t = nullptr;   // segment maxima [V/128, B*L] (fused) / tile maxima [V/256, B*L]
  float* mref = nullptr;     // fused pass: reference maxima of the range partials [Q, B*L]
  uint32_t* vp_sync = nullptr;
  uint32_t* err = nullptr;
  // tensor-core step without top-k: where the Gumbel race runs (inside the self-conditioning
  // launch, with its queue counters gq[2], or as a launch of its own): -1 by shape (race_in_sc),
  // 0 / 1 forced by DS_GUMBEL_IN_SELFCOND
  int gumbel_in_sc = -1;
  uint32_t* gq = nullptr;
  uint32_t* row_flags = nullptr;  // [max_batch * L]: rows merged inside the launch (generation)
  int32_t* iter = nullptr;
  int last_batch = 0;
  // device staging for ds_sampler_step_host (allocated on first use)
  void* stage = nullptr;
  size_t stage_bytes = 0;
  void* hstage = nullptr;  // pinned host mirror of the small per-step buffers
  cudaStream_t capture_stream = nullptr;
  std::vector<LoopGraph> graphs;
  std::vector<BlockGraph> block_graphs;
  // block-autoregressive control words: [0] block index (0 outside ds_block_loop; every random
  // draw's counter carries it), [1..3] the driver's action, committed block and iterations
  int32_t* blk = nullptr;
  std::vector<void*> allocations;
  // phase timing (ds_sampler_set_phase_timing)
  int timing = 0;  // 0 off, 1 every phase, 2 the coarse boundaries only (coarse_phase)
  std::vector<cudaEvent_t> events;  // kPhaseEvents per timed step
  int timed_steps = 0;
  cudaStream_t timed_stream = nullptr;
  int64_t launches = 0;
};

namespace {

constexpr int kPhases = 7;
constexpr int kPhaseEvents = kPhases + 1;

// Event marking the end of `phase` (or the start of the step for phase -1) in the current
// timed step; nullptr when timing is off.
// Phases whose end is marked in coarse timing: the logits GEMM, everything up to the
// self-conditioning GEMM, the GEMM itself, and everything after it (fewer events between the
// kernels of a step: an event between two kernels costs more than its own record, since the
// second kernel can no longer be launched as the first retires).
bool coarse_phase(int phase) { return phase == 0 || phase == 3 || phase == 4 || phase == 6; }

void mark(ds_sampler* s, int phase, cudaStream_t st) {
  if (!s->timing) return;
  if (s->timing == 2 && phase >= 0 && !coarse_phase(phase)) return;
  const size_t need = (size_t)(s->timed_steps + 1) * kPhaseEvents;
  while (s->events.size() < need) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) {
      s->timing = 0;
      return;
    }
    s->events.push_back(e);
  }
  cudaEventRecord(s->events[(size_t)s->timed_steps * kPhaseEvents + (phase + 1)], st);
}

int esize(int dtype) { return dtype == DS_DTYPE_FP32 ? 4 : 2; }

// Whether a step's Gumbel race runs on warps of the self-conditioning launch. Measured on GB300
// (step time, race inside / own launch), d = 2816: B = 1, V = 262144: 0.886 / 0.892 ms and on
// another box 0.904 / 0.913; V = 65536 and 131072: 0.276 / 0.293 and 0.469 / 0.481 ms. B = 1,
// V = 32768, d = 1024: 0.154 / 0.116 ms (a short GEMM leaves the race to a few warps). At
// V = 262144 and larger batches the answer depends on the clocks: in short runs at 2070 MHz
// (same box, two repeats) B = 2: 1.51 / 1.556 ms, B = 4: 2.905 / 2.979, B = 8: 5.884 / 6.000,
// B = 16: 12.02-12.51 / 12.02-12.33; in runs of 2-3 s under the power cap B = 2: 1.661 / 1.668-
// 1.675, B = 4: 3.304-3.308 / 3.261-3.268, B = 8: 6.669-6.725 / 6.637-6.657, B = 16: 13.51 /
// 13.43-13.46 (the race inside draws more power, and the cap lowers the clock further). So
// inside for up to two canvases of rows (faster in both regimes), with d >= 2048.
bool race_in_selfcond(const ds_sampler* s, int R, int d) {
  if (s->gumbel_in_sc >= 0) return s->gumbel_in_sc == 1;
  return R <= 512 && d >= 2048;
}

int splits_for(const ds_sampler* s, int batch) {
  const int R = batch * s->cfg.canvas_len;
  const int64_t V = s->cfg.vocab;
  const int d = s->cfg.d_model;
  if (s->impl != DS_IMPL_SIMT) {
    // DS_SELFCOND_SPLITS=n (read once) overrides the choice, for measurements; the workspace is
    // sized with the same function, so the override holds for a sampler's whole life
    static const int forced = [] {
      const char* e = getenv("DS_SELFCOND_SPLITS");
      return e ? atoi(e) : 0;
    }();
    if (forced >= 1)
      return (int)std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(forced, 64), V / 256));
    return selfcond_tc_splits(R, V, d, s->num_sms);
  }
  // CUDA-core GEMM: aim at about four waves of 128 x 64 tiles, >= 1024 tokens per split
  const long tiles = (long)(d / 64) * (R / 128);
  long S = (4L * s->num_sms + tiles - 1) / tiles;
  S = std::max(1L, std::min(S, std::min(64L, (long)(V / 1024))));
  return (int)std::max(1L, S);
}

thread_local cudaError_t t_last_cuda_error = cudaSuccess;

ds_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DS_OK;
  t_last_cuda_error = e;
  if (e == cudaErrorMemoryAllocation) return DS_ERR_OOM;
  return DS_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

ds_status check_step_args(const ds_sampler* s, const ds_step_args* a) {
  if (!a) return DS_ERR_INVALID_ARG;
  if (a->batch < 1 || a->batch > s->cfg.max_batch) return DS_ERR_INVALID_ARG;
  if (!a->H || !a->E || !a->temperature || !a->tau || !a->step || !a->canvas || !a->lock ||
      !a->done || !a->s || !a->sampled || !a->conf || !a->entropy || !a->argmax)
    return DS_ERR_INVALID_ARG;
  if (!aligned(a->H, 16) || !aligned(a->E, 16) || !aligned(a->s, 16)) return DS_ERR_INVALID_ARG;
  if (s->cfg.lock_rule == DS_LOCK_ENTROPY_BUDGET && !a->prev_argmax) return DS_ERR_INVALID_ARG;
  return DS_OK;
}

ds_status enqueue_step(ds_sampler* s, const ds_step_args* a, cudaStream_t st) {
  const int L = s->cfg.canvas_len, d = s->cfg.d_model, B = a->batch;
  const int64_t V = s->cfg.vocab;
  const int R = B * L;
  const bool fp32 = s->cfg.dtype == DS_DTYPE_FP32;
  const int k = s->cfg.top_k;
  const int S = splits_for(s, B);
  s->last_batch = B;
  mark(s, -1, st);
  const float* T = a->temperature;
  if (s->cfg.t_start > 0.f) {
    launch_temperature(a->step, B, s->cfg.t_start, s->cfg.t_end, s->cfg.max_steps, s->Teff, st);
    T = s->Teff;
    s->launches += 1;
  }
  if (s->fused) {
    const VocabPassShape sh = vocab_pass_shape(R, V, d, s->num_sms, s->vp_producers);
    cudaError_t e = launch_vocab_pass_tc(
        sh, static_cast<const uint16_t*>(a->H), static_cast<const uint16_t*>(a->E), R, V, d, L,
        T, a->done, a->step, a->seed, s->Phi, s->Plo, s->seg, s->mseg_t, s->Opart, s->mref,
        s->vp_sync, s->err, st);
    if (e != cudaSuccess) return cuda_status(e);
    mark(s, 0, st);
    launch_row_merge(s->seg, (int)(V / kVpSegment), R, L, a->done, s->rs, st);
    mark(s, 1, st);
    mark(s, 2, st);
    launch_gumbel_items(s->Phi, s->Plo, s->seg, s->rs, R, V, L, a->done, a->step, a->seed, s->blk,
                      false, s->best, st);
    mark(s, 3, st);
    mark(s, 4, st);
    launch_finalize_with_s(s->rs, s->best, nullptr, s->n_chunks, 0, R, L, a->done, a->step,
                           a->seed, s->blk, a->sampled, a->conf, a->entropy, a->argmax, s->Opart,
                           sh.n_ranges, d, a->s, s->mref, st);
    s->launches += 4;
  } else if (s->impl != DS_IMPL_SIMT) {
    // the logits leave the GEMM as tile-relative probabilities; no y, no convert pass. Without
    // top-k the Gumbel race runs over all of them; with top-k each chunk's k most probable
    // tokens become the candidates that finalize draws among.
    cudaError_t e = launch_logits_p_tc(static_cast<const uint16_t*>(a->H),
                                       static_cast<const uint16_t*>(a->E), R, V, d, L, T, a->done,
                                       s->Phi, s->Plo, s->cs, s->mseg_t, s->err, st);
    if (e != cudaSuccess) return cuda_status(e);
    mark(s, 0, st);
    // with the race inside the self-conditioning launch, the row merge is the first work of its
    // racing warps (the GEMM does not need it); otherwise a launch of its own
    const bool race_in_sc = k == 0 && race_in_selfcond(s, R, d);
    if (!race_in_sc) launch_row_merge(s->cs, (int)(V / kTcSegment), R, L, a->done, s->rs, st);
    mark(s, 1, st);
    if (k > 0)
      launch_topk_row(s->Phi, s->Plo, s->cs, s->mseg_t, s->rs, R, V, L, a->done, k, s->cand, st);
    mark(s, 2, st);
    if (k == 0 && !race_in_sc)
      launch_gumbel_items(s->Phi, s->Plo, s->cs, s->rs, R, V, L, a->done, a->step, a->seed, s->blk,
                        true, s->best, st);
    mark(s, 3, st);
    const GumbelWork gw{s->Phi, s->Plo, s->cs,  s->rs, a->done, a->step, s->blk,
                        a->seed, s->best, s->gq, R,    L,       s->n_chunks, 1,
                        s->rs,   s->row_flags, s->err};
    e = launch_selfcond_tc(s->Phi, s->Plo, static_cast<const uint16_t*>(a->E), R, V, d, L,
                           a->done, S, s->Opart, s->mseg_t, s->mref, s->err,
                           race_in_sc ? &gw : nullptr, st);
    if (e != cudaSuccess) return cuda_status(e);
    mark(s, 4, st);
    // with top-k the candidate pool of a row is its k candidates (one "chunk")
    launch_finalize_with_s(s->rs, s->best, k > 0 ? s->cand : nullptr, k > 0 ? 1 : s->n_chunks, k,
                           R, L, a->done, a->step, a->seed, s->blk, a->sampled, a->conf,
                           a->entropy, a->argmax, s->Opart, S, d, a->s, s->mref, st);
    s->launches += race_in_sc ? 3 : 5;
  } else {
    launch_logits_simt(a->H, a->E, fp32, R, V, d, L, T, a->done, s->Y, st);
    mark(s, 0, st);
    launch_chunk_stats(s->Y, R, V, L, a->done, s->cs, st);
    launch_row_merge(s->cs, s->n_chunks, R, L, a->done, s->rs, st);
  }
  if (!s->fused && s->impl == DS_IMPL_SIMT) {
    // CUDA-core path: y materialised, split into hi / lo by the convert pass
    mark(s, 1, st);
    if (k > 0) launch_topk_chunk(s->Y, R, V, L, a->done, k, s->cand, st);
    mark(s, 2, st);
    launch_convert(s->Y, s->rs, R, V, L, a->done, a->step, a->seed, s->blk, k == 0, s->Phi,
                   s->Plo, s->best, st);
    mark(s, 3, st);
    launch_selfcond_simt(s->Phi, s->Plo, a->E, fp32, R, V, d, L, a->done, S, s->Opart, st);
    mark(s, 4, st);
    launch_finalize_with_s(s->rs, s->best, s->cand, s->n_chunks, k, R, L, a->done, a->step,
                           a->seed, s->blk, a->sampled, a->conf, a->entropy, a->argmax, s->Opart,
                           S, d, a->s, nullptr, st);
    s->launches += 6 + (k > 0 ? 1 : 0);
  }
  mark(s, 5, st);
  if (s->cfg.lock_rule == DS_LOCK_ENTROPY_BUDGET)
    launch_lock_entropy(B, L, V, s->cfg.max_steps, a->seed, s->blk, s->cfg.entropy_budget,
                        s->cfg.stop_entropy, a->sampled, a->entropy, a->argmax, a->prev_argmax,
                        a->step, a->canvas, a->lock, a->done, st);
  else
    launch_lock(B, L, V, s->cfg.max_steps, a->seed, s->blk, a->tau, a->sampled, a->conf,
                a->step, a->canvas, a->lock, a->done, st);
  mark(s, 6, st);
  if (s->timing) {
    ++s->timed_steps;
    s->timed_stream = st;
  }
  s->launches += 1;
  return cuda_status(cudaGetLastError());
}

ds_status enqueue_standin(ds_sampler* s, const void* W, const float* s_prev, const void* E,
                          const int32_t* canvas, const uint8_t* done, void* H_out, int batch,
                          cudaStream_t st) {
  const int d = s->cfg.d_model, L = s->cfg.canvas_len, R = batch * L;
  if (s->impl != DS_IMPL_SIMT && s->U && d % 256 == 0) {
    launch_standin_gather(s_prev, static_cast<const uint16_t*>(E), canvas, done, R, d, L,
                          s->cfg.vocab, s->err, s->U, st);
    cudaError_t e = launch_standin_tc(s->U, static_cast<const uint16_t*>(W), R, d, L, done,
                                      static_cast<uint16_t*>(H_out), s->err, st);
    s->launches += 2;
    return cuda_status(e == cudaSuccess ? cudaGetLastError() : e);
  }
  launch_standin_simt(static_cast<const uint16_t*>(W), s_prev, static_cast<const uint16_t*>(E),
                      canvas, done, batch * s->cfg.canvas_len, s->cfg.d_model, s->cfg.canvas_len,
                      s->cfg.vocab, s->err, static_cast<uint16_t*>(H_out), st);
  s->launches += 1;
  return cuda_status(cudaGetLastError());
}

ds_status enqueue_iteration(ds_sampler* s, const ds_loop_args* a, cudaStream_t st) {
  if (a->h_mode == DS_H_STANDIN) {
    ds_status r = enqueue_standin(s, a->W, a->step.s, a->step.E, a->step.canvas, a->step.done,
                                  a->H_buf, a->step.batch, st);
    if (r != DS_OK) return r;
    ds_step_args sa = a->step;
    sa.H = a->H_buf;
    return enqueue_step(s, &sa, st);
  }
  return enqueue_step(s, &a->step, st);
}

template <class T>
T* carve(ds_sampler* s, size_t count, cudaError_t* e) {
  void* p = nullptr;
  if (*e != cudaSuccess || count == 0) return nullptr;
  *e = cudaMalloc(&p, count * sizeof(T));
  if (*e == cudaSuccess) {
    s->allocations.push_back(p);
    s->ws_bytes += count * sizeof(T);
  }
  return static_cast<T*>(p);
}

void free_all(ds_sampler* s) {
  for (auto& g : s->graphs) {
    if (g.exec) cudaGraphExecDestroy(g.exec);
    if (g.graph) cudaGraphDestroy(g.graph);
  }
  s->graphs.clear();
  for (auto& g : s->block_graphs) {
    if (g.exec) cudaGraphExecDestroy(g.exec);
    if (g.graph) cudaGraphDestroy(g.graph);
  }
  s->block_graphs.clear();
  for (cudaEvent_t e : s->events) cudaEventDestroy(e);
  s->events.clear();
  for (void* p : s->allocations) cudaFree(p);
  s->allocations.clear();
  if (s->stage) cudaFree(s->stage);
  s->stage = nullptr;
  if (s->hstage) cudaFreeHost(s->hstage);
  s->hstage = nullptr;
  if (s->capture_stream) cudaStreamDestroy(s->capture_stream);
  s->capture_stream = nullptr;
}

}  // namespace

namespace ds {

ds_status validate_config(const ds_sampler_config& c) {
  if (c.canvas_len < 128 || c.canvas_len > 1024 || c.canvas_len % 128) return DS_ERR_INVALID_ARG;
  if (c.vocab < 256 || c.vocab > (1 << 24) || c.vocab % 256) return DS_ERR_INVALID_ARG;
  if (c.d_model < 64 || c.d_model > 16384 || c.d_model % 64) return DS_ERR_INVALID_ARG;
  if (c.dtype != DS_DTYPE_BF16 && c.dtype != DS_DTYPE_FP32) return DS_ERR_INVALID_ARG;
  if (c.top_k < 0 || c.top_k > kMaxTopK) return DS_ERR_INVALID_ARG;
  if (c.max_steps < 1 || c.max_steps > (1 << 28)) return DS_ERR_INVALID_ARG;
  if (c.impl != DS_IMPL_AUTO && c.impl != DS_IMPL_TENSOR && c.impl != DS_IMPL_SIMT &&
      c.impl != DS_IMPL_FUSED)
    return DS_ERR_INVALID_ARG;
  if (c.lock_rule != DS_LOCK_THRESHOLD && c.lock_rule != DS_LOCK_ENTROPY_BUDGET)
    return DS_ERR_INVALID_ARG;
  if (!(c.entropy_budget >= 0.f) || !(c.stop_entropy >= 0.f) || !(c.t_end == c.t_end) ||
      (c.t_start > 0.f && !(c.t_end > 0.f)))
    return DS_ERR_INVALID_ARG;
  if (c.top_k > 0 && (int64_t)n_chunks_of(c.vocab) * c.top_k > kMaxTopKPool)
    return DS_ERR_UNSUPPORTED;
  return DS_OK;
}

}  // namespace ds

extern "C" {

int32_t ds_abi_version(void) { return DS_SAMPLER_ABI_VERSION; }

const char* ds_last_cuda_error(void) { return cudaGetErrorString(t_last_cuda_error); }

const char* ds_status_string(ds_status status) {
  switch (status) {
    case DS_OK: return "ok";
    case DS_ERR_INVALID_ARG: return "invalid argument";
    case DS_ERR_UNSUPPORTED: return "unsupported configuration";
    case DS_ERR_CUDA: return "CUDA runtime error";
    case DS_ERR_TIMEOUT: return "a device-side bounded wait ran out";
    case DS_ERR_OOM: return "out of device memory";
    case DS_ERR_DEVICE: return "device-side check failed";
  }
  return "unknown status";
}

ds_status ds_sampler_create(const ds_sampler_config* cfg, ds_sampler** out) {
  if (!cfg || !out) return DS_ERR_INVALID_ARG;
  *out = nullptr;
  const ds_sampler_config& c = *cfg;
  if (c.max_batch < 1 || (int64_t)c.max_batch * c.canvas_len > 65535) return DS_ERR_INVALID_ARG;
  const ds_status vs = ds::validate_config(c);
  if (vs != DS_OK) return vs;
  const int n_chunks = n_chunks_of(c.vocab);

  ds_sampler* s = new (std::nothrow) ds_sampler();
  if (!s) return DS_ERR_OOM;
  s->cfg = c;
  s->n_chunks = n_chunks;
  cudaError_t e = cudaGetDevice(&s->device);
  if (e != cudaSuccess) {
    delete s;
    return DS_ERR_CUDA;
  }
  if (c.impl == DS_IMPL_SIMT) {
    s->impl = DS_IMPL_SIMT;
  } else {
    const bool tc_ok = c.dtype == DS_DTYPE_BF16 && tc_available();
    if ((c.impl == DS_IMPL_TENSOR || c.impl == DS_IMPL_FUSED) && !tc_ok) {
      delete s;
      return DS_ERR_UNSUPPORTED;
    }
    s->impl = tc_ok ? DS_IMPL_TENSOR : DS_IMPL_SIMT;
  }
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, s->device);
  s->num_sms = sms > 0 ? sms : 1;

  const size_t Rm = (size_t)c.max_batch * c.canvas_len;
  const size_t V = (size_t)c.vocab, d = (size_t)c.d_model;
  if (c.impl == DS_IMPL_FUSED) {
    if (c.top_k != 0 || vocab_pass_shape((int)Rm, c.vocab, c.d_model, s->num_sms, 0).grid == 0) {
      delete s;
      return DS_ERR_UNSUPPORTED;
    }
    s->fused = true;
    s->impl = DS_IMPL_FUSED;
    // producer / consumer split of the fused pass (a tuning knob; 0 = in proportion to work)
    if (const char* env = getenv("DS_VP_PRODUCERS")) s->vp_producers = atoi(env);
  }
  if (const char* env = getenv("DS_GUMBEL_IN_SELFCOND")) s->gumbel_in_sc = env[0] == '0' ? 0 : 1;
  size_t opart = 0, nref = 0;
  for (int b = 1; b <= c.max_batch; ++b) {
    const size_t Rb = (size_t)b * c.canvas_len;
    if (s->fused) {
      const VocabPassShape sh = vocab_pass_shape((int)Rb, c.vocab, c.d_model, s->num_sms, 0);
      opart = std::max(opart, (size_t)sh.n_ranges * Rb * d);
      nref = std::max(nref, (size_t)sh.n_ranges * Rb);
    } else {
      opart = std::max(opart, (size_t)splits_for(s, b) * Rb * d);
    }
  }
  e = cudaSuccess;
  // the tensor-core step never materialises y (tile-relative probabilities)
  const bool seg_path = s->impl == DS_IMPL_TENSOR;
  if (s->fused) {
    const VocabPassShape sh = vocab_pass_shape((int)Rm, c.vocab, c.d_model, s->num_sms, 0);
    s->seg = carve<ChunkStat>(s, Rm * (V / kVpSegment), &e);
    s->mseg_t = carve<float>(s, Rm * (V / kVpSegment), &e);
    s->mref = carve<float>(s, nref, &e);
    s->vp_sync = carve<uint32_t>(s, vocab_pass_sync_words(sh), &e);
  } else if (seg_path) {
    s->mseg_t = carve<float>(s, Rm * (V / 256), &e);  // tile maxima [V/256, R]
    for (int b = 1; b <= c.max_batch; ++b) nref = std::max(nref, (size_t)splits_for(s, b) * b * c.canvas_len);
    s->mref = carve<float>(s, nref, &e);
  } else {
    s->Y = carve<float>(s, Rm * V, &e);
  }
  s->Phi = carve<uint16_t>(s, Rm * V, &e);
  s->Plo = carve<uint16_t>(s, Rm * V, &e);
  if (!s->fused) s->cs = carve<ChunkStat>(s, Rm * std::max<size_t>(n_chunks, V / kTcSegment), &e);
  s->rs = carve<RowStat>(s, Rm, &e);
  // best / cand also hold a shard merge's records (one per shard, or k candidates per shard)
  s->best = carve<Best>(s, Rm * std::max(n_chunks, kMaxShards), &e);
  if (c.top_k > 0)
    s->cand = carve<Cand>(
        s, Rm * std::max(n_chunks, std::min(kMaxShards, kMaxTopKPool / c.top_k)) * c.top_k, &e);
  s->Opart = carve<float>(s, opart, &e);
  s->Teff = carve<float>(s, (size_t)c.max_batch, &e);
  if (s->impl != DS_IMPL_SIMT && c.d_model % 256 == 0) s->U = carve<uint16_t>(s, Rm * 2 * d, &e);
  s->opart_floats = opart;
  s->err = carve<uint32_t>(s, 4, &e);
  s->iter = carve<int32_t>(s, 4, &e);
  s->blk = carve<int32_t>(s, 4, &e);
  s->gq = carve<uint32_t>(s, 4, &e);
  s->row_flags = carve<uint32_t>(s, Rm, &e);
  if (e == cudaSuccess) e = cudaMemset(s->err, 0, 4 * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(s->gq, 0, 4 * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(s->row_flags, 0, Rm * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(s->blk, 0, 4 * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s->capture_stream, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    free_all(s);
    delete s;
    cudaGetLastError();
    return cuda_status(e);
  }
  *out = s;
  return DS_OK;
}

ds_status ds_sampler_destroy(ds_sampler* s) {
  if (!s) return DS_OK;
  cudaDeviceSynchronize();
  free_all(s);
  delete s;
  return DS_OK;
}

ds_status ds_sampler_workspace_bytes(const ds_sampler* s, size_t* bytes) {
  if (!s || !bytes) return DS_ERR_INVALID_ARG;
  *bytes = s->ws_bytes;
  return DS_OK;
}

ds_status ds_sampler_impl(const ds_sampler* s, int32_t* impl) {
  if (!s || !impl) return DS_ERR_INVALID_ARG;
  *impl = s->impl;
  return DS_OK;
}

ds_status ds_sampler_step(ds_sampler* s, const ds_step_args* a, void* stream) {
  NvtxRange nvtx_range("ds_sampler_step");
  if (!s) return DS_ERR_INVALID_ARG;
  ds_status r = check_step_args(s, a);
  if (r != DS_OK) return r;
  return enqueue_step(s, a, static_cast<cudaStream_t>(stream));
}

ds_status ds_sampler_step_host(ds_sampler* s, const ds_step_args* h, void* stream) {
  NvtxRange nvtx_range("ds_sampler_step_host");
  if (!s) return DS_ERR_INVALID_ARG;
  if (!h || h->batch < 1 || h->batch > s->cfg.max_batch || !h->E) return DS_ERR_INVALID_ARG;
  if (!h->H || !h->temperature || !h->tau || !h->step || !h->canvas || !h->lock || !h->done ||
      !h->s || !h->sampled || !h->conf || !h->entropy || !h->argmax)
    return DS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t B = (size_t)h->batch, L = (size_t)s->cfg.canvas_len, d = (size_t)s->cfg.d_model;
  const size_t Bm = (size_t)s->cfg.max_batch;
  // the canvas is in host memory here, so its tokens are checked before anything is enqueued
  // (the device step itself never indexes E by them; the stand-in does)
  {
    const int32_t* cv = static_cast<const int32_t*>(h->canvas);
    for (size_t i = 0; i < B * L; ++i)
      if (cv[i] < 0 || (int64_t)cv[i] >= s->cfg.vocab) return DS_ERR_INVALID_ARG;
  }
  const size_t es = esize(s->cfg.dtype);
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  auto up16 = [](size_t x) { return (x + 15) & ~size_t(15); };
  // The small per-step buffers travel as one block, mirrored in pinned host memory: [T | tau |
  // step | canvas | lock | done | prev_argmax | sampled | conf | entropy | argmax] laid out for
  // this batch. The inputs go in with one copy (T .. prev_argmax), the updated state and the
  // outputs come back with one (step .. argmax); H and s move directly between the caller's
  // buffers and the device. Four copies a step instead of one per buffer.
  size_t o = 0;
  auto seg = [&](size_t n) {
    const size_t at = o;
    o += up16(n);
    return at;
  };
  const size_t oT = seg(B * 4), otau = seg(B * 4), ostep = seg(B * 4), ocanvas = seg(B * L * 4),
               olock = seg(B * L), odone = seg(B), oprev = seg(h->prev_argmax ? B * L * 4 : 0),
               osampled = seg(B * L * 4), oconf = seg(B * L * 4), oent = seg(B * L * 4),
               oarg = seg(B * L * 4);
  const size_t oend = o;
  // block size at max_batch (the largest any call needs)
  const size_t nblock = up(9 * up16(Bm * L * 4) + 4 * up16(Bm * 4) + up16(Bm * L) + up16(Bm));
  const size_t nH = up(Bm * L * d * es), nS = up(Bm * L * d * 4);
  const size_t total = nH + nS + nblock;
  if (!s->stage) {
    cudaError_t e = cudaMalloc(&s->stage, total);
    if (e != cudaSuccess) {
      s->stage = nullptr;
      return cuda_status(e);
    }
    s->stage_bytes = total;
  }
  if (!s->hstage) {
    cudaError_t e = cudaMallocHost(&s->hstage, nblock);
    if (e != cudaSuccess) {
      s->hstage = nullptr;
      return cuda_status(e);
    }
  }
  uint8_t* dev = static_cast<uint8_t*>(s->stage);
  uint8_t* blk_d = dev + nH + nS;
  uint8_t* blk_h = static_cast<uint8_t*>(s->hstage);
  std::memcpy(blk_h + oT, h->temperature, B * 4);
  std::memcpy(blk_h + otau, h->tau, B * 4);
  std::memcpy(blk_h + ostep, h->step, B * 4);
  std::memcpy(blk_h + ocanvas, h->canvas, B * L * 4);
  std::memcpy(blk_h + olock, h->lock, B * L);
  std::memcpy(blk_h + odone, h->done, B);
  if (h->prev_argmax) std::memcpy(blk_h + oprev, h->prev_argmax, B * L * 4);
  ds_step_args a{};
  a.batch = h->batch;
  a.seed = h->seed;
  a.E = h->E;
  a.H = dev;
  a.s = reinterpret_cast<float*>(dev + nH);
  // s in page-locked host memory that the device can address (cudaHostAlloc'd or registered as
  // mapped): the finalize kernel writes it there directly, instead of a copy after the step
  bool s_direct = false;
  {
    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, h->s) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
        pa.devicePointer != nullptr && (reinterpret_cast<uintptr_t>(pa.devicePointer) & 15) == 0) {
      a.s = static_cast<float*>(pa.devicePointer);
      s_direct = true;
    }
    cudaGetLastError();  // a pointer the runtime does not know is not an error here
  }
  a.temperature = reinterpret_cast<const float*>(blk_d + oT);
  a.tau = reinterpret_cast<const float*>(blk_d + otau);
  a.step = reinterpret_cast<int32_t*>(blk_d + ostep);
  a.canvas = reinterpret_cast<int32_t*>(blk_d + ocanvas);
  a.lock = blk_d + olock;
  a.done = blk_d + odone;
  a.prev_argmax = h->prev_argmax ? reinterpret_cast<int32_t*>(blk_d + oprev) : nullptr;
  a.sampled = reinterpret_cast<int32_t*>(blk_d + osampled);
  a.conf = reinterpret_cast<float*>(blk_d + oconf);
  a.entropy = reinterpret_cast<float*>(blk_d + oent);
  a.argmax = reinterpret_cast<int32_t*>(blk_d + oarg);
  cudaError_t e = cudaMemcpyAsync(dev, h->H, B * L * d * es, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(blk_d, blk_h, osampled, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_status(e);
  ds_status r = check_step_args(s, &a);
  if (r != DS_OK) return r;
  r = enqueue_step(s, &a, st);
  if (r != DS_OK) return r;
  // Like the device entry point, the outputs of sequences that were done before the step are
  // left as the caller had them: s comes back for each run of consecutive live sequences (one
  // copy when all are live), the small outputs row by row from the staging mirror.
  const uint8_t* done_in = blk_h + odone;  // the flags as they were before the step
  for (size_t b0 = 0; b0 < B && e == cudaSuccess && !s_direct;) {
    if (done_in[b0]) {
      ++b0;
      continue;
    }
    size_t b1 = b0;
    while (b1 < B && !done_in[b1]) ++b1;
    e = cudaMemcpyAsync(h->s + b0 * L * d, a.s + b0 * L * d, (b1 - b0) * L * d * 4,
                        cudaMemcpyDeviceToHost, st);
    b0 = b1;
  }
  std::vector<uint8_t> live(B);
  for (size_t b = 0; b < B; ++b) live[b] = !done_in[b];
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(blk_h + ostep, blk_d + ostep, oend - ostep, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  std::memcpy(h->step, blk_h + ostep, B * 4);
  std::memcpy(h->canvas, blk_h + ocanvas, B * L * 4);
  std::memcpy(h->lock, blk_h + olock, B * L);
  std::memcpy(h->done, blk_h + odone, B);
  if (h->prev_argmax) std::memcpy(h->prev_argmax, blk_h + oprev, B * L * 4);
  for (size_t b = 0; b < B; ++b) {
    if (!live[b]) continue;
    std::memcpy(h->sampled + b * L, blk_h + osampled + b * L * 4, L * 4);
    std::memcpy(h->conf + b * L, blk_h + oconf + b * L * 4, L * 4);
    std::memcpy(h->entropy + b * L, blk_h + oent + b * L * 4, L * 4);
    std::memcpy(h->argmax + b * L, blk_h + oarg + b * L * 4, L * 4);
  }
  return DS_OK;
}

static_assert(sizeof(ds_shard_row) == sizeof(RowStat) && sizeof(ds_shard_best) == sizeof(Best) &&
                  sizeof(ds_shard_cand) == sizeof(Cand),
              "the shard records are the kernels' row, winner and candidate records");

ds_status ds_sampler_step_shard(ds_sampler* s, const ds_step_args* a, int32_t token_offset,
                               int64_t vocab_total, const ds_shard_partial* out, void* stream) {
  NvtxRange nvtx_range("ds_sampler_step_shard");
  if (!s || !a || !out) return DS_ERR_INVALID_ARG;
  if (a->batch < 1 || a->batch > s->cfg.max_batch) return DS_ERR_INVALID_ARG;
  if (!a->H || !a->E || !a->temperature || !a->step || !a->done || !out->rows || !out->best ||
      !out->O || (s->cfg.top_k > 0 && !out->cand))
    return DS_ERR_INVALID_ARG;
  if (!aligned(a->H, 16) || !aligned(a->E, 16) || !aligned(out->O, 16)) return DS_ERR_INVALID_ARG;
  if (token_offset < 0 || token_offset % 256 || vocab_total > (1 << 24) ||
      (int64_t)token_offset + s->cfg.vocab > vocab_total)
    return DS_ERR_INVALID_ARG;
  // the shard step runs the tensor-core path (logits as tile-relative probabilities)
  if (s->impl != DS_IMPL_TENSOR || s->fused) return DS_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int L = s->cfg.canvas_len, d = s->cfg.d_model, B = a->batch, R = B * L;
  const int64_t V = s->cfg.vocab;
  const int k = s->cfg.top_k;
  const int S = splits_for(s, B);
  s->last_batch = B;
  const float* T = a->temperature;
  if (s->cfg.t_start > 0.f) {
    launch_temperature(a->step, B, s->cfg.t_start, s->cfg.t_end, s->cfg.max_steps, s->Teff, st);
    T = s->Teff;
    s->launches += 1;
  }
  cudaError_t e = launch_logits_p_tc(static_cast<const uint16_t*>(a->H),
                                     static_cast<const uint16_t*>(a->E), R, V, d, L, T, a->done,
                                     s->Phi, s->Plo, s->cs, s->mseg_t, s->err, st);
  if (e != cudaSuccess) return cuda_status(e);
  const bool race_in_sc = k == 0 && race_in_selfcond(s, R, d);
  if (!race_in_sc) launch_row_merge(s->cs, (int)(V / kTcSegment), R, L, a->done, s->rs, st);
  if (k > 0)
    launch_topk_row(s->Phi, s->Plo, s->cs, s->mseg_t, s->rs, R, V, L, a->done, k, s->cand, st,
                    token_offset);
  if (k == 0 && !race_in_sc)
    launch_gumbel_items(s->Phi, s->Plo, s->cs, s->rs, R, V, L, a->done, a->step, a->seed, s->blk,
                        true, s->best, st, token_offset);
  GumbelWork gw{s->Phi, s->Plo, s->cs,  s->rs, a->done, a->step, s->blk,
                a->seed, s->best, s->gq, R,    L,       s->n_chunks, 1,
                s->rs,   s->row_flags, s->err};
  gw.j_offset = token_offset;
  e = launch_selfcond_tc(s->Phi, s->Plo, static_cast<const uint16_t*>(a->E), R, V, d, L, a->done,
                         S, s->Opart, s->mseg_t, s->mref, s->err, race_in_sc ? &gw : nullptr, st);
  if (e != cudaSuccess) return cuda_status(e);
  launch_shard_export(s->rs, s->best, s->n_chunks, s->cand, k, R, L, a->done, s->Opart, S, d,
                      s->mref, token_offset, reinterpret_cast<RowStat*>(out->rows),
                      reinterpret_cast<Best*>(out->best), out->O,
                      reinterpret_cast<Cand*>(out->cand), st);
  // logits, [row merge], [top-k | race], self-conditioning, export
  s->launches += 3 + (race_in_sc ? 0 : 1) + ((k > 0 || !race_in_sc) ? 1 : 0);
  return cuda_status(cudaGetLastError());
}

ds_status ds_merge_shards(ds_sampler* s, const ds_step_args* a, int32_t n_shards,
                          const ds_shard_partial* parts, int64_t vocab_total, void* stream) {
  NvtxRange nvtx_range("ds_merge_shards");
  if (!s || !parts || !a) return DS_ERR_INVALID_ARG;
  // the merge reads no H, E or temperature: only the state, tau and the outputs are checked
  if (a->batch < 1 || a->batch > s->cfg.max_batch) return DS_ERR_INVALID_ARG;
  if (!a->tau || !a->step || !a->canvas || !a->lock || !a->done || !a->s || !a->sampled ||
      !a->conf || !a->entropy || !a->argmax || !aligned(a->s, 16))
    return DS_ERR_INVALID_ARG;
  if (s->cfg.lock_rule == DS_LOCK_ENTROPY_BUDGET && !a->prev_argmax) return DS_ERR_INVALID_ARG;
  const int k = s->cfg.top_k;
  if (n_shards < 1 || n_shards > kMaxShards || !parts->rows || !parts->best || !parts->O ||
      (k > 0 && !parts->cand) || !aligned(parts->O, 16))
    return DS_ERR_INVALID_ARG;
  if (vocab_total < 256 || vocab_total > (1 << 24)) return DS_ERR_INVALID_ARG;
  // the merge keeps one record (or k candidates) per shard and row in the workspace
  if (k > 0 && (int64_t)n_shards * k > kMaxTopKPool) return DS_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int L = s->cfg.canvas_len, d = s->cfg.d_model, B = a->batch, R = B * L;
  launch_shard_merge(n_shards, reinterpret_cast<const RowStat*>(parts->rows),
                     reinterpret_cast<const Best*>(parts->best), parts->O,
                     reinterpret_cast<const Cand*>(parts->cand), k, R, d, L, a->done, s->rs,
                     s->best, s->cand, a->s, st);
  launch_finalize(s->rs, s->best, k > 0 ? s->cand : nullptr, n_shards, k, R, L, a->done, a->step,
                  a->seed, s->blk, a->sampled, a->conf, a->entropy, a->argmax, st);
  if (s->cfg.lock_rule == DS_LOCK_ENTROPY_BUDGET)
    launch_lock_entropy(B, L, vocab_total, s->cfg.max_steps, a->seed, s->blk,
                        s->cfg.entropy_budget, s->cfg.stop_entropy, a->sampled, a->entropy,
                        a->argmax, a->prev_argmax, a->step, a->canvas, a->lock, a->done, st);
  else
    launch_lock(B, L, vocab_total, s->cfg.max_steps, a->seed, s->blk, a->tau, a->sampled,
                a->conf, a->step, a->canvas, a->lock, a->done, st);
  s->launches += 3;
  return cuda_status(cudaGetLastError());
}

ds_status ds_standin_hidden(ds_sampler* s, const void* W, const float* s_prev, const void* E,
                            const int32_t* canvas, const uint8_t* done, void* H_out, int32_t batch,
                            void* stream) {
  if (!s || !W || !s_prev || !E || !canvas || !H_out) return DS_ERR_INVALID_ARG;
  if (batch < 1 || batch > s->cfg.max_batch || s->cfg.dtype != DS_DTYPE_BF16)
    return DS_ERR_INVALID_ARG;
  return enqueue_standin(s, W, s_prev, E, canvas, done, H_out, batch,
                         static_cast<cudaStream_t>(stream));
}

ds_status ds_denoise_loop(ds_sampler* s, const ds_loop_args* a, void* stream) {
  NvtxRange nvtx_range("ds_denoise_loop");
  if (!s || !a) return DS_ERR_INVALID_ARG;
  if (a->max_iters < 1 || a->max_iters > s->cfg.max_steps) return DS_ERR_INVALID_ARG;
  if (a->h_mode != DS_H_FIXED && a->h_mode != DS_H_STANDIN) return DS_ERR_INVALID_ARG;
  ds_step_args sa = a->step;
  if (a->h_mode == DS_H_STANDIN) {
    if (!a->W || !a->H_buf || s->cfg.dtype != DS_DTYPE_BF16) return DS_ERR_INVALID_ARG;
    sa.H = a->H_buf;
  }
  ds_status r = check_step_args(s, &sa);
  if (r != DS_OK) return r;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!a->use_graph) {
    for (int it = 0; it < a->max_iters; ++it) {
      r = enqueue_iteration(s, a, st);
      if (r != DS_OK) return r;
    }
    return DS_OK;
  }
  const int was_timing = s->timing;
  s->timing = 0;
  struct Restore {
    ds_sampler* s;
    int v;
    ~Restore() { s->timing = v; }
  } restore{s, was_timing};
  LoopGraph* g = nullptr;
  for (auto& e : s->graphs)
    if (std::memcmp(&e.key, a, sizeof(ds_loop_args)) == 0) g = &e;
  if (!g) {
    LoopGraph ng;
    std::memcpy(&ng.key, a, sizeof(ds_loop_args));
    ng.batch = a->step.batch;
    cudaError_t e = cudaGraphCreate(&ng.graph, 0);
    cudaGraphConditionalHandle h = 0;
    if (e == cudaSuccess) e = cudaGraphConditionalHandleCreate(&h, ng.graph, 0, 0);
    cudaStream_t cs = s->capture_stream;
    if (e == cudaSuccess)
      e = cudaStreamBeginCaptureToGraph(cs, ng.graph, nullptr, nullptr, 0,
                                        cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
      launch_loop_begin(a->step.done, a->step.batch, s->iter, a->max_iters, h, cs);
      s->launches += 1;
      cudaGraph_t outg = nullptr;
      e = cudaStreamEndCapture(cs, &outg);
    }
    cudaGraphNode_t begin_node = nullptr;
    size_t n_nodes = 1;
    if (e == cudaSuccess) e = cudaGraphGetNodes(ng.graph, &begin_node, &n_nodes);
    cudaGraphNodeParams cp{};
    cudaGraphNode_t cond_node = nullptr;
    if (e == cudaSuccess) {
      cp.type = cudaGraphNodeTypeConditional;
      cp.conditional.handle = h;
      cp.conditional.type = cudaGraphCondTypeWhile;
      cp.conditional.size = 1;
      e = cudaGraphAddNode(&cond_node, ng.graph, &begin_node, nullptr, 1, &cp);
    }
    if (e == cudaSuccess) {
      cudaGraph_t body = cp.conditional.phGraph_out[0];
      e = cudaStreamBeginCaptureToGraph(cs, body, nullptr, nullptr, 0,
                                        cudaStreamCaptureModeThreadLocal);
      if (e == cudaSuccess) {
        ds_status rr = enqueue_iteration(s, a, cs);
        launch_loop_end(a->step.done, a->step.batch, s->iter, a->max_iters, h, cs);
        s->launches += 1;
        cudaGraph_t outb = nullptr;
        cudaError_t e2 = cudaStreamEndCapture(cs, &outb);
        e = (rr != DS_OK) ? cudaErrorUnknown : e2;
      }
    }
    if (e == cudaSuccess) e = cudaGraphInstantiate(&ng.exec, ng.graph, 0);
    if (e != cudaSuccess) {
      if (ng.exec) cudaGraphExecDestroy(ng.exec);
      if (ng.graph) cudaGraphDestroy(ng.graph);
      cudaGetLastError();
      return DS_ERR_CUDA;
    }
    s->graphs.push_back(ng);
    g = &s->graphs.back();
  }
  return cuda_status(cudaGraphLaunch(g->exec, st));
}

ds_status ds_block_loop(ds_sampler* s, const ds_block_args* a, void* stream) {
  NvtxRange nvtx_range("ds_block_loop");
  if (!s || !a) return DS_ERR_INVALID_ARG;
  const ds_loop_args& lp = a->loop;
  if (a->n_blocks < 1 || a->first_block < 0 || (int64_t)a->first_block + a->n_blocks > 65536)
    return DS_ERR_INVALID_ARG;
  if (!a->init_canvas || !a->out_canvas || !a->out_steps) return DS_ERR_INVALID_ARG;
  if (lp.max_iters < 1 || lp.max_iters > s->cfg.max_steps) return DS_ERR_INVALID_ARG;
  if (lp.h_mode != DS_H_FIXED && lp.h_mode != DS_H_STANDIN) return DS_ERR_INVALID_ARG;
  ds_step_args sa = lp.step;
  if (lp.h_mode == DS_H_STANDIN) {
    if (!lp.W || !lp.H_buf || s->cfg.dtype != DS_DTYPE_BF16) return DS_ERR_INVALID_ARG;
    sa.H = lp.H_buf;
  }
  ds_status r = check_step_args(s, &sa);
  if (r != DS_OK) return r;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int B = sa.batch, L = s->cfg.canvas_len, d = s->cfg.d_model;
  const int total = a->n_blocks * lp.max_iters;
  const BlockState bs{sa.canvas, sa.lock, sa.step, sa.done, sa.prev_argmax, sa.s};
  auto body = [&](cudaStream_t cs, bool use_cond, cudaGraphConditionalHandle h) -> ds_status {
    ds_status rr = enqueue_iteration(s, &lp, cs);
    if (rr != DS_OK) return rr;
    launch_block_check(s->blk, sa.done, B, a->first_block, a->n_blocks, total, use_cond, h, cs);
    launch_block_rollover(s->blk, a->init_canvas, a->out_canvas, a->out_steps, bs, B, L, d, cs);
    s->launches += 2;
    return cuda_status(cudaGetLastError());
  };
  auto finish = [&](cudaStream_t cs) {
    // outside a block run every draw is block 0's
    return cuda_status(cudaMemsetAsync(s->blk, 0, sizeof(int32_t), cs));
  };
  if (!lp.use_graph) {
    launch_block_start(s->blk, a->first_block, a->init_canvas, bs, B, L, d, st);
    s->launches += 1;
    for (int it = 0; it < total; ++it) {
      r = body(st, false, 0);
      if (r != DS_OK) return r;
    }
    return finish(st);
  }
  const int was_timing = s->timing;
  s->timing = 0;
  struct Restore {
    ds_sampler* s;
    int v;
    ~Restore() { s->timing = v; }
  } restore{s, was_timing};
  BlockGraph* g = nullptr;
  for (auto& e : s->block_graphs)
    if (std::memcmp(&e.key, a, sizeof(ds_block_args)) == 0) g = &e;
  if (!g) {
    BlockGraph ng;
    std::memcpy(&ng.key, a, sizeof(ds_block_args));
    cudaError_t e = cudaGraphCreate(&ng.graph, 0);
    cudaGraphConditionalHandle h = 0;
    // the loop runs at least one step: the condition starts at 1 on every launch
    if (e == cudaSuccess)
      e = cudaGraphConditionalHandleCreate(&h, ng.graph, 1, cudaGraphCondAssignDefault);
    cudaStream_t cs = s->capture_stream;
    if (e == cudaSuccess)
      e = cudaStreamBeginCaptureToGraph(cs, ng.graph, nullptr, nullptr, 0,
                                        cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
      launch_block_start(s->blk, a->first_block, a->init_canvas, bs, B, L, d, cs);
      s->launches += 1;
      cudaGraph_t outg = nullptr;
      e = cudaStreamEndCapture(cs, &outg);
    }
    cudaGraphNode_t start_node = nullptr;
    size_t n_nodes = 1;
    if (e == cudaSuccess) e = cudaGraphGetNodes(ng.graph, &start_node, &n_nodes);
    cudaGraphNodeParams cp{};
    cudaGraphNode_t cond_node = nullptr;
    if (e == cudaSuccess) {
      cp.type = cudaGraphNodeTypeConditional;
      cp.conditional.handle = h;
      cp.conditional.type = cudaGraphCondTypeWhile;
      cp.conditional.size = 1;
      e = cudaGraphAddNode(&cond_node, ng.graph, &start_node, nullptr, 1, &cp);
    }
    if (e == cudaSuccess) {
      cudaGraph_t bodyg = cp.conditional.phGraph_out[0];
      e = cudaStreamBeginCaptureToGraph(cs, bodyg, nullptr, nullptr, 0,
                                        cudaStreamCaptureModeThreadLocal);
      if (e == cudaSuccess) {
        ds_status rr = body(cs, true, h);
        cudaGraph_t outb = nullptr;
        cudaError_t e2 = cudaStreamEndCapture(cs, &outb);
        e = (rr != DS_OK) ? cudaErrorUnknown : e2;
      }
    }
    if (e == cudaSuccess) {
      cudaGraphNode_t reset_node = nullptr;
      cudaMemsetParams mp{};
      mp.dst = s->blk;
      mp.value = 0;
      mp.elementSize = sizeof(int32_t);
      mp.width = 1;
      mp.height = 1;
      e = cudaGraphAddMemsetNode(&reset_node, ng.graph, &cond_node, 1, &mp);
    }
    if (e == cudaSuccess) e = cudaGraphInstantiate(&ng.exec, ng.graph, 0);
    if (e != cudaSuccess) {
      if (ng.exec) cudaGraphExecDestroy(ng.exec);
      if (ng.graph) cudaGraphDestroy(ng.graph);
      t_last_cuda_error = e;
      cudaGetLastError();
      return DS_ERR_CUDA;
    }
    s->block_graphs.push_back(ng);
    g = &s->block_graphs.back();
  }
  return cuda_status(cudaGraphLaunch(g->exec, st));
}

ds_status ds_sampler_device_status(ds_sampler* s, ds_status* out) {
  if (!s || !out) return DS_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return DS_ERR_CUDA;
  uint32_t w = 0;
  e = cudaMemcpy(&w, s->err, sizeof(w), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return DS_ERR_CUDA;
  cudaMemset(s->err, 0, sizeof(uint32_t));
  *out = (w & kErrTimeout) ? DS_ERR_TIMEOUT : (w ? DS_ERR_DEVICE : DS_OK);
  return DS_OK;
}

ds_status ds_philox4x32_10(const uint32_t* ctr, uint64_t seed, uint32_t* out, int64_t n,
                           void* stream) {
  if (n < 0 || (n > 0 && (!ctr || !out))) return DS_ERR_INVALID_ARG;
  if (!aligned(ctr, 16) || !aligned(out, 16)) return DS_ERR_INVALID_ARG;
  launch_philox(ctr, seed, out, n, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

ds_status ds_sampler_set_phase_timing(ds_sampler* s, int32_t enable) {
  if (!s) return DS_ERR_INVALID_ARG;
  if (enable < 0 || enable > 2) return DS_ERR_INVALID_ARG;
  s->timing = enable;
  s->timed_steps = 0;
  return DS_OK;
}

ds_status ds_sampler_phase_times(ds_sampler* s, float* ms, int32_t n, int32_t* steps) {
  if (!s || (n > 0 && !ms)) return DS_ERR_INVALID_ARG;
  double acc[kPhases] = {0};
  if (s->timed_steps > 0) {
    cudaError_t e = cudaStreamSynchronize(s->timed_stream);
    if (e != cudaSuccess) return DS_ERR_CUDA;
    for (int t = 0; t < s->timed_steps; ++t) {
      // each recorded phase end, from the previous recorded event (the step's start first)
      const size_t base = (size_t)t * kPhaseEvents;
      size_t prev = base;
      for (int p = 0; p < kPhases; ++p) {
        if (s->timing == 2 && !coarse_phase(p)) continue;
        float x = 0.f;
        if (cudaEventElapsedTime(&x, s->events[prev], s->events[base + p + 1]) == cudaSuccess)
          acc[p] += x;
        prev = base + p + 1;
      }
    }
  }
  for (int p = 0; p < n && p < kPhases; ++p) ms[p] = (float)acc[p];
  if (steps) *steps = s->timed_steps;
  s->timed_steps = 0;
  return DS_OK;
}

ds_status ds_sampler_launch_count(const ds_sampler* s, int64_t* count) {
  if (!s || !count) return DS_ERR_INVALID_ARG;
  *count = s->launches;
  return DS_OK;
}

ds_status ds_sampler_selftest_wait(ds_sampler* s, int64_t limit_ns, void* stream) {
  if (!s || limit_ns < 1000 || limit_ns > 1000000000) return DS_ERR_INVALID_ARG;
  launch_wait_selftest((uint64_t)limit_ns, s->err, static_cast<cudaStream_t>(stream));
  s->launches += 1;
  return cuda_status(cudaGetLastError());
}

ds_status ds_sampler_debug_buffer(ds_sampler* s, int32_t which, const void** ptr, size_t* bytes) {
  if (!s || !ptr || !bytes) return DS_ERR_INVALID_ARG;
  const size_t R = (size_t)std::max(1, s->last_batch) * s->cfg.canvas_len;
  const size_t V = (size_t)s->cfg.vocab;
  switch (which) {
    case 0:
      if (!s->Y) return DS_ERR_UNSUPPORTED;
      *ptr = s->Y;
      *bytes = R * V * 4;
      return DS_OK;
    case 1: *ptr = s->rs; *bytes = R * sizeof(RowStat); return DS_OK;
    case 2: *ptr = s->Phi; *bytes = R * V * 2; return DS_OK;
    case 3: *ptr = s->Plo; *bytes = R * V * 2; return DS_OK;
    case 4: {
      // segment records exist on the paths that keep P relative to each segment's maximum
      const ChunkStat* seg = s->seg ? s->seg : (s->mseg_t ? s->cs : nullptr);
      if (!seg) return DS_ERR_UNSUPPORTED;
      *ptr = seg;
      *bytes = R * (V / kVpSegment) * sizeof(ChunkStat);
      return DS_OK;
    }
  }
  return DS_ERR_INVALID_ARG;
}

}  // extern "C"
