// The sampler step without any device allocation.
//
// Some callers cannot allocate device memory when they want a step: a serving engine that
// reserves (almost) all HBM for its own pools at start-up and forbids later allocations, or a
// latency-critical path where cudaMalloc / cudaFree would synchronise the device and stall
// other streams. ds_sampler_create allocates a workspace, so such callers get this entry
// point instead: it needs no sampler object and takes its scratch from one fixed array below.
//
// The scratch array is a file-scope __device__ array, so every GPU that loads the library
// holds it until the process exits. Host code cannot use the array's name as a device
// address (on the host it names a stand-in object); the address is looked up with
// cudaGetSymbolAddress once per device context, while that device is current, and passed to the
// kernels. The lookup is keyed on the context's unique id, so a device reset (which unloads the
// module and may place the array elsewhere) leads to a fresh lookup instead of a stale pointer.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "../../include/ds_sampler.h"
#include "ds_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;  // 64 MiB
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
// The first 256 bytes of the array hold the device error word of the last call (cleared at the
// start of every call), at a fixed place so that ds_sampler_noalloc_status can read it.
constexpr size_t kErrWordBytes = 256;

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
struct ScratchAddr {
  unsigned long long ctx_id = 0;  // the context the address belongs to (0: none yet)
  void* addr = nullptr;
};
ScratchAddr g_noalloc_addr[kMaxDevices];

// Driver entry points for the current context's unique id (resolved once; a device reset or a
// new primary context gives a new id, and the array may then sit at a new address).
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

void resolve_ctx_entry_points() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
}

// The unique id of the calling thread's current context; false when none is current.
bool current_ctx_id(unsigned long long* id) {
  std::call_once(g_ctx_once, resolve_ctx_entry_points);
  CUcontext ctx = nullptr;
  return g_ctx_current && g_ctx_id && g_ctx_current(&ctx) == CUDA_SUCCESS && ctx &&
         g_ctx_id(ctx, id) == CUDA_SUCCESS && *id != 0;
}

// Device address of the scratch array in the current device's context: looked up with
// cudaGetSymbolAddress (which also makes the device's primary context current) the first time a
// context is seen on the device, and kept while that context lives.
ds_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DS_ERR_CUDA;
  unsigned long long id = 0;
  const bool have = current_ctx_id(&id);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  ScratchAddr& a = g_noalloc_addr[dev];
  if (!have || a.ctx_id != id || !a.addr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return DS_ERR_CUDA;
    }
    if (!current_ctx_id(&id)) return DS_ERR_CUDA;
    a.addr = p;
    a.ctx_id = id;
  }
  *out = a.addr;
  return DS_OK;
}

struct Carver {
  unsigned char* base;
  size_t used = 0;
  template <class T>
  T* take(size_t count) {
    T* p = reinterpret_cast<T*>(base + used);
    used += (count * sizeof(T) + 255) & ~size_t(255);
    return p;
  }
};

}  // namespace

extern "C" ds_status ds_sampler_step_noalloc(const ds_sampler_config* cfg,
                                             const ds_step_args* a, void* stream) {
  using namespace ds;
  if (!cfg || !a) return DS_ERR_INVALID_ARG;
  const ds_sampler_config& c = *cfg;
  const ds_status vs = validate_config(c);
  if (vs != DS_OK) return vs;
  // the fused vocabulary pass needs a control block and range partials of its own, which this
  // entry point does not carve: it is refused rather than replaced by another path
  if (c.impl == DS_IMPL_FUSED) return DS_ERR_UNSUPPORTED;
  if (c.lock_rule == DS_LOCK_ENTROPY_BUDGET && !a->prev_argmax) return DS_ERR_INVALID_ARG;
  if (a->batch < 1 || (int64_t)a->batch * c.canvas_len > 65535) return DS_ERR_INVALID_ARG;
  if (!a->H || !a->E || !a->temperature || !a->tau || !a->step || !a->canvas || !a->lock ||
      !a->done || !a->s || !a->sampled || !a->conf || !a->entropy || !a->argmax)
    return DS_ERR_INVALID_ARG;
  auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!aligned16(a->H) || !aligned16(a->E) || !aligned16(a->s)) return DS_ERR_INVALID_ARG;
  const int nc = n_chunks_of(c.vocab);

  bool tensor = false;
  if (c.impl != DS_IMPL_SIMT) {
    const bool ok = c.dtype == DS_DTYPE_BF16 && tc_available();
    if (c.impl == DS_IMPL_TENSOR && !ok) return DS_ERR_UNSUPPORTED;
    tensor = ok;
  }
  int dev = 0, sms = 1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DS_ERR_CUDA;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  sms = std::max(1, sms);

  const int L = c.canvas_len, d = c.d_model, B = a->batch, R = B * L, k = c.top_k;
  const int64_t V = c.vocab;
  int S;
  if (tensor) {
    S = selfcond_tc_splits(R, V, d, sms);
  } else {
    const long tiles = (long)(d / 64) * (R / 128);
    long s = (4L * sms + tiles - 1) / tiles;
    S = (int)std::max(1L, std::min(s, std::min(64L, (long)(V / 1024))));
  }

  // The scratch this step needs, laid out with 256-byte alignment; refuse what does not fit.
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t RV = (size_t)R * (size_t)V;
  const size_t nstat = std::max<size_t>(nc, (size_t)(V / kTcSegment));
  const size_t need = up(RV * 4) + 2 * up(RV * 2) + up((size_t)R * nstat * sizeof(ChunkStat)) +
                      up((size_t)R * sizeof(RowStat)) + up((size_t)R * nc * sizeof(Best)) +
                      (k > 0 ? up((size_t)R * nc * k * sizeof(Cand)) : 0) +
                      up((size_t)S * R * d * 4) + up((size_t)B * 4) + kErrWordBytes;
  if (need > kNoAllocScratchBytes) return DS_ERR_UNSUPPORTED;

  void* base = nullptr;
  ds_status st = scratch_address(&base);
  if (st != DS_OK) return st;
  Carver cv{static_cast<unsigned char*>(base)};
  uint32_t* err = cv.take<uint32_t>(kErrWordBytes / sizeof(uint32_t));
  float* Y = cv.take<float>(RV);
  uint16_t* Phi = cv.take<uint16_t>(RV);
  uint16_t* Plo = cv.take<uint16_t>(RV);
  ChunkStat* cs = cv.take<ChunkStat>((size_t)R * nstat);
  RowStat* rs = cv.take<RowStat>((size_t)R);
  Best* best = cv.take<Best>((size_t)R * nc);
  Cand* cand = k > 0 ? cv.take<Cand>((size_t)R * nc * k) : nullptr;
  float* Opart = cv.take<float>((size_t)S * R * d);
  float* Teff = cv.take<float>((size_t)B);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the error word must start at zero. Every
  // other region is fully written before it is read in this step.
  if (cudaMemsetAsync(err, 0, sizeof(uint32_t), s) != cudaSuccess) return DS_ERR_CUDA;
  const bool fp32 = c.dtype == DS_DTYPE_FP32;
  const float* T = a->temperature;
  if (c.t_start > 0.f) {
    launch_temperature(a->step, B, c.t_start, c.t_end, c.max_steps, Teff, s);
    T = Teff;
  }
  if (tensor) {
    if (launch_logits_tc(static_cast<const uint16_t*>(a->H), static_cast<const uint16_t*>(a->E), R,
                         V, d, L, T, a->done, Y, cs, err, s) != cudaSuccess)
      return DS_ERR_CUDA;
    launch_row_merge(cs, (int)(V / kTcSegment), R, L, a->done, rs, s);
  } else {
    launch_logits_simt(a->H, a->E, fp32, R, V, d, L, T, a->done, Y, s);
    launch_chunk_stats(Y, R, V, L, a->done, cs, s);
    launch_row_merge(cs, nc, R, L, a->done, rs, s);
  }
  if (k > 0) launch_topk_chunk(Y, R, V, L, a->done, k, cand, s);
  launch_convert(Y, rs, R, V, L, a->done, a->step, a->seed, nullptr, k == 0, Phi, Plo, best, s);
  if (tensor) {
    if (launch_selfcond_tc(Phi, Plo, static_cast<const uint16_t*>(a->E), R, V, d, L, a->done, S,
                           Opart, nullptr, nullptr, err, nullptr, s) != cudaSuccess)
      return DS_ERR_CUDA;
  } else {
    launch_selfcond_simt(Phi, Plo, a->E, fp32, R, V, d, L, a->done, S, Opart, s);
  }
  launch_reduce_s(Opart, S, R, d, L, a->done, rs, a->s, s);
  launch_finalize(rs, best, cand, nc, k, R, L, a->done, a->step, a->seed, nullptr, a->sampled,
                  a->conf, a->entropy, a->argmax, s);
  if (c.lock_rule == DS_LOCK_ENTROPY_BUDGET)
    launch_lock_entropy(B, L, V, c.max_steps, a->seed, nullptr, c.entropy_budget, c.stop_entropy,
                        a->sampled, a->entropy, a->argmax, a->prev_argmax, a->step, a->canvas,
                        a->lock, a->done, s);
  else
    launch_lock(B, L, V, c.max_steps, a->seed, nullptr, a->tau, a->sampled, a->conf, a->step,
                a->canvas, a->lock, a->done, s);
  return cudaGetLastError() == cudaSuccess ? DS_OK : DS_ERR_CUDA;
}

extern "C" ds_status ds_sampler_noalloc_status(void* stream, ds_status* out) {
  if (!out) return DS_ERR_INVALID_ARG;
  void* base = nullptr;
  const ds_status st = scratch_address(&base);
  if (st != DS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t w = 0;
  // pageable host memory: the copy completes before cudaMemcpyAsync returns or at the
  // synchronisation below; nothing is allocated
  if (cudaMemcpyAsync(&w, base, sizeof(w), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemsetAsync(base, 0, sizeof(uint32_t), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return DS_ERR_CUDA;
  *out = (w & ds::kErrTimeout) ? DS_ERR_TIMEOUT : (w ? DS_ERR_DEVICE : DS_OK);
  return DS_OK;
}
