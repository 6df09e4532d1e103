/*
 * ds_sampler.h -- C ABI of the GB300 (sm_103a) canvas sampler for uniform-state text diffusion.
 *
 * One sampler step over a batch of 256-token canvases:
 *   logits  z = H . E^T over the whole vocabulary, y = z / T;
 *   full-precision softmax over the vocabulary and the self-conditioning vector
 *   s = softmax(y) . E                       -- DiffusionGemma Technical Report, section 6,
 *                                               "Sampling" (softmax over the full canvas, a
 *                                               "self-conditioning embedding matmul", vocabulary
 *                                               262k, full precision); section 8, "Finetuning
 *                                               procedure" (z_t from a previous forward pass);
 *   Gumbel-max sample x with its probability c, optional top-k truncation of the sampling step
 *                                            -- report section 6, "Multi-user throughput";
 *   lock positions with c >= tau (at least one per step), re-noise every other position with a
 *   uniform token, stop per sequence when all positions are locked or the step budget is spent
 *                                            -- "DiffusionGemma: Google's open diffusion LLM",
 *                                               sections "A diffusion language model refines 256
 *                                               tokens in 12 steps" and "Tokens stay editable
 *                                               within a canvas, then freeze"; "Google DeepMind's
 *                                               DiffusionGemma Generates Text 4x Faster by
 *                                               Ditching Tokens", "How text diffusion actually
 *                                               works";
 *   the loop runs on the GPU with no host synchronisation
 *                                            -- report section 6, "Eliminating CPU-GPU
 *                                               synchronization".
 *
 * Conventions for every entry point:
 *   - Pointers marked [device] are CUDA device pointers on the device the sampler was created
 *     on; [host] pointers are ordinary host memory. The caller owns every buffer it passes;
 *     the library owns its workspace and any CUDA graphs it instantiates.
 *   - Layouts are dense row-major. B = batch (sequences), L = canvas length, V = vocabulary,
 *     d = hidden width. bf16 values are IEEE bfloat16 bit patterns (uint16).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Step and
 *     loop calls only enqueue work; they return before the GPU finishes.
 *   - Argument errors are found synchronously and returned as a ds_status; nothing is
 *     enqueued then. Errors found by a kernel (a bounded wait that ran out) set a device error
 *     word that ds_sampler_device_status reports. No call throws across the ABI.
 *   - One sampler must not be used from two streams at once (its workspace is shared).
 *   - Launch shapes (the SM count and how many CTA pairs can be resident) are read once per
 *     process, from the device that is current at the first call; samplers on GPUs of another
 *     kind in the same process are not supported.
 */
#ifndef DS_SAMPLER_H
#define DS_SAMPLER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DS_SAMPLER_ABI_VERSION 4

typedef enum ds_status {
  DS_OK = 0,
  DS_ERR_INVALID_ARG = 1,  /* null pointer, bad size or bad enum value */
  DS_ERR_UNSUPPORTED = 2,  /* valid request the library cannot serve (e.g. shape constraints) */
  DS_ERR_CUDA = 3,         /* a CUDA runtime call failed; the sampler may be unusable */
  DS_ERR_TIMEOUT = 4,      /* a kernel's bounded wait ran out (reported by device_status) */
  DS_ERR_OOM = 5,          /* workspace allocation failed */
  DS_ERR_DEVICE = 6        /* another device-side check failed (reported by device_status) */
} ds_status;

enum { DS_DTYPE_BF16 = 0, DS_DTYPE_FP32 = 1 };
/* Kernel family: TENSOR = tcgen05/TMEM/TMA tensor-core kernels (bf16 inputs, d % 64 == 0);
 * SIMT = CUDA-core fp32 kernels (any supported dtype); FUSED = the tensor-core step with the
 * logits and self-conditioning GEMMs in one persistent cooperative kernel that never writes the
 * logits (bf16 inputs, top_k == 0, d % 256 == 0; else DS_ERR_UNSUPPORTED; the no-allocation
 * step runs it as TENSOR); AUTO = TENSOR where it applies, else SIMT. */
enum { DS_IMPL_AUTO = 0, DS_IMPL_TENSOR = 1, DS_IMPL_SIMT = 2, DS_IMPL_FUSED = 3 };
enum { DS_H_FIXED = 0, DS_H_STANDIN = 1 };
/* Lock rule. THRESHOLD: lock unlocked positions with c >= tau (at least one per step, sticky),
 * re-noise the rest, done when all are locked. ENTROPY_BUDGET: the pages' default sampler --
 * accept positions from the lowest to the highest entropy until entropy_budget is spent (at
 * least one), re-noise all others, decided afresh every step; stop when the mean entropy is
 * below stop_entropy and the argmax equals the previous step's, or at the last step, with the
 * canvas set to the argmax ("DiffusionGemma: Google's open diffusion LLM", "A diffusion
 * language model refines 256 tokens in 12 steps" and Table 2). */
enum { DS_LOCK_THRESHOLD = 0, DS_LOCK_ENTROPY_BUDGET = 1 };

/* Sampler shape and options, fixed at creation.
 *   canvas_len  L, a multiple of 128 and at most 1024 (256 on the pages);
 *   vocab       V, a multiple of 256, at most 2^24;
 *   d_model     d, a multiple of 64, at most 16384;
 *   max_batch   largest B a call may pass (the workspace is sized for it);
 *   dtype       storage type of H and E (DS_DTYPE_*);
 *   top_k       0 = sample from the full softmax, else 1..256: sample among the k largest logits;
 *   max_steps   step budget per canvas (48 on the pages); the last step locks every position;
 *   impl        DS_IMPL_*;
 *   lock_rule   DS_LOCK_*; entropy_budget (0.1 on the pages) and stop_entropy (0.005) are used
 *               by DS_LOCK_ENTROPY_BUDGET;
 *   t_start, t_end  temperature schedule: when t_start > 0 the temperature of a sequence at
 *               step k is t_start + (t_end - t_start) k / (max_steps - 1) (0.8 -> 0.4 on the
 *               pages) and the per-call temperature is ignored; t_start <= 0 turns it off. */
typedef struct ds_sampler_config {
  int32_t max_batch;
  int32_t canvas_len;
  int32_t d_model;
  int32_t dtype;
  int64_t vocab;
  int32_t top_k;
  int32_t max_steps;
  int32_t impl;
  int32_t lock_rule;
  float entropy_budget;
  float stop_entropy;
  float t_start;
  float t_end;
} ds_sampler_config;

typedef struct ds_sampler ds_sampler;

/* Arguments of one step. All pointers [device] unless a host entry point says otherwise.
 *   H           [B, L, d] dtype     hidden states of the canvas positions (input)
 *   E           [V, d] dtype        embedding table, used as both keys and values (input)
 *   temperature [B] float           T_b > 0 (input)
 *   tau         [B] float           lock threshold (input)
 *   step        [B] int32           steps already taken by each sequence (in/out)
 *   canvas      [B, L] int32        canvas tokens in [0, V) (in/out); ds_sampler_step_host
 *                                   refuses others (DS_ERR_INVALID_ARG); in device memory the
 *                                   stand-in, the one reader that indexes E by them, clamps an
 *                                   out-of-range token into E and records DS_ERR_DEVICE for
 *                                   ds_sampler_device_status
 *   lock        [B, L] uint8        1 = locked (in/out)
 *   done        [B] uint8           1 = finished; finished sequences are left untouched (in/out)
 *   s           [B, L, d] float     self-conditioning vector (out)
 *   sampled     [B, L] int32        Gumbel-max sample x (out)
 *   conf        [B, L] float        probability of x under the sampled distribution (out)
 *   entropy     [B, L] float        softmax entropy in nats (out)
 *   argmax      [B, L] int32        most likely token, lowest index on ties (out)
 *   prev_argmax [B, L] int32        the previous step's argmax (in/out; DS_LOCK_ENTROPY_BUDGET
 *                                   only, else may be NULL; any values at step 0)
 *   seed        key of the counter-based generator (Philox4x32-10); draws depend only on
 *               (seed, sequence, position, token, step), so any step boundary is a checkpoint. */
typedef struct ds_step_args {
  int32_t batch;
  int32_t reserved;
  uint64_t seed;
  const void* H;
  const void* E;
  const float* temperature;
  const float* tau;
  int32_t* step;
  int32_t* canvas;
  uint8_t* lock;
  uint8_t* done;
  float* s;
  int32_t* sampled;
  float* conf;
  float* entropy;
  int32_t* argmax;
  int32_t* prev_argmax;
} ds_step_args;

/* Arguments of a denoising loop: steps repeat on the GPU until every sequence is done or
 * max_iters steps have run.
 *   h_mode   DS_H_FIXED: every step uses step.H;
 *            DS_H_STANDIN: before each step H = bf16(tanh(W . [bf16(s); E[canvas]])) is written
 *            to H_buf (a stand-in for the model's decoder, which is out of scope); `s` must hold
 *            the previous step's self-conditioning vector (zeros for a fresh canvas).
 *   W        [d, 2d] bf16 [device] (DS_H_STANDIN only)
 *   H_buf    [B, L, d] bf16 [device] work buffer (DS_H_STANDIN only)
 *   max_iters 1 .. max_steps
 *   use_graph 1: the whole loop is one CUDA graph launch whose while-node condition is set by
 *            the lock kernel (no host synchronisation); 0: plain launches of the same kernels.
 * Graphs are cached per argument set; buffers must outlive the sampler or the next call with
 * different pointers. */
typedef struct ds_loop_args {
  ds_step_args step;
  int32_t h_mode;
  int32_t max_iters;
  int32_t use_graph;
  int32_t reserved;
  const void* W;
  void* H_buf;
} ds_loop_args;

/* Block-autoregressive generation ("DiffusionGemma: Google's open diffusion LLM": generation
 * continues block by block, each new canvas starting from noise once the previous one is
 * committed). loop describes the per-block loop: loop.step holds the working state and outputs
 * (canvas, lock, step, done, prev_argmax, s, ...), loop.max_iters bounds each block's steps,
 * h_mode / W / H_buf as for ds_denoise_loop (the stand-in sees only the current block: the
 * model's attention to committed blocks is out of scope).
 * For k = 0 .. n_blocks - 1: the state is reset (canvas = init_canvas[k], no locks, step 0,
 * done 0, prev_argmax -1, s = 0), the block's steps run until every sequence is done, and the
 * block is committed: out_canvas[k] = canvas, out_steps[k] = step. Block k draws its random
 * numbers with counter word 2 = sequence + 2^16 (first_block + k); block 0 draws exactly as a
 * single canvas does. The whole run is one graph launch when loop.use_graph is set (a while
 * node over all blocks' steps, no host synchronisation), else plain launches of
 * n_blocks * max_iters steps (finished blocks and sequences are skipped).
 *   init_canvas [n_blocks, B, L] int32, out_canvas [n_blocks, B, L] int32,
 *   out_steps [n_blocks, B] int32, all [device]; 1 <= n_blocks, first_block >= 0,
 *   first_block + n_blocks <= 65536. */
typedef struct ds_block_args {
  ds_loop_args loop;
  int32_t n_blocks;
  int32_t first_block;
  const int32_t* init_canvas;
  int32_t* out_canvas;
  int32_t* out_steps;
} ds_block_args;

/* Version of this ABI (DS_SAMPLER_ABI_VERSION). */
int32_t ds_abi_version(void);

/* Static string for a status code; never NULL. */
const char* ds_status_string(ds_status status);

/* Message of the last CUDA runtime error seen by an entry point on the calling thread (the
 * detail behind DS_ERR_CUDA / DS_ERR_OOM); "no error" if none. Static storage; never NULL. */
const char* ds_last_cuda_error(void);

/* Create a sampler on the current CUDA device: validates `cfg`, allocates the workspace for
 * cfg->max_batch. On success *out owns the sampler (free it with ds_sampler_destroy). */
ds_status ds_sampler_create(const ds_sampler_config* cfg, ds_sampler** out);

/* Free the workspace and graphs. Synchronises the device first. NULL is accepted. */
ds_status ds_sampler_destroy(ds_sampler* sampler);

/* Bytes of device workspace the sampler holds. */
ds_status ds_sampler_workspace_bytes(const ds_sampler* sampler, size_t* bytes);

/* The kernel family the sampler runs (DS_IMPL_TENSOR, DS_IMPL_SIMT or DS_IMPL_FUSED; AUTO is
 * resolved at creation). */
ds_status ds_sampler_impl(const ds_sampler* sampler, int32_t* impl);

/* Enqueue one sampler step on `stream` (see ds_step_args). 1 <= batch <= max_batch. */
ds_status ds_sampler_step(ds_sampler* sampler, const ds_step_args* args, void* stream);

/* The same step with every per-step buffer in [host] memory (page-locked memory gives
 * asynchronous copies) and only E on the device: copies the inputs in, runs the step, copies
 * the outputs and the updated state back, and synchronises `stream` before returning. As with
 * ds_sampler_step, the outputs (s, sampled, conf, entropy, argmax) of sequences with done == 1
 * on entry are left as the caller had them. Uses a device staging area and a page-locked host
 * staging block of the sampler (allocated on the first call), so calls on one sampler must not
 * overlap. When s is page-locked host memory the device can address (cudaHostAlloc, or
 * cudaHostRegister with the mapped flag), the step writes s into it directly instead of copying
 * it back after the step. */
ds_status ds_sampler_step_host(ds_sampler* sampler, const ds_step_args* host_args, void* stream);

/* Enqueue a denoising loop on `stream` (see ds_loop_args). */
ds_status ds_denoise_loop(ds_sampler* sampler, const ds_loop_args* args, void* stream);

/* Enqueue a block-autoregressive run on `stream` (see ds_block_args). */
ds_status ds_block_loop(ds_sampler* sampler, const ds_block_args* args, void* stream);

/* Enqueue the hidden-state stand-in alone: H_out = bf16(tanh(W . [bf16(s_prev); E[canvas]]))
 * for sequences with done == 0 (done may be NULL). W [d, 2d] bf16, s_prev [B, L, d] float,
 * E [V, d] bf16, canvas [B, L] int32, H_out [B, L, d] bf16, all [device]. */
ds_status ds_standin_hidden(ds_sampler* sampler, const void* W, const float* s_prev,
                            const void* E, const int32_t* canvas, const uint8_t* done,
                            void* H_out, int32_t batch, void* stream);

/* ---- vocabulary shards ----------------------------------------------------------------
 * The step over a vocabulary split into shards (contiguous token ranges, e.g. one per GPU):
 * the softmax statistics, the entropy, s = softmax(y) . E and the Gumbel-max sample of the
 * full vocabulary decompose over any partition of it ("DiffusionGemma Technical Report",
 * section 6 "Sampling": softmax and self-conditioning matmul over the full vocabulary; the
 * pages give no multi-GPU sampler, the decomposition is the plain identity). Each shard runs
 * ds_sampler_step_shard on its rows of E and writes a partial record; the records of all
 * shards, gathered on one device in token order, are combined by ds_merge_shards, which writes
 * the step's outputs and the state update exactly as ds_sampler_step does. Draws use global
 * token indices, so the merged sample is the full-vocabulary one.
 *
 * Partial record of one shard (caller-owned [device] buffers; R = B * L rows):
 *   rows  [R] ds_shard_row   the shard's softmax statistics: maximum m_q of y, normaliser
 *                            l_q = sum exp(y - m_q), entropy of the shard's renormalised
 *                            softmax, and its argmax (global token, lowest on ties)
 *   best  [R] ds_shard_best  top_k == 0: the shard's Gumbel-max race winner: score = -key
 *                            (key = E_j / exp(y_j - m_q), the exponential-race form), token
 *                            (global), lnp = y_token - m_q
 *   O     [R, d] float       sum_j exp(y_j - m_q) E_j over the shard (not divided by l_q)
 *   cand  [R, top_k]         top_k > 0: the shard's top_k candidates {y, global token}
 *                            (unused slots: token INT32_MAX); NULL when top_k == 0
 * For ds_merge_shards the four pointers address n_shards records stacked in token order
 * (rows [n, R], best [n, R], O [n, R, d], cand [n, R, top_k]). */
typedef struct ds_shard_row {
  float m;
  float l;
  float entropy;
  int32_t argmax;
} ds_shard_row;
typedef struct ds_shard_best {
  float score;
  int32_t token;
  float lnp;
  int32_t reserved;
} ds_shard_best;
typedef struct ds_shard_cand {
  float y;
  int32_t token;
} ds_shard_cand;
typedef struct ds_shard_partial {
  ds_shard_row* rows;
  ds_shard_best* best;
  float* O;
  ds_shard_cand* cand;
} ds_shard_partial;

/* Enqueue the partial record of one shard: the sampler's vocab is the shard's size (a multiple
 * of 256), args->E its rows [vocab, d] (bf16, tensor-core path only: else DS_ERR_UNSUPPORTED),
 * token_offset the global index of its first token (a multiple of 256) and vocab_total the
 * full vocabulary (token_offset + vocab <= vocab_total <= 2^24; else DS_ERR_INVALID_ARG).
 * Uses args->batch, seed, H, E, temperature, step and done; canvas, lock and the outputs are
 * neither read nor written. Finished sequences' records are left untouched. */
ds_status ds_sampler_step_shard(ds_sampler* sampler, const ds_step_args* args,
                                int32_t token_offset, int64_t vocab_total,
                                const ds_shard_partial* out, void* stream);

/* Enqueue the merge of n_shards partial records (1 <= n_shards <= 64, else
 * DS_ERR_INVALID_ARG; n_shards * top_k <= 8192, else DS_ERR_UNSUPPORTED) into the
 * step's outputs (s, sampled, conf, entropy, argmax) and the lock / re-noise / stop update of
 * args (all [device], as for ds_sampler_step; H, E and temperature are not read and may be
 * NULL), re-noising over vocab_total tokens. The sampler
 * must have the shards' canvas_len, d_model, top_k, max_steps and lock rule (its vocab is not
 * used). With top_k > 0 the sample is drawn from the top_k of the shards' pooled candidates. */
ds_status ds_merge_shards(ds_sampler* sampler, const ds_step_args* args, int32_t n_shards,
                          const ds_shard_partial* parts, int64_t vocab_total, void* stream);

/* Synchronise the sampler's device and report (then clear) the device error word:
 * DS_OK, DS_ERR_TIMEOUT or DS_ERR_DEVICE. */
ds_status ds_sampler_device_status(ds_sampler* sampler, ds_status* out);

/* Philox4x32-10 blocks on the device, for checking the generator: out[i] = Philox(ctr[i], key)
 * with key = (seed low word, seed high word). ctr and out are [n, 4] uint32 [device]. */
ds_status ds_philox4x32_10(const uint32_t* ctr, uint64_t seed, uint32_t* out, int64_t n,
                           void* stream);

/* Per-phase device timing of ds_sampler_step, for profiling. enable = 1: every step records
 * CUDA events on its stream around each phase and accumulates the elapsed times:
 *   0 logits GEMM, 1 softmax statistics, 2 top-k candidates, 3 exp(y - m) split + Gumbel-max,
 *   4 self-conditioning GEMM, 5 reduction of s + finalize, 6 lock / re-noise / stop.
 * enable = 2 (coarse): only the ends of phases 0, 3, 4 and 6 are marked, so phases 1-3 are
 * accumulated under 3 and phases 5-6 under 6 (fewer events between the kernels, which then
 * run closer to their untimed schedule). enable = 0 switches timing off; other values are
 * DS_ERR_INVALID_ARG. ds_sampler_phase_times synchronises the stream of the last timed step,
 * writes up to n accumulated milliseconds (per phase, summed over *steps steps) and resets the
 * totals. Not for use inside stream capture. */
ds_status ds_sampler_set_phase_timing(ds_sampler* sampler, int32_t enable);
ds_status ds_sampler_phase_times(ds_sampler* sampler, float* ms, int32_t n, int32_t* steps);

/* Number of kernels the sampler has enqueued since creation (steps, loops, stand-in calls;
 * a loop captured in a graph counts its kernels once per capture). */
ds_status ds_sampler_launch_count(const ds_sampler* sampler, int64_t* count);

/* One sampler step that allocates no device memory.
 * The paper has no counterpart to this entry point; it exists for callers that cannot allocate
 * when they run a step: a serving engine that reserves (almost) all HBM for its own pools at
 * start-up and forbids later allocations, or a latency-critical path where cudaMalloc/cudaFree
 * would synchronise the device and stall other streams. Such callers cannot use
 * ds_sampler_create (it allocates a workspace), so this call needs no sampler at all.
 *   cfg   shapes and options as for ds_sampler_create (max_batch is not used);
 *   args  inputs and outputs exactly as for ds_sampler_step (all [device]); args->batch >= 1.
 * The step's scratch (logits, statistics, the probability split, partial sums) is carved from
 * one fixed 64 MiB array inside the library, which every GPU that loads the library holds until
 * the process exits. A step whose scratch would not fit returns DS_ERR_UNSUPPORTED and enqueues
 * nothing; the scratch is about 8*B*L*V + 4*S*B*L*d bytes (S = vocabulary splits of the
 * self-conditioning GEMM), e.g. B=1, L=256, V=32768, d=1024 does not fit and V=16384 does.
 * The first call on a device looks up the array's device address (a one-time set-up with that
 * device current, repeated only if the device's context is replaced, e.g. after a device
 * reset); make that first call before any stream capture. Every call shares the one array and
 * it keeps the last call's contents (the call clears what must start at zero): calls whose work
 * overlaps on the GPU -- two streams, or two host threads -- race on it and must be serialised
 * by the caller. Nothing is allocated: no cudaMalloc, cudaFree or allocating library routine is
 * called. The configuration is checked as by ds_sampler_create (max_batch aside);
 * cfg->impl == DS_IMPL_FUSED is refused with DS_ERR_UNSUPPORTED (this entry point runs the
 * separate logits and self-conditioning GEMMs only). A bounded wait that runs out inside the
 * step's kernels is not reported by the return value (the call returns once the work is
 * enqueued): read it with ds_sampler_noalloc_status after the step's work has completed. */
ds_status ds_sampler_step_noalloc(const ds_sampler_config* cfg, const ds_step_args* args,
                                  void* stream);

/* Device status of the last ds_sampler_step_noalloc call on the current device: synchronises
 * `stream` (the stream that call used), reads the device error word kept in the same fixed
 * array and clears it. *out = DS_OK, DS_ERR_TIMEOUT (a kernel's bounded wait ran out, so that
 * step's outputs and state update are not valid) or DS_ERR_DEVICE (another device-side check
 * failed). Each no-allocation step clears the word when it starts, so read it before the next
 * one. Allocates nothing. */
ds_status ds_sampler_noalloc_status(void* stream, ds_status* out);

/* Self-test of the kernels' bounded waits: enqueues one small kernel that waits on an
 * mbarrier no thread will ever complete, gives up after limit_ns nanoseconds (1 us .. 1 s),
 * records DS_ERR_TIMEOUT in the device error word and returns normally. The context stays
 * usable; ds_sampler_device_status then reports (and clears) the time-out. This is how the
 * time-out path of the pipelines is exercised without faulting or hanging a GPU. */
ds_status ds_sampler_selftest_wait(ds_sampler* sampler, int64_t limit_ns, void* stream);

/* Read-only view of an internal buffer of the last step, for tests and profiling.
 * which: 0 = scaled logits y [B*L, V] float (only where the step materialises them: top_k > 0
 * or the CUDA-core path; else DS_ERR_UNSUPPORTED); 1 = row statistics [B*L] x {m, l, entropy,
 * argmax}; 2 = bf16 high part of the probabilities [B*L, V]; 3 = bf16 low part. Their reference:
 * exp(y - m) with m the row maximum where y is materialised (CUDA-core path); on the tensor-core
 * path (DS_IMPL_TENSOR / AUTO), exp(y - m_t) with m_t the row's maximum over the token's
 * 256-token tile; in the fused pass (DS_IMPL_FUSED), exp(y - m_g) with m_g the maximum of the
 * token's 128-token segment. 4 = the 128-token segment records of the tensor-core paths
 * [B*L, V/128] x {m_g, sum exp(y - m_g), sum exp(y - m_g)(y - m_g), argmax_g} (16 bytes each;
 * DS_ERR_UNSUPPORTED on the other paths). *ptr is [device]. */
ds_status ds_sampler_debug_buffer(ds_sampler* sampler, int32_t which, const void** ptr,
                                  size_t* bytes);

#ifdef __cplusplus
}
#endif
#endif /* DS_SAMPLER_H */
