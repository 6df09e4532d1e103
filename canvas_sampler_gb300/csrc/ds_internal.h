// Host-side interface between the C ABI (ds_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/ds_sampler.h"
#include "ds_common.cuh"

namespace ds {

// Vocabulary chunk handled by one CTA of the row kernels (256 threads x 32 values).
constexpr int kChunk = 8192;
// Most partial sums of s that the finalize kernel combines.
constexpr int kMaxSplits = 256;
// Most vocabulary shards one merge combines.
constexpr int kMaxShards = 64;
// Largest top-k the sampler supports, and the largest candidate pool its merge takes.
constexpr int kMaxTopK = 256;
constexpr int kMaxTopKPool = 8192;

inline int n_chunks_of(int64_t V) { return (int)((V + kChunk - 1) / kChunk); }

// Whether kernels of a step are launched with programmatic stream serialisation (each may start
// while its predecessor finishes; it waits in-kernel before using the predecessor's results).
// On unless DS_PDL=0 in the environment.
bool pdl_enabled();

// Launch `kernel` on `st`, with programmatic stream serialisation when pdl_enabled().
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Checks of a sampler configuration shared by ds_sampler_create and the no-allocation step
// (everything but max_batch): DS_OK, DS_ERR_INVALID_ARG or DS_ERR_UNSUPPORTED (a top-k candidate
// pool beyond kMaxTopKPool).
ds_status validate_config(const ds_sampler_config& c);

// ---- row kernels (ds_rows.cu) ----
void launch_chunk_stats(const float* Y, int R, int64_t V, int L, const uint8_t* done,
                        ChunkStat* cs, cudaStream_t st);
void launch_row_merge(const ChunkStat* cs, int n_chunks, int R, int L, const uint8_t* done,
                      RowStat* rs, cudaStream_t st);
// blk: the block index of a block-autoregressive run (device int32, or nullptr for 0); every
// launcher that draws random numbers takes it (counter word 2 = sequence + 2^16 block).
void launch_convert(const float* Y, const RowStat* rs, int R, int64_t V, int L,
                    const uint8_t* done, const int32_t* step, uint64_t seed, const int32_t* blk,
                    bool gumbel, uint16_t* Phi, uint16_t* Plo, Best* best, cudaStream_t st);
void launch_topk_chunk(const float* Y, int R, int64_t V, int L, const uint8_t* done, int k,
                       Cand* cand, cudaStream_t st);
// The row's top k from the stored probabilities (bf16 hi + lo relative to the tile maxima
// mtile_t [V/256, R]), pruned by the 128-token segment maxima seg [R, V/128]: k candidates per
// row (cand [R, k]) carrying y = m + ln p.
void launch_topk_row(const uint16_t* Phi, const uint16_t* Plo, const ChunkStat* seg,
                     const float* mtile_t, const RowStat* rs, int R, int64_t V, int L,
                     const uint8_t* done, int k, Cand* cand, cudaStream_t st,
                     int64_t j_offset = 0);
void launch_finalize(const RowStat* rs, const Best* best, const Cand* cand, int n_chunks, int k,
                     int R, int L, const uint8_t* done, const int32_t* step, uint64_t seed,
                     const int32_t* blk, int32_t* sampled, float* conf, float* entropy,
                     int32_t* argmax, cudaStream_t st);
// launch_finalize plus the reduction of s (launch_reduce_s) in the same per-row kernel.
void launch_finalize_with_s(const RowStat* rs, const Best* best, const Cand* cand, int n_chunks,
                            int k, int R, int L, const uint8_t* done, const int32_t* step,
                            uint64_t seed, const int32_t* blk, int32_t* sampled, float* conf,
                            float* entropy, int32_t* argmax, const float* Opart, int S, int d,
                            float* s, const float* mref, cudaStream_t st);
// The Gumbel race of a step over (row, 8192-token chunk) items, each raced by one warp (see
// gumbel_chunk_warp). As a queue (inside the self-conditioning launch): ctr[0] is the next item,
// ctr[1] counts the CTAs of the launch that have finished; the last CTA returns both to zero, so
// they are zero between launches, and advances the generation ctr[2] (zero all three once when
// allocated).
struct GumbelWork {
  const uint16_t* Phi;
  const uint16_t* Plo;
  const ChunkStat* seg;  // segment statistics [R, V/128]
  const RowStat* rs;
  const uint8_t* done;
  const int32_t* step;
  const int32_t* blk;
  uint64_t seed;
  Best* best;  // [R, n_chunks]
  uint32_t* ctr;
  int R, L, n_chunks;
  int tile_ref;  // probabilities relative to 256-token tile maxima (else to segment maxima)
  // In the queue only: with rs_out, the queue's first R items merge the rows' segment statistics
  // into rs_out (= rs) as k_row_merge does, bit for bit, and each row's race items wait until
  // row_flags[r] holds this launch's generation (ctr[2] + 1); a wait that runs out sets
  // kErrTimeout in err.
  RowStat* rs_out;
  uint32_t* row_flags;  // [R], zero when allocated
  uint32_t* err;
  // Global index of the first token of the vocabulary the probabilities cover (a vocabulary
  // shard's step): the race's draws and its winners use global token indices.
  int64_t j_offset;
};

// Gumbel-max sample per (row, chunk) from probabilities stored relative to each 128-token
// segment's maximum (tile_ref = false, the fused pass) or to the maximum over each 256-token
// tile (tile_ref = true), with the segment statistics seg [R, V/128] (Best records).
void launch_gumbel_items(const uint16_t* Phi, const uint16_t* Plo, const ChunkStat* seg,
                       const RowStat* rs, int R, int64_t V, int L, const uint8_t* done,
                       const int32_t* step, uint64_t seed, const int32_t* blk, bool tile_ref,
                       Best* best, cudaStream_t st, int64_t j_offset = 0);
void launch_reduce_s(const float* Opart, int S, int R, int d, int L, const uint8_t* done,
                     const RowStat* rs, float* s, cudaStream_t st);
// A vocabulary shard's step record (k_shard_export) and the merge of n shards' records
// (k_shard_merge, then launch_finalize over its row statistics and winner / candidate pool);
// see ds_rows.cu.
void launch_shard_export(const RowStat* rs, const Best* best, int n_chunks, const Cand* cand,
                         int k, int R, int L, const uint8_t* done, const float* Opart, int S,
                         int d, const float* mref, int64_t j_offset, RowStat* rows_out,
                         Best* best_out, float* O_out, Cand* cand_out, cudaStream_t st);
void launch_shard_merge(int n, const RowStat* rows, const Best* best, const float* O,
                        const Cand* cand, int k, int R, int d, int L, const uint8_t* done,
                        RowStat* rs_out, Best* best_out, Cand* pool_out, float* s_out,
                        cudaStream_t st);
void launch_lock(int B, int L, int64_t V, int max_steps, uint64_t seed, const int32_t* blk,
                 const float* tau, const int32_t* sampled, const float* conf, int32_t* step,
                 int32_t* canvas, uint8_t* lock, uint8_t* done, cudaStream_t st);
void launch_temperature(const int32_t* step, int B, float t_start, float t_end, int max_steps,
                        float* T, cudaStream_t st);
void launch_lock_entropy(int B, int L, int64_t V, int max_steps, uint64_t seed,
                         const int32_t* blk, float budget, float stop_entropy,
                         const int32_t* sampled, const float* entropy, const int32_t* argmax,
                         int32_t* prev_argmax, int32_t* step, int32_t* canvas, uint8_t* lock,
                         uint8_t* done, cudaStream_t st);
void launch_wait_selftest(uint64_t limit_ns, uint32_t* err, cudaStream_t st);
void launch_philox(const uint32_t* ctr, uint64_t seed, uint32_t* out, int64_t n, cudaStream_t st);
void launch_loop_begin(const uint8_t* done, int B, int32_t* iter, int max_iters,
                       cudaGraphConditionalHandle h, cudaStream_t st);
void launch_loop_end(const uint8_t* done, int B, int32_t* iter, int max_iters,
                     cudaGraphConditionalHandle h, cudaStream_t st);
// Block-autoregressive driver (ds_block_loop). ctl[0] = block index (the blk word of the
// kernels above), ctl[1] = action of the last check (0 continue, 1 commit and start the next
// block, 2 commit, all blocks finished), ctl[2] = local index of the block to commit, ctl[3] =
// iterations. start: block first_block, state from init_canvas[0]; check (one warp): decide and,
// when use_cond, set the loop condition; rollover: commit and reset per the decision.
struct BlockState {
  int32_t* canvas;
  uint8_t* lock;
  int32_t* step;
  uint8_t* done;
  int32_t* prev_argmax;  // may be nullptr
  float* s;
};
void launch_block_start(int32_t* ctl, int first_block, const int32_t* init_canvas, BlockState bs,
                        int B, int L, int d, cudaStream_t st);
void launch_block_check(int32_t* ctl, const uint8_t* done, int B, int first_block, int n_blocks,
                        int max_iters, bool use_cond, cudaGraphConditionalHandle h,
                        cudaStream_t st);
void launch_block_rollover(const int32_t* ctl, const int32_t* init_canvas, int32_t* out_canvas,
                           int32_t* out_steps, BlockState bs, int B, int L, int d,
                           cudaStream_t st);

// ---- CUDA-core GEMMs (ds_simt.cu) ----
void launch_logits_simt(const void* H, const void* E, bool fp32_inputs, int R, int64_t V, int d,
                        int L, const float* T, const uint8_t* done, float* Y, cudaStream_t st);
void launch_selfcond_simt(const uint16_t* Phi, const uint16_t* Plo, const void* E,
                          bool fp32_inputs, int R, int64_t V, int d, int L, const uint8_t* done,
                          int S, float* Opart, cudaStream_t st);
// Both stand-in launchers read E[canvas[r]]: a token outside [0, V) is clamped into E and sets
// kErrBounds in err.
void launch_standin_simt(const uint16_t* W, const float* s_prev, const uint16_t* E,
                         const int32_t* canvas, const uint8_t* done, int R, int d, int L,
                         int64_t V, uint32_t* err, uint16_t* H_out, cudaStream_t st);

// ---- tensor-core GEMMs (ds_tc.cu host side, ds_tc_logits.cu, ds_tc_selfcond.cu) ----
// Resolves the driver's tensor-map encoder; false when unavailable.
bool tc_available();
int tc_num_sms();
// 2-D tensor maps (128-byte swizzle) over a row-major [rows, cols] array, box [box_rows, box_cols].
bool tc_make_map_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                      uint32_t box_rows, uint32_t box_cols);
bool tc_make_map_f32(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows, uint32_t box_cols);
// The same with a 64-byte swizzle (boxes of 32 bf16 columns).
bool tc_make_map_bf16_sw64(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint32_t box_rows, uint32_t box_cols);
void tc_prepare_logits();
void tc_prepare_selfcond();
// Also writes the softmax statistics of every 128-token segment of every row:
// seg_stats [R, V / kTcSegment].
constexpr int kTcSegment = 128;
cudaError_t launch_logits_tc(const uint16_t* H, const uint16_t* E, int R, int64_t V, int d, int L,
                             const float* T, const uint8_t* done, float* Y, ChunkStat* seg_stats,
                             uint32_t* err, cudaStream_t st);
// Whether the logits GEMMs run as CTA pairs (M = 256 tiles over two SMs) for R rows: R % 256 ==
// 0 and not switched off by DS_LOGITS_PAIR=0 in the environment.
bool logits_pair_enabled(int R);
// The same GEMM writing, instead of y, P = exp(y - m_t) as bf16 hi + lo (m_t the row's maximum
// over the token's 256-token tile) and m_t tile-major in mtile_t [V/256, R].
cudaError_t launch_logits_p_tc(const uint16_t* H, const uint16_t* E, int R, int64_t V, int d,
                               int L, const float* T, const uint8_t* done, uint16_t* Phi,
                               uint16_t* Plo, ChunkStat* seg_stats, float* mtile_t, uint32_t* err,
                               cudaStream_t st);
// H = bf16(tanh(U . W^T)) for U [R, 2d] bf16, W [d, 2d] bf16 (d % 256 == 0).
cudaError_t launch_standin_tc(const uint16_t* U, const uint16_t* W, int R, int d, int L,
                              const uint8_t* done, uint16_t* H_out, uint32_t* err,
                              cudaStream_t st);
// U [R, 2d] = [bf16(s_prev) | E[canvas]] for the stand-in (rows of done sequences skipped).
void launch_standin_gather(const float* s_prev, const uint16_t* E, const int32_t* canvas,
                           const uint8_t* done, int R, int d, int L, int64_t V, uint32_t* err,
                           uint16_t* U, cudaStream_t st);
// With mtile_t set, P is relative to the row's maximum over each 256-token tile (mtile_t
// [V/256, R]) and the reference maximum of each split's partial goes to mref [S, R] (see
// ds_tc_selfcond.cu).
// With gw (not nullptr; tensor-core step without top-k) the same launch also runs the Gumbel race
// of the step (the work of launch_gumbel_items with tile_ref) on warps of its own beside the GEMM.
cudaError_t launch_selfcond_tc(const uint16_t* Phi, const uint16_t* Plo, const uint16_t* E, int R,
                               int64_t V, int d, int L, const uint8_t* done, int S, float* Opart,
                               const float* mtile_t, float* mref, uint32_t* err,
                               const GumbelWork* gw, cudaStream_t st);
// Split count of the tensor-core self-conditioning GEMM for a shape.
int selfcond_tc_splits(int R, int64_t V, int d, int num_sms);

// ---- fused vocabulary pass (ds_tc_fused.cu) ----
// One cooperative persistent kernel: logits, segment statistics and the bf16 hi/lo
// probabilities (producer CTAs), and the self-conditioning partials per vocabulary range with
// their reference maxima (consumer CTAs).
constexpr int kVpSegment = 128;  // tokens per segment of SegStat
struct VocabPassShape {
  int n_rt, n_vt, n_dt;  // row tiles (128), vocabulary tiles (256), d tiles (256)
  int kvt;               // vocabulary tiles per consumer range
  int n_ranges;          // consumer ranges
  int producers;         // CTAs that start as producers
  int grid;              // CTAs (one per SM)
};
void tc_prepare_vocab_pass();
// Shape of the pass for R rows (0 grid when the fused pass cannot run: d % 256 != 0 or the
// kernel does not fit one CTA per SM). `producers` <= 0 picks the default split.
VocabPassShape vocab_pass_shape(int R, int64_t V, int d, int num_sms, int producers);
// Words of the control block (queue counters, ready flags); zeroed before every launch.
size_t vocab_pass_sync_words(const VocabPassShape& sh);
cudaError_t launch_vocab_pass_tc(const VocabPassShape& sh, const uint16_t* H, const uint16_t* E,
                                 int R, int64_t V, int d, int L, const float* T,
                                 const uint8_t* done, const int32_t* step, uint64_t seed,
                                 uint16_t* Phi, uint16_t* Plo, ChunkStat* seg, float* mseg_t,
                                 float* Opart, float* mref, uint32_t* sync, uint32_t* err,
                                 cudaStream_t st);


}  // namespace ds
