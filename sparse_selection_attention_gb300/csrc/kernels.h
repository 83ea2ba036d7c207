// Kernel parameter blocks and launchers (internal to the library).
#pragma once

#include "common.cuh"

namespace qsa {

struct ScoresParams {
  PoolDev pools[QSA_MAX_POOLS];
  int unit_begin[QSA_MAX_POOLS + 1];  // prefix sums of each pool's block count
  int row_pool[QSA_MAX_DECODE_ROWS];
  int n_pools, total_units;
  int n_rows, n_q_heads, n_kv_heads, block_cells, max_blocks;
  int q_rows_per_batch;   // rows of q staged in shared memory at a time
  int frag_smem;          // decode window: 1 when the scores kernel stages the q fragments in shared memory
  int own_frag;           // decode window: 1 when each scores CTA makes the q fragments itself (small windows)
  const float* q;
  float* scores;
  int* err;               // device error word (bounded waits of the staged kernel)
  unsigned long long wait_limit_ns;
};

struct TopkParams {
  const float* scores;
  int max_blocks;
  int n_filled[QSA_MAX_DECODE_ROWS];
  int n_rows, block_cells, k_cells;
  int32_t* ids;
  int32_t* n_sel;
};

struct AttnParams {
  PoolDev pools[QSA_MAX_POOLS];
  int row_pool[QSA_MAX_DECODE_ROWS];
  const float* q;
  const int32_t* row_pos;
  const int32_t* ids;
  const int32_t* n_sel;
  int n_rows, n_q_heads, n_kv_heads, k_cells, chunk_cells, n_chunks;
  float* ml;  // [n_rows][n_q_heads][n_chunks][2]
  float* o;   // [n_rows][n_q_heads][n_chunks][128]
};

// Byte offset of the o region in a chunk-partials buffer of n (row, head, chunk) entries: the
// (m, l) pairs first, then o from the next 256-byte boundary, so that o is aligned for vector
// stores whatever n is.
inline size_t partials_o_offset(size_t n) { return (sizeof(float) * 2 * n + 255) & ~(size_t)255; }

struct MergeParams {
  const float* ml;
  const float* o;
  const int32_t* n_sel;
  int n_rows, n_q_heads, chunk_cells, n_chunks;
  float* out;
  float* lse;
};

struct PromptParams {
  PoolDev pool;
  int n_kv_heads, n_q_heads, n_q, q_pos0;
  const float* q;
  float* out;
  float* lse;
  uint8_t* scratch;   // header, tile images and part records (prompt_scratch_bytes)
  int n_tiles;        // 64-cell tiles the call reads: (q_pos0 + n_q - 1) / 64 + 1
  // Work units: (block of qpc queries, KV head), unit u = kv_head * n_qb + query block.  Units below
  // n_whole run as one CTA each; each later unit runs as n_split CTAs over equal tile ranges whose
  // partial rows go to part_o / part_ml and are combined by prompt_merge_kernel.
  int qpc, n_qb, n_whole, n_split;
  float* part_o;      // [n_parts][128 rows][128]  unnormalised O of a part, in output units
  float* part_ml;     // [n_parts][128 rows][2]    (running max m in log2 units, row sum l)
  unsigned long long wait_limit_ns;
};

// Quantise-on-append of new cells (qsa_kv_append): the pool read through `pool`, its code and
// scale arrays written through the other pointers.
struct AppendParams {
  PoolDev pool;
  int8_t* k_codes;
  uint8_t* v_codes;
  float* k_scales;
  float* v_scales;
  const float* k;   // [n_new][n_kv_heads][128]
  const float* v;
  int n_kv_heads, first_cell, n_new;
};

// How a prompt call is cut into CTAs for a device with n_sm SMs, and the scratch it needs.
struct PromptPlan {
  int qpc, n_qb, n_units, n_whole, n_split, n_parts;
  size_t images_offset, parts_offset, ml_offset, bytes;
};

// Split attention + fused merge of a decode window (qsa_decode_window).
struct WinAttnParams {
  PoolDev pools[QSA_MAX_POOLS];
  int row_pool[QSA_MAX_DECODE_ROWS];
  const float* q;
  const int32_t* row_pos;
  const int32_t* ids;
  const int32_t* n_sel;
  int n_rows, n_q_heads, n_kv_heads, k_cells;
  int split_cells;   // cells of one split (multiple of 16)
  int n_splits;      // splits per (row, q head) in the workspace
  float* part_ml;    // [n_rows][n_q_heads][n_splits][2]
  float* part_o;     // [n_rows][n_q_heads][n_splits][128]
  float* out;        // [n_rows][n_q_heads][128]
  float* lse;        // [n_rows][n_q_heads] or nullptr
};

// Byte offsets of the parts of a decode-window workspace.
struct WindowLayout {
  size_t frag, inv_f, part_ml, part_o, q_in, pos_in, total;
  int split_cells, n_splits;
};

struct WindowArgs {
  ScoresParams scores;
  TopkParams topk;
  int max_nb;
  WinAttnParams attn;
  WindowLayout layout;
  void* workspace;
  // Inputs in page-locked host memory (device aliases), staged into the workspace's q_in / pos_in by
  // the window's first launch; the other launches then read the staged copies.  NULL: q and row_pos
  // are device memory, read in place.
  const float* q_src;
  const int32_t* pos_src;
};

WindowLayout window_layout(int n_rows, int n_q_heads, int n_kv_heads, int k_cells, int n_sm);
bool window_scores_supported(int n_rows, int n_kv_heads, int block_cells);
cudaError_t launch_decode_window(const WindowArgs& a, cudaStream_t stream, cudaEvent_t* ev = nullptr);
// Top-k launch; with pdl the launch may start before the preceding kernel of the stream ends.
cudaError_t launch_topk_ex(const TopkParams& p, int max_nb, cudaStream_t stream, bool pdl);

bool prompt_plan(int v_bits, int n_kv_heads, int n_q_heads, int n_q, int q_pos0, int n_sm, PromptPlan* plan);
size_t block_scores_smem_bytes(int n_rows, int n_q_heads, int n_kv_heads, int block_cells);
bool block_scores_supported(int n_kv_heads, int block_cells);
int block_scores_q_rows_per_batch(int n_rows, int n_q_heads, int n_kv_heads, int block_cells);
size_t topk_smem_bytes(int max_nb);
cudaError_t launch_block_scores(const ScoresParams& p, cudaStream_t stream);
cudaError_t launch_topk(const TopkParams& p, int max_nb, cudaStream_t stream);
cudaError_t launch_decode_attn(const AttnParams& p, cudaStream_t stream);
// qsa_decode_attn through the decode window's attention kernels (4-bit K; decode_window.cu).
cudaError_t launch_chunk_attn_window_kernels(const AttnParams& p, cudaStream_t stream);
cudaError_t launch_attn_merge(const MergeParams& p, cudaStream_t stream);
cudaError_t launch_attn_merge_ex(const MergeParams& p, cudaStream_t stream, bool pdl);
cudaError_t launch_prompt_attn(const PromptParams& p, cudaStream_t stream);
cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream);
// Block summaries (block_sums.cu): (re)writes the summaries of the 64-cell blocks that cells
// first_cell .. first_cell + n_cells - 1 fall in, each over its cells below first_cell + n_cells;
// block scores from the summaries when every pool keeps them and block_cells is a multiple of 64.
cudaError_t launch_summarise(const PoolDev& pool, float* k_sums, int n_kv_heads, int first_cell, int n_cells,
                             cudaStream_t stream);
bool block_sums_usable(const ScoresParams& p);
cudaError_t launch_sum_scores(const ScoresParams& p, cudaStream_t stream, bool pdl);
cudaError_t read_and_clear_device_error(int32_t* code, cudaStream_t stream);
// Dense tcgen05 rate (tc_rate.cu): times `passes` x 4 MMAs of M = 128, N = 256 per SM on the
// legacy default stream; *ms the launch's event time, *ops the operations it performed.
cudaError_t run_tc_rate(int kind_i8, int passes, float* ms, double* ops);
unsigned long long wait_limit_ns();
// Device address of the library's error word on the current device (for kernels of other
// translation units), or nullptr.
int* device_error_word();

}  // namespace qsa
