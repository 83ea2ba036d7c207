/*
 * qsa.h -- C ABI of the GB300 (sm_103a) QSA attention library.
 *
 * QSA ("sparse selection") attention reads a paged KV cache whose K and V are
 * stored as int8 codes (or int8 K with 4-bit V) with one fp32 scale per
 * (cell, KV head, dim group).  The decode side scores 64-cell blocks, keeps
 * the cells of the top-scoring blocks, runs split-KV attention over them in
 * chunks and merges the chunks by log-sum-exp.  The prompt side runs causal
 * attention of a chunk of many queries over the whole cached context.
 *
 * Sources (pull-request pages of the "Strata" inference engine):
 *   #1888  "QSA decode attention: split each query's cells across blocks on
 *           the int8 mma path" -- Summary, What changed.
 *   #2075  "QSA decode attention: PR #540's two-cells-per-step chunk kernel on
 *           every CUDA card and a bounded merge" -- Summary, Bit for bit.
 *   #600   "qsa_prompt_attn: tensor-core kernel for Volta" -- description.
 *   #2806  "sycl: decode QSA selection and attention in fewer, shorter
 *           launches" -- Summary (switch table), What changed.
 *   #1367  "prompt attention: STRATA_PROMPT_ATTN_IMMA=1 - the int8-KV kernel
 *           on INT8 tensor cores" -- What it does.
 *
 * Conventions shared by every call
 *   - Memory is owned by the caller.  Pointers marked (dev) are device
 *     pointers on the current CUDA device, (host) are host pointers read
 *     before the call returns.  No call allocates device memory.
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream.  Work is enqueued asynchronously on it.
 *   - Arguments are validated on the host before anything is enqueued.  Any
 *     status other than QSA_OK means nothing was enqueued, except
 *     QSA_ERR_CUDA, which reports a failed launch (as #1888 What changed:
 *     the launcher returns without launching when it cannot serve a call).
 *   - head_dim is 128.  K scales cover 64-dim groups; int8 V scales 64-dim
 *     groups, 4-bit V scales 32-dim groups.
 *   - Results are deterministic: the same inputs and sizes give the same bits
 *     on every run (fixed reduction orders; #2075 Bit for bit).
 */
#ifndef QSA_GB300_H
#define QSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QSA_OK = 0,
  QSA_ERR_ARG = 1,          /* invalid argument (null pointer, bad size, misaligned) */
  QSA_ERR_UNSUPPORTED = 2,  /* valid request outside this build's limits */
  QSA_ERR_SCRATCH = 3,      /* caller's scratch buffer is too small */
  QSA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  QSA_ERR_DEVICE = 5        /* a kernel reported an error through the device error word */
} qsa_status;

/* Limits of this build (host-validated). */
#define QSA_HEAD_DIM 128
#define QSA_MAX_POOLS 4          /* pool sets per launch (#2806 What changed: up to four) */
#define QSA_MAX_DECODE_ROWS 32   /* rows of one decode window */
#define QSA_MAX_GROUP 8          /* q heads per KV head on the decode side */
#define QSA_MAX_TOPK_BLOCKS 16384
#define QSA_MAX_KV_HEADS 16      /* KV heads of a pool */
#define QSA_MAX_CHUNKS 8192      /* chunks per (row, q head) of the chunk partials */

/*
 * One slot's paged KV pool.  All pointers (dev), 16-byte aligned, caller-owned.
 *   k_codes    k_bits 8: int8 [n_pages][n_kv_heads][page_cells][128]
 *              k_bits 4: uint8 [n_pages][n_kv_heads][page_cells][64], packed as
 *              4-bit V codes are (the q4_0 layout with v_bits 4)
 *   v_codes    v_bits 8: int8 [n_pages][n_kv_heads][page_cells][128]
 *              v_bits 4: uint8 [n_pages][n_kv_heads][page_cells][64]; byte j
 *              holds dim 2j in its low nibble and dim 2j+1 in its high nibble,
 *              nibble = code + 8 (code in [-8, 7])
 *   k_scales   fp32   [n_pages][n_kv_heads][page_cells][128 / k_group],
 *              k_group = 64 (k_bits 8) or 32 (k_bits 4)
 *   v_scales   fp32   [n_pages][n_kv_heads][page_cells][128 / v_group],
 *              v_group = 64 (v_bits 8) or 32 (v_bits 4)
 * Every call serves 4-bit K.  The pools of one call share k_bits.
 *   page_table int32  [ceil(capacity / page_cells)] logical -> physical page
 *   k_sums     fp32   [n_pages][n_kv_heads][page_cells / 64][128], or NULL:
 *              optional block summaries, for each 64-cell block of a page the
 *              sum over its cells of the dequantised K rows (kcode * kscale),
 *              in ascending cell order.  When every pool of a call keeps them
 *              and block_cells is a multiple of 64, qsa_block_scores and
 *              qsa_decode_window score blocks from them (the same S[t,b],
 *              512 bytes per 64 cells and KV head read instead of the codes
 *              and scales).  They must describe exactly cells 0 .. n_filled-1:
 *              qsa_kv_append keeps them so for in-order appends;
 *              qsa_kv_summarise (re)builds them.
 * Logical cell c is at physical page page_table[c / page_cells], offset
 * c % page_cells.  Cells 0 .. n_filled-1 hold data; others are never read.
 * (Per-(cell, KV head, 64-dim group) scales: #600 description; paged pool and
 * one pool per slot: #2806 Summary.)
 */
typedef struct {
  const int8_t* k_codes;
  const void* v_codes;
  const float* k_scales;
  const float* v_scales;
  const int32_t* page_table;
  int32_t n_filled;
  int32_t capacity;
  int32_t page_cells;   /* multiple of 64 */
  int32_t n_kv_heads;   /* 1..16 */
  int32_t head_dim;     /* must be 128 */
  int32_t v_bits;       /* 8 or 4 */
  int32_t k_bits;       /* 8, or 4 for 4-bit K (the q4_0 layout) */
  const float* k_sums;  /* optional block summaries (see above), 16-byte aligned, or NULL */
} qsa_pool;

/*
 * qsa_block_scores -- decode block scores of every row of a window, one
 * launch over all slots' pools (#2806 Summary: scores once per slot; a
 * block's (query, head) sums reduced together).
 *   S[t,b] = sum_h (1/n_b) sum_{c in b} sum_{g in G(h)} q[t,g] . K[c,h] / sqrt(128)
 * where block b holds logical cells [b*B, min((b+1)*B, n_filled)), n_b of
 * them, K[c,h,d] = kcode * kscale[c,h,d/64], and q head g reads KV head
 * g / (n_q_heads / n_kv_heads).  (The pages name the step but print no
 * formula; this is the library's stated definition.)
 *   pools      (host) [n_pools] descriptors, 1 <= n_pools <= QSA_MAX_POOLS
 *   row_pool   (host) int32 [n_rows]: pool index of each row
 *   q          (dev)  fp32 [n_rows][n_q_heads][128], 16-byte aligned
 *   scores     (dev)  fp32 [n_rows][max_blocks]; entries b < ceil(n_filled/B)
 *              of each row's pool are written, the rest are left untouched
 *   block_cells B in {32, 64, 128, 256}, dividing every pool's page_cells
 *   max_blocks >= ceil(n_filled / B) of every row's pool
 * Errors: QSA_ERR_ARG on null/misaligned pointers or bad sizes;
 * QSA_ERR_UNSUPPORTED past the limits above.
 */
qsa_status qsa_block_scores(const qsa_pool* pools, int n_pools, const int32_t* row_pool,
                            const float* q, int n_rows, int n_q_heads, int block_cells,
                            float* scores, int max_blocks, void* stream);

/*
 * qsa_topk -- per row, the cells of the k_cells / B highest-scoring blocks,
 * in ascending cell id (#2806 Summary: one top-k per window; radix digits on
 * integer keys, so the ids are the same whatever the kernel).
 * Order: score descending, ties by block id ascending; -0.0 equals +0.0; a
 * NaN score ranks below -inf.  Blocks are those b < ceil(n_filled[t] / B).
 *   scores     (dev)  fp32 [n_rows][max_blocks]
 *   n_filled   (host) int32 [n_rows]: filled cells of each row's pool
 *   ids        (dev)  int32 [n_rows][k_cells]: entries [0, n_sel[t]) written
 *   n_sel      (dev)  int32 [n_rows]: number of ids of each row
 *   k_cells    multiple of block_cells, >= 0
 * Errors: QSA_ERR_ARG (bad sizes, k_cells not a multiple of block_cells);
 * QSA_ERR_UNSUPPORTED when ceil(n_filled/B) > QSA_MAX_TOPK_BLOCKS.
 */
qsa_status qsa_topk(const float* scores, int max_blocks, const int32_t* n_filled, int n_rows,
                    int block_cells, int k_cells, int32_t* ids, int32_t* n_sel, void* stream);

/*
 * Partials of the decode attention (caller scratch).  For n_rows rows,
 * n_q_heads heads and n_chunks chunks per (row, head), N = n_rows *
 * n_q_heads * n_chunks, the buffer holds
 *   float ml[n_rows][n_q_heads][n_chunks][2]      (m, l) of each chunk, at byte 0
 *   float o [n_rows][n_q_heads][n_chunks][128]    unnormalised sum p * V, at
 *                                                 byte 8 * N rounded up to a
 *                                                 multiple of 256
 * The buffer must be 16-byte aligned.  An empty chunk (no visible cell) has
 * m = -inf, l = 0, o = 0.  Returns 0 for sizes below 1.
 */
size_t qsa_decode_partials_bytes(int n_rows, int n_q_heads, int n_chunks);

/*
 * qsa_decode_attn -- split-KV chunk attention over the selected cells
 * (#2075 Summary: chunk kernel over the selection, empty chunks marked;
 * #1888 Summary: one query's cells split among blocks, ~2 blocks per SM).
 * Chunk j of row t is ids[t][j*C .. min((j+1)*C, n_sel[t])).  For every q
 * head g and chunk j < ceil(n_sel[t] / C), over the chunk's cells c with
 * c <= row_pos[t]:
 *   z_c = q[t,g] . K[c, kv(g)] / sqrt(128),  m = max z,  l = sum exp(z - m),
 *   o = sum exp(z - m) V[c, kv(g)]
 * with V[c,h,d] = vcode * vscale[c,h,d/v_group].  Chunks at or past
 * ceil(n_sel[t] / C) are not written.
 *   pools, row_pool  as qsa_block_scores
 *   q          (dev)  fp32 [n_rows][n_q_heads][128], 16-byte aligned
 *   row_pos    (dev)  int32 [n_rows]: each row's own cell (causal, inclusive)
 *   ids        (dev)  int32 [n_rows][k_cells], ids < the row pool's n_filled
 *   n_sel      (dev)  int32 [n_rows], 0 <= n_sel <= k_cells
 *   chunk_cells C: multiple of 16, 16 <= C <= 1024
 *   n_chunks   chunks per (row, head) in the partials, >= ceil(k_cells / C)
 *   partials   (dev)  scratch, partials_bytes >= qsa_decode_partials_bytes()
 * Errors: QSA_ERR_ARG, QSA_ERR_UNSUPPORTED (group > QSA_MAX_GROUP, rows >
 * QSA_MAX_DECODE_ROWS, n_chunks > QSA_MAX_CHUNKS), QSA_ERR_SCRATCH
 * (partials too small).
 */
qsa_status qsa_decode_attn(const qsa_pool* pools, int n_pools, const int32_t* row_pool,
                           const float* q, const int32_t* row_pos, const int32_t* ids,
                           const int32_t* n_sel, int n_rows, int n_q_heads, int k_cells,
                           int chunk_cells, int n_chunks, void* partials, size_t partials_bytes,
                           void* stream);

/*
 * qsa_attn_merge -- log-sum-exp merge of the chunk partials in chunk order,
 * visiting only chunks j < ceil(n_sel[t] / C) and skipping empty ones
 * (#1888 What changed: splits merged in split order; #2075 Summary:
 * attn_merge_v2 skips chunks marked empty; #2806 Summary: the merge folds
 * only the chunks its selection reaches).
 *   M = max m_j, L = sum l_j exp(m_j - M), out = sum o_j exp(m_j - M) / L,
 *   lse = M + ln L; no live chunk: out = 0, lse = -inf.
 *   partials   (dev)  as written by qsa_decode_attn with the same sizes
 *   n_sel      (dev)  int32 [n_rows]
 *   out        (dev)  fp32 [n_rows][n_q_heads][128]
 *   lse        (dev)  fp32 [n_rows][n_q_heads], may be NULL
 * Errors: QSA_ERR_ARG (null or misaligned pointers, bad sizes),
 * QSA_ERR_UNSUPPORTED (n_rows > QSA_MAX_DECODE_ROWS, n_chunks >
 * QSA_MAX_CHUNKS).
 */
qsa_status qsa_attn_merge(const void* partials, const int32_t* n_sel, int n_rows, int n_q_heads,
                          int chunk_cells, int n_chunks, float* out, float* lse, void* stream);

/*
 * qsa_decode_window -- one whole decode window in one call: block scores ->
 * top-k -> split-KV attention -> log-sum-exp merge (the four steps above),
 * enqueued as five launches chained by programmatic dependent launch on
 * `stream` (q preparation, block scores, top-k, split attention, merge; in
 * windows of at most 152 blocks the block-score launch prepares q itself and
 * there are four; when the pools keep block summaries the scores come from
 * them and there are four;
 * "#2806 sycl: decode QSA selection and attention in fewer, shorter
 * launches", Summary: selection and attention of a window in fewer, shorter
 * launches).  scores, ids and n_sel are written exactly as qsa_block_scores
 * and qsa_topk write them.  The attention splits each (row, KV head)'s
 * selection into splits of a multiple of 16 cells chosen by the library for
 * this GPU (about four CTAs per SM, at most 256 splits), and the merge
 * folds the splits in split order, skipping empty ones; out and lse follow
 * the qsa_attn_merge definition (equal to the chunked result up to
 * rounding; bitwise reproducible run to run on the same GPU).
 *   pools, row_pool, q, n_rows, n_q_heads, block_cells, max_blocks
 *              as qsa_block_scores
 *   row_pos    (dev)  int32 [n_rows], as qsa_decode_attn
 *   k_cells    multiple of block_cells, >= 0
 *   scores     (dev)  fp32 [n_rows][max_blocks]   (output)
 *   ids        (dev)  int32 [n_rows][max(k_cells, 1)] (output)
 *   n_sel      (dev)  int32 [n_rows]              (output)
 *   out        (dev)  fp32 [n_rows][n_q_heads][128] (output)
 *   lse        (dev)  fp32 [n_rows][n_q_heads], may be NULL (output)
 *   workspace  (dev)  caller-owned, 256-byte aligned, workspace_bytes >=
 *              qsa_decode_window_workspace_bytes(); needs no initialisation.
 * Calls on one stream may reuse one workspace; calls that run concurrently
 * need their own.
 * Errors: as qsa_block_scores / qsa_topk / qsa_decode_attn, and
 * QSA_ERR_SCRATCH when the workspace is too small.
 */
size_t qsa_decode_window_workspace_bytes(int n_rows, int n_q_heads, int n_kv_heads, int k_cells);
qsa_status qsa_decode_window(const qsa_pool* pools, int n_pools, const int32_t* row_pool,
                             const float* q, const int32_t* row_pos, int n_rows, int n_q_heads,
                             int block_cells, int k_cells, float* scores, int max_blocks,
                             int32_t* ids, int32_t* n_sel, float* out, float* lse,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * qsa_decode_window_host -- qsa_decode_window whose per-step inputs and
 * results live in page-locked host memory: q, row_pos, out and lse (when not
 * NULL) are host pointers from cudaHostAlloc / cudaMallocHost or a range
 * registered with cudaHostRegister, in the layouts of qsa_decode_window.  The
 * window's first launch reads q and row_pos through the device's mapping of
 * those pages (on Grace-Blackwell, over the coherent host link) into the
 * workspace, and the later launches read that copy; the merge writes out and
 * lse straight into host memory.  No DMA copy is enqueued.  Everything else
 * (pools, scores, ids, n_sel, workspace) is device memory as for
 * qsa_decode_window, and the workspace size is the same.  The results are in
 * host memory once `stream` has completed the call.
 * Errors: QSA_ERR_ARG, with nothing enqueued, when one of the four host
 * buffers is not page-locked (pageable memory, device memory or NULL; lse may
 * be NULL); otherwise as qsa_decode_window.
 */
qsa_status qsa_decode_window_host(const qsa_pool* pools, int n_pools, const int32_t* row_pool,
                                  const float* q, const int32_t* row_pos, int n_rows,
                                  int n_q_heads, int block_cells, int k_cells, float* scores,
                                  int max_blocks, int32_t* ids, int32_t* n_sel, float* out,
                                  float* lse, void* workspace, size_t workspace_bytes,
                                  void* stream);

/*
 * qsa_decode_window_profile -- qsa_decode_window for measurement: the same
 * launches (q fragments, block scores, top-k, split attention, merge), each
 * started only after the previous one has finished, with CUDA events between
 * them.  Synchronises `stream`, then writes the five steps' times in
 * microseconds to kernel_us (host, 5 floats; a step without a launch of its
 * own, such as the q fragments of a small window, reads about 0).  Outputs as
 * qsa_decode_window.
 * Errors: as qsa_decode_window; QSA_ERR_ARG when kernel_us is NULL.
 */
qsa_status qsa_decode_window_profile(const qsa_pool* pools, int n_pools, const int32_t* row_pool,
                                     const float* q, const int32_t* row_pos, int n_rows,
                                     int n_q_heads, int block_cells, int k_cells, float* scores,
                                     int max_blocks, int32_t* ids, int32_t* n_sel, float* out,
                                     float* lse, void* workspace, size_t workspace_bytes,
                                     void* stream, float* kernel_us);

/*
 * qsa_prompt_attn -- causal attention of a chunk of n_q queries over the
 * cached context, on the tensor cores (#1367 What it does: both products on
 * the tensor cores with an exact split of the non-code operand; #600
 * description: a chunk of queries against the whole context).
 * Query i sits at position q_pos0 + i and sees cells 0 .. q_pos0 + i:
 *   out[i,g] = sum_c softmax_c(q[i,g] . K[c,kv(g)] / sqrt(128)) V[c,kv(g)]
 *   lse[i,g] = ln sum_c exp(...)
 *   pool       (host) one descriptor; page_cells multiple of 64
 *   q          (dev)  fp32 [n_q][n_q_heads][128], 16-byte aligned
 *   scratch    (dev)  caller-owned work space of scratch_bytes >=
 *                     qsa_prompt_scratch_bytes(pool, n_q, q_pos0, n_q_heads), 256-byte
 *                     aligned.  The call first converts every 64-cell tile it reads,
 *                     once per KV head, into the operand images the tensor
 *                     cores load: K' = kcode * kscale * 2^a and V' = vcode *
 *                     vscale * 2^b as fp16 hi + lo, with powers of two a, b
 *                     per KV head.  Work runs as one CTA per (block of
 *                     128 / group queries, KV head); when the last round of
 *                     CTAs would leave SMs idle, its units are cut into equal
 *                     ranges of tiles whose partial rows (unnormalised output,
 *                     running max, row sum) also live in scratch and are
 *                     combined by log-sum-exp in range order.
 *   out        (dev)  fp32 [n_q][n_q_heads][128], 16-byte aligned
 *   lse        (dev)  fp32 [n_q][n_q_heads], may be NULL
 *   q_pos0 >= 0, q_pos0 + n_q <= pool->n_filled
 * Errors: QSA_ERR_ARG, QSA_ERR_UNSUPPORTED (n_q_heads / n_kv_heads > 128),
 * QSA_ERR_SCRATCH (scratch missing, misaligned or too small).
 * A kernel whose internal wait runs out sets the device error word (see
 * qsa_get_device_error) and leaves its outputs incomplete.
 */
qsa_status qsa_prompt_attn(const qsa_pool* pool, const float* q, int n_q, int q_pos0,
                           int n_q_heads, void* scratch, size_t scratch_bytes, float* out,
                           float* lse, void* stream);

/*
 * qsa_prompt_scratch_bytes -- device scratch bytes qsa_prompt_attn needs for
 * a call of n_q >= 1 queries of n_q_heads heads from position q_pos0 over
 * `pool`, on the current device: a 256-byte header, 65,536 bytes per 64-cell
 * tile of cells 0 .. q_pos0 + n_q - 1 per KV head (int8 and 4-bit V alike),
 * and 66,560 bytes per partial range of a cut unit (their number depends on
 * the device's SM count; none without a device).  Returns 0 for invalid
 * arguments.
 */
size_t qsa_prompt_scratch_bytes(const qsa_pool* pool, int n_q, int q_pos0, int n_q_heads);

/*
 * qsa_kv_append -- quantise n_new new cells into a pool: cell first_cell + i
 * of KV head h takes the rows k[i][h] and v[i][h] ("#2806 sycl: decode QSA
 * selection and attention in fewer, shorter launches", What it leaves alone:
 * the per-row K/V appends; storage format of "#1367 prompt attention",
 * Operands, and "#2075 QSA decode attention", Bit for bit).  Each group of a
 * row (64 dims; 32 for 4-bit V) is quantised symmetrically by its largest
 * magnitude amax:
 *   scale = amax / 127 (4-bit V: amax / 7), stored as the group's fp32 scale;
 *   code  = x / scale rounded to nearest with ties to even, clamped to +-127
 *           (+-7; stored as the nibble code + 8, the even dim in the low
 *           nibble); amax = 0 gives scale 0 and codes 0.
 * The division and rounding are IEEE fp32, so the codes are exact integers.
 * A pool with k_sums has the summaries of the 64-cell blocks the new cells
 * fall in rewritten, each over its cells below first_cell + n_new.
 *   pool        (host) descriptor; the call WRITES its code and scale arrays
 *                      for the appended cells (the const in qsa_pool marks
 *                      the attention calls' read-only use).  n_filled is the
 *                      caller's: raise it to first_cell + n_new before reading
 *                      the new cells.
 *   k, v        (dev)  fp32 [n_new][n_kv_heads][128], 16-byte aligned
 *   first_cell >= 0, first_cell + n_new <= pool->capacity
 * Errors: QSA_ERR_ARG, QSA_ERR_UNSUPPORTED (as for the pool elsewhere).
 * Non-finite inputs give unspecified codes for their group (no fault).
 */
qsa_status qsa_kv_append(const qsa_pool* pool, const float* k, const float* v, int first_cell,
                         int n_new, void* stream);

/*
 * qsa_kv_summarise -- (re)writes a pool's block summaries (qsa_pool.k_sums)
 * of the 64-cell blocks that cells first_cell .. first_cell + n_cells - 1
 * fall in, each over its cells below first_cell + n_cells (so a call with
 * first_cell 0 and n_cells = n_filled builds them for the whole fill).  An
 * index of the pool's blocks kept beside the K/V cells ("#2806 sycl: decode
 * QSA selection and attention in fewer, shorter launches", What it leaves
 * alone: the K/V and indexer appends).
 *   pool   (host) descriptor with k_sums set; the call WRITES k_sums
 *   first_cell >= 0, n_cells >= 0, first_cell + n_cells <= capacity
 * Errors: QSA_ERR_ARG (no k_sums, bad range), QSA_ERR_UNSUPPORTED.
 */
qsa_status qsa_kv_summarise(const qsa_pool* pool, int first_cell, int n_cells, void* stream);

/* Size of the library-owned scratch of qsa_decode_attn_noalloc (8 MiB). */
#define QSA_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * qsa_decode_attn_noalloc -- qsa_decode_attn followed by qsa_attn_merge, for
 * callers that cannot allocate device memory: it takes inputs and outputs
 * only and keeps the chunk partials in a fixed array of
 * QSA_NOALLOC_SCRATCH_BYTES that the library owns on every GPU it is loaded
 * on (held until the process exits).  The pages have no counterpart of this
 * call; it exists for engines whose device memory is all reserved up front
 * and for plugins whose interface carries no allocator.
 *   Arguments as qsa_decode_attn and qsa_attn_merge, with
 *   n_chunks = ceil(k_cells / chunk_cells) (at least 1).
 *   Requires qsa_decode_partials_bytes(n_rows, n_q_heads, n_chunks) <=
 *   QSA_NOALLOC_SCRATCH_BYTES, else QSA_ERR_SCRATCH.  Every refusal (ARG,
 *   UNSUPPORTED, SCRATCH) comes with nothing enqueued.  No cudaMalloc /
 *   cudaFree.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 *   All calls share the one array: calls that overlap on the GPU (other
 *   streams, other threads) race on it and must be serialised by the caller.
 *   Nothing in it needs clearing between calls.
 */
qsa_status qsa_decode_attn_noalloc(const qsa_pool* pools, int n_pools, const int32_t* row_pool,
                                   const float* q, const int32_t* row_pos, const int32_t* ids,
                                   const int32_t* n_sel, int n_rows, int n_q_heads, int k_cells,
                                   int chunk_cells, float* out, float* lse, void* stream);

/*
 * qsa_get_device_error -- synchronises `stream`, then reads and clears the
 * device error word of the current device.  *code = 0 when no kernel
 * reported an error; otherwise a nonzero code (1 = a bounded wait inside
 * the prompt kernel ran out).  Returns QSA_ERR_DEVICE when *code != 0.
 */
qsa_status qsa_get_device_error(int32_t* code, void* stream);

/* Test hook: limit, in nanoseconds, of each bounded wait inside the kernels
 * (default 2e9).  0 makes the first wait give up at once, which exercises the
 * error path without a hang.  Affects later launches on all devices. */
void qsa_set_wait_limit_ns(uint64_t ns);

/*
 * Context-sharded decode (several GPUs, each holding a range of every slot's
 * cells).  The split and its merge follow "#1888 QSA decode attention: split
 * each query's cells across blocks on the int8 mma path", Summary: the cells
 * of a query are split, each split yields (m, l, o) partials, and the splits
 * are merged by the log-sum-exp rescale in split order.  Here a split is a
 * rank's cell range.  A rank describes its range [lo, hi) of a slot as a pool
 * view (page_table advanced by lo / page_cells pages, n_filled = min(hi,
 * n_filled) - lo; lo and hi multiples of page_cells) and runs:
 *   qsa_block_scores on its views; an all-gather of the scores (the caller's
 *   collective); qsa_topk over the gathered scores (one global selection,
 *   the same on every rank and equal to a single GPU's); qsa_ids_in_range;
 *   qsa_decode_attn on its views; an all-gather of the chunk partials and of
 *   the ranks' n_sel; qsa_attn_merge_shards.
 */

/*
 * qsa_ids_in_range -- per row t, the selected ids in [lo[t], hi[t]) (the
 * rank's range of the row's slot), shifted by -lo[t] (the range's own cell
 * numbering), and the row's position shifted by -lo[t].
 *   ids        (dev)  int32 [n_rows][k_cells], ascending in [0, n_sel)
 *   n_sel      (dev)  int32 [n_rows]
 *   row_pos    (dev)  int32 [n_rows]
 *   lo, hi     (host) int32 [n_rows], 0 <= lo <= hi
 *   ids_out    (dev)  int32 [n_rows][k_cells]: entries [0, n_sel_out) written
 *   n_sel_out, row_pos_out (dev) int32 [n_rows]
 * Errors: QSA_ERR_ARG, QSA_ERR_UNSUPPORTED (n_rows > QSA_MAX_DECODE_ROWS).
 */
qsa_status qsa_ids_in_range(const int32_t* ids, const int32_t* n_sel, const int32_t* row_pos, int n_rows,
                            int k_cells, const int32_t* lo, const int32_t* hi, int32_t* ids_out,
                            int32_t* n_sel_out, int32_t* row_pos_out, void* stream);

/*
 * qsa_attn_merge_shards -- the log-sum-exp merge of qsa_attn_merge over the
 * chunk partials of n_shards ranks, folded in rank order, then chunk order,
 * visiting for rank s only chunks j < ceil(n_sel[s][t] / C) and skipping
 * empty ones.  out and lse as qsa_attn_merge.
 *   partials   (dev)  n_shards buffers back to back, each
 *                     qsa_decode_partials_bytes(n_rows, n_q_heads, n_chunks)
 *                     bytes in the chunk-partials layout (as written by
 *                     qsa_decode_attn with these sizes), 16-byte aligned
 *   n_sel      (dev)  int32 [n_shards][n_rows]: each rank's n_sel_out
 * Errors: QSA_ERR_ARG, QSA_ERR_UNSUPPORTED (n_rows > QSA_MAX_DECODE_ROWS,
 * n_chunks > QSA_MAX_CHUNKS).
 */
qsa_status qsa_attn_merge_shards(const void* partials, int n_shards, const int32_t* n_sel, int n_rows,
                                 int n_q_heads, int chunk_cells, int n_chunks, float* out, float* lse,
                                 void* stream);

/*
 * qsa_measure_tc_rate -- measurement utility (the pages have no counterpart):
 * the dense tensor-core rate of the current GPU for one operand kind, timed
 * with CUDA events on the legacy default stream after one warm-up launch.
 *   QSA_TC_KIND_F16: one CTA per SM issues `passes` x 4 back-to-back
 *     tcgen05.mma kind::f16 (f16 x f16 -> f32, M = 128, N = 256, K = 16)
 *     from shared memory into tensor memory (about 1 ms per 3,000 passes);
 *   QSA_TC_KIND_I8: tcgen05 has no int8 kind on sm_103a, so 16 warps per SM
 *     each issue `passes` x 8 independent mma.sync.m16n8k32 s8 x s8 -> s32
 *     (about 1 ms per 10 passes).
 * Writes 2 * M * N * K * MMAs / seconds to *ops_per_second (host).
 * Synchronous; occupies every SM for the launch.  Errors: QSA_ERR_ARG (kind,
 * passes outside 1 .. 2^20, NULL output), QSA_ERR_CUDA, QSA_ERR_DEVICE (the
 * f16 launch's bounded wait ran out).
 */
#define QSA_TC_KIND_F16 0
#define QSA_TC_KIND_I8 1
qsa_status qsa_measure_tc_rate(int kind, int passes, double* ops_per_second);

const char* qsa_status_str(qsa_status s);

/* ABI version of this header (major * 100 + minor). */
int qsa_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* QSA_GB300_H */
