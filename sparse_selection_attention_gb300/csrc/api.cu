// C ABI of the QSA library: host-side validation and launches.
//
// Every entry point validates all host-visible arguments before it enqueues
// anything; a non-OK status (other than QSA_ERR_CUDA) means nothing was
// enqueued ("#1888 QSA decode attention", What changed: the launcher returns
// without launching when it cannot serve the call).
#include <cstdio>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "kernels.h"

namespace qsa {

namespace {
unsigned long long g_wait_limit_ns = 2000000000ull;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DeviceInfo {
  int sms = 0;
  int smem_optin = 0;
};

DeviceInfo& device_info() {
  static std::mutex mu;
  static std::vector<DeviceInfo> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  if ((int)cache.size() <= dev) cache.resize(dev + 1);
  DeviceInfo& d = cache[dev];
  if (d.sms == 0) {
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (d.sms <= 0) d.sms = 1;
  }
  return d;
}

qsa_status check_pool(const qsa_pool& p, bool need_v) {
  if (!p.k_codes || !p.k_scales || !p.page_table || (need_v && (!p.v_codes || !p.v_scales))) return QSA_ERR_ARG;
  if (!aligned16(p.k_codes) || !aligned16(p.k_scales) || (need_v && (!aligned16(p.v_codes) || !aligned16(p.v_scales))))
    return QSA_ERR_ARG;
  if (p.head_dim != QSA_HEAD_DIM) return QSA_ERR_UNSUPPORTED;
  if (p.v_bits != 8 && p.v_bits != 4) return QSA_ERR_ARG;
  if (p.k_bits != 8 && p.k_bits != 4) return QSA_ERR_ARG;
  if (p.page_cells <= 0 || p.page_cells % 64 != 0) return QSA_ERR_ARG;
  if (p.n_kv_heads < 1 || p.n_kv_heads > QSA_MAX_KV_HEADS) return QSA_ERR_UNSUPPORTED;
  if (p.capacity < 0 || p.n_filled < 0 || p.n_filled > p.capacity) return QSA_ERR_ARG;
  if (p.k_sums && !aligned16(p.k_sums)) return QSA_ERR_ARG;
  return QSA_OK;
}

PoolDev to_dev(const qsa_pool& p) {
  PoolDev d;
  d.k_codes = p.k_codes;
  d.v_codes = static_cast<const uint8_t*>(p.v_codes);
  d.k_scales = p.k_scales;
  d.v_scales = p.v_scales;
  d.page_table = p.page_table;
  d.n_filled = p.n_filled;
  d.page_cells = p.page_cells;
  d.page_shift = (p.page_cells & (p.page_cells - 1)) == 0 ? __builtin_ctz((unsigned)p.page_cells) : -1;
  d.v_bits = p.v_bits;
  d.k_bits = p.k_bits;
  d.k_sums = p.k_sums;
  return d;
}

// Shared checks of the pool set and row mapping of a decode window.
qsa_status check_window(const qsa_pool* pools, int n_pools, const int32_t* row_pool, int n_rows,
                        int n_q_heads, bool need_v) {
  if (!pools || !row_pool) return QSA_ERR_ARG;
  if (n_pools < 1 || n_pools > QSA_MAX_POOLS) return QSA_ERR_UNSUPPORTED;
  if (n_rows < 1) return QSA_ERR_ARG;
  if (n_rows > QSA_MAX_DECODE_ROWS) return QSA_ERR_UNSUPPORTED;
  for (int i = 0; i < n_pools; ++i) {
    const qsa_status s = check_pool(pools[i], need_v);
    if (s != QSA_OK) return s;
    if (pools[i].n_kv_heads != pools[0].n_kv_heads || pools[i].k_bits != pools[0].k_bits) return QSA_ERR_ARG;
  }
  for (int t = 0; t < n_rows; ++t)
    if (row_pool[t] < 0 || row_pool[t] >= n_pools) return QSA_ERR_ARG;
  const int Hkv = pools[0].n_kv_heads;
  if (n_q_heads < 1 || n_q_heads % Hkv != 0) return QSA_ERR_ARG;
  if (n_q_heads / Hkv > QSA_MAX_GROUP) return QSA_ERR_UNSUPPORTED;
  return QSA_OK;
}

qsa_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return QSA_OK;
  fprintf(stderr, "qsa: CUDA error %s\n", cudaGetErrorString(e));
  return QSA_ERR_CUDA;
}

}  // namespace

int device_sm_count() { return device_info().sms; }

cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  size_t& cur = done[{dev, kernel}];
  if (bytes <= cur) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) cur = bytes;
  return e;
}
int device_max_smem_optin() { return device_info().smem_optin; }
unsigned long long wait_limit_ns() { return g_wait_limit_ns; }
void set_wait_limit_ns(unsigned long long ns) { g_wait_limit_ns = ns; }

}  // namespace qsa

using namespace qsa;

extern "C" {

qsa_status qsa_block_scores(const qsa_pool* pools, int n_pools, const int32_t* row_pool, const float* q,
                            int n_rows, int n_q_heads, int block_cells, float* scores, int max_blocks,
                            void* stream) {
  qsa_status s = check_window(pools, n_pools, row_pool, n_rows, n_q_heads, false);
  if (s != QSA_OK) return s;
  if (!q || !scores || !aligned16(q)) return QSA_ERR_ARG;
  if (block_cells != 32 && block_cells != 64 && block_cells != 128 && block_cells != 256) return QSA_ERR_ARG;
  ScoresParams p{};
  p.n_pools = n_pools;
  p.unit_begin[0] = 0;
  for (int i = 0; i < n_pools; ++i) {
    if (pools[i].page_cells % block_cells != 0) return QSA_ERR_ARG;
    const int nb = (pools[i].n_filled + block_cells - 1) / block_cells;
    if (nb > max_blocks) return QSA_ERR_ARG;
    p.pools[i] = to_dev(pools[i]);
    p.unit_begin[i + 1] = p.unit_begin[i] + nb;
  }
  p.total_units = p.unit_begin[n_pools];
  for (int t = 0; t < n_rows; ++t) p.row_pool[t] = row_pool[t];
  p.n_rows = n_rows;
  p.n_q_heads = n_q_heads;
  p.n_kv_heads = pools[0].n_kv_heads;
  p.block_cells = block_cells;
  p.max_blocks = max_blocks;
  p.q = q;
  p.scores = scores;
  p.err = device_error_word();
  p.wait_limit_ns = wait_limit_ns();
  if (!p.err) return QSA_ERR_CUDA;
  if (block_sums_usable(p)) return from_cuda(launch_sum_scores(p, static_cast<cudaStream_t>(stream), false));
  if (pools[0].k_bits == 4) return from_cuda(launch_block_scores(p, static_cast<cudaStream_t>(stream)));
  if (!block_scores_supported(p.n_kv_heads, block_cells)) return QSA_ERR_UNSUPPORTED;
  p.q_rows_per_batch = block_scores_q_rows_per_batch(n_rows, n_q_heads, p.n_kv_heads, block_cells);
  if (block_scores_smem_bytes(n_rows, n_q_heads, p.n_kv_heads, block_cells) > (size_t)device_max_smem_optin())
    return QSA_ERR_UNSUPPORTED;
  return from_cuda(launch_block_scores(p, static_cast<cudaStream_t>(stream)));
}

qsa_status qsa_topk(const float* scores, int max_blocks, const int32_t* n_filled, int n_rows, int block_cells,
                    int k_cells, int32_t* ids, int32_t* n_sel, void* stream) {
  if (!scores || !n_filled || !ids || !n_sel) return QSA_ERR_ARG;
  if (n_rows < 1) return QSA_ERR_ARG;
  if (n_rows > QSA_MAX_DECODE_ROWS) return QSA_ERR_UNSUPPORTED;
  if (block_cells < 1 || k_cells < 0 || k_cells % block_cells != 0) return QSA_ERR_ARG;
  TopkParams p{};
  int max_nb = 1;
  for (int t = 0; t < n_rows; ++t) {
    if (n_filled[t] < 0) return QSA_ERR_ARG;
    const int nb = (n_filled[t] + block_cells - 1) / block_cells;
    if (nb > max_blocks) return QSA_ERR_ARG;
    if (nb > QSA_MAX_TOPK_BLOCKS) return QSA_ERR_UNSUPPORTED;
    max_nb = nb > max_nb ? nb : max_nb;
    p.n_filled[t] = n_filled[t];
  }
  p.scores = scores;
  p.max_blocks = max_blocks;
  p.n_rows = n_rows;
  p.block_cells = block_cells;
  p.k_cells = k_cells;
  p.ids = ids;
  p.n_sel = n_sel;
  if (topk_smem_bytes(max_nb) > (size_t)device_max_smem_optin()) return QSA_ERR_UNSUPPORTED;
  return from_cuda(launch_topk(p, max_nb, static_cast<cudaStream_t>(stream)));
}

size_t qsa_decode_partials_bytes(int n_rows, int n_q_heads, int n_chunks) {
  if (n_rows <= 0 || n_q_heads <= 0 || n_chunks <= 0) return 0;
  const size_t n = (size_t)n_rows * n_q_heads * n_chunks;
  return partials_o_offset(n) + sizeof(float) * n * QSA_HEAD_DIM;
}

qsa_status qsa_decode_attn(const qsa_pool* pools, int n_pools, const int32_t* row_pool, const float* q,
                           const int32_t* row_pos, const int32_t* ids, const int32_t* n_sel, int n_rows,
                           int n_q_heads, int k_cells, int chunk_cells, int n_chunks, void* partials,
                           size_t partials_bytes, void* stream) {
  qsa_status s = check_window(pools, n_pools, row_pool, n_rows, n_q_heads, true);
  if (s != QSA_OK) return s;
  if (!q || !row_pos || !ids || !n_sel || !partials) return QSA_ERR_ARG;
  if (!aligned16(partials) || !aligned16(q)) return QSA_ERR_ARG;
  if (k_cells < 0 || chunk_cells < 16 || chunk_cells > 1024 || chunk_cells % 16 != 0) return QSA_ERR_ARG;
  const long long need_chunks = ((long long)k_cells + chunk_cells - 1) / chunk_cells;
  if (n_chunks < need_chunks || n_chunks < 1) return QSA_ERR_ARG;
  if (n_chunks > QSA_MAX_CHUNKS) return QSA_ERR_UNSUPPORTED;
  if (partials_bytes < qsa_decode_partials_bytes(n_rows, n_q_heads, n_chunks)) return QSA_ERR_SCRATCH;
  AttnParams p{};
  for (int i = 0; i < n_pools; ++i) p.pools[i] = to_dev(pools[i]);
  for (int t = 0; t < n_rows; ++t) p.row_pool[t] = row_pool[t];
  p.q = q;
  p.row_pos = row_pos;
  p.ids = ids;
  p.n_sel = n_sel;
  p.n_rows = n_rows;
  p.n_q_heads = n_q_heads;
  p.n_kv_heads = pools[0].n_kv_heads;
  p.k_cells = k_cells;
  p.chunk_cells = chunk_cells;
  p.n_chunks = n_chunks;
  p.ml = static_cast<float*>(partials);
  p.o = reinterpret_cast<float*>(static_cast<uint8_t*>(partials) +
                                 partials_o_offset((size_t)n_rows * n_q_heads * n_chunks));
  if (pools[0].k_bits == 4) return from_cuda(launch_chunk_attn_window_kernels(p, static_cast<cudaStream_t>(stream)));
  return from_cuda(launch_decode_attn(p, static_cast<cudaStream_t>(stream)));
}

qsa_status qsa_attn_merge(const void* partials, const int32_t* n_sel, int n_rows, int n_q_heads,
                          int chunk_cells, int n_chunks, float* out, float* lse, void* stream) {
  if (!partials || !n_sel || !out) return QSA_ERR_ARG;
  if (!aligned16(partials)) return QSA_ERR_ARG;
  if (n_rows < 1 || n_q_heads < 1 || n_chunks < 1) return QSA_ERR_ARG;
  if (n_rows > QSA_MAX_DECODE_ROWS || n_chunks > QSA_MAX_CHUNKS) return QSA_ERR_UNSUPPORTED;
  if (chunk_cells < 16 || chunk_cells > 1024 || chunk_cells % 16 != 0) return QSA_ERR_ARG;
  MergeParams p{};
  p.ml = static_cast<const float*>(partials);
  p.o = reinterpret_cast<const float*>(static_cast<const uint8_t*>(partials) +
                                       partials_o_offset((size_t)n_rows * n_q_heads * n_chunks));
  p.n_sel = n_sel;
  p.n_rows = n_rows;
  p.n_q_heads = n_q_heads;
  p.chunk_cells = chunk_cells;
  p.n_chunks = n_chunks;
  p.out = out;
  p.lse = lse;
  return from_cuda(launch_attn_merge(p, static_cast<cudaStream_t>(stream)));
}

size_t qsa_decode_window_workspace_bytes(int n_rows, int n_q_heads, int n_kv_heads, int k_cells) {
  if (n_rows < 1 || n_rows > QSA_MAX_DECODE_ROWS || n_kv_heads < 1 || n_q_heads < 1 || n_q_heads % n_kv_heads != 0 ||
      k_cells < 0)
    return 0;
  return window_layout(n_rows, n_q_heads, n_kv_heads, k_cells, device_sm_count()).total;
}

static qsa_status decode_window_impl(const qsa_pool* pools, int n_pools, const int32_t* row_pool, const float* q,
                              const int32_t* row_pos, int n_rows, int n_q_heads, int block_cells, int k_cells,
                              float* scores, int max_blocks, int32_t* ids, int32_t* n_sel, float* out, float* lse,
                              void* workspace, size_t workspace_bytes, void* stream, float* kernel_us,
                              bool host_inputs = false) {
  qsa_status s = check_window(pools, n_pools, row_pool, n_rows, n_q_heads, true);
  if (s != QSA_OK) return s;
  if (!q || !row_pos || !scores || !ids || !n_sel || !out || !workspace) return QSA_ERR_ARG;
  if (!aligned16(q) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return QSA_ERR_ARG;
  if (block_cells != 32 && block_cells != 64 && block_cells != 128 && block_cells != 256) return QSA_ERR_ARG;
  if (k_cells < 0 || k_cells % block_cells != 0) return QSA_ERR_ARG;
  const int Hkv = pools[0].n_kv_heads;
  WindowArgs a{};
  // block scores
  ScoresParams& sp = a.scores;
  sp.n_pools = n_pools;
  sp.unit_begin[0] = 0;
  for (int i = 0; i < n_pools; ++i) {
    if (pools[i].page_cells % block_cells != 0) return QSA_ERR_ARG;
    const int nb = (pools[i].n_filled + block_cells - 1) / block_cells;
    if (nb > max_blocks) return QSA_ERR_ARG;
    if (nb > QSA_MAX_TOPK_BLOCKS) return QSA_ERR_UNSUPPORTED;
    sp.pools[i] = to_dev(pools[i]);
    sp.unit_begin[i + 1] = sp.unit_begin[i] + nb;
  }
  sp.total_units = sp.unit_begin[n_pools];
  for (int t = 0; t < n_rows; ++t) sp.row_pool[t] = row_pool[t];
  sp.n_rows = n_rows;
  sp.n_q_heads = n_q_heads;
  sp.n_kv_heads = Hkv;
  sp.block_cells = block_cells;
  sp.max_blocks = max_blocks;
  sp.q = q;
  sp.scores = scores;
  sp.err = device_error_word();
  sp.wait_limit_ns = wait_limit_ns();
  if (!sp.err) return QSA_ERR_CUDA;
  if (!block_sums_usable(sp) && !window_scores_supported(n_rows, Hkv, block_cells)) return QSA_ERR_UNSUPPORTED;
  // top-k
  TopkParams& tp = a.topk;
  int max_nb = 1;
  for (int t = 0; t < n_rows; ++t) {
    const int nf = pools[row_pool[t]].n_filled;
    const int nb = (nf + block_cells - 1) / block_cells;
    max_nb = nb > max_nb ? nb : max_nb;
    tp.n_filled[t] = nf;
  }
  tp.scores = scores;
  tp.max_blocks = max_blocks;
  tp.n_rows = n_rows;
  tp.block_cells = block_cells;
  tp.k_cells = k_cells;
  tp.ids = ids;
  tp.n_sel = n_sel;
  a.max_nb = max_nb;
  if (topk_smem_bytes(max_nb) > (size_t)device_max_smem_optin()) return QSA_ERR_UNSUPPORTED;
  // attention + merge
  a.layout = window_layout(n_rows, n_q_heads, Hkv, k_cells, device_sm_count());
  if (workspace_bytes < a.layout.total) return QSA_ERR_SCRATCH;
  WinAttnParams& ap = a.attn;
  for (int i = 0; i < n_pools; ++i) ap.pools[i] = to_dev(pools[i]);
  for (int t = 0; t < n_rows; ++t) ap.row_pool[t] = row_pool[t];
  ap.q = q;
  ap.row_pos = row_pos;
  ap.ids = ids;
  ap.n_sel = n_sel;
  ap.n_rows = n_rows;
  ap.n_q_heads = n_q_heads;
  ap.n_kv_heads = Hkv;
  ap.k_cells = k_cells;
  ap.out = out;
  ap.lse = lse;
  a.workspace = workspace;
  if (host_inputs) {   // q and row_pos are staged into the workspace by the window's first launch
    a.q_src = q;
    a.pos_src = row_pos;
    sp.q = ap.q = reinterpret_cast<const float*>(static_cast<uint8_t*>(workspace) + a.layout.q_in);
    ap.row_pos = reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(workspace) + a.layout.pos_in);
  }
  if (!kernel_us) return from_cuda(launch_decode_window(a, static_cast<cudaStream_t>(stream)));
  cudaEvent_t ev[6] = {};
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 6 && e == cudaSuccess; ++i) e = cudaEventCreate(&ev[i]);
  if (e == cudaSuccess) e = launch_decode_window(a, static_cast<cudaStream_t>(stream), ev);
  if (e == cudaSuccess) e = cudaEventSynchronize(ev[5]);
  for (int i = 0; i < 5 && e == cudaSuccess; ++i) {
    float ms = 0.f;
    e = cudaEventElapsedTime(&ms, ev[i], ev[i + 1]);
    kernel_us[i] = 1000.f * ms;
  }
  for (int i = 0; i < 6; ++i)
    if (ev[i]) cudaEventDestroy(ev[i]);
  return from_cuda(e);
}

qsa_status qsa_decode_window(const qsa_pool* pools, int n_pools, const int32_t* row_pool, const float* q,
                             const int32_t* row_pos, int n_rows, int n_q_heads, int block_cells, int k_cells,
                             float* scores, int max_blocks, int32_t* ids, int32_t* n_sel, float* out, float* lse,
                             void* workspace, size_t workspace_bytes, void* stream) {
  return decode_window_impl(pools, n_pools, row_pool, q, row_pos, n_rows, n_q_heads, block_cells, k_cells, scores,
                            max_blocks, ids, n_sel, out, lse, workspace, workspace_bytes, stream, nullptr);
}

// The device's alias of a page-locked host buffer, or NULL for anything else.
static const void* host_alias(const void* ptr) {
  if (!ptr) return nullptr;
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

qsa_status qsa_decode_window_host(const qsa_pool* pools, int n_pools, const int32_t* row_pool, const float* q,
                                  const int32_t* row_pos, int n_rows, int n_q_heads, int block_cells, int k_cells,
                                  float* scores, int max_blocks, int32_t* ids, int32_t* n_sel, float* out, float* lse,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  const float* qd = static_cast<const float*>(host_alias(q));
  const int32_t* pd = static_cast<const int32_t*>(host_alias(row_pos));
  float* od = static_cast<float*>(const_cast<void*>(host_alias(out)));
  float* ld = lse ? static_cast<float*>(const_cast<void*>(host_alias(lse))) : nullptr;
  if (!qd || !pd || !od || (lse && !ld)) return QSA_ERR_ARG;
  return decode_window_impl(pools, n_pools, row_pool, qd, pd, n_rows, n_q_heads, block_cells, k_cells, scores,
                            max_blocks, ids, n_sel, od, ld, workspace, workspace_bytes, stream, nullptr, true);
}

qsa_status qsa_decode_window_profile(const qsa_pool* pools, int n_pools, const int32_t* row_pool, const float* q,
                                     const int32_t* row_pos, int n_rows, int n_q_heads, int block_cells,
                                     int k_cells, float* scores, int max_blocks, int32_t* ids, int32_t* n_sel,
                                     float* out, float* lse, void* workspace, size_t workspace_bytes, void* stream,
                                     float* kernel_us) {
  if (!kernel_us) return QSA_ERR_ARG;
  return decode_window_impl(pools, n_pools, row_pool, q, row_pos, n_rows, n_q_heads, block_cells, k_cells, scores,
                            max_blocks, ids, n_sel, out, lse, workspace, workspace_bytes, stream, kernel_us);
}

size_t qsa_prompt_scratch_bytes(const qsa_pool* pool, int n_q, int q_pos0, int n_q_heads) {
  PromptPlan plan;
  if (!pool || !prompt_plan(pool->v_bits, pool->n_kv_heads, n_q_heads, n_q, q_pos0, device_sm_count(), &plan))
    return 0;
  return plan.bytes;
}

qsa_status qsa_prompt_attn(const qsa_pool* pool, const float* q, int n_q, int q_pos0, int n_q_heads, void* scratch,
                           size_t scratch_bytes, float* out, float* lse, void* stream) {
  if (!pool || !q || !out || !aligned16(q) || !aligned16(out)) return QSA_ERR_ARG;
  qsa_status s = check_pool(*pool, true);
  if (s != QSA_OK) return s;
  if (n_q < 0 || q_pos0 < 0 || (long long)q_pos0 + n_q > pool->n_filled) return QSA_ERR_ARG;
  if (n_q_heads < 1 || n_q_heads % pool->n_kv_heads != 0) return QSA_ERR_ARG;
  if (n_q_heads / pool->n_kv_heads > 128) return QSA_ERR_UNSUPPORTED;
  if (n_q == 0) return QSA_OK;
  PromptPlan plan;
  if (!prompt_plan(pool->v_bits, pool->n_kv_heads, n_q_heads, n_q, q_pos0, device_sm_count(), &plan))
    return QSA_ERR_ARG;
  if (!scratch || (reinterpret_cast<uintptr_t>(scratch) & 255u) != 0 || scratch_bytes < plan.bytes)
    return QSA_ERR_SCRATCH;
  PromptParams p{};
  p.scratch = static_cast<uint8_t*>(scratch);
  p.qpc = plan.qpc;
  p.n_qb = plan.n_qb;
  p.n_whole = plan.n_whole;
  p.n_split = plan.n_split;
  p.part_o = reinterpret_cast<float*>(p.scratch + plan.parts_offset);
  p.part_ml = reinterpret_cast<float*>(p.scratch + plan.ml_offset);
  p.n_tiles = (q_pos0 + n_q - 1) / 64 + 1;
  p.pool = to_dev(*pool);
  p.n_kv_heads = pool->n_kv_heads;
  p.n_q_heads = n_q_heads;
  p.n_q = n_q;
  p.q_pos0 = q_pos0;
  p.q = q;
  p.out = out;
  p.lse = lse;
  p.wait_limit_ns = wait_limit_ns();
  return from_cuda(launch_prompt_attn(p, static_cast<cudaStream_t>(stream)));
}

qsa_status qsa_get_device_error(int32_t* code, void* stream) {
  if (!code) return QSA_ERR_ARG;
  const qsa_status s = from_cuda(read_and_clear_device_error(code, static_cast<cudaStream_t>(stream)));
  if (s != QSA_OK) return s;
  return *code ? QSA_ERR_DEVICE : QSA_OK;
}

void qsa_set_wait_limit_ns(uint64_t ns) { set_wait_limit_ns(ns); }

const char* qsa_status_str(qsa_status s) {
  switch (s) {
    case QSA_OK: return "ok";
    case QSA_ERR_ARG: return "invalid argument";
    case QSA_ERR_UNSUPPORTED: return "unsupported by this build";
    case QSA_ERR_SCRATCH: return "scratch buffer too small";
    case QSA_ERR_CUDA: return "CUDA error";
    case QSA_ERR_DEVICE: return "device error word set";
  }
  return "unknown status";
}

qsa_status qsa_kv_append(const qsa_pool* pool, const float* k, const float* v, int first_cell, int n_new,
                         void* stream) {
  if (!pool || !k || !v || !aligned16(k) || !aligned16(v)) return QSA_ERR_ARG;
  qsa_status s = check_pool(*pool, true);
  if (s != QSA_OK) return s;
  if (first_cell < 0 || n_new < 0 || (long long)first_cell + n_new > pool->capacity) return QSA_ERR_ARG;
  if (n_new == 0) return QSA_OK;
  AppendParams p{};
  p.pool = to_dev(*pool);
  p.k_codes = const_cast<int8_t*>(pool->k_codes);
  p.v_codes = static_cast<uint8_t*>(const_cast<void*>(pool->v_codes));
  p.k_scales = const_cast<float*>(pool->k_scales);
  p.v_scales = const_cast<float*>(pool->v_scales);
  p.k = k;
  p.v = v;
  p.n_kv_heads = pool->n_kv_heads;
  p.first_cell = first_cell;
  p.n_new = n_new;
  qsa_status st = from_cuda(launch_kv_append(p, static_cast<cudaStream_t>(stream)));
  if (st != QSA_OK || !pool->k_sums) return st;
  return from_cuda(launch_summarise(p.pool, const_cast<float*>(pool->k_sums), pool->n_kv_heads, first_cell, n_new,
                                    static_cast<cudaStream_t>(stream)));
}

qsa_status qsa_kv_summarise(const qsa_pool* pool, int first_cell, int n_cells, void* stream) {
  if (!pool) return QSA_ERR_ARG;
  qsa_status s = check_pool(*pool, false);
  if (s != QSA_OK) return s;
  if (!pool->k_sums) return QSA_ERR_ARG;
  if (first_cell < 0 || n_cells < 0 || (long long)first_cell + n_cells > pool->capacity) return QSA_ERR_ARG;
  if (n_cells == 0) return QSA_OK;
  return from_cuda(launch_summarise(to_dev(*pool), const_cast<float*>(pool->k_sums), pool->n_kv_heads, first_cell,
                                    n_cells, static_cast<cudaStream_t>(stream)));
}

qsa_status qsa_measure_tc_rate(int kind, int passes, double* ops_per_second) {
  if (!ops_per_second || (kind != QSA_TC_KIND_F16 && kind != QSA_TC_KIND_I8) || passes < 1 || passes > (1 << 20))
    return QSA_ERR_ARG;
  float ms = 0.f;
  double ops = 0.0;
  const qsa_status s = from_cuda(run_tc_rate(kind == QSA_TC_KIND_I8, passes, &ms, &ops));
  if (s != QSA_OK) return s;
  int32_t code = 0;
  if (read_and_clear_device_error(&code, nullptr) != cudaSuccess) return QSA_ERR_CUDA;
  if (code != 0) return QSA_ERR_DEVICE;
  *ops_per_second = ms > 0.f ? ops / (1e-3 * ms) : 0.0;
  return QSA_OK;
}

int qsa_abi_version(void) { return 109; }

}  // extern "C"
