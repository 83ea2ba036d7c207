// qsa_decode_attn_noalloc: the decode chunk attention and its merge, with the
// chunk partials kept in a scratch array that the library itself owns.
//
// Who needs it: callers that can hand the library their inputs and outputs
// but no scratch buffer.  An inference engine that reserves all device
// memory up front for its KV pool and activations has no allocator to lend;
// a host plugin whose interface carries only input and output pointers has
// none either; and cudaMalloc on a decode step would synchronise the device
// and can fail under memory pressure.  This entry point allocates nothing:
// the partials live in a fixed-size __device__ array that every GPU loading
// the library holds until the process exits.
//
// The array's name is only a host-side stand-in in host code, so its device
// address is looked up once per device (cudaGetSymbolAddress, with that
// device current) and passed to the kernels.  The existing kernels run
// unchanged on that address.
#include <mutex>
#include <vector>

#include "kernels.h"

namespace qsa {
namespace {

static __device__ __align__(256) float g_noalloc_partials[QSA_NOALLOC_SCRATCH_BYTES / sizeof(float)];

std::mutex g_noalloc_mu;
std::vector<void*> g_noalloc_ptr;   // device address of the array, per device ordinal

// Device address of the scratch array on the current device (set up on first use).
qsa_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if ((int)g_noalloc_ptr.size() <= dev) g_noalloc_ptr.resize(dev + 1, nullptr);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_partials);
    if (e != cudaSuccess || p == nullptr) return QSA_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return QSA_OK;
}

}  // namespace
}  // namespace qsa

extern "C" qsa_status qsa_decode_attn_noalloc(const qsa_pool* pools, int n_pools, const int32_t* row_pool,
                                              const float* q, const int32_t* row_pos, const int32_t* ids,
                                              const int32_t* n_sel, int n_rows, int n_q_heads, int k_cells,
                                              int chunk_cells, float* out, float* lse, void* stream) {
  // Every check of both steps comes first: a refused call enqueues nothing.
  if (!out || !n_sel) return QSA_ERR_ARG;
  if (k_cells < 0 || chunk_cells < 16 || chunk_cells > 1024 || chunk_cells % 16 != 0) return QSA_ERR_ARG;
  if (n_rows < 1 || n_q_heads < 1) return QSA_ERR_ARG;
  long long n_chunks = ((long long)k_cells + chunk_cells - 1) / chunk_cells;
  if (n_chunks < 1) n_chunks = 1;
  if (n_rows > QSA_MAX_DECODE_ROWS || n_chunks > QSA_MAX_CHUNKS) return QSA_ERR_UNSUPPORTED;
  // Sizes past the fixed scratch are refused before anything is looked up or enqueued.
  if (qsa_decode_partials_bytes(n_rows, n_q_heads, (int)n_chunks) > (size_t)QSA_NOALLOC_SCRATCH_BYTES)
    return QSA_ERR_SCRATCH;
  void* scratch = nullptr;
  qsa_status s = qsa::noalloc_scratch(&scratch);
  if (s != QSA_OK) return s;
  // Nothing in the scratch has to start at zero: every chunk the merge reads
  // was written by the attention launch just before it on the same stream.
  s = qsa_decode_attn(pools, n_pools, row_pool, q, row_pos, ids, n_sel, n_rows, n_q_heads, k_cells, chunk_cells,
                      (int)n_chunks, scratch, QSA_NOALLOC_SCRATCH_BYTES, stream);
  if (s != QSA_OK) return s;
  return qsa_attn_merge(scratch, n_sel, n_rows, n_q_heads, chunk_cells, (int)n_chunks, out, lse, stream);
}
