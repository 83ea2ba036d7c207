// Context-sharded decode: the two steps a rank adds around the single-GPU calls when the cells of
// every slot are split into ranges held by different GPUs ("#1888 QSA decode attention: split each
// query's cells across blocks", Summary: the splits of a query's cells are merged by the
// log-sum-exp rescale, in split order; here a split is a rank's range).
//
//  ids_in_range_kernel: per row, the selected ids that fall in the row's range [lo, hi) of its
//      slot, shifted to the range's own cell numbering, and the row's position in that numbering
//      (the ids are ascending, so they form one contiguous run of the list).
//  merge_shards_kernel: per (row, q head), the log-sum-exp fold of every rank's chunk partials in
//      rank order, then chunk order, visiting only the chunks each rank's selection reaches and
//      skipping empty ones.
#include "kernels.h"

namespace qsa {
namespace {

struct RangeParams {
  const int32_t* ids;
  const int32_t* n_sel;
  const int32_t* row_pos;
  int k_cells;
  int lo[QSA_MAX_DECODE_ROWS], hi[QSA_MAX_DECODE_ROWS];   // each row's range (its pool's)
  int32_t* ids_out;
  int32_t* n_sel_out;
  int32_t* row_pos_out;
};

__global__ void __launch_bounds__(256) ids_in_range_kernel(const RangeParams p) {
  __shared__ int s_a, s_b;
  const int t = blockIdx.x, tid = threadIdx.x;
  const int k_cells = p.k_cells, lo = p.lo[t], hi = p.hi[t];
  const int32_t* ids = p.ids;
  const int32_t* row = ids + (size_t)t * k_cells;
  const int n = min(max(__ldg(p.n_sel + t), 0), k_cells);
  if (tid == 0) {
    // first index with id >= lo, and first with id >= hi (binary searches over the ascending ids)
    int a = 0, b = n;
    while (a < b) {
      const int m = (a + b) >> 1;
      if (__ldg(row + m) < lo) a = m + 1; else b = m;
    }
    int c = a, d = n;
    while (c < d) {
      const int m = (c + d) >> 1;
      if (__ldg(row + m) < hi) c = m + 1; else d = m;
    }
    s_a = a;
    s_b = c;
    p.n_sel_out[t] = c - a;
    p.row_pos_out[t] = __ldg(p.row_pos + t) - lo;
  }
  __syncthreads();
  const int a = s_a, cnt = s_b - s_a;
  int32_t* out = p.ids_out + (size_t)t * k_cells;
  for (int j = tid; j < cnt; j += blockDim.x) out[j] = __ldg(row + a + j) - lo;
}

struct MergeShardsParams {
  const uint8_t* partials;    // n_shards buffers of shard_bytes, each in the chunk-partials layout
  size_t shard_bytes, o_offset;
  const int32_t* n_sel;       // [n_shards][n_rows]
  int n_shards, n_rows, n_q_heads, chunk_cells, n_chunks;
  float* out;
  float* lse;
};

__global__ void __launch_bounds__(kD) merge_shards_kernel(const MergeShardsParams p) {
  const int g = blockIdx.x, t = blockIdx.y, d = threadIdx.x;
  const size_t base = ((size_t)t * p.n_q_heads + g) * p.n_chunks;
  float M = -INFINITY;
  for (int s = 0; s < p.n_shards; ++s) {
    const float* ml = reinterpret_cast<const float*>(p.partials + s * p.shard_bytes);
    const int n_act = min(p.n_chunks, (max(__ldg(p.n_sel + (size_t)s * p.n_rows + t), 0) + p.chunk_cells - 1) /
                                          p.chunk_cells);
    for (int j = 0; j < n_act; ++j) M = fmaxf(M, __ldg(ml + (base + j) * 2));
  }
  float* out = p.out + ((size_t)t * p.n_q_heads + g) * kD;
  if (M == -INFINITY) {
    out[d] = 0.f;
    if (p.lse && d == 0) p.lse[(size_t)t * p.n_q_heads + g] = -INFINITY;
    return;
  }
  float L = 0.f, O = 0.f;
  for (int s = 0; s < p.n_shards; ++s) {
    const uint8_t* sb = p.partials + s * p.shard_bytes;
    const float* ml = reinterpret_cast<const float*>(sb);
    const float* o = reinterpret_cast<const float*>(sb + p.o_offset);
    const int n_act = min(p.n_chunks, (max(__ldg(p.n_sel + (size_t)s * p.n_rows + t), 0) + p.chunk_cells - 1) /
                                          p.chunk_cells);
    for (int j = 0; j < n_act; ++j) {
      const float mj = __ldg(ml + (base + j) * 2);
      if (mj == -INFINITY) continue;   // empty chunk
      const float w = expf(mj - M);
      L = fmaf(__ldg(ml + (base + j) * 2 + 1), w, L);
      O = fmaf(__ldg(o + (base + j) * kD + d), w, O);
    }
  }
  out[d] = O / L;
  if (p.lse && d == 0) p.lse[(size_t)t * p.n_q_heads + g] = M + logf(L);
}

}  // namespace
}  // namespace qsa

using namespace qsa;

extern "C" {

qsa_status qsa_ids_in_range(const int32_t* ids, const int32_t* n_sel, const int32_t* row_pos, int n_rows,
                            int k_cells, const int32_t* lo, const int32_t* hi, int32_t* ids_out, int32_t* n_sel_out,
                            int32_t* row_pos_out, void* stream) {
  if (!ids || !n_sel || !row_pos || !lo || !hi || !ids_out || !n_sel_out || !row_pos_out) return QSA_ERR_ARG;
  if (n_rows < 1 || k_cells < 0) return QSA_ERR_ARG;
  if (n_rows > QSA_MAX_DECODE_ROWS) return QSA_ERR_UNSUPPORTED;
  RangeParams p{};
  for (int t = 0; t < n_rows; ++t) {
    if (lo[t] < 0 || hi[t] < lo[t]) return QSA_ERR_ARG;
    p.lo[t] = lo[t];
    p.hi[t] = hi[t];
  }
  p.ids = ids;
  p.n_sel = n_sel;
  p.row_pos = row_pos;
  p.k_cells = k_cells;
  p.ids_out = ids_out;
  p.n_sel_out = n_sel_out;
  p.row_pos_out = row_pos_out;
  ids_in_range_kernel<<<n_rows, 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}

qsa_status qsa_attn_merge_shards(const void* partials, int n_shards, const int32_t* n_sel, int n_rows,
                                 int n_q_heads, int chunk_cells, int n_chunks, float* out, float* lse,
                                 void* stream) {
  if (!partials || !n_sel || !out) return QSA_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(partials) & 15u) != 0) return QSA_ERR_ARG;
  if (n_shards < 1 || n_rows < 1 || n_q_heads < 1 || n_chunks < 1) return QSA_ERR_ARG;
  if (chunk_cells < 16 || chunk_cells > 1024 || chunk_cells % 16 != 0) return QSA_ERR_ARG;
  if (n_rows > QSA_MAX_DECODE_ROWS || n_chunks > QSA_MAX_CHUNKS) return QSA_ERR_UNSUPPORTED;
  MergeShardsParams p{};
  p.partials = static_cast<const uint8_t*>(partials);
  const size_t n = (size_t)n_rows * n_q_heads * n_chunks;
  p.o_offset = partials_o_offset(n);
  p.shard_bytes = qsa_decode_partials_bytes(n_rows, n_q_heads, n_chunks);
  p.n_sel = n_sel;
  p.n_shards = n_shards;
  p.n_rows = n_rows;
  p.n_q_heads = n_q_heads;
  p.chunk_cells = chunk_cells;
  p.n_chunks = n_chunks;
  p.out = out;
  p.lse = lse;
  merge_shards_kernel<<<dim3(n_q_heads, n_rows), kD, 0, static_cast<cudaStream_t>(stream)>>>(p);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}

}  // extern "C"
