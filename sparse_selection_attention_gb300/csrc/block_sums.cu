// Block summaries of K and the block scores computed from them.
//
// The library's block score is linear in K:
//     S[t, b] = 1 / (n_b sqrt(128)) * sum_h qbar[t, h] . Kbar[b, h],   qbar[t, h] = sum_{g in G(h)} q[t, g],
//     Kbar[b, h, d] = sum_{c in b} K[c, h, d],   K[c, h, d] = kcode[c, h, d] * kscale[c, h, d / group].
// A pool may keep Kbar per 64-cell summary block and KV head (k_sums, fp32 [pages][heads][page_cells
// / 64][128]), written when cells are appended ("#2806 sycl: decode QSA selection and attention in
// fewer, shorter launches", What it leaves alone: the K/V and indexer appends of a window, per row).
// A block of B cells (B a multiple of 64) is then scored from its B / 64 summaries, 512 bytes per
// (summary block, KV head) instead of the 8,704 bytes of int8 codes and scales.
//
//  summarise_kernel: one 128-thread CTA per (summary block, KV head); thread d sums its dim over the
//      block's cells in ascending order (fmaf), int8 or 4-bit codes.
//  sum_scores_kernel: one CTA per (pool, block), one warp per KV head; lane l holds dims 4l .. 4l + 3
//      of the block's summaries and of qbar of each row (the group's q heads summed in head order);
//      a fixed butterfly per (row, head), then the heads added in head order.
#include "kernels.h"

namespace qsa {
namespace {

constexpr int kSumCells = 64;   // cells per summary block

struct SummariseParams {
  PoolDev pool;
  float* k_sums;
  int n_kv_heads, first_block, end_cell;   // blocks first_block .. ; cells below end_cell count
};

__global__ void __launch_bounds__(kD) summarise_kernel(const SummariseParams p) {
  const int j = p.first_block + blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const PoolDev& pool = p.pool;
  const int c0 = j * kSumCells;
  const int n = min(kSumCells, p.end_cell - c0);
  const int page = __ldg(pool.page_table + c0 / pool.page_cells);
  const int off = c0 % pool.page_cells;
  const long long slot0 = ((long long)page * p.n_kv_heads + h) * pool.page_cells + off;
  float acc = 0.f;
  if (pool.k_bits == 8) {
    for (int c = 0; c < n; ++c) {
      const float code = (float)pool.k_codes[(slot0 + c) * kD + d];
      acc = fmaf(__ldg(pool.k_scales + (slot0 + c) * 2 + (d >> 6)), code, acc);
    }
  } else {
    for (int c = 0; c < n; ++c) {
      const uint32_t byte = (uint8_t)pool.k_codes[(slot0 + c) * (kD / 2) + (d >> 1)];
      const float code = (float)((int)((d & 1) ? (byte >> 4) : (byte & 15u)) - 8);
      acc = fmaf(__ldg(pool.k_scales + (slot0 + c) * 4 + (d >> 5)), code, acc);
    }
  }
  const long long srow = ((long long)page * p.n_kv_heads + h) * (pool.page_cells / kSumCells) + off / kSumCells;
  p.k_sums[srow * kD + d] = acc;
}

// One CTA per (pool, block), one warp per KV head (all heads' loads in flight together): warp h adds
// the block's summaries of head h (lane l: dims 4l .. 4l + 3), forms qbar of each row of the pool
// from q and reduces the dot product over the warp; the heads' sums meet in shared memory and are
// added in head order.
__global__ void __launch_bounds__(32 * QSA_MAX_KV_HEADS) sum_scores_kernel(const ScoresParams p) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // the top-k may start its CTAs
  __shared__ float part[QSA_MAX_KV_HEADS][QSA_MAX_DECODE_ROWS];
  const int lane = threadIdx.x & 31, h = threadIdx.x >> 5;
  const int unit = blockIdx.x;
  int pi = 0;
  while (pi + 1 < p.n_pools && unit >= p.unit_begin[pi + 1]) ++pi;
  const PoolDev& pool = p.pools[pi];
  const int B = p.block_cells, Hkv = p.n_kv_heads, R = p.n_rows, G = p.n_q_heads / Hkv;
  const int b = unit - p.unit_begin[pi];
  const int cell0 = b * B;
  const int n_b = min(B, pool.n_filled - cell0);
  const int n_sum = (n_b + kSumCells - 1) / kSumCells;   // summary blocks holding the block's filled cells
  const int page = __ldg(pool.page_table + cell0 / pool.page_cells);
  const int spp = pool.page_cells / kSumCells;           // summary blocks per page
  const int s0 = (cell0 % pool.page_cells) / kSumCells;
  const float4* ks = reinterpret_cast<const float4*>(pool.k_sums + (((long long)page * Hkv + h) * spp + s0) * kD) + lane;
  float4 kb = __ldg(ks);
  for (int j = 1; j < n_sum; ++j) {
    const float4 x = __ldg(ks + j * (kD / 4));
    kb.x += x.x;
    kb.y += x.y;
    kb.z += x.z;
    kb.w += x.w;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");   // q staged by a preceding launch (else a no-op)
  for (int t = 0; t < R; ++t) {
    if (p.row_pool[t] != pi) continue;
    const float4* qg = reinterpret_cast<const float4*>(p.q + ((size_t)t * p.n_q_heads + (size_t)h * G) * kD) + lane;
    float4 qb = __ldg(qg);
    for (int g = 1; g < G; ++g) {
      const float4 x = __ldg(qg + (size_t)g * (kD / 4));
      qb.x += x.x;
      qb.y += x.y;
      qb.z += x.z;
      qb.w += x.w;
    }
    float v = qb.x * kb.x;
    v = fmaf(qb.y, kb.y, v);
    v = fmaf(qb.z, kb.z, v);
    v = fmaf(qb.w, kb.w, v);
    v = warp_sum(v);
    if (lane == 0) part[h][t] = v;
  }
  __syncthreads();
  if (threadIdx.x < R && p.row_pool[threadIdx.x] == pi) {
    const int t = threadIdx.x;
    float sum = 0.f;
    for (int hh = 0; hh < Hkv; ++hh) sum += part[hh][t];
    p.scores[(size_t)t * p.max_blocks + b] = sum * (kInvSqrtD / (float)n_b);
  }
}

}  // namespace

cudaError_t launch_summarise(const PoolDev& pool, float* k_sums, int n_kv_heads, int first_cell, int n_cells,
                             cudaStream_t stream) {
  if (n_cells <= 0) return cudaSuccess;
  SummariseParams p{};
  p.pool = pool;
  p.k_sums = k_sums;
  p.n_kv_heads = n_kv_heads;
  p.first_block = first_cell / kSumCells;
  p.end_cell = first_cell + n_cells;
  const int last_block = (p.end_cell - 1) / kSumCells;
  summarise_kernel<<<dim3(last_block - p.first_block + 1, n_kv_heads), kD, 0, stream>>>(p);
  return cudaGetLastError();
}

bool block_sums_usable(const ScoresParams& p) {
  if (p.block_cells % kSumCells != 0) return false;
  for (int i = 0; i < p.n_pools; ++i)
    if (!p.pools[i].k_sums) return false;
  return true;
}

cudaError_t launch_sum_scores(const ScoresParams& p, cudaStream_t stream, bool pdl) {
  if (p.total_units == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.total_units);
  cfg.blockDim = dim3(32 * p.n_kv_heads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, sum_scores_kernel, p);
}

}  // namespace qsa
