// Decode block scores (qsa_block_scores).
//
// S[t,b] = sum_h (1/n_b) sum_{c in b} sum_{g in G(h)} q[t,g] . K[c,h] / sqrt(D).
// The score is linear in K, so a block is read once per window: the kernel
// forms the fp32 per-dim block sum ksum[h][d] = sum_c kcode*kscale of each KV
// head, then dots it with qbar[t][h][d] = sum_{g in G(h)} q[t,g,d] for every
// row of the block's pool ("#2806 sycl: decode QSA selection and attention in
// fewer, shorter launches", Summary: a block's (query, head) sums are reduced
// together; scores run once per slot).  HBM-bound: every filled K code and
// scale is read exactly once per call.
//
// Work unit = (pool, block).  A persistent grid walks the units; each CTA
// builds qbar for all rows once.  Reductions run in a fixed order (lane
// butterflies, then warps 0..7), so results are bitwise reproducible.
#include "kernels.h"

namespace qsa {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCellsPerThread = 8;  // block_cells <= 256 over 32 cell slots

__global__ void __launch_bounds__(kThreads) block_scores_kernel(const ScoresParams p) {
  extern __shared__ float smem[];
  const int Hkv = p.n_kv_heads;
  const int G = p.n_q_heads / Hkv;
  float* qbar = smem;                                  // [n_rows][Hkv][128]
  float* red = qbar + p.n_rows * Hkv * kD;             // [kWarps][Hkv][128]
  float* ksum = red + kWarps * Hkv * kD;               // [Hkv][128]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int i = tid; i < p.n_rows * Hkv * kD; i += kThreads) {
    const int t = i / (Hkv * kD), h = (i / kD) % Hkv, d = i % kD;
    const float* qg = p.q + ((size_t)t * p.n_q_heads + h * G) * kD + d;
    float s = 0.f;
    for (int g = 0; g < G; ++g) s += __ldg(qg + (size_t)g * kD);
    qbar[i] = s;
  }
  __syncthreads();

  const int dq = lane & 7;                    // 16-dim slice of the 128 dims
  const int cs = (lane >> 3) + 4 * warp;      // cell slot 0..31
  const int B = p.block_cells;

  for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
    int pi = 0;
    while (pi + 1 < p.n_pools && u >= p.unit_begin[pi + 1]) ++pi;
    const PoolDev& pool = p.pools[pi];
    const int b = u - p.unit_begin[pi];
    const int cell0 = b * B;
    const int n_b = min(B, pool.n_filled - cell0);
    const int page = __ldg(pool.page_table + cell0 / pool.page_cells);
    const int off0 = cell0 % pool.page_cells;

    for (int h = 0; h < Hkv; ++h) {
      const long long slot0 = ((long long)page * Hkv + h) * pool.page_cells + off0;
      uint4 cv[kMaxCellsPerThread];
      float sv[kMaxCellsPerThread];
#pragma unroll
      for (int k = 0; k < kMaxCellsPerThread; ++k) {
        const int c = cs + 32 * k;
        if (c < n_b) {
          cv[k] = __ldg(reinterpret_cast<const uint4*>(pool.k_codes + (slot0 + c) * kD) + dq);
          sv[k] = __ldg(pool.k_scales + (slot0 + c) * 2 + (dq >> 2));
        }
      }
      float acc[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[j] = 0.f;
#pragma unroll
      for (int k = 0; k < kMaxCellsPerThread; ++k) {
        if (cs + 32 * k < n_b) {
          const uint32_t w[4] = {cv[k].x, cv[k].y, cv[k].z, cv[k].w};
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[j] = fmaf(s8_to_f32(w[j >> 2], j & 3), sv[k], acc[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], 8);
        acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], 16);
      }
      if (lane < 8) {
#pragma unroll
        for (int j = 0; j < 16; ++j) red[(warp * Hkv + h) * kD + dq * 16 + j] = acc[j];
      }
    }
    __syncthreads();
    for (int i = tid; i < Hkv * kD; i += kThreads) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += red[w * Hkv * kD + i];
      ksum[i] = s;
    }
    __syncthreads();
    const float inv = kInvSqrtD / (float)n_b;
    for (int t = warp; t < p.n_rows; t += kWarps) {
      if (p.row_pool[t] != pi) continue;
      float s = 0.f;
      for (int h = 0; h < Hkv; ++h) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int d = lane + 32 * j;
          s = fmaf(qbar[(t * Hkv + h) * kD + d], ksum[h * kD + d], s);
        }
      }
      s = warp_sum(s);
      if (lane == 0) p.scores[(size_t)t * p.max_blocks + b] = s * inv;
    }
    __syncthreads();
  }
}

}  // namespace

size_t block_scores_smem_bytes(int n_rows, int n_kv_heads) {
  return sizeof(float) * (size_t)(n_rows * n_kv_heads * kD + kWarps * n_kv_heads * kD + n_kv_heads * kD);
}

cudaError_t launch_block_scores(const ScoresParams& p, cudaStream_t stream) {
  const size_t smem = block_scores_smem_bytes(p.n_rows, p.n_kv_heads);
  if (p.total_units == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(block_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = min(p.total_units, device_sm_count() * 4);
  block_scores_kernel<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace qsa
