// Split-KV decode attention over the selected cells (qsa_decode_attn) and the
// log-sum-exp merge of its chunks (qsa_attn_merge).
//
// Chunk kernel: one CTA per (chunk j, KV head h, row t).  It computes, for
// the G q heads of h, the partial (m, l, o) of the chunk's visible cells
// ("#2075 QSA decode attention: ... a bounded merge", Summary: a chunk kernel
// over the selected cells; "#1888 QSA decode attention: split each query's
// cells across blocks", Summary: each query's cells split among blocks, the
// splits merged by the log-sum-exp rescale).  A KV head's K/V rows are read
// once for all of its q heads.  Chunks past the row's selection launch no
// work and are never written; the merge does not visit them ("#2806 sycl",
// Summary: the merge folds only the chunks its selection reaches).
//
// Determinism: every dot product is summed lane-locally in dim order, then by
// a fixed xor butterfly; p.V folds cells in chunk order with fmaf; the merge
// folds chunks in chunk order with fmaf ("#2075", Bit for bit).
#include "kernels.h"

namespace qsa {

namespace {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;

__global__ void __launch_bounds__(kAttnThreads) decode_chunk_kernel(const AttnParams p) {
  const int j = blockIdx.x, h = blockIdx.y, t = blockIdx.z;
  const int n_sel = min(__ldg(p.n_sel + t), p.k_cells);   // ids past k_cells are never read
  const int C = p.chunk_cells;
  if (j * C >= n_sel) return;
  const int G = p.n_q_heads / p.n_kv_heads;
  const int n = min(C, n_sel - j * C);
  const int pos = __ldg(p.row_pos + t);
  const PoolDev& pool = p.pools[p.row_pool[t]];
  const int Hkv = p.n_kv_heads;

  extern __shared__ float smem[];
  float* qs = smem;                        // [G][128]
  float* z = qs + G * kD;                  // [G][C]  logits, then probabilities
  long long* slot = reinterpret_cast<long long*>(z + G * C);  // [C] cell slots (-1: masked)
  __shared__ float s_m[QSA_MAX_GROUP], s_l[QSA_MAX_GROUP];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* qrow = p.q + ((size_t)t * p.n_q_heads + h * G) * kD;
  for (int i = tid; i < G * kD; i += kAttnThreads) qs[i] = __ldg(qrow + i);
  const int32_t* idrow = p.ids + (size_t)t * p.k_cells + (size_t)j * C;
  for (int i = tid; i < n; i += kAttnThreads) {
    const int c = __ldg(idrow + i);
    // Cells past the row's position are masked; ids outside the pool's fill are ignored.
    slot[i] = (c <= pos && c >= 0 && c < pool.n_filled) ? cell_slot(pool, Hkv, h, c) : -1;
  }
  __syncthreads();

  // Logits: a warp per cell, lane l holds dims 4l..4l+3.
  for (int i = warp; i < n; i += kAttnWarps) {
    const long long s = slot[i];
    if (s < 0) {
      if (lane < G) z[lane * C + i] = -INFINITY;
      continue;
    }
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(pool.k_codes + s * kD) + lane);
    const float ks = __ldg(pool.k_scales + s * 2 + (lane >> 4));
    const float k0 = s8_to_f32(w, 0), k1 = s8_to_f32(w, 1), k2 = s8_to_f32(w, 2), k3 = s8_to_f32(w, 3);
    for (int g = 0; g < G; ++g) {
      const float* qg = qs + g * kD + 4 * lane;
      float d = qg[0] * k0;
      d = fmaf(qg[1], k1, d);
      d = fmaf(qg[2], k2, d);
      d = fmaf(qg[3], k3, d);
      d = warp_sum(d * ks);
      if (lane == 0) z[g * C + i] = d * kInvSqrtD;
    }
  }
  __syncthreads();

  // Softmax statistics: warp g handles q head g.
  for (int g = warp; g < G; g += kAttnWarps) {
    float m = -INFINITY;
    for (int i = lane; i < n; i += 32) m = fmaxf(m, z[g * C + i]);
    m = warp_max(m);
    float l = 0.f;
    if (m != -INFINITY) {
      for (int i = lane; i < n; i += 32) {
        const float e = (z[g * C + i] == -INFINITY) ? 0.f : expf(z[g * C + i] - m);
        z[g * C + i] = e;
        l += e;
      }
      l = warp_sum(l);
    }
    if (lane == 0) { s_m[g] = m; s_l[g] = l; }
  }
  __syncthreads();

  // p.V: thread -> dim d, q heads g = gs, gs + 2, ...
  const int d = tid & (kD - 1);
  const int gs = tid >> 7;
  float acc[QSA_MAX_GROUP / 2];
#pragma unroll
  for (int k = 0; k < QSA_MAX_GROUP / 2; ++k) acc[k] = 0.f;
  const bool live = s_m[0] != -INFINITY;   // a chunk is empty for all heads or none
  if (live) {
    for (int i = 0; i < n; ++i) {
      const long long s = slot[i];
      if (s < 0) continue;
      float v;
      if (pool.v_bits == 8) {
        v = (float)__ldg(reinterpret_cast<const int8_t*>(pool.v_codes) + s * kD + d) *
            __ldg(pool.v_scales + s * 2 + (d >> 6));
      } else {
        const uint8_t b = __ldg(pool.v_codes + s * (kD / 2) + (d >> 1));
        const int code = (int)((d & 1) ? (b >> 4) : (b & 0xF)) - 8;
        v = (float)code * __ldg(pool.v_scales + s * 4 + (d >> 5));
      }
#pragma unroll
      for (int k = 0; k < QSA_MAX_GROUP / 2; ++k) {
        const int g = gs + 2 * k;
        if (g < G) acc[k] = fmaf(z[g * C + i], v, acc[k]);
      }
    }
  }
  const size_t base = ((size_t)t * p.n_q_heads + h * G) * p.n_chunks + j;
#pragma unroll
  for (int k = 0; k < QSA_MAX_GROUP / 2; ++k) {
    const int g = gs + 2 * k;
    if (g < G) p.o[(base + (size_t)g * p.n_chunks) * kD + d] = acc[k];
  }
  if (tid < G) {
    p.ml[(base + (size_t)tid * p.n_chunks) * 2 + 0] = s_m[tid];
    p.ml[(base + (size_t)tid * p.n_chunks) * 2 + 1] = s_l[tid];
  }
}

__global__ void __launch_bounds__(kD) attn_merge_kernel(const MergeParams p) {
  const int g = blockIdx.x, t = blockIdx.y, d = threadIdx.x;
  const int n_sel = __ldg(p.n_sel + t);
  const int n_act = min(p.n_chunks, (n_sel + p.chunk_cells - 1) / p.chunk_cells);
  const size_t base = ((size_t)t * p.n_q_heads + g) * p.n_chunks;
  float M = -INFINITY;
  for (int j = 0; j < n_act; ++j) M = fmaxf(M, __ldg(p.ml + (base + j) * 2));
  float* out = p.out + ((size_t)t * p.n_q_heads + g) * kD;
  if (M == -INFINITY) {
    out[d] = 0.f;
    if (p.lse && d == 0) p.lse[(size_t)t * p.n_q_heads + g] = -INFINITY;
    return;
  }
  float L = 0.f, acc = 0.f;
  for (int j = 0; j < n_act; ++j) {
    const float mj = __ldg(p.ml + (base + j) * 2);
    if (mj == -INFINITY) continue;
    const float w = expf(mj - M);
    L = fmaf(__ldg(p.ml + (base + j) * 2 + 1), w, L);
    acc = fmaf(__ldg(p.o + (base + j) * kD + d), w, acc);
  }
  out[d] = acc / L;
  if (p.lse && d == 0) p.lse[(size_t)t * p.n_q_heads + g] = M + logf(L);
}

}  // namespace

cudaError_t launch_decode_attn(const AttnParams& p, cudaStream_t stream) {
  const int G = p.n_q_heads / p.n_kv_heads;
  const int n_chunks_max = (p.k_cells + p.chunk_cells - 1) / p.chunk_cells;
  if (n_chunks_max == 0) return cudaSuccess;
  const size_t smem = sizeof(float) * (size_t)(G * kD + G * p.chunk_cells) + sizeof(long long) * p.chunk_cells;
  cudaError_t e = cudaFuncSetAttribute(decode_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(n_chunks_max, p.n_kv_heads, p.n_rows);
  decode_chunk_kernel<<<grid, kAttnThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attn_merge(const MergeParams& p, cudaStream_t stream) {
  dim3 grid(p.n_q_heads, p.n_rows);
  attn_merge_kernel<<<grid, kD, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace qsa
