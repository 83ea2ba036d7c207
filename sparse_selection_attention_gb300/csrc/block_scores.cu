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
// A persistent grid of one 512-thread CTA per SM walks the (pool, block)
// units, several units at a time when a unit needs fewer than 512 threads.
// Thread (head h, 16-dim slice dq, cell group cg) accumulates 8 cells
// cg + (B/8) k in registers; the int8 codes become fp32 through the exponent
// bias (2^23 + 128 + code is exact, so subtracting 2^23 + 128 gives the code).
// The next units' loads are in flight while the current ones are reduced.
// Reductions run in a fixed order (cells in order, lane butterflies over 4
// cell groups, then warps in index order): bitwise reproducible.
#include "kernels.h"

namespace qsa {

namespace {

constexpr int kThreads = 512;
constexpr int kCellsPerThread = 8;

struct Slice {
  uint4 codes[kCellsPerThread];
  float scale[kCellsPerThread];
  int pi, n_b, b;
  bool live;
};

// Unit us of super-unit su: pool, block, and this thread's 8 code slices.
__device__ __forceinline__ void load_slice(const ScoresParams& p, int unit, bool active, Slice& s) {
  const int B = p.block_cells, Hkv = p.n_kv_heads;
  s.live = active && unit < p.total_units;
  if (!s.live) return;
  int pi = 0;
  while (pi + 1 < p.n_pools && unit >= p.unit_begin[pi + 1]) ++pi;
  const PoolDev& pool = p.pools[pi];
  const int b = unit - p.unit_begin[pi];
  const int cell0 = b * B;
  const int n_b = min(B, pool.n_filled - cell0);
  const int page = __ldg(pool.page_table + cell0 / pool.page_cells);
  const int off0 = cell0 % pool.page_cells;
  const int i = threadIdx.x % (Hkv * B);
  const int dq = i & 7, ncg = B / 8, cg = (i >> 3) % ncg, h = (i >> 3) / ncg;
  const long long slot0 = ((long long)page * Hkv + h) * pool.page_cells + off0;
#pragma unroll
  for (int k = 0; k < kCellsPerThread; ++k) {
    const int c = cg + ncg * k;
    if (c < n_b) {
      s.codes[k] = __ldg(reinterpret_cast<const uint4*>(pool.k_codes + (slot0 + c) * kD) + dq);
      s.scale[k] = __ldg(pool.k_scales + (slot0 + c) * 2 + (dq >> 2));
    } else {
      s.codes[k] = make_uint4(0u, 0u, 0u, 0u);
      s.scale[k] = 0.f;
    }
  }
  s.pi = pi;
  s.n_b = n_b;
  s.b = b;
}

// Byte j of a biased word (code + 128) -> exact float of the code.
__device__ __forceinline__ float biased_byte_to_f32(uint32_t u, int j) {
  return __int_as_float(__byte_perm(u, 0x4B000000u, 0x7540 | j)) - 8388736.0f;
}

__global__ void __launch_bounds__(kThreads, 1) block_scores_kernel(const ScoresParams p) {
  extern __shared__ float smem[];
  const int Hkv = p.n_kv_heads;
  const int G = p.n_q_heads / Hkv;
  const int B = p.block_cells;
  const int U = Hkv * B;                   // threads per unit
  const int upi = kThreads / U;            // units per iteration
  const int wph = B / 32;                  // warps per head (4 cell groups each)
  float* qbar = smem;                                  // [n_rows][Hkv][128]
  float* red = qbar + p.n_rows * Hkv * kD;             // [upi][Hkv][wph][128]
  float* ksum = red + upi * Hkv * wph * kD;            // [upi][Hkv][128]
  const int tid = threadIdx.x, lane = tid & 31;
  const int us = tid / U;                  // unit slot of this thread
  const bool active = us < upi;
  const int i = tid % U;
  const int dq = i & 7, h = (i >> 3) / (B / 8), wl = ((i >> 3) % (B / 8)) / 4;
  const int n_super = (p.total_units + upi - 1) / upi;

  if ((int)blockIdx.x >= n_super) return;
  Slice cur, nxt;
  load_slice(p, blockIdx.x * upi + us, active, cur);

  // q -> shared memory in one coalesced pass (every load in flight at once), then
  // qbar[t][h][d] = sum over the group's q heads, in head order.
  {
    float* qs = red;   // the work area is free until the first unit is reduced
    const int row_floats = p.n_q_heads * kD;
    const int rb = p.q_rows_per_batch;
    for (int r0 = 0; r0 < p.n_rows; r0 += rb) {
      const int nr = min(rb, p.n_rows - r0);
      const float4* q4 = reinterpret_cast<const float4*>(p.q + (size_t)r0 * row_floats);
      for (int k = tid; k < nr * row_floats / 4; k += kThreads) reinterpret_cast<float4*>(qs)[k] = __ldg(q4 + k);
      __syncthreads();
      for (int k = tid; k < nr * Hkv * kD; k += kThreads) {
        const int t = k / (Hkv * kD), hh = (k / kD) % Hkv, d = k % kD;
        const float* qg = qs + (size_t)t * row_floats + hh * G * kD + d;
        float s = 0.f;
        for (int g = 0; g < G; ++g) s += qg[(size_t)g * kD];
        qbar[(size_t)r0 * Hkv * kD + k] = s;
      }
      __syncthreads();
    }
  }

  for (int su = blockIdx.x; su < n_super; su += gridDim.x) {
    const bool more = su + (int)gridDim.x < n_super;
    if (more) load_slice(p, (su + gridDim.x) * upi + us, active, nxt);
    else nxt.live = false;

    if (active) {   // warp-uniform: U is a multiple of 32
      float acc[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[j] = 0.f;
      if (cur.live) {
#pragma unroll
        for (int k = 0; k < kCellsPerThread; ++k) {
          const uint32_t w[4] = {cur.codes[k].x ^ 0x80808080u, cur.codes[k].y ^ 0x80808080u,
                                 cur.codes[k].z ^ 0x80808080u, cur.codes[k].w ^ 0x80808080u};
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[j] = fmaf(biased_byte_to_f32(w[j >> 2], j & 3), cur.scale[k], acc[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], 8);
        acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], 16);
      }
      if (lane < 8) {
        float4* dst = reinterpret_cast<float4*>(red + ((us * Hkv + h) * wph + wl) * kD + dq * 16);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        dst[2] = make_float4(acc[8], acc[9], acc[10], acc[11]);
        dst[3] = make_float4(acc[12], acc[13], acc[14], acc[15]);
      }
    }
    __syncthreads();
    for (int k = tid; k < upi * Hkv * kD; k += kThreads) {
      const int uh = k / kD, d = k % kD;
      float s = 0.f;
      for (int w = 0; w < wph; ++w) s += red[(uh * wph + w) * kD + d];
      ksum[k] = s;
    }
    __syncthreads();
    // Dots: warp -> (unit slot, row) pairs of rows in the unit's pool.
    for (int pr = tid >> 5; pr < upi * p.n_rows; pr += kThreads / 32) {
      const int u_s = pr / p.n_rows, t = pr % p.n_rows;
      const int unit = su * upi + u_s;
      if (unit >= p.total_units) continue;
      int pi = 0;
      while (pi + 1 < p.n_pools && unit >= p.unit_begin[pi + 1]) ++pi;
      if (p.row_pool[t] != pi) continue;
      const int b = unit - p.unit_begin[pi];
      const int n_b = min(B, p.pools[pi].n_filled - b * B);
      float s = 0.f;
      for (int hh = 0; hh < Hkv; ++hh) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int d = lane + 32 * j;
          s = fmaf(qbar[(t * Hkv + hh) * kD + d], ksum[(u_s * Hkv + hh) * kD + d], s);
        }
      }
      s = warp_sum(s);
      if (lane == 0) p.scores[(size_t)t * p.max_blocks + b] = s * (kInvSqrtD / (float)n_b);
    }
    if (more) cur = nxt;
    __syncthreads();
  }
}

}  // namespace

// Floats of the work area: the reduction buffers, or at least one row of q (staged there first).
static size_t block_scores_work_floats(int n_rows, int n_q_heads, int n_kv_heads, int block_cells) {
  const int upi = kThreads / (n_kv_heads * block_cells);
  size_t work = (size_t)upi * n_kv_heads * (block_cells / 32) * kD + (size_t)upi * n_kv_heads * kD;
  const size_t q_row = (size_t)n_q_heads * kD;
  const size_t q_all = q_row * n_rows;
  const size_t want = q_all < 16384 ? q_all : (q_row > 16384 ? q_row : 16384);   // up to 64 KB of q at once
  return work > want ? work : want;
}

int block_scores_q_rows_per_batch(int n_rows, int n_q_heads, int n_kv_heads, int block_cells) {
  const size_t area = block_scores_work_floats(n_rows, n_q_heads, n_kv_heads, block_cells);
  const int rb = (int)(area / ((size_t)n_q_heads * kD));
  return rb < 1 ? 1 : (rb > n_rows ? n_rows : rb);
}

size_t block_scores_smem_bytes(int n_rows, int n_q_heads, int n_kv_heads, int block_cells) {
  return sizeof(float) * ((size_t)n_rows * n_kv_heads * kD +
                          block_scores_work_floats(n_rows, n_q_heads, n_kv_heads, block_cells));
}

bool block_scores_supported(int n_kv_heads, int block_cells) {
  return n_kv_heads * block_cells <= kThreads && block_cells == kCellsPerThread * (block_cells / 8) &&
         (n_kv_heads * block_cells) % 32 == 0 && block_cells >= 32;
}

cudaError_t launch_block_scores(const ScoresParams& p, cudaStream_t stream) {
  const size_t smem = block_scores_smem_bytes(p.n_rows, p.n_q_heads, p.n_kv_heads, p.block_cells);
  if (p.total_units == 0) return cudaSuccess;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(block_scores_kernel), (size_t)smem);
  if (e != cudaSuccess) return e;
  const int upi = kThreads / (p.n_kv_heads * p.block_cells);
  const int n_super = (p.total_units + upi - 1) / upi;
  const int grid = min(n_super, device_sm_count());
  block_scores_kernel<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace qsa
