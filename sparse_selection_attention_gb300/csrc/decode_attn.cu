// Split-KV decode attention over the selected cells (qsa_decode_attn) and the
// log-sum-exp merge of its chunks (qsa_attn_merge).
//
// Chunk kernel: 128-thread CTAs, each bound to one (row t, KV head h) pair
// (t fastest across CTAs, so that a window's rows, which select mostly the
// same cells, read them close together in time) and walking a strided set of
// that pair's chunks; the next 64-cell sub-tile's cp.async copies are in
// flight while the current one is computed.  For the G <= 8 q heads of h it computes the
// chunk's partial (m, l, o) ("#2075 QSA decode attention: ... a bounded
// merge", Summary: a chunk kernel over the selected cells; "#1888 QSA decode
// attention: split each query's cells across blocks", Summary: a query's
// cells split among blocks and merged by the log-sum-exp rescale).  A KV
// head's K/V rows are read once for all of its q heads.  Chunks past the
// row's selection launch no work and are never written; the merge does not
// visit them ("#2806 sycl", Summary: the merge folds only the chunks its
// selection reaches).
//
// Both products run as mma.sync m16n8k16 (fp16 operands, fp32 accumulate)
// on 64-cell sub-tiles staged in shared memory by cp.async:
//   S^T[cells x heads] = Kcode[cells x dims] . (q f)^T, per 64-dim K-scale
//     group, q f split into fp16 hi + lo (both accumulate into one fp32 sum);
//   O^T[dims x heads] += Vcode^T[dims x cells] . W[cells x heads],
//     W = p * vscale * 2^k split into fp16 hi + lo, per V-scale group.
// int8 and 4-bit codes convert to fp16 exactly in registers.  The chunk's
// softmax is exact within the chunk (online across its 64-cell sub-tiles).
// Determinism: fixed MMA order, fixed shuffle and warp reduction order.
#include <cuda_fp16.h>

#include "kernels.h"
#include "mma_sync.cuh"

namespace qsa {

namespace {

constexpr int kThreads = 128;
constexpr int kSub = 64;   // cells per sub-tile

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Two bytes of u (chosen by sel, 0x64 placed above each) -> fp16 pair 1024 + b - bias, exact.
__device__ __forceinline__ uint32_t byte_pair_h2(uint32_t u, uint32_t sel, uint32_t bias) {
  return h2u(__hsub2(u2h(__byte_perm(u, 0x64646464u, sel)), u2h(bias)));
}

__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 back = __half22float2(h);
  hi = h2u(h);
  lo = h2u(__floats2half2_rn(a - back.x, b - back.y));
}

// 2^e as a float (e clamped to the normal range), for exact power-of-two scaling.
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + max(-126, min(127, e))) << 23); }

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_group1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// One 64-cell sub-tile of K/V codes and scales in shared memory.
struct Stage {
  int8_t k[kSub * kD];
  uint8_t v[kSub * kD];
  float ks[kSub * 2];
  float vs[kSub * 4];
  int valid[kSub];
};

// Position in the CTA's sequence of (chunk, sub-tile) work items.
struct Item {
  int j, st;
};

__device__ __forceinline__ int chunk_cells_of(int j, int C, int n_sel) { return min(C, n_sel - j * C); }

// Issues the copies of item `it` into stage `sg`: thread (cell c = tid / 2, half) copies half of
// the cell's K and V pieces and one of its scale rows; invisible cells copy nothing.
__device__ __forceinline__ void prefetch(const AttnParams& p, const PoolDev& pool, Stage& sg, Item it, int t, int h,
                                         int n_sel, int pos, bool v4) {
  const int C = p.chunk_cells;
  const int c = threadIdx.x >> 1, half = threadIdx.x & 1;
  const int n_j = chunk_cells_of(it.j, C, n_sel);
  const int idx = it.st * kSub + c;
  bool valid = false;
  long long slot = 0;
  if (idx < n_j) {
    const int cell = __ldg(p.ids + (size_t)t * p.k_cells + (size_t)it.j * C + idx);
    // Cells past the row's position are masked; ids outside the pool's fill are ignored.
    valid = cell <= pos && cell >= 0 && cell < pool.n_filled;
    if (valid) slot = cell_slot(pool, p.n_kv_heads, h, cell);
  }
  if (valid) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int pc = 4 * half + k;
      cp_async16(sg.k + c * kD + pc * 16, pool.k_codes + slot * kD + pc * 16);
    }
    if (!v4) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int pc = 4 * half + k;
        cp_async16(sg.v + c * kD + pc * 16, pool.v_codes + slot * kD + pc * 16);
      }
      if (half) cp_async8(sg.vs + 2 * c, pool.v_scales + slot * 2);
    } else {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int pc = 2 * half + k;
        cp_async16(sg.v + c * 64 + pc * 16, pool.v_codes + slot * 64 + pc * 16);
      }
      if (half) cp_async16(sg.vs + 4 * c, pool.v_scales + slot * 4);
    }
    if (!half) cp_async8(sg.ks + 2 * c, pool.k_scales + slot * 2);
  }
  if (!half) sg.valid[c] = valid;
  cp_async_commit();
}

__global__ void __launch_bounds__(kThreads, 5) decode_chunk_kernel(const AttnParams p) {
  const int R = p.n_rows, Hkv = p.n_kv_heads;
  const int n_pairs = R * Hkv;
  const int pair = blockIdx.x % n_pairs, ci = blockIdx.x / n_pairs, cpp = gridDim.x / n_pairs;
  const int t = pair % R, h = pair / R;
  const int n_sel = min(__ldg(p.n_sel + t), p.k_cells);   // ids past k_cells are never read
  const int C = p.chunk_cells;
  const int n_act = (n_sel + C - 1) / C;
  if (ci >= n_act) return;
  const int G = p.n_q_heads / Hkv;
  const int pos = __ldg(p.row_pos + t);
  const PoolDev& pool = p.pools[p.row_pool[t]];
  const bool v4 = pool.v_bits == 4;
  const int n_vg = v4 ? 4 : 2;

  __shared__ __align__(16) Stage stages[2];
  __shared__ __align__(16) float p_s[8][kSub];
  __shared__ float red_s[2][4][8];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tq = lane & 3;

  Item it{ci, 0};
  prefetch(p, pool, stages[0], it, t, h, n_sel, pos, v4);

  // ---- q of head g (this thread's B columns): dims 16s + 4tq .. +3, s = 0..7,
  // scaled by 2^fe (max |q 2^fe| in [64, 128)) and split into fp16 hi + lo.
  uint32_t qh[8][2], ql[8][2];
  float lam_lo, lam_hi;   // logit scale of heads 2tq and 2tq+1
  {
    float qv[8][4];
    float amax = 0.f;
    const float* qrow = p.q + ((size_t)t * p.n_q_heads + h * G + min(g, G - 1)) * kD + 4 * tq;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (g < G) v = __ldg(reinterpret_cast<const float4*>(qrow + 16 * s));
      qv[s][0] = v.x; qv[s][1] = v.y; qv[s][2] = v.z; qv[s][3] = v.w;
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int e = 0;
    if (amax > 0.f) frexpf(amax, &e);
    const int fe = amax > 0.f ? max(-126, min(127, 7 - e)) : 0;
    const float f = pow2i(fe);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      split_pair(qv[s][0] * f, qv[s][1] * f, qh[s][0], ql[s][0]);
      split_pair(qv[s][2] * f, qv[s][3] * f, qh[s][1], ql[s][1]);
    }
    const float lam = kInvSqrtD * pow2i(-fe);
    lam_lo = __shfl_sync(0xffffffffu, lam, 4 * (2 * tq));
    lam_hi = __shfl_sync(0xffffffffu, lam, 4 * (2 * tq + 1));
  }
  const int vgrp = v4 ? warp : (warp >> 1);   // V-scale group of this warp's 32 dims

  float m_run[2], l_run[2], o_acc[2][4];
  for (int k = 0;; ++k) {
    const int sg = k & 1;
    Stage& S = stages[sg];
    // Next item: the chunk's next sub-tile, else the CTA's next chunk.
    Item nx{it.j, it.st + 1};
    if (nx.st * kSub >= chunk_cells_of(it.j, C, n_sel)) nx = Item{it.j + cpp, 0};
    const bool has_next = nx.j < n_act;
    if (has_next) {
      prefetch(p, pool, stages[sg ^ 1], nx, t, h, n_sel, pos, v4);
      cp_async_wait_group1();
    } else {
      cp_async_wait_all();
    }
    __syncthreads();
    if (it.st == 0) {
      m_run[0] = m_run[1] = -INFINITY;
      l_run[0] = l_run[1] = 0.f;
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) o_acc[i][q] = 0.f;
    }

    // ---- S^T = Kcode . (q f)^T on this warp's 16 cells, per K-scale group.
    const int cb = 16 * warp;
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint32_t w0 = *reinterpret_cast<const uint32_t*>(S.k + (cb + g) * kD + 16 * s + 4 * tq) ^ 0x80808080u;
      const uint32_t w1 = *reinterpret_cast<const uint32_t*>(S.k + (cb + g + 8) * kD + 16 * s + 4 * tq) ^ 0x80808080u;
      uint32_t a[4];
      a[0] = byte_pair_h2(w0, 0x4140, 0x64806480u);
      a[2] = byte_pair_h2(w0, 0x4342, 0x64806480u);
      a[1] = byte_pair_h2(w1, 0x4140, 0x64806480u);
      a[3] = byte_pair_h2(w1, 0x4342, 0x64806480u);
      if (s < 4) {
        mma16816(d0, a, qh[s][0], qh[s][1]);
        mma16816(d0, a, ql[s][0], ql[s][1]);
      } else {
        mma16816(d1, a, qh[s][0], qh[s][1]);
        mma16816(d1, a, ql[s][0], ql[s][1]);
      }
    }
    // ---- logits of cells cb+g, cb+g+8 for heads 2tq, 2tq+1; masked cells -> -inf.
    float z[4];
    {
      const bool va = S.valid[cb + g], vb = S.valid[cb + g + 8];
      const float2 ka = *reinterpret_cast<const float2*>(S.ks + 2 * (cb + g));
      const float2 kb = *reinterpret_cast<const float2*>(S.ks + 2 * (cb + g + 8));
      z[0] = va ? fmaf(d1[0], ka.y, d0[0] * ka.x) * lam_lo : -INFINITY;
      z[1] = va ? fmaf(d1[1], ka.y, d0[1] * ka.x) * lam_hi : -INFINITY;
      z[2] = vb ? fmaf(d1[2], kb.y, d0[2] * kb.x) * lam_lo : -INFINITY;
      z[3] = vb ? fmaf(d1[3], kb.y, d0[3] * kb.x) * lam_hi : -INFINITY;
    }
    float mx0 = fmaxf(z[0], z[2]), mx1 = fmaxf(z[1], z[3]);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    if (g == 0) {
      red_s[0][warp][2 * tq] = mx0;
      red_s[0][warp][2 * tq + 1] = mx1;
    }
    __syncthreads();
    float mt0 = red_s[0][0][2 * tq], mt1 = red_s[0][0][2 * tq + 1];
#pragma unroll
    for (int w = 1; w < 4; ++w) {
      mt0 = fmaxf(mt0, red_s[0][w][2 * tq]);
      mt1 = fmaxf(mt1, red_s[0][w][2 * tq + 1]);
    }
    const float mn0 = fmaxf(m_run[0], mt0), mn1 = fmaxf(m_run[1], mt1);
    const float al0 = (mn0 == -INFINITY) ? 1.f : expf(m_run[0] - mn0);
    const float al1 = (mn1 == -INFINITY) ? 1.f : expf(m_run[1] - mn1);
    float pr[4];
    pr[0] = (z[0] == -INFINITY) ? 0.f : expf(z[0] - mn0);
    pr[1] = (z[1] == -INFINITY) ? 0.f : expf(z[1] - mn1);
    pr[2] = (z[2] == -INFINITY) ? 0.f : expf(z[2] - mn0);
    pr[3] = (z[3] == -INFINITY) ? 0.f : expf(z[3] - mn1);
    float ls0 = pr[0] + pr[2], ls1 = pr[1] + pr[3];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      ls0 += __shfl_xor_sync(0xffffffffu, ls0, o);
      ls1 += __shfl_xor_sync(0xffffffffu, ls1, o);
    }
    if (g == 0) {
      red_s[1][warp][2 * tq] = ls0;
      red_s[1][warp][2 * tq + 1] = ls1;
    }
    p_s[2 * tq][cb + g] = pr[0];
    p_s[2 * tq + 1][cb + g] = pr[1];
    p_s[2 * tq][cb + g + 8] = pr[2];
    p_s[2 * tq + 1][cb + g + 8] = pr[3];
    __syncthreads();
    float lt0 = red_s[1][0][2 * tq], lt1 = red_s[1][0][2 * tq + 1];
#pragma unroll
    for (int w = 1; w < 4; ++w) {
      lt0 += red_s[1][w][2 * tq];
      lt1 += red_s[1][w][2 * tq + 1];
    }
    l_run[0] = fmaf(l_run[0], al0, lt0);
    l_run[1] = fmaf(l_run[1], al1, lt1);
    m_run[0] = mn0;
    m_run[1] = mn1;

    // ---- power of two 2^k for this warp's V-scale group: max |vs| 2^k in [8, 16).
    float vmax = 0.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int c = lane + 32 * q;
      if (S.valid[c]) vmax = fmaxf(vmax, fabsf(S.vs[c * n_vg + vgrp]));
    }
    vmax = warp_max(vmax);
    int ve = 0;
    if (vmax > 0.f) frexpf(vmax, &ve);
    const int vk = vmax > 0.f ? max(-126, min(127, 4 - ve)) : 0;
    const float vup = pow2i(vk), vdown = pow2i(-vk);

    // ---- O^T[32 dims of this warp x heads] = Vcode^T . W over the sub-tile's 64 cells.
    float pv[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int c0 = 16 * s + 4 * tq;
      const float4 pp = *reinterpret_cast<const float4*>(&p_s[g][c0]);
      float w[4] = {pp.x, pp.y, pp.z, pp.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) w[q] = S.valid[c0 + q] ? w[q] * (S.vs[(c0 + q) * n_vg + vgrp] * vup) : 0.f;
      uint32_t bh0, bl0, bh1, bl1;
      split_pair(w[0], w[1], bh0, bl0);
      split_pair(w[2], w[3], bh1, bl1);
      uint32_t x[4];
      uint32_t bias;
      if (!v4) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          x[q] = *reinterpret_cast<const uint32_t*>(S.v + (c0 + q) * kD + 32 * warp + 4 * g) ^ 0x80808080u;
        bias = 0x64806480u;
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t b = *reinterpret_cast<const uint16_t*>(S.v + (c0 + q) * 64 + 16 * warp + 2 * g);
          x[q] = __byte_perm(b & 0x0F0Fu, (b >> 4) & 0x0F0Fu, 0x5140);   // nibbles -> bytes, dim order
        }
        bias = 0x64086408u;
      }
      // m-tile 0: dims 32w + 4g + {0, 1}; m-tile 1: dims 32w + 4g + {2, 3}
      const uint32_t y01l = __byte_perm(x[0], x[1], 0x5140), y01h = __byte_perm(x[0], x[1], 0x7362);
      const uint32_t y23l = __byte_perm(x[2], x[3], 0x5140), y23h = __byte_perm(x[2], x[3], 0x7362);
      uint32_t a0[4], a1[4];
      a0[0] = byte_pair_h2(y01l, 0x4140, bias);
      a0[1] = byte_pair_h2(y01l, 0x4342, bias);
      a0[2] = byte_pair_h2(y23l, 0x4140, bias);
      a0[3] = byte_pair_h2(y23l, 0x4342, bias);
      a1[0] = byte_pair_h2(y01h, 0x4140, bias);
      a1[1] = byte_pair_h2(y01h, 0x4342, bias);
      a1[2] = byte_pair_h2(y23h, 0x4140, bias);
      a1[3] = byte_pair_h2(y23h, 0x4342, bias);
      mma16816(pv[0], a0, bh0, bh1);
      mma16816(pv[0], a0, bl0, bl1);
      mma16816(pv[1], a1, bh0, bh1);
      mma16816(pv[1], a1, bl0, bl1);
    }
    // ---- fold: O = O * alpha + PV / 2^k (columns: heads 2tq, 2tq+1)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      o_acc[i][0] = fmaf(o_acc[i][0], al0, pv[i][0] * vdown);
      o_acc[i][1] = fmaf(o_acc[i][1], al1, pv[i][1] * vdown);
      o_acc[i][2] = fmaf(o_acc[i][2], al0, pv[i][2] * vdown);
      o_acc[i][3] = fmaf(o_acc[i][3], al1, pv[i][3] * vdown);
    }

    // ---- last sub-tile of the chunk: write its partials (heads 2tq, 2tq+1 < G; dims 32w + 4g ..).
    if (nx.st == 0) {
      const size_t base = ((size_t)t * p.n_q_heads + h * G) * p.n_chunks + it.j;
      if (2 * tq < G) {
        float* o = p.o + (base + (size_t)(2 * tq) * p.n_chunks) * kD + 32 * warp + 4 * g;
        *reinterpret_cast<float4*>(o) = make_float4(o_acc[0][0], o_acc[0][2], o_acc[1][0], o_acc[1][2]);
        if (warp == 0 && g == 0) {
          p.ml[(base + (size_t)(2 * tq) * p.n_chunks) * 2 + 0] = m_run[0];
          p.ml[(base + (size_t)(2 * tq) * p.n_chunks) * 2 + 1] = l_run[0];
        }
      }
      if (2 * tq + 1 < G) {
        float* o = p.o + (base + (size_t)(2 * tq + 1) * p.n_chunks) * kD + 32 * warp + 4 * g;
        *reinterpret_cast<float4*>(o) = make_float4(o_acc[0][1], o_acc[0][3], o_acc[1][1], o_acc[1][3]);
        if (warp == 0 && g == 0) {
          p.ml[(base + (size_t)(2 * tq + 1) * p.n_chunks) * 2 + 0] = m_run[1];
          p.ml[(base + (size_t)(2 * tq + 1) * p.n_chunks) * 2 + 1] = l_run[1];
        }
      }
    }
    __syncthreads();
    if (!has_next) break;
    it = nx;
  }
}

// Merge: one CTA per (q head, row), 4 x 128 threads.  The chunk weights
// exp(m_j - M) are computed in parallel; quarter k of the CTA folds the live
// chunks j = k (mod 4) of its dim in chunk order with fmaf (independent loads,
// so they pipeline), and the four partial sums and the l sums are combined in
// a fixed order.
constexpr int kMergeThreads = 512;

__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const MergeParams p) {
  extern __shared__ float w_s[];   // [n_chunks]
  __shared__ float red[kMergeThreads / 32];
  __shared__ float part[4][kD];
  __shared__ float s_M, s_L;
  const int g = blockIdx.x, t = blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int d = tid & (kD - 1), qtr = tid >> 7;
  ms::pdl_wait();   // partials of the preceding launch (a no-op without that dependency)
  const int n_sel = __ldg(p.n_sel + t);
  const size_t base = ((size_t)t * p.n_q_heads + g) * p.n_chunks;
  // Chunk partials of this quarter's first chunks and this thread's (m, l), loaded before their
  // weights are known and, inside the partials buffer, before n_sel is: chunks past the selection
  // are dropped below without being read for anything.
  constexpr int kPre = 16;
  float o_pre[kPre];
  const float* o = p.o + base * kD + d;
#pragma unroll
  for (int i = 0; i < kPre; ++i) {
    const int jj = qtr + 4 * i;
    o_pre[i] = jj < p.n_chunks ? __ldg(o + (size_t)jj * kD) : 0.f;
  }
  const float2 ml_first =
      tid < p.n_chunks ? __ldg(reinterpret_cast<const float2*>(p.ml) + base + tid) : make_float2(-INFINITY, 0.f);
  const int n_act = min(p.n_chunks, (max(n_sel, 0) + p.chunk_cells - 1) / p.chunk_cells);
  float M = -INFINITY, lsum_self = 0.f, m_self = -INFINITY;
  for (int jj = tid; jj < n_act; jj += kMergeThreads) {
    const float2 ml = jj == tid ? ml_first : __ldg(reinterpret_cast<const float2*>(p.ml) + base + jj);
    w_s[jj] = ml.x;
    M = fmaxf(M, ml.x);
    if (jj == tid) { m_self = ml.x; lsum_self = ml.y; }
  }
  M = warp_max(M);
  if (lane == 0) red[warp] = M;
  __syncthreads();
  if (tid == 0) {
    float mm = red[0];
    for (int w = 1; w < kMergeThreads / 32; ++w) mm = fmaxf(mm, red[w]);
    s_M = mm;
  }
  __syncthreads();
  M = s_M;
  float* out = p.out + ((size_t)t * p.n_q_heads + g) * kD;
  if (M == -INFINITY) {
    if (tid < kD) out[tid] = 0.f;
    if (p.lse && tid == 0) p.lse[(size_t)t * p.n_q_heads + g] = -INFINITY;
    return;
  }
  float lsum = 0.f;
  for (int jj = tid; jj < n_act; jj += kMergeThreads) {
    const float mj = (jj == tid) ? m_self : w_s[jj];
    const float w = (mj == -INFINITY) ? 0.f : expf(mj - M);
    w_s[jj] = w;
    const float lj = (jj == tid) ? lsum_self : __ldg(p.ml + (base + jj) * 2 + 1);
    lsum = fmaf(lj, w, lsum);
  }
  lsum = warp_sum(lsum);
  __syncthreads();
  if (lane == 0) red[warp] = lsum;
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kPre; ++i) {
    const int jj = qtr + 4 * i;
    if (jj < n_act) acc = fmaf(o_pre[i], w_s[jj], acc);
  }
#pragma unroll 8
  for (int jj = qtr + 4 * kPre; jj < n_act; jj += 4) acc = fmaf(__ldg(o + (size_t)jj * kD), w_s[jj], acc);
  part[qtr][d] = acc;
  __syncthreads();
  if (tid == 0) {
    float L = 0.f;
    for (int w = 0; w < kMergeThreads / 32; ++w) L += red[w];
    s_L = L;
  }
  __syncthreads();
  if (tid < kD) {
    const float L = s_L;
    out[tid] = (((part[0][tid] + part[1][tid]) + part[2][tid]) + part[3][tid]) / L;
    if (p.lse && tid == 0) p.lse[(size_t)t * p.n_q_heads + g] = M + logf(L);
  }
}

}  // namespace

cudaError_t launch_decode_attn(const AttnParams& p, cudaStream_t stream) {
  const int n_chunks_max = (p.k_cells + p.chunk_cells - 1) / p.chunk_cells;
  if (n_chunks_max == 0) return cudaSuccess;
  // (row, KV head) pairs x CTAs per pair, filling about 5 resident CTAs per SM.
  const int n_pairs = p.n_kv_heads * p.n_rows;
  const int cpp = max(1, min(n_chunks_max, device_sm_count() * 5 / n_pairs));
  decode_chunk_kernel<<<n_pairs * cpp, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attn_merge_ex(const MergeParams& p, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_q_heads, p.n_rows);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = sizeof(float) * p.n_chunks;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_merge_kernel, p);
}

cudaError_t launch_attn_merge(const MergeParams& p, cudaStream_t stream) { return launch_attn_merge_ex(p, stream, false); }

}  // namespace qsa
