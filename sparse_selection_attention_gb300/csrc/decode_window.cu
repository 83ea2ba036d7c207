// One decode window in one call (qsa_decode_window): q fragments -> block scores -> top-k ->
// split-KV attention -> log-sum-exp merge, as five launches chained on one stream with
// programmatic dependent launch, so that each launch's start-up and prologue overlap the tail of
// the one before ("#2806 sycl: decode QSA selection and attention in fewer, shorter launches",
// Summary and What changed: selection and attention of a window in fewer launches; "#1888 QSA
// decode attention: split each query's cells across blocks", Summary: each query's cells split
// among blocks and merged by the log-sum-exp rescale in split order).
//
//  1. win_qprep_kernel: per (row, KV head) qbar = sum of the group's q heads, scaled by a power
//     of two and split into fp16 hi + lo, laid out as the block-score kernel's mma B fragments
//     (computed once per window instead of once per CTA).
//  2. win_scores_kernel: one CTA per (pool, block); all of the block's K codes and scales are
//     copied into shared memory (cp.async) before the kernel waits for step 1; warp items of two
//     16-cell m-tiles of one KV head share every fragment load.  S^T = Kcode . qbar on mma.sync
//     (int8 codes, or 4-bit codes of the q4_0 layout); cell weights by K scale, fixed butterflies
//     over cells, then over heads and m-tiles.  The result is the qsa_block_scores definition.
//  3. topk_kernel (topk.cu), unchanged arithmetic.
//  4. win_attn8_kernel<K4, V4> (each warp owns its 16-cell slices; int8 or 4-bit K and V, one
//     format per launch) or, for a window whose pools mix V formats, win_attn_kernel (the warps
//     share 64-cell sub-tiles): one CTA per (row, KV head, split of the selection); each split's
//     partial (m, l, o) per q head goes to the workspace in the qsa_decode_attn partials layout (a
//     split of the window is a chunk of that layout).  Splits past the selection launch no work.
//  5. attn_merge_kernel (decode_attn.cu): the log-sum-exp merge in split order, skipping empty
//     splits; bitwise reproducible.
#include "kernels.h"
#include "mma_sync.cuh"

namespace qsa {

namespace {

using namespace ms;

constexpr int kAttnThreads = 128;
constexpr int kSub = 64;   // cells per sub-tile of the attention
constexpr int kMaxSplits = 256;   // splits per (row, KV head)

__device__ __forceinline__ int pool_index(const int* unit_begin, int n_pools, int unit) {
  int pi = 0;
  while (pi + 1 < n_pools && unit >= unit_begin[pi + 1]) ++pi;
  return pi;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int w) {
  return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
}

// ------------------------------------------------------------------------------------------ 1
// Fragment layout (uint4 per lane): frag[((h * NT + nt) * 8 + s) * 32 + lane] holds, for row
// 8 nt + lane / 4, four dims d0 .. d0 + 3 of k-step s as {hi(d0, d0+1), hi(d0+2, d0+3),
// lo(d0, d0+1), lo(d0+2, d0+3)}: the B operand of mma.m16n8k16 for the same permutation of dims
// that the A fragments of the codes use.  int8 K: k-step s = 4 grp + sp takes, in lane column
// group tq = lane % 4, dims 64 grp + 16 tq + 4 sp (inside one 64-dim scale group).  4-bit K
// (k4): k-step s = 2 gq + j takes dims 32 gq + 8 tq + 4 j (inside one 32-dim scale group).
// The fragment of row t and KV head h for this lane (a whole warp calls it): qbar = the sum of the
// head's q heads (dims 4 lane .. + 3), max |qbar 2^fe| in [64, 128), split into fp16 hi + lo; rows
// at or past n_rows give zero fragments.
__device__ __forceinline__ void q_fragment(const float* __restrict__ q, int t, int h, int n_rows, int n_q_heads,
                                           int n_kv_heads, int NT, int k4, int lane, uint4* frag, float* inv_f) {
  const int G = n_q_heads / n_kv_heads;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (t < n_rows) {
    const float* qg = q + ((size_t)t * n_q_heads + (size_t)h * G) * kD + 4 * lane;
    for (int gg = 0; gg < G; ++gg) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(qg + (size_t)gg * kD));
      v[0] += x.x;
      v[1] += x.y;
      v[2] += x.z;
      v[3] += x.w;
    }
  }
  const float amax = warp_max(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
  const int fe = scale_exp_128(amax);
  const float f = pow2i(fe);
  if (lane == 0 && t < n_rows) inv_f[t * n_kv_heads + h] = pow2i(-fe);
  const int d0 = 4 * lane;
  const int s = k4 ? 2 * (d0 >> 5) + ((d0 >> 2) & 1) : 4 * (d0 >> 6) + ((d0 >> 2) & 3);
  const int tqp = k4 ? (d0 >> 3) & 3 : (d0 >> 4) & 3;
  const int nt = t >> 3, gp = t & 7;
  uint32_t h01, l01, h23, l23;
  split_pair(v[0] * f, v[1] * f, h01, l01);
  split_pair(v[2] * f, v[3] * f, h23, l23);
  frag[((h * NT + nt) * 8 + s) * 32 + gp * 4 + tqp] = make_uint4(h01, h23, l01, l23);
}

__global__ void __launch_bounds__(32) win_qprep_kernel(const float* __restrict__ q, int n_rows, int n_q_heads,
                                                       int n_kv_heads, int NT, int k4, uint4* frag, float* inv_f) {
  pdl_trigger();
  pdl_wait();   // q staged by the preceding launch (a no-op without that dependency)
  q_fragment(q, blockIdx.x, blockIdx.y, n_rows, n_q_heads, n_kv_heads, NT, k4, threadIdx.x, frag, inv_f);
}

// ------------------------------------------------------------------------------------------ 2
// One 256-thread CTA per unit (pool, block).  Thread i copies 64 bytes of one cell's K codes (and
// half 0 its two K scales) into shared memory with cp.async before the kernel waits for step 1, so
// every read of the CTA is in flight at once and no register is held across the wait; warp tasks
// (KV head, 16-cell m-tile) then take their operands from shared memory.
constexpr int kScoreThreads = 256;
constexpr size_t kFragSmemMax = 16384;   // q fragments staged in shared memory up to this size
// Score CTAs make their own q fragments in windows of up to this many blocks (at most one CTA per
// SM): the tiny dense window takes 15.6 instead of 17.7 us; at 512 blocks (the verify window) the
// per-CTA fragment work costs more than the launch it saves (31.8 against 29.7 us).
constexpr int kOwnFragUnits = 152;
constexpr int kMaxInvF = 2 * kScoreThreads;   // (row, KV head) factors in shared memory (R * Hkv <= 32 * 16)

// K4: 4-bit K codes (the q4_0 layout): rows of 64 bytes, four scales per cell.
template <int NT, bool K4>
__global__ void __launch_bounds__(kScoreThreads, 4) win_scores_kernel(const ScoresParams p,
                                                                       const uint4* __restrict__ frag,
                                                                       const float* __restrict__ inv_f) {
  extern __shared__ __align__(16) uint8_t sm[];
  constexpr int kRow = K4 ? kD / 2 : kD, kNs = K4 ? 4 : 2;   // code bytes and scales per (head, cell)
  const int B = p.block_cells, Hkv = p.n_kv_heads, R = p.n_rows;
  const int lgB = 31 - __clz(B);   // B is a power of two
  const int mts = B >> 4, tpu = Hkv * mts;
  uint8_t* codes = sm;                                                    // [Hkv][B][kRow]
  float* kscale = reinterpret_cast<float*>(sm + (size_t)Hkv * B * kRow);  // [Hkv][B][kNs]
  float* part = kscale + (size_t)Hkv * B * kNs;                           // [tpu][NT * 8]
  float* invf_s = part + (size_t)tpu * NT * 8;                            // [R][Hkv]
  uint4* frag_s = reinterpret_cast<uint4*>(invf_s + kMaxInvF);            // [Hkv][NT][8][32] (frag_smem)
  const int unit = blockIdx.x;
  const int pi = pool_index(p.unit_begin, p.n_pools, unit);
  const PoolDev& pool = p.pools[pi];
  const int b = unit - p.unit_begin[pi];
  const int cell0 = b * B;
  const int n_b = min(B, pool.n_filled - cell0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tq = lane & 3;
  {
    const int page = __ldg(pool.page_table + cell0 / pool.page_cells);
    const long long slot00 = (long long)page * Hkv * pool.page_cells + cell0 % pool.page_cells;
    for (int item = tid; item < 2 * Hkv * B; item += kScoreThreads) {
      const int half = item & 1, hc = item >> 1, h = hc >> lgB, c = hc & (B - 1);
      if (c < n_b) {
        const long long slot = slot00 + (long long)h * pool.page_cells + c;
        if constexpr (K4) {
          const int8_t* src = pool.k_codes + slot * kRow + 32 * half;
          uint8_t* dst = codes + (size_t)hc * kRow + 32 * half;
          cp_async16(dst, src);
          cp_async16(dst + 16, src + 16);
          if (!half) cp_async16(kscale + 4 * hc, pool.k_scales + slot * 4);
        } else {
          const int8_t* src = pool.k_codes + slot * kD + 64 * half;
          uint8_t* dst = codes + (size_t)hc * kD + 64 * (half ^ (c & 1));   // odd rows: halves swapped
#pragma unroll
          for (int k = 0; k < 4; ++k) cp_async16(dst + 16 * k, src + 16 * k);
          if (!half) cp_async8(kscale + 2 * hc, pool.k_scales + slot * 2);
        }
      } else if (!half) {
#pragma unroll
        for (int k = 0; k < kNs; ++k) kscale[kNs * hc + k] = 0.f;   // cells past the fill weigh nothing
      }
    }
    cp_async_commit();
  }
  pdl_trigger();
  pdl_wait();   // q fragments (or, with host inputs, q) of the preceding launch
  const bool fsm = p.frag_smem != 0;
  if (p.own_frag) {
    // Small windows: every CTA makes the q fragments and factors itself, from q, while its codes
    // are in flight (the values of win_qprep_kernel, without its launch).
    for (int task = warp; task < NT * 8 * Hkv; task += kScoreThreads / 32)
      q_fragment(p.q, task / Hkv, task % Hkv, R, p.n_q_heads, Hkv, NT, K4 ? 1 : 0, lane, frag_s, invf_s);
    cp_async_wait_all();
  } else {
    // The fragments every task reads, copied once into shared memory while the codes are in flight.
    if (fsm) {
      for (int i = tid; i < Hkv * NT * 8 * 32; i += kScoreThreads) cp_async16(frag_s + i, frag + i);
      cp_async_commit();
    }
    // per-(row, head) factors 2^-fe of the fragments, read while the codes arrive
    const float invf0 = tid < R * Hkv ? __ldg(inv_f + tid) : 0.f;
    const float invf1 = tid + kScoreThreads < R * Hkv ? __ldg(inv_f + tid + kScoreThreads) : 0.f;
    cp_async_wait_all();
    if (tid < R * Hkv) invf_s[tid] = invf0;
    if (tid + kScoreThreads < R * Hkv) invf_s[tid + kScoreThreads] = invf1;
  }
  __syncthreads();

  if constexpr (!K4) {
  // Warp work item: TPW consecutive m-tiles of one KV head, which share every fragment load.
  constexpr int TPW = NT == 1 ? 2 : 1;
  const int ipb = (mts + TPW - 1) / TPW;   // items per head
  for (int item = warp; item < Hkv * ipb; item += kScoreThreads / 32) {
    const int h = item / ipb, mt0 = TPW * (item % ipb);
    const int cnt = min(TPW, mts - mt0);
    float d[TPW][NT][2][4];   // [m-tile][n-tile][K-scale group]: hi and lo parts of qbar accumulate together
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int gr = 0; gr < 2; ++gr)
#pragma unroll
          for (int i = 0; i < 4; ++i) d[tt][nt][gr][i] = 0.f;
    const size_t fo = (size_t)h * NT * 8 * 32 + lane;
#pragma unroll
    for (int gr = 0; gr < 2; ++gr) {
      // codes of dims 64 gr .. + 63 of the lane's cells g and g + 8 (rows of odd cells hold the two
      // 64-byte halves swapped, so the eight lanes of each load phase hit eight different chunks)
      uint4 c[TPW][2];
#pragma unroll
      for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
        for (int ab = 0; ab < 2; ++ab) {
          const int row = h * B + 16 * (mt0 + tt) + g + 8 * ab;
          c[tt][ab] = tt < cnt ? *reinterpret_cast<const uint4*>(codes + (size_t)row * kD + 64 * (gr ^ (g & 1)) + 16 * tq)
                               : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int s = 4 * gr + w;
        uint32_t a[TPW][4];
#pragma unroll
        for (int tt = 0; tt < TPW; ++tt) {
          const uint32_t wa = word_of(c[tt][0], w) ^ 0x80808080u;
          const uint32_t wb = word_of(c[tt][1], w) ^ 0x80808080u;
          a[tt][0] = byte_pair_h2(wa, 0x4140, kBiasS8);
          a[tt][2] = byte_pair_h2(wa, 0x4342, kBiasS8);
          a[tt][1] = byte_pair_h2(wb, 0x4140, kBiasS8);
          a[tt][3] = byte_pair_h2(wb, 0x4342, kBiasS8);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint4 bf = fsm ? frag_s[fo + (nt * 8 + s) * 32] : __ldg(frag + fo + (nt * 8 + s) * 32);
#pragma unroll
          for (int tt = 0; tt < TPW; ++tt) {
            if (tt < cnt) {
              mma16816(d[tt][nt][gr], a[tt], bf.x, bf.y);
              mma16816(d[tt][nt][gr], a[tt], bf.z, bf.w);
            }
          }
        }
      }
    }
    // cell weights by K scale, the lane's two cells summed, then a butterfly over the 8 cell pairs
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt) {
      if (tt < cnt) {
        const int task = h * mts + mt0 + tt;
        const int row0 = h * B + 16 * (mt0 + tt) + g;
        const float2 ks0 = *reinterpret_cast<const float2*>(kscale + 2 * row0);
        const float2 ks1 = *reinterpret_cast<const float2*>(kscale + 2 * (row0 + 8));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float(&x)[2][4] = d[tt][nt];
          float e0 = fmaf(ks0.y, x[1][0], ks0.x * x[0][0]);
          e0 += fmaf(ks1.y, x[1][2], ks1.x * x[0][2]);
          float e1 = fmaf(ks0.y, x[1][1], ks0.x * x[0][1]);
          e1 += fmaf(ks1.y, x[1][3], ks1.x * x[0][3]);
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            e0 += __shfl_xor_sync(0xffffffffu, e0, o);
            e1 += __shfl_xor_sync(0xffffffffu, e1, o);
          }
          if (g == 0) {
            const int row = nt * 8 + 2 * tq;
            part[task * NT * 8 + row] = row < R ? e0 * invf_s[row * Hkv + h] : 0.f;
            part[task * NT * 8 + row + 1] = row + 1 < R ? e1 * invf_s[(row + 1) * Hkv + h] : 0.f;
          }
        }
      }
    }
  }
  } else {
  // 4-bit K: lane column group tq holds, in 32-dim scale group gq, dims 32 gq + 8 tq .. + 7 (one 32-bit
  // word: byte 16 gq + 4 tq of the 64-byte row); k-step s = 2 gq + j takes its dims 4 j .. 4 j + 3.
  constexpr int TPW = NT == 1 ? 2 : 1;
  const int ipb = (mts + TPW - 1) / TPW;   // items per head
  for (int item = warp; item < Hkv * ipb; item += kScoreThreads / 32) {
    const int h = item / ipb, mt0 = TPW * (item % ipb);
    const int cnt = min(TPW, mts - mt0);
    float d[TPW][NT][4][4];   // [m-tile][n-tile][32-dim K-scale group]
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int gq = 0; gq < 4; ++gq)
#pragma unroll
          for (int i = 0; i < 4; ++i) d[tt][nt][gq][i] = 0.f;
    const size_t fo = (size_t)h * NT * 8 * 32 + lane;
#pragma unroll
    for (int gq = 0; gq < 4; ++gq) {
      uint32_t c[TPW][2];
#pragma unroll
      for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
        for (int ab = 0; ab < 2; ++ab) {
          const int row = h * B + 16 * (mt0 + tt) + g + 8 * ab;
          c[tt][ab] = tt < cnt ? *reinterpret_cast<const uint32_t*>(codes + (size_t)row * kRow + 16 * gq + 4 * tq) : 0u;
        }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int s = 2 * gq + j;
        uint32_t a[TPW][4];
#pragma unroll
        for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
          for (int ab = 0; ab < 2; ++ab) {
            // low nibbles = even dims, high nibbles = odd dims; bytes in dim order for this k-step
            const uint32_t lo = c[tt][ab] & 0x0F0F0F0Fu, hi = (c[tt][ab] >> 4) & 0x0F0F0F0Fu;
            const uint32_t pr = __byte_perm(lo, hi, j ? 0x7362 : 0x5140);
            a[tt][ab] = byte_pair_h2(pr, 0x4140, kBiasNibble);
            a[tt][2 + ab] = byte_pair_h2(pr, 0x4342, kBiasNibble);
          }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint4 bf = fsm ? frag_s[fo + (nt * 8 + s) * 32] : __ldg(frag + fo + (nt * 8 + s) * 32);
#pragma unroll
          for (int tt = 0; tt < TPW; ++tt) {
            if (tt < cnt) {
              mma16816(d[tt][nt][gq], a[tt], bf.x, bf.y);
              mma16816(d[tt][nt][gq], a[tt], bf.z, bf.w);
            }
          }
        }
      }
    }
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt) {
      if (tt < cnt) {
        const int task = h * mts + mt0 + tt;
        const int row0 = h * B + 16 * (mt0 + tt) + g;
        const float4 ks0 = *reinterpret_cast<const float4*>(kscale + 4 * row0);
        const float4 ks1 = *reinterpret_cast<const float4*>(kscale + 4 * (row0 + 8));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float(&x)[4][4] = d[tt][nt];
          float e0 = ks0.x * x[0][0];
          e0 = fmaf(ks0.y, x[1][0], e0);
          e0 = fmaf(ks0.z, x[2][0], e0);
          e0 = fmaf(ks0.w, x[3][0], e0);
          float e0b = ks1.x * x[0][2];
          e0b = fmaf(ks1.y, x[1][2], e0b);
          e0b = fmaf(ks1.z, x[2][2], e0b);
          e0b = fmaf(ks1.w, x[3][2], e0b);
          e0 += e0b;
          float e1 = ks0.x * x[0][1];
          e1 = fmaf(ks0.y, x[1][1], e1);
          e1 = fmaf(ks0.z, x[2][1], e1);
          e1 = fmaf(ks0.w, x[3][1], e1);
          float e1b = ks1.x * x[0][3];
          e1b = fmaf(ks1.y, x[1][3], e1b);
          e1b = fmaf(ks1.z, x[2][3], e1b);
          e1b = fmaf(ks1.w, x[3][3], e1b);
          e1 += e1b;
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            e0 += __shfl_xor_sync(0xffffffffu, e0, o);
            e1 += __shfl_xor_sync(0xffffffffu, e1, o);
          }
          if (g == 0) {
            const int rw = nt * 8 + 2 * tq;
            part[task * NT * 8 + rw] = rw < R ? e0 * invf_s[rw * Hkv + h] : 0.f;
            part[task * NT * 8 + rw + 1] = rw + 1 < R ? e1 * invf_s[(rw + 1) * Hkv + h] : 0.f;
          }
        }
      }
    }
  }
  }
  __syncthreads();
  // S[t, b] for the rows of this pool: lane l holds task l (head-major), then a fixed butterfly.
  for (int t = warp; t < R; t += kScoreThreads / 32) {
    if (p.row_pool[t] != pi) continue;
    float sum = lane < tpu ? part[lane * NT * 8 + t] : 0.f;
    sum = warp_sum(sum);
    if (lane == 0) p.scores[(size_t)t * p.max_blocks + b] = sum * (kInvSqrtD / (float)n_b);
  }
}

// ------------------------------------------------------------------------------------------ 4
struct Stage {
  int8_t k[kSub * kD];   // int8 K rows, or 64-byte 4-bit K rows at the same stride
  uint8_t v[kSub * kD];
  float ks[kSub * 4];    // 2 (int8 K) or 4 (4-bit K) scales per cell
  float vs[kSub * 4];
  int valid[kSub];
};

// Copies of sub-tile `st` of the split into `sg`: thread (cell c = tid / 2, half) copies half of
// the cell's K and V pieces and one of its scale rows; invisible cells copy nothing.
__device__ __forceinline__ void prefetch_sub(const WinAttnParams& p, const PoolDev& pool, Stage& sg, int base, int n_cells,
                                             int st, int t, int h, int pos, bool v4) {
  const int c = threadIdx.x >> 1, half = threadIdx.x & 1;
  const int idx = st * kSub + c;
  bool valid = false;
  long long slot = 0;
  if (idx < n_cells) {
    const int cell = __ldg(p.ids + (size_t)t * p.k_cells + base + idx);
    valid = cell <= pos && cell >= 0 && cell < pool.n_filled;
    if (valid) slot = cell_slot(pool, p.n_kv_heads, h, cell);
  }
  const bool k4 = pool.k_bits == 4;
  if (valid) {
    if (!k4) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int pc = 4 * half + k;
        cp_async16(sg.k + c * kD + pc * 16, pool.k_codes + slot * kD + pc * 16);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int pc = 2 * half + k;
        cp_async16(sg.k + c * kD + pc * 16, pool.k_codes + slot * (kD / 2) + pc * 16);
      }
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
    if (!half) {
      if (k4) cp_async16(sg.ks + 4 * c, pool.k_scales + slot * 4);
      else cp_async8(sg.ks + 4 * c, pool.k_scales + slot * 2);
    }
  }
  if (!half) sg.valid[c] = valid;
  cp_async_commit();
}

__global__ void __launch_bounds__(kAttnThreads, 5) win_attn_kernel(const WinAttnParams p) {
  const int R = p.n_rows, Hkv = p.n_kv_heads;
  const int n_pairs = R * Hkv;
  const int pair = blockIdx.x % n_pairs, split = blockIdx.x / n_pairs;
  const int t = pair % R, h = pair / R;
  const int G = p.n_q_heads / Hkv;
  const int pos = __ldg(p.row_pos + t);
  const PoolDev& pool = p.pools[p.row_pool[t]];
  const bool v4 = pool.v_bits == 4;
  const bool k4 = pool.k_bits == 4;   // the same for every pool of the window
  const int n_vg = v4 ? 4 : 2;

  __shared__ __align__(16) Stage stages[2];
  __shared__ __align__(16) float p_s[8][kSub];
  __shared__ float red_s[2][4][8];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tq = lane & 3;

  // ---- q of head g (this thread's B columns) for k-step s = 0..7: int8 K, dims 16s + 4tq .. +3;
  // 4-bit K, dims 32 (s/2) + 8 tq + 4 (s%2) .. +3 (inside one 32-dim scale group), scaled by 2^fe
  // (max |q 2^fe| in [64, 128)) and split into fp16 hi + lo.  q is an input of the window, so this
  // runs before the wait for the selection.
  uint32_t qh[8][2], ql[8][2];
  float lam_lo, lam_hi;   // logit scale of heads 2tq and 2tq+1
  {
    float qv[8][4];
    float amax = 0.f;
    const float* qrow = p.q + ((size_t)t * p.n_q_heads + h * G + min(g, G - 1)) * kD;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      const int d0 = k4 ? 32 * (s >> 1) + 8 * tq + 4 * (s & 1) : 16 * s + 4 * tq;
      if (g < G) v = __ldg(reinterpret_cast<const float4*>(qrow + d0));
      qv[s][0] = v.x; qv[s][1] = v.y; qv[s][2] = v.z; qv[s][3] = v.w;
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int fe = scale_exp_128(amax);
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

  pdl_wait();   // ids and n_sel of the preceding launch
  const int n_sel = min(__ldg(p.n_sel + t), p.k_cells);
  const int n_act = (n_sel + p.split_cells - 1) / p.split_cells;
  if (split >= n_act) return;   // past the selection: nothing to read, nothing the merge reads
  const int base = split * p.split_cells;
  const int n_cells = min(p.split_cells, n_sel - base);
  const int n_sub = (n_cells + kSub - 1) / kSub;
  prefetch_sub(p, pool, stages[0], base, n_cells, 0, t, h, pos, v4);

  const int vgrp = v4 ? warp : (warp >> 1);   // V-scale group of this warp's 32 dims
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o_acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  for (int st = 0; st < n_sub; ++st) {
    Stage& S = stages[st & 1];
    if (st + 1 < n_sub) {
      prefetch_sub(p, pool, stages[(st + 1) & 1], base, n_cells, st + 1, t, h, pos, v4);
      cp_async_wait_group1();
    } else {
      cp_async_wait_all();
    }
    __syncthreads();

    // ---- S^T = Kcode . (q f)^T on this warp's 16 cells, one accumulator per K-scale group (two
    // 64-dim groups for int8 K, four 32-dim groups for 4-bit K).
    const int cb = 16 * warp;
    float dk[4][4];
#pragma unroll
    for (int gq = 0; gq < 4; ++gq)
#pragma unroll
      for (int i = 0; i < 4; ++i) dk[gq][i] = 0.f;
    if (!k4) {
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(S.k + (cb + g) * kD + 16 * s + 4 * tq) ^ 0x80808080u;
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(S.k + (cb + g + 8) * kD + 16 * s + 4 * tq) ^ 0x80808080u;
        uint32_t a[4];
        a[0] = byte_pair_h2(w0, 0x4140, kBiasS8);
        a[2] = byte_pair_h2(w0, 0x4342, kBiasS8);
        a[1] = byte_pair_h2(w1, 0x4140, kBiasS8);
        a[3] = byte_pair_h2(w1, 0x4342, kBiasS8);
        mma16816(dk[s >> 2], a, qh[s][0], qh[s][1]);
        mma16816(dk[s >> 2], a, ql[s][0], ql[s][1]);
      }
    } else {
#pragma unroll
      for (int gq = 0; gq < 4; ++gq) {
        // one word per row: dims 32 gq + 8 tq .. + 7 (low nibble = even dim)
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(S.k + (cb + g) * kD + 16 * gq + 4 * tq);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(S.k + (cb + g + 8) * kD + 16 * gq + 4 * tq);
        const uint32_t lo0 = w0 & 0x0F0F0F0Fu, hi0 = (w0 >> 4) & 0x0F0F0F0Fu;
        const uint32_t lo1 = w1 & 0x0F0F0F0Fu, hi1 = (w1 >> 4) & 0x0F0F0F0Fu;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int s = 2 * gq + j;
          const uint32_t p0 = __byte_perm(lo0, hi0, j ? 0x7362 : 0x5140);
          const uint32_t p1 = __byte_perm(lo1, hi1, j ? 0x7362 : 0x5140);
          uint32_t a[4];
          a[0] = byte_pair_h2(p0, 0x4140, kBiasNibble);
          a[2] = byte_pair_h2(p0, 0x4342, kBiasNibble);
          a[1] = byte_pair_h2(p1, 0x4140, kBiasNibble);
          a[3] = byte_pair_h2(p1, 0x4342, kBiasNibble);
          mma16816(dk[gq], a, qh[s][0], qh[s][1]);
          mma16816(dk[gq], a, ql[s][0], ql[s][1]);
        }
      }
    }
    // ---- logits of cells cb+g, cb+g+8 for heads 2tq, 2tq+1; masked cells -> -inf.
    float z[4];
    {
      const bool va = S.valid[cb + g], vb = S.valid[cb + g + 8];
      const float4 ka = *reinterpret_cast<const float4*>(S.ks + 4 * (cb + g));
      const float4 kb = *reinterpret_cast<const float4*>(S.ks + 4 * (cb + g + 8));
      float x[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 k = i < 2 ? ka : kb;
        x[i] = fmaf(dk[1][i], k.y, dk[0][i] * k.x);
        if (k4) x[i] = fmaf(dk[3][i], k.w, fmaf(dk[2][i], k.z, x[i]));
      }
      z[0] = va ? x[0] * lam_lo : -INFINITY;
      z[1] = va ? x[1] * lam_hi : -INFINITY;
      z[2] = vb ? x[2] * lam_lo : -INFINITY;
      z[3] = vb ? x[3] * lam_hi : -INFINITY;
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
    for (int q2 = 0; q2 < 2; ++q2) {
      const int c = lane + 32 * q2;
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
      for (int q2 = 0; q2 < 4; ++q2) w[q2] = S.valid[c0 + q2] ? w[q2] * (S.vs[(c0 + q2) * n_vg + vgrp] * vup) : 0.f;
      uint32_t bh0, bl0, bh1, bl1;
      split_pair(w[0], w[1], bh0, bl0);
      split_pair(w[2], w[3], bh1, bl1);
      uint32_t x[4];
      uint32_t bias;
      if (!v4) {
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2)
          x[q2] = *reinterpret_cast<const uint32_t*>(S.v + (c0 + q2) * kD + 32 * warp + 4 * g) ^ 0x80808080u;
        bias = kBiasS8;
      } else {
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) {
          const uint32_t bb = *reinterpret_cast<const uint16_t*>(S.v + (c0 + q2) * 64 + 16 * warp + 2 * g);
          x[q2] = __byte_perm(bb & 0x0F0Fu, (bb >> 4) & 0x0F0Fu, 0x5140);   // nibbles -> bytes, dim order
        }
        bias = kBiasNibble;
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
    __syncthreads();   // the stage and p_s are rewritten by the sub-tile after next
  }

  // ---- this split's partial (qsa_decode_attn layout, split = chunk): heads 2tq, 2tq+1 < G,
  // dims 32w + 4g ..
  const size_t cbase = ((size_t)t * p.n_q_heads + h * G) * p.n_splits + split;
  if (2 * tq < G) {
    const size_t ci = cbase + (size_t)(2 * tq) * p.n_splits;
    *reinterpret_cast<float4*>(p.part_o + ci * kD + 32 * warp + 4 * g) =
        make_float4(o_acc[0][0], o_acc[0][2], o_acc[1][0], o_acc[1][2]);
    if (warp == 0 && g == 0) *reinterpret_cast<float2*>(p.part_ml + ci * 2) = make_float2(m_run[0], l_run[0]);
  }
  if (2 * tq + 1 < G) {
    const size_t ci = cbase + (size_t)(2 * tq + 1) * p.n_splits;
    *reinterpret_cast<float4*>(p.part_o + ci * kD + 32 * warp + 4 * g) =
        make_float4(o_acc[0][1], o_acc[0][3], o_acc[1][1], o_acc[1][3]);
    if (warp == 0 && g == 0) *reinterpret_cast<float2*>(p.part_ml + ci * 2) = make_float2(m_run[1], l_run[1]);
  }
}

// ------------------------------------------------------------------------------------------ 4'
// Warp-owned cells (int8 or 4-bit K, int8 or 4-bit V; one format per launch): the four warps of a
// CTA own their cells.  Warp w walks the 16-cell slices w, w + 4, ...
// of the split through its own two-stage cp.async ring and keeps its own online softmax (base-2
// logits) and O^T accumulators, so no CTA barrier sits in the loop; the W = p * vscale operand is
// formed once per (cell, head, V group).  The warps' states are combined in warp order at the end
// of the split.
//   QK^T: A = K codes of the slice (16 cells x 16 dims per k-step, converted exactly to fp16),
//         B = q of the 8 heads scaled by 2^fe and split into fp16 hi + lo; one accumulator per
//         K-scale group: int8 K, k-step s = 4 gr + w takes dims 64 gr + 16 tq + 4 w .. + 3 (two
//         64-dim groups); 4-bit K, s = 2 gq + j takes dims 32 gq + 8 tq + 4 j .. + 3 (four 32-dim
//         groups).
//   PV:   A = V^T (16 dims x 16 cells), B = W of the slice in fp16 hi + lo per V-scale group,
//         accumulated in O^T (dims x heads).  m-tile mt holds, in row r (and r + 8, the next dim):
//         int8 V, dim 64 (mt / 4) + 8 r + 2 (mt % 4); 4-bit V, dim 32 (mt / 2) + 4 r + 2 (mt % 2);
//         so every m-tile lies in one V-scale group.
//   W is scaled by 2^kv[group] (max |vscale| 2^kv in [8, 16) over the slices seen so far; kv only
//   decreases, and O's rows of that group are rescaled when it does).
constexpr int kSlice = 16;
constexpr int kPageCache = 1024;   // page-table entries the attention keeps in shared memory

// Code rows at a 128-byte stride (a 4-bit row uses 64 bytes of it); 2 (int8) or 4 (4-bit) scales
// per cell.
template <bool K4, bool V4>
struct WarpStage {
  int8_t k[kSlice * kD];
  int8_t v[kSlice * kD];
  float ks[kSlice * (K4 ? 4 : 2)];
  float vs[kSlice * (V4 ? 4 : 2)];
};

// Id of this lane's cell (lane / 2) of the slice starting at split entry `first`, or -1 past the
// split.  The read stays inside the row's k_cells ids, so it may be issued before n_sel is known.
__device__ __forceinline__ int slice_cell_id(const WinAttnParams& p, const int32_t* row_ids, int base, int first,
                                             int n_cells) {
  const int idx = first + ((threadIdx.x & 31) >> 1);
  return (idx < n_cells && base + idx < p.k_cells) ? __ldg(row_ids + idx) : -1;
}

// Copies the slice's cells (ids from slice_cell_id; lane: cell lane / 2, half lane % 2) into `sg`,
// pages looked up in `pt` (the pool's page table, in shared memory when it fits); returns the warp's
// ballot of visible cells (bit 2c + half for cell c).
template <bool K4, bool V4>
__device__ __forceinline__ uint32_t prefetch_slice(const WinAttnParams& p, const PoolDev& pool, const int32_t* pt,
                                                   WarpStage<K4, V4>& sg, int cell, int h, int pos) {
  const int lane = threadIdx.x & 31, c = lane >> 1, half = lane & 1;
  const bool valid = cell >= 0 && cell <= pos && cell < pool.n_filled;
  long long slot = 0;
  if (valid) {
    int pg, off;
    if (pool.page_shift >= 0) {
      pg = cell >> pool.page_shift;
      off = cell & (pool.page_cells - 1);
    } else {
      pg = cell / pool.page_cells;
      off = cell - pg * pool.page_cells;
    }
    slot = ((long long)pt[pg] * p.n_kv_heads + h) * pool.page_cells + off;
  }
  if (valid) {
    // 16-byte chunks swizzled within the 128-byte row so that the fragment reads below are free of
    // bank conflicts: int8 K chunk pc of cell c at pc ^ 4 (c & 1), 4-bit K chunk pc at pc ^ (c & 7);
    // int8 V chunk pc at pc ^ 2 ((c >> 1) & 3), 4-bit V chunk pc at pc ^ ((c >> 1) & 3).
    if constexpr (!K4) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int pc = 4 * half + k;
        cp_async16(sg.k + c * kD + ((pc ^ (4 * (c & 1))) << 4), pool.k_codes + slot * kD + pc * 16);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int pc = 2 * half + k;
        cp_async16(sg.k + c * kD + ((pc ^ (c & 7)) << 4), pool.k_codes + slot * (kD / 2) + pc * 16);
      }
    }
    if constexpr (!V4) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int pc = 4 * half + k;
        cp_async16(sg.v + c * kD + ((pc ^ (2 * ((c >> 1) & 3))) << 4), pool.v_codes + slot * kD + pc * 16);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int pc = 2 * half + k;
        cp_async16(sg.v + c * kD + ((pc ^ ((c >> 1) & 3)) << 4), pool.v_codes + slot * (kD / 2) + pc * 16);
      }
    }
    if (!half) {
      if constexpr (K4)
        cp_async16(sg.ks + 4 * c, pool.k_scales + slot * 4);
      else
        cp_async8(sg.ks + 2 * c, pool.k_scales + slot * 2);
    } else {
      if constexpr (V4)
        cp_async16(sg.vs + 4 * c, pool.v_scales + slot * 4);
      else
        cp_async8(sg.vs + 2 * c, pool.v_scales + slot * 2);
    }
  }
  cp_async_commit();
  return __ballot_sync(0xffffffffu, valid);
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float f4_at(const float4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// P.V of one slice for 4-bit V (four 32-dim V-scale groups): the V-scale exponents kv (max |vscale|
// 2^kv in [8, 16) over the slices seen so far, only decreasing), O rescaled by alpha (columns) and
// by the change of kv (rows of the group), then per group W = p vscale 2^kv in fp16 hi + lo (b0 =
// cells 2tq, 2tq+1, b1 = cells 2tq+8, 2tq+9) and O^T += V^T . W over its two m-tiles.  Lane (g, tq)
// reads, of each of those cells, the two bytes of dims 32 gv + 4 g .. + 3 (chunk gv at gv ^ tq).
template <typename StageT>
__device__ __forceinline__ void pv_slice_v4(const StageT& S, float2 pA, float2 pB, bool c0, bool c1, bool c2,
                                            bool c3, float al0, float al1, int g, int tq, int (&kv)[4],
                                            bool (&have_kv)[4], float (&O)[8][4]) {
  const float4 vs0 = *reinterpret_cast<const float4*>(S.vs + 4 * (2 * tq));
  const float4 vs1 = *reinterpret_cast<const float4*>(S.vs + 4 * (2 * tq + 1));
  const float4 vs2 = *reinterpret_cast<const float4*>(S.vs + 4 * (2 * tq + 8));
  const float4 vs3 = *reinterpret_cast<const float4*>(S.vs + 4 * (2 * tq + 9));
  float fac[4] = {1.f, 1.f, 1.f, 1.f};
#pragma unroll
  for (int gv = 0; gv < 4; ++gv) {
    float vx = 0.f;
    if (c0) vx = fmaxf(vx, fabsf(f4_at(vs0, gv)));
    if (c1) vx = fmaxf(vx, fabsf(f4_at(vs1, gv)));
    if (c2) vx = fmaxf(vx, fabsf(f4_at(vs2, gv)));
    if (c3) vx = fmaxf(vx, fabsf(f4_at(vs3, gv)));
    vx = fmaxf(vx, __shfl_xor_sync(0xffffffffu, vx, 1));
    vx = fmaxf(vx, __shfl_xor_sync(0xffffffffu, vx, 2));
    if (vx > 0.f) {   // warp-uniform: the lanes of one tq see the same cells
      int e = 0;
      frexpf(vx, &e);
      const int k = max(-126, min(127, 4 - e));
      if (!have_kv[gv]) {
        kv[gv] = k;
        have_kv[gv] = true;
      } else if (k < kv[gv]) {
        fac[gv] = pow2i(k - kv[gv]);
        kv[gv] = k;
      }
    }
  }
  if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f) || fac[0] != 1.f || fac[1] != 1.f || fac[2] != 1.f ||
      fac[3] != 1.f) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const float f = fac[mt >> 1];
      O[mt][0] *= al0 * f;
      O[mt][1] *= al1 * f;
      O[mt][2] *= al0 * f;
      O[mt][3] *= al1 * f;
    }
  }
#pragma unroll
  for (int gv = 0; gv < 4; ++gv) {
    const float sv = pow2i(kv[gv]);
    uint32_t bh0, bl0, bh1, bl1;
    split_pair(c0 ? pA.x * (f4_at(vs0, gv) * sv) : 0.f, c1 ? pA.y * (f4_at(vs1, gv) * sv) : 0.f, bh0, bl0);
    split_pair(c2 ? pB.x * (f4_at(vs2, gv) * sv) : 0.f, c3 ? pB.y * (f4_at(vs3, gv) * sv) : 0.f, bh1, bl1);
    const int off = ((gv ^ tq) << 4) + 2 * g;
    uint32_t x[4];
#pragma unroll
    for (int q2 = 0; q2 < 4; ++q2) {
      const int cell = 2 * tq + (q2 & 1) + 8 * (q2 >> 1);
      const uint32_t bb = *reinterpret_cast<const uint16_t*>(S.v + cell * kD + off);
      x[q2] = __byte_perm(bb & 0x0F0Fu, (bb >> 4) & 0x0F0Fu, 0x5140);   // nibbles -> bytes, dim order
    }
    // m-tile 2 gv: dims 32 gv + 4 g + {0, 1}; m-tile 2 gv + 1: + {2, 3}
    const uint32_t y01l = __byte_perm(x[0], x[1], 0x5140), y01h = __byte_perm(x[0], x[1], 0x7362);
    const uint32_t y23l = __byte_perm(x[2], x[3], 0x5140), y23h = __byte_perm(x[2], x[3], 0x7362);
    uint32_t a0[4], a1[4];
    a0[0] = byte_pair_h2(y01l, 0x4140, kBiasNibble);
    a0[1] = byte_pair_h2(y01l, 0x4342, kBiasNibble);
    a0[2] = byte_pair_h2(y23l, 0x4140, kBiasNibble);
    a0[3] = byte_pair_h2(y23l, 0x4342, kBiasNibble);
    a1[0] = byte_pair_h2(y01h, 0x4140, kBiasNibble);
    a1[1] = byte_pair_h2(y01h, 0x4342, kBiasNibble);
    a1[2] = byte_pair_h2(y23h, 0x4140, kBiasNibble);
    a1[3] = byte_pair_h2(y23h, 0x4342, kBiasNibble);
    mma16816(O[2 * gv], a0, bh0, bh1);
    mma16816(O[2 * gv], a0, bl0, bl1);
    mma16816(O[2 * gv + 1], a1, bh0, bh1);
    mma16816(O[2 * gv + 1], a1, bl0, bl1);
  }
}

template <bool K4, bool V4>
__global__ void __launch_bounds__(kAttnThreads, 4) win_attn8_kernel(const WinAttnParams p) {
  const int R = p.n_rows, Hkv = p.n_kv_heads;
  const int n_pairs = R * Hkv;
  const int pair = blockIdx.x % n_pairs, split = blockIdx.x / n_pairs;
  const int t = pair % R, h = pair / R;
  const int G = p.n_q_heads / Hkv;
  const int pos = __ldg(p.row_pos + t);
  const PoolDev& pool = p.pools[p.row_pool[t]];

  using Stage8 = WarpStage<K4, V4>;
  __shared__ __align__(16) Stage8 ring[4][2];
  __shared__ __align__(16) float pbuf[4][8][kSlice];
  __shared__ float wm[4][8], wl[4][8];
  __shared__ int32_t pt_s[kPageCache];
  __shared__ uint4 qf_s[8][32];    // warp 0's q fragments: (hi pair, lo pair) per k-step and lane
  __shared__ float2 lam_s[32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tq = lane & 3;

  // ---- q of head g: for k-step s the dims of the K layout (int8: 64 gr + 16 tq + 4 w .. + 3 for
  // s = 4 gr + w; 4-bit: 32 gq + 8 tq + 4 j .. + 3 for s = 2 gq + j), scaled by 2^fe (max |q 2^fe|
  // in [64, 128)) and split into fp16 hi + lo.  q is an input of the window, so
  // this runs before the wait for the selection; warp 0 makes the fragments, the other warps of
  // the CTA (the same row and KV head) take them from shared memory.
  uint32_t qh[8][2], ql[8][2];
  float lam0, lam1;   // base-2 logit scale of heads 2tq and 2tq+1
  if (warp == 0) {
    float qv[8][4];
    float amax = 0.f;
    const float* qrow = p.q + ((size_t)t * p.n_q_heads + h * G + min(g, G - 1)) * kD;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      const int d0 = K4 ? 32 * (s >> 1) + 8 * tq + 4 * (s & 1) : 64 * (s >> 2) + 16 * tq + 4 * (s & 3);
      if (g < G) v = __ldg(reinterpret_cast<const float4*>(qrow + d0));
      qv[s][0] = v.x; qv[s][1] = v.y; qv[s][2] = v.z; qv[s][3] = v.w;
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int fe = scale_exp_128(amax);
    const float f = pow2i(fe);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      split_pair(qv[s][0] * f, qv[s][1] * f, qh[s][0], ql[s][0]);
      split_pair(qv[s][2] * f, qv[s][3] * f, qh[s][1], ql[s][1]);
    }
    const float lam = kInvSqrtD * kLog2e * pow2i(-fe);
    lam0 = __shfl_sync(0xffffffffu, lam, 4 * (2 * tq));
    lam1 = __shfl_sync(0xffffffffu, lam, 4 * (2 * tq + 1));
#pragma unroll
    for (int s = 0; s < 8; ++s) qf_s[s][lane] = make_uint4(qh[s][0], qh[s][1], ql[s][0], ql[s][1]);
    lam_s[lane] = make_float2(lam0, lam1);
  }

  // The pool's page table (an input of the window) into shared memory when it fits.
  const int n_pages = (pool.n_filled + pool.page_cells - 1) / pool.page_cells;
  const int32_t* pt = pool.page_table;
  if (n_pages <= kPageCache) {
    for (int i = tid; i < n_pages; i += kAttnThreads) pt_s[i] = __ldg(pool.page_table + i);
    pt = pt_s;
  }
  __syncthreads();
  if (warp != 0) {
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint4 f = qf_s[s][lane];
      qh[s][0] = f.x;
      qh[s][1] = f.y;
      ql[s][0] = f.z;
      ql[s][1] = f.w;
    }
    const float2 lm = lam_s[lane];
    lam0 = lm.x;
    lam1 = lm.y;
  }
  pdl_wait();   // ids and n_sel of the preceding launch
  const int base = split * p.split_cells;
  const int32_t* row_ids = p.ids + (size_t)t * p.k_cells + base;
  // The ids of the warp's first two slices are read together with n_sel (inside the row's ids, so
  // before the split's extent is known); later ids are read one slice ahead of their copy.
  int id_a = slice_cell_id(p, row_ids, base, kSlice * warp, p.split_cells);
  int id_b = slice_cell_id(p, row_ids, base, kSlice * (warp + 4), p.split_cells);
  const int n_sel = min(__ldg(p.n_sel + t), p.k_cells);
  const int n_act = (n_sel + p.split_cells - 1) / p.split_cells;
  if (split >= n_act) return;   // past the selection: nothing to read, nothing the merge reads
  const int n_cells = min(p.split_cells, n_sel - base);
  const int n_slices = (n_cells + kSlice - 1) / kSlice;
  const int my_n = n_slices > warp ? (n_slices - warp + 3) / 4 : 0;
  if (kSlice * warp + (lane >> 1) >= n_cells) id_a = -1;
  if (kSlice * (warp + 4) + (lane >> 1) >= n_cells) id_b = -1;
  Stage8* rg = ring[warp];
  float(*pb)[kSlice] = pbuf[warp];

  float m2[2] = {-INFINITY, -INFINITY};   // running max (base 2) of heads 2tq, 2tq+1
  float lp[2] = {0.f, 0.f};               // this lane's share of the running sums
  float O[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) O[mt][i] = 0.f;
  constexpr int kVG = V4 ? 4 : 2;   // V-scale groups
  int kv[kVG];
  bool have_kv[kVG];
#pragma unroll
  for (int gv = 0; gv < kVG; ++gv) {
    kv[gv] = 0;
    have_kv[gv] = false;
  }
  uint32_t vmask[2] = {0u, 0u};
  if (my_n > 0) vmask[0] = prefetch_slice(p, pool, pt, rg[0], id_a, h, pos);

  for (int j = 0; j < my_n; ++j) {
    const int st = j & 1;
    if (j + 1 < my_n) {
      vmask[st ^ 1] = prefetch_slice(p, pool, pt, rg[st ^ 1], id_b, h, pos);
      id_b = slice_cell_id(p, row_ids, base, kSlice * (warp + 4 * (j + 2)), n_cells);
      cp_async_wait_group1();
    } else {
      cp_async_wait_all();
    }
    __syncwarp();
    const Stage8& S = rg[st];
    const uint32_t vm = vmask[st];

    // ---- S^T = Kcode . (q f)^T, one accumulator per K-scale group
    constexpr int kKG = K4 ? 4 : 2;
    float dk[kKG][4];
#pragma unroll
    for (int gq = 0; gq < kKG; ++gq)
#pragma unroll
      for (int i = 0; i < 4; ++i) dk[gq][i] = 0.f;
    if constexpr (K4) {
#pragma unroll
      for (int gq = 0; gq < 4; ++gq) {
        // one word per row: dims 32 gq + 8 tq .. + 7 (low nibble = even dim); rows g and g + 8 share
        // the swizzle (chunk gq at gq ^ g)
        const int off = ((gq ^ g) << 4) + 4 * tq;
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(S.k + g * kD + off);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(S.k + (g + 8) * kD + off);
        const uint32_t lo0 = w0 & 0x0F0F0F0Fu, hi0 = (w0 >> 4) & 0x0F0F0F0Fu;
        const uint32_t lo1 = w1 & 0x0F0F0F0Fu, hi1 = (w1 >> 4) & 0x0F0F0F0Fu;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int s = 2 * gq + j;
          const uint32_t p0 = __byte_perm(lo0, hi0, j ? 0x7362 : 0x5140);
          const uint32_t p1 = __byte_perm(lo1, hi1, j ? 0x7362 : 0x5140);
          uint32_t a[4];
          a[0] = byte_pair_h2(p0, 0x4140, kBiasNibble);
          a[2] = byte_pair_h2(p0, 0x4342, kBiasNibble);
          a[1] = byte_pair_h2(p1, 0x4140, kBiasNibble);
          a[3] = byte_pair_h2(p1, 0x4342, kBiasNibble);
          mma16816(dk[gq], a, qh[s][0], qh[s][1]);
          mma16816(dk[gq], a, ql[s][0], ql[s][1]);
        }
      }
    } else {
      float(&d0)[4] = dk[0];
      float(&d1)[4] = dk[kKG - 1];
      const int sk = 4 * (g & 1);   // rows g and g + 8 share the swizzle
      const uint4 ca0 = *reinterpret_cast<const uint4*>(S.k + g * kD + ((tq ^ sk) << 4));
      const uint4 ca1 = *reinterpret_cast<const uint4*>(S.k + g * kD + (((4 + tq) ^ sk) << 4));
      const uint4 cb0 = *reinterpret_cast<const uint4*>(S.k + (g + 8) * kD + ((tq ^ sk) << 4));
      const uint4 cb1 = *reinterpret_cast<const uint4*>(S.k + (g + 8) * kD + (((4 + tq) ^ sk) << 4));
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int w = s & 3;
        const uint32_t wa = word_of(s < 4 ? ca0 : ca1, w) ^ 0x80808080u;
        const uint32_t wb = word_of(s < 4 ? cb0 : cb1, w) ^ 0x80808080u;
        uint32_t a[4];
        a[0] = byte_pair_h2(wa, 0x4140, kBiasS8);
        a[2] = byte_pair_h2(wa, 0x4342, kBiasS8);
        a[1] = byte_pair_h2(wb, 0x4140, kBiasS8);
        a[3] = byte_pair_h2(wb, 0x4342, kBiasS8);
        if (s < 4) {
          mma16816(d0, a, qh[s][0], qh[s][1]);
          mma16816(d0, a, ql[s][0], ql[s][1]);
        } else {
          mma16816(d1, a, qh[s][0], qh[s][1]);
          mma16816(d1, a, ql[s][0], ql[s][1]);
        }
      }
    }
    // ---- base-2 logits of cells g, g+8 for heads 2tq, 2tq+1; masked cells -> -inf
    const bool va = (vm >> (2 * g)) & 1u, vb = (vm >> (2 * g + 16)) & 1u;
    float z[4];
    if constexpr (K4) {
      const float4 ka = *reinterpret_cast<const float4*>(S.ks + 4 * g);
      const float4 kb = *reinterpret_cast<const float4*>(S.ks + 4 * (g + 8));
      float x[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 k = i < 2 ? ka : kb;
        x[i] = fmaf(dk[3][i], k.w, fmaf(dk[2][i], k.z, fmaf(dk[1][i], k.y, dk[0][i] * k.x)));
      }
      z[0] = va ? x[0] * lam0 : -INFINITY;
      z[1] = va ? x[1] * lam1 : -INFINITY;
      z[2] = vb ? x[2] * lam0 : -INFINITY;
      z[3] = vb ? x[3] * lam1 : -INFINITY;
    } else {
      const float2 ka = *reinterpret_cast<const float2*>(S.ks + 2 * g);
      const float2 kb = *reinterpret_cast<const float2*>(S.ks + 2 * (g + 8));
      z[0] = va ? fmaf(dk[1][0], ka.y, dk[0][0] * ka.x) * lam0 : -INFINITY;
      z[1] = va ? fmaf(dk[1][1], ka.y, dk[0][1] * ka.x) * lam1 : -INFINITY;
      z[2] = vb ? fmaf(dk[1][2], kb.y, dk[0][2] * kb.x) * lam0 : -INFINITY;
      z[3] = vb ? fmaf(dk[1][3], kb.y, dk[0][3] * kb.x) * lam1 : -INFINITY;
    }
    float mx0 = fmaxf(z[0], z[2]), mx1 = fmaxf(z[1], z[3]);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float mn0 = fmaxf(m2[0], mx0), mn1 = fmaxf(m2[1], mx1);
    const float al0 = (mn0 == -INFINITY) ? 1.f : ex2f(m2[0] - mn0);
    const float al1 = (mn1 == -INFINITY) ? 1.f : ex2f(m2[1] - mn1);
    const float p0 = (z[0] == -INFINITY) ? 0.f : ex2f(z[0] - mn0);
    const float p1 = (z[1] == -INFINITY) ? 0.f : ex2f(z[1] - mn1);
    const float p2 = (z[2] == -INFINITY) ? 0.f : ex2f(z[2] - mn0);
    const float p3 = (z[3] == -INFINITY) ? 0.f : ex2f(z[3] - mn1);
    lp[0] = fmaf(lp[0], al0, p0 + p2);
    lp[1] = fmaf(lp[1], al1, p1 + p3);
    m2[0] = mn0;
    m2[1] = mn1;

    // ---- p to the B layout: this lane needs cells 2tq, 2tq+1, 2tq+8, 2tq+9 of head g
    pb[2 * tq][g] = p0;
    pb[2 * tq + 1][g] = p1;
    pb[2 * tq][g + 8] = p2;
    pb[2 * tq + 1][g + 8] = p3;
    __syncwarp();
    const float2 pA = *reinterpret_cast<const float2*>(&pb[g][2 * tq]);
    const float2 pB = *reinterpret_cast<const float2*>(&pb[g][2 * tq + 8]);
    const bool c0 = (vm >> (4 * tq)) & 1u, c1 = (vm >> (4 * tq + 2)) & 1u;
    const bool c2 = (vm >> (4 * tq + 16)) & 1u, c3 = (vm >> (4 * tq + 18)) & 1u;
    if constexpr (V4) {
      pv_slice_v4(S, pA, pB, c0, c1, c2, c3, al0, al1, g, tq, kv, have_kv, O);
    } else {
    const float4 vsA = *reinterpret_cast<const float4*>(S.vs + 4 * tq);         // cells 2tq, 2tq+1: (g0, g1)
    const float4 vsB = *reinterpret_cast<const float4*>(S.vs + 4 * tq + 16);    // cells 2tq+8, 2tq+9

    // ---- V-scale exponent per group (slice maximum over visible cells; kv only decreases)
    float fac[2] = {1.f, 1.f};
    {
      float vx0 = 0.f, vx1 = 0.f;
      if (c0) { vx0 = fmaxf(vx0, fabsf(vsA.x)); vx1 = fmaxf(vx1, fabsf(vsA.y)); }
      if (c1) { vx0 = fmaxf(vx0, fabsf(vsA.z)); vx1 = fmaxf(vx1, fabsf(vsA.w)); }
      if (c2) { vx0 = fmaxf(vx0, fabsf(vsB.x)); vx1 = fmaxf(vx1, fabsf(vsB.y)); }
      if (c3) { vx0 = fmaxf(vx0, fabsf(vsB.z)); vx1 = fmaxf(vx1, fabsf(vsB.w)); }
      vx0 = fmaxf(vx0, __shfl_xor_sync(0xffffffffu, vx0, 1));
      vx0 = fmaxf(vx0, __shfl_xor_sync(0xffffffffu, vx0, 2));
      vx1 = fmaxf(vx1, __shfl_xor_sync(0xffffffffu, vx1, 1));
      vx1 = fmaxf(vx1, __shfl_xor_sync(0xffffffffu, vx1, 2));
      const float vx[2] = {vx0, vx1};
#pragma unroll
      for (int gv = 0; gv < 2; ++gv) {
        if (vx[gv] > 0.f) {   // warp-uniform
          int e = 0;
          frexpf(vx[gv], &e);
          const int k = max(-126, min(127, 4 - e));
          if (!have_kv[gv]) {
            kv[gv] = k;
            have_kv[gv] = true;
          } else if (k < kv[gv]) {
            fac[gv] = pow2i(k - kv[gv]);
            kv[gv] = k;
          }
        }
      }
    }
    // ---- O = O * alpha (columns) * 2^(kv change) (rows of the group), when anything changed
    if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f) || fac[0] != 1.f || fac[1] != 1.f) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const float f = fac[mt >> 2];
        O[mt][0] *= al0 * f;
        O[mt][1] *= al1 * f;
        O[mt][2] *= al0 * f;
        O[mt][3] *= al1 * f;
      }
    }
    // ---- W = p vscale 2^kv per group, fp16 hi + lo: b0 = cells (2tq, 2tq+1), b1 = (2tq+8, 2tq+9)
    uint32_t bh[2][2], bl[2][2];
    {
      const float s0 = pow2i(kv[0]), s1 = pow2i(kv[1]);
      const float w00 = c0 ? pA.x * (vsA.x * s0) : 0.f, w01 = c1 ? pA.y * (vsA.z * s0) : 0.f;
      const float w02 = c2 ? pB.x * (vsB.x * s0) : 0.f, w03 = c3 ? pB.y * (vsB.z * s0) : 0.f;
      const float w10 = c0 ? pA.x * (vsA.y * s1) : 0.f, w11 = c1 ? pA.y * (vsA.w * s1) : 0.f;
      const float w12 = c2 ? pB.x * (vsB.y * s1) : 0.f, w13 = c3 ? pB.y * (vsB.w * s1) : 0.f;
      split_pair(w00, w01, bh[0][0], bl[0][0]);
      split_pair(w02, w03, bh[0][1], bl[0][1]);
      split_pair(w10, w11, bh[1][0], bl[1][0]);
      split_pair(w12, w13, bh[1][1], bl[1][1]);
    }
    // ---- O^T += V^T . W: lane (g, tq) reads dims 8g .. 8g+7 and 64 + 8g .. of cells 2tq, 2tq+1,
    // 2tq+8, 2tq+9
    {
      // 8-byte column g (dims 8g..) and g + 8 (dims 64 + 8g..) of rows 2tq, 2tq+1, 2tq+8, 2tq+9,
      // all four with the row swizzle 2 tq on 16-byte chunks = 4 tq on 8-byte columns
      const int oa = 8 * (g ^ (4 * tq)), ob = 8 * ((g + 8) ^ (4 * tq));
      const int8_t* vr = S.v;
      const uint2 x0a = *reinterpret_cast<const uint2*>(vr + (2 * tq) * kD + oa);
      const uint2 x0b = *reinterpret_cast<const uint2*>(vr + (2 * tq) * kD + ob);
      const uint2 x1a = *reinterpret_cast<const uint2*>(vr + (2 * tq + 1) * kD + oa);
      const uint2 x1b = *reinterpret_cast<const uint2*>(vr + (2 * tq + 1) * kD + ob);
      const uint2 x2a = *reinterpret_cast<const uint2*>(vr + (2 * tq + 8) * kD + oa);
      const uint2 x2b = *reinterpret_cast<const uint2*>(vr + (2 * tq + 8) * kD + ob);
      const uint2 x3a = *reinterpret_cast<const uint2*>(vr + (2 * tq + 9) * kD + oa);
      const uint2 x3b = *reinterpret_cast<const uint2*>(vr + (2 * tq + 9) * kD + ob);
      // words of each group: [gv][half word] for the four cells
      const uint32_t wc0[2][2] = {{x0a.x, x0a.y}, {x0b.x, x0b.y}};
      const uint32_t wc1[2][2] = {{x1a.x, x1a.y}, {x1b.x, x1b.y}};
      const uint32_t wc2[2][2] = {{x2a.x, x2a.y}, {x2b.x, x2b.y}};
      const uint32_t wc3[2][2] = {{x3a.x, x3a.y}, {x3b.x, x3b.y}};
#pragma unroll
      for (int gv = 0; gv < 2; ++gv) {
#pragma unroll
        for (int hw = 0; hw < 2; ++hw) {
          const uint32_t u0 = wc0[gv][hw] ^ 0x80808080u, u1 = wc1[gv][hw] ^ 0x80808080u;
          const uint32_t u2 = wc2[gv][hw] ^ 0x80808080u, u3 = wc3[gv][hw] ^ 0x80808080u;
          // bytes 0,1 -> m-tile j = 2 hw; bytes 2,3 -> j = 2 hw + 1
          const uint32_t ylo = __byte_perm(u0, u1, 0x5140), yhi = __byte_perm(u0, u1, 0x7362);
          const uint32_t zlo = __byte_perm(u2, u3, 0x5140), zhi = __byte_perm(u2, u3, 0x7362);
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const uint32_t y = jj ? yhi : ylo, zz = jj ? zhi : zlo;
            uint32_t a[4];
            a[0] = byte_pair_h2(y, 0x4140, kBiasS8);
            a[1] = byte_pair_h2(y, 0x4342, kBiasS8);
            a[2] = byte_pair_h2(zz, 0x4140, kBiasS8);
            a[3] = byte_pair_h2(zz, 0x4342, kBiasS8);
            const int mt = 4 * gv + 2 * hw + jj;
            mma16816(O[mt], a, bh[gv][0], bh[gv][1]);
            mma16816(O[mt], a, bl[gv][0], bl[gv][1]);
          }
        }
      }
    }
    }   // int8 V
    __syncwarp();   // the stage and pb are rewritten by the slice after next
  }

  // ---- combine the warps (in warp order) and write the split's partial
  lp[0] += __shfl_xor_sync(0xffffffffu, lp[0], 4);
  lp[0] += __shfl_xor_sync(0xffffffffu, lp[0], 8);
  lp[0] += __shfl_xor_sync(0xffffffffu, lp[0], 16);
  lp[1] += __shfl_xor_sync(0xffffffffu, lp[1], 4);
  lp[1] += __shfl_xor_sync(0xffffffffu, lp[1], 8);
  lp[1] += __shfl_xor_sync(0xffffffffu, lp[1], 16);
  cp_async_wait_all();
  __syncwarp();
  float* wo = reinterpret_cast<float*>(rg);   // this warp's ring: O^T as [head][128]
  {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const float u = pow2i(-kv[V4 ? mt >> 1 : mt >> 2]);
      const int dim = V4 ? 32 * (mt >> 1) + 4 * g + 2 * (mt & 1) : 64 * (mt >> 2) + 8 * g + 2 * (mt & 3);
      wo[(2 * tq) * kD + dim] = O[mt][0] * u;
      wo[(2 * tq + 1) * kD + dim] = O[mt][1] * u;
      wo[(2 * tq) * kD + dim + 1] = O[mt][2] * u;
      wo[(2 * tq + 1) * kD + dim + 1] = O[mt][3] * u;
    }
    if (g == 0) {
      wm[warp][2 * tq] = m2[0];
      wm[warp][2 * tq + 1] = m2[1];
      wl[warp][2 * tq] = lp[0];
      wl[warp][2 * tq + 1] = lp[1];
    }
  }
  __syncthreads();
  const size_t cbase = ((size_t)t * p.n_q_heads + h * G) * p.n_splits + split;
  for (int hh = 0; hh < G; ++hh) {
    float M = wm[0][hh];
#pragma unroll
    for (int w = 1; w < 4; ++w) M = fmaxf(M, wm[w][hh]);
    float o = 0.f, l = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float mw = wm[w][hh];
        const float sc = (mw == -INFINITY) ? 0.f : ex2f(mw - M);
        o = fmaf(reinterpret_cast<const float*>(ring[w])[hh * kD + tid], sc, o);
        l = fmaf(wl[w][hh], sc, l);
      }
    }
    const size_t ci = cbase + (size_t)hh * p.n_splits;
    p.part_o[ci * kD + tid] = o;
    if (tid == 0) *reinterpret_cast<float2*>(p.part_ml + ci * 2) = make_float2(M * kLn2, l);
  }
}

}  // namespace

// ---------------------------------------------------------------------------------------------
// Host side

int window_split_cells(int n_rows, int n_kv_heads, int k_cells, int n_sm) {
  // about four 128-thread CTAs per SM in one wave (the most the registers allow: the more warps per
  // SM, the more of the gathers' latency is hidden; splits of whole 64-cell rounds, with fewer CTAs,
  // measured 2 us slower on the verify window), splits a multiple of the 16-cell slice, at most
  // kMaxSplits splits per (row, KV head)
  constexpr long long kUnit = 16;
  const long long total = (long long)n_rows * n_kv_heads * (k_cells > 0 ? k_cells : 1);
  const long long target = 4LL * (n_sm > 0 ? n_sm : 1);
  long long sc = kUnit * ((total + kUnit * target - 1) / (kUnit * target));
  const long long min_sc = kUnit * (((long long)k_cells + kUnit * kMaxSplits - 1) / (kUnit * kMaxSplits));
  if (sc < min_sc) sc = min_sc;
  if (sc < kUnit) sc = kUnit;
  return (int)sc;
}

// ------------------------------------------------------------------------------------------ 0
// Inputs in page-locked host memory: one load of each 16 bytes of q and of the row positions across
// the host link, stored into the workspace, so that no later launch of the window (the split
// attention reads q and row_pos in every CTA) waits on the host link.
__global__ void __launch_bounds__(256) stage_inputs_kernel(const float4* __restrict__ q_src, int n_q4,
                                                           const int32_t* __restrict__ pos_src, int n_rows,
                                                           float4* q_dst, int32_t* pos_dst) {
  pdl_trigger();   // the next launch may start its CTAs; it waits for this grid before reading q
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_q4; i += gridDim.x * blockDim.x) q_dst[i] = q_src[i];
  if (blockIdx.x == 0 && threadIdx.x < n_rows) pos_dst[threadIdx.x] = pos_src[threadIdx.x];
}

WindowLayout window_layout(int n_rows, int n_q_heads, int n_kv_heads, int k_cells, int n_sm) {
  WindowLayout L{};
  const int NT = (n_rows + 7) / 8;
  L.split_cells = window_split_cells(n_rows, n_kv_heads, k_cells, n_sm);
  L.n_splits = (k_cells + L.split_cells - 1) / L.split_cells;
  if (L.n_splits < 1) L.n_splits = 1;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  size_t off = 0;
  L.frag = off;
  off = up(off + (size_t)16 * n_kv_heads * NT * 8 * 32);
  L.inv_f = off;
  off = up(off + sizeof(float) * (size_t)n_rows * n_kv_heads);
  L.part_ml = off;   // the qsa_decode_attn partials layout (ml, then o), o 256-byte aligned for vector access
  off = up(off + sizeof(float) * 2 * (size_t)n_rows * n_q_heads * L.n_splits);
  L.part_o = off;
  off = up(off + sizeof(float) * kD * (size_t)n_rows * n_q_heads * L.n_splits);
  L.q_in = off;   // staged q and row positions (calls with host inputs)
  off = up(off + sizeof(float) * kD * (size_t)n_rows * n_q_heads);
  L.pos_in = off;
  off = up(off + sizeof(int32_t) * (size_t)n_rows);
  L.total = off;
  return L;
}

bool window_scores_supported(int n_rows, int n_kv_heads, int block_cells) {
  return n_rows <= 32 && block_cells % 16 == 0 && n_kv_heads * (block_cells / 16) <= 32;
}

template <typename... KArgs, typename... Args>
static cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_chunk_attn_window_kernels(const AttnParams& a, cudaStream_t stream) {
  // A chunk of qsa_decode_attn is a split of this file's attention kernels: same (m, l, o) per
  // (row, q head, chunk) in the same layout, chunks past the selection not written.
  WinAttnParams p{};
  for (int i = 0; i < QSA_MAX_POOLS; ++i) p.pools[i] = a.pools[i];
  bool same_v = true;
  for (int t = 0; t < a.n_rows; ++t) {
    p.row_pool[t] = a.row_pool[t];
    same_v = same_v && a.pools[a.row_pool[t]].v_bits == a.pools[a.row_pool[0]].v_bits;
  }
  p.q = a.q;
  p.row_pos = a.row_pos;
  p.ids = a.ids;
  p.n_sel = a.n_sel;
  p.n_rows = a.n_rows;
  p.n_q_heads = a.n_q_heads;
  p.n_kv_heads = a.n_kv_heads;
  p.k_cells = a.k_cells;
  p.split_cells = a.chunk_cells;
  p.n_splits = a.n_chunks;
  p.part_ml = a.ml;
  p.part_o = a.o;
  const bool k4 = a.pools[a.row_pool[0]].k_bits == 4;
  const bool v4 = a.pools[a.row_pool[0]].v_bits == 4;
  const dim3 grid(a.n_rows * a.n_kv_heads * a.n_chunks);
  if (!same_v) return launch_ex(win_attn_kernel, grid, dim3(kAttnThreads), 0, stream, false, p);
  if (k4)
    return v4 ? launch_ex(win_attn8_kernel<true, true>, grid, dim3(kAttnThreads), 0, stream, false, p)
              : launch_ex(win_attn8_kernel<true, false>, grid, dim3(kAttnThreads), 0, stream, false, p);
  return v4 ? launch_ex(win_attn8_kernel<false, true>, grid, dim3(kAttnThreads), 0, stream, false, p)
            : launch_ex(win_attn8_kernel<false, false>, grid, dim3(kAttnThreads), 0, stream, false, p);
}

cudaError_t launch_decode_window(const WindowArgs& a, cudaStream_t stream, cudaEvent_t* ev) {
  // With `ev` (6 events) the launches are not chained (each starts after the previous one ends) and
  // ev[i] is recorded before launch i, ev[5] after the last: per-kernel times.
  const bool pdl = ev == nullptr;
  auto mark = [&](int i) { return ev ? cudaEventRecord(ev[i], stream) : cudaSuccess; };
  const ScoresParams& sp = a.scores;
  const int R = sp.n_rows, Hkv = sp.n_kv_heads, NT = (R + 7) / 8;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  uint4* frag = reinterpret_cast<uint4*>(ws + a.layout.frag);
  float* inv_f = reinterpret_cast<float*>(ws + a.layout.inv_f);
  WinAttnParams ap = a.attn;
  ap.part_ml = reinterpret_cast<float*>(ws + a.layout.part_ml);
  ap.part_o = reinterpret_cast<float*>(ws + a.layout.part_o);
  ap.split_cells = a.layout.split_cells;
  ap.n_splits = a.layout.n_splits;
  const int n_pairs = R * Hkv;

  // 1. q fragments: an ordinary launch, ordered after everything before it on the stream (the
  //    previous window may still read the workspace).  With host inputs an ordinary launch first
  //    stages q and row_pos into the workspace, and the q fragments follow it chained.
  cudaError_t e = mark(0);
  if (e != cudaSuccess) return e;
  const bool staged = a.q_src != nullptr;
  if (staged) {
    const int n_q4 = R * sp.n_q_heads * (kD / 4);
    const int blocks = (n_q4 + 255) / 256;
    stage_inputs_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(a.q_src), n_q4, a.pos_src, R,
                                                    reinterpret_cast<float4*>(ws + a.layout.q_in),
                                                    reinterpret_cast<int32_t*>(ws + a.layout.pos_in));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int k4 = sp.pools[0].k_bits == 4 ? 1 : 0;   // the pools of a window share k_bits
  const bool sums = block_sums_usable(sp);           // scores from the pools' block summaries: no q prep
  const size_t frag_bytes = (size_t)Hkv * NT * 8 * 32 * sizeof(uint4);
  // Windows of at most kOwnFragUnits blocks: the score CTAs make the q fragments themselves (each
  // reads all of q), which takes the q-preparation launch out of the chain.
  const bool own_frag = !sums && frag_bytes <= kFragSmemMax && sp.total_units <= kOwnFragUnits;
  if (!sums && !own_frag)
    e = launch_ex(win_qprep_kernel, dim3(NT * 8, Hkv), dim3(32), 0, stream, pdl && staged, sp.q, R, sp.n_q_heads, Hkv,
                  NT, k4, frag, inv_f);
  if (e != cudaSuccess) return e;
  e = mark(1);
  if (e != cudaSuccess) return e;
  // 2. block scores
  if (sums) {
    e = launch_sum_scores(sp, stream, pdl && staged);
    if (e != cudaSuccess) return e;
  } else if (sp.total_units > 0) {
    const int tpu = Hkv * (sp.block_cells / 16);
    ScoresParams spx = sp;
    spx.frag_smem = frag_bytes <= kFragSmemMax;
    spx.own_frag = own_frag ? 1 : 0;
    const size_t row_bytes = k4 ? kD / 2 + 16 : kD + 8;   // codes + scales of one (head, cell)
    const size_t smem = (size_t)Hkv * sp.block_cells * row_bytes + sizeof(float) * ((size_t)tpu * NT * 8 + kMaxInvF) +
                        (spx.frag_smem ? frag_bytes : 0);
    using Kern = void (*)(ScoresParams, const uint4*, const float*);
    const Kern k8_kerns[4] = {win_scores_kernel<1, false>, win_scores_kernel<2, false>, win_scores_kernel<3, false>,
                              win_scores_kernel<4, false>};
    const Kern k4_kerns[4] = {win_scores_kernel<1, true>, win_scores_kernel<2, true>, win_scores_kernel<3, true>,
                              win_scores_kernel<4, true>};
    const Kern kern = k4 ? k4_kerns[NT - 1] : k8_kerns[NT - 1];
    e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    e = launch_ex(kern, dim3(sp.total_units), dim3(kScoreThreads), smem, stream, own_frag ? pdl && staged : pdl, spx,
                  (const uint4*)frag, (const float*)inv_f);
    if (e != cudaSuccess) return e;
  }
  e = mark(2);
  if (e != cudaSuccess) return e;
  // 3. top-k
  e = launch_topk_ex(a.topk, a.max_nb, stream, pdl);
  if (e != cudaSuccess) return e;
  e = mark(3);
  if (e != cudaSuccess) return e;
  // 4. split attention: warp-owned cells when the window's pools share one V format (the K format
  //    is shared by validation); the chunk-style kernel for pools of mixed V formats
  bool same_v = true;
  for (int i = 1; i < sp.n_pools; ++i) same_v = same_v && sp.pools[i].v_bits == sp.pools[0].v_bits;
  const dim3 agrid(n_pairs * ap.n_splits);
  if (!same_v)
    e = launch_ex(win_attn_kernel, agrid, dim3(kAttnThreads), 0, stream, pdl, ap);
  else if (sp.pools[0].v_bits == 8)
    e = k4 ? launch_ex(win_attn8_kernel<true, false>, agrid, dim3(kAttnThreads), 0, stream, pdl, ap)
           : launch_ex(win_attn8_kernel<false, false>, agrid, dim3(kAttnThreads), 0, stream, pdl, ap);
  else
    e = k4 ? launch_ex(win_attn8_kernel<true, true>, agrid, dim3(kAttnThreads), 0, stream, pdl, ap)
           : launch_ex(win_attn8_kernel<false, true>, agrid, dim3(kAttnThreads), 0, stream, pdl, ap);
  if (e != cudaSuccess) return e;
  e = mark(4);
  if (e != cudaSuccess) return e;
  // 5. merge of the splits
  MergeParams mp{};
  mp.ml = ap.part_ml;
  mp.o = ap.part_o;
  mp.n_sel = ap.n_sel;
  mp.n_rows = R;
  mp.n_q_heads = sp.n_q_heads;
  mp.chunk_cells = ap.split_cells;
  mp.n_chunks = ap.n_splits;
  mp.out = ap.out;
  mp.lse = ap.lse;
  e = launch_attn_merge_ex(mp, stream, pdl);
  if (e != cudaSuccess) return e;
  return mark(5);
}

}  // namespace qsa
