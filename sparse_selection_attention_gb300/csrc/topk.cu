// Block top-k selection (qsa_topk).
//
// Per row: the k_cells / B highest-scoring blocks, emitted as their filled
// cells in ascending cell id.  Scores become order-preserving uint32 keys
// (-0.0 -> +0.0, NaN -> 0, below -inf), so the selection is integer work and
// its ids are exact ("#2806 sycl: decode QSA selection and attention in
// fewer, shorter launches", Summary: the wide top-k's radix passes find each
// digit with a work-group scan over the bins; integers only, so the same ids).
//
// One CTA per row; thread i holds the keys of blocks [i*K, (i+1)*K) in
// registers.  The threshold T (the kb-th largest key) is found one bit at a
// time from the most significant: T | bit is kept when at least kb keys are
// >= it.  Each step is one CTA-wide count: __syncthreads_count when a thread
// holds one key, else a warp reduction and one barrier.  Blocks with key > T
// are taken, then the lowest-id blocks with key == T.  Two CTA prefix sums in
// block-id order give each chosen block its rank j; every block but the row's
// last holds exactly B cells, so chosen block j fills ids[j*B ..], written
// coalesced by the whole CTA.
#include "kernels.h"

namespace qsa {

namespace {

constexpr int kMaxThreads = 1024;
constexpr int kMaxKeys = 16;   // keys per thread

__device__ __forceinline__ uint32_t score_key(float x) {
  if (x != x) return 0u;                 // NaN ranks below every number
  if (x == 0.0f) x = 0.0f;               // -0.0 == +0.0
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive CTA-wide prefix sum of one int per thread; `tot` receives the total.  The warp totals
// are scanned lane-parallel by every warp (no serial loop over warps).
__device__ __forceinline__ int cta_exclusive_scan(int v, int* warp_tot, int& tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  int wt = lane < n_warps ? warp_tot[lane] : 0;
  int winc = wt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, winc, o);
    if (lane >= o) winc += n;
  }
  const int base = __shfl_sync(0xffffffffu, winc - wt, warp);
  tot = __shfl_sync(0xffffffffu, winc, 31);
  __syncthreads();
  return base + inc - v;
}

// Number of this CTA's keys >= cand (every thread gets the total).
__device__ __forceinline__ int cta_count_ge(const uint32_t (&key)[kMaxKeys], int K, int b0, int nb, uint32_t cand,
                                            int* wsum, int parity) {
  if (K == 1) return __syncthreads_count(b0 < nb && key[0] >= cand);
  int c = 0;
#pragma unroll
  for (int i = 0; i < kMaxKeys; ++i) c += (i < K && b0 + i < nb && key[i] >= cand) ? 1 : 0;
  c = __reduce_add_sync(0xffffffffu, c);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
  if (lane == 0) wsum[parity * 32 + warp] = c;
  __syncthreads();
  // wsum[parity] is rewritten two steps later, after the next barrier
  return __reduce_add_sync(0xffffffffu, lane < n_warps ? wsum[parity * 32 + lane] : 0);
}

__global__ void __launch_bounds__(kMaxThreads) topk_kernel(const TopkParams p) {
  extern __shared__ int smem[];          // chosen list [kb]
  __shared__ int warp_tot[32];
  __shared__ int wsum[64];
  const int t = blockIdx.x, tid = threadIdx.x;
  const int n_threads = blockDim.x;
  const int B = p.block_cells;
  const int n_filled = p.n_filled[t];
  const int nb = (n_filled + B - 1) / B;
  const int kb = min(p.k_cells / B, nb);
  int32_t* ids = p.ids + (size_t)t * p.k_cells;
  if (kb == 0) {
    if (tid == 0) p.n_sel[t] = 0;
    return;
  }
  int* sel = smem;
  const int K = (nb + n_threads - 1) / n_threads;   // <= kMaxKeys
  const int b0 = tid * K;
  const float* sc = p.scores + (size_t)t * p.max_blocks;
  uint32_t key[kMaxKeys];
#pragma unroll
  for (int i = 0; i < kMaxKeys; ++i) key[i] = (i < K && b0 + i < nb) ? score_key(__ldg(sc + b0 + i)) : 0u;

  const bool take_all = (kb == nb);
  uint32_t T = 0;
  int need = 0;
  if (!take_all) {
    for (int bit = 31; bit >= 0; --bit) {
      const uint32_t cand = T | (1u << bit);
      if (cta_count_ge(key, K, b0, nb, cand, wsum, bit & 1) >= kb) T = cand;
    }
    // keys > T (T + 1 does not wrap: the largest key, +inf's, is 0xFF800000); parity 1 follows bit 0's 0
    need = kb - cta_count_ge(key, K, b0, nb, T + 1u, wsum, 1);
  }

  int tot = 0;
  int eq = 0;
  if (!take_all) {
#pragma unroll
    for (int i = 0; i < kMaxKeys; ++i) eq += (i < K && b0 + i < nb && key[i] == T);
  }
  int e = take_all ? 0 : cta_exclusive_scan(eq, warp_tot, tot);
  int chosen = 0;
  uint32_t chosen_bits = 0;
#pragma unroll
  for (int i = 0; i < kMaxKeys; ++i) {
    if (i < K && b0 + i < nb) {
      bool c = take_all || key[i] > T;
      if (!take_all && key[i] == T) { c = e < need; ++e; }
      if (c) { ++chosen; chosen_bits |= 1u << i; }
    }
  }
  int j = cta_exclusive_scan(chosen, warp_tot, tot);
#pragma unroll
  for (int i = 0; i < kMaxKeys; ++i)
    if (chosen_bits & (1u << i)) sel[j++] = b0 + i;
  __syncthreads();
  // ids[j*B + i] = sel[j]*B + i, four at a time when the row's ids start 16-byte aligned (ids aligned,
  // k_cells and B multiples of 4); cells past n_filled (the row's last block) are not written.
  if ((B & 3) == 0 && (p.k_cells & 3) == 0 && (reinterpret_cast<uintptr_t>(p.ids) & 15) == 0) {
    for (int i4 = tid; i4 < kb * B / 4; i4 += n_threads) {
      const int idx = 4 * i4;
      const int cell = sel[idx / B] * B + idx % B;
      if (cell + 3 < n_filled) {
        *reinterpret_cast<int4*>(ids + idx) = make_int4(cell, cell + 1, cell + 2, cell + 3);
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (cell + u < n_filled) ids[idx + u] = cell + u;
      }
    }
  } else {
    for (int idx = tid; idx < kb * B; idx += n_threads) {
      const int cell = sel[idx / B] * B + idx % B;
      if (cell < n_filled) ids[idx] = cell;
    }
  }
  if (tid == 0) {
    const int n_last = n_filled - (nb - 1) * B;
    p.n_sel[t] = kb * B - (sel[kb - 1] == nb - 1 ? (B - n_last) : 0);
  }
}

int topk_threads(int max_nb) {
  // one key per thread up to 1,024 blocks (the count is then one __syncthreads_count), else 1,024
  // threads with up to kMaxKeys keys each
  int th = (max_nb + 31) / 32 * 32;
  th = th < 128 ? 128 : (th > kMaxThreads ? kMaxThreads : th);
  return th;
}

}  // namespace

size_t topk_smem_bytes(int max_nb) { return sizeof(int) * (size_t)max_nb; }

cudaError_t launch_topk(const TopkParams& p, int max_nb, cudaStream_t stream) {
  const int th = topk_threads(max_nb);
  if ((max_nb + th - 1) / th > kMaxKeys) return cudaErrorInvalidValue;
  const size_t smem = topk_smem_bytes(max_nb);
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(topk_kernel), smem);
  if (e != cudaSuccess) return e;
  topk_kernel<<<p.n_rows, th, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace qsa
