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
// registers.  Four radix passes of 8 bits (most significant first) find the
// threshold key T.  A pass histograms the digit of the keys still matching
// the prefix into per-warp bins (shared atomics, aggregated over lanes with
// equal digits; integer counts do not depend on their order), then 256
// threads each sum one digit over the warps and scan the bins from the
// highest digit down to find the digit holding the k-th key.  Blocks with
// key > T are taken, then the lowest-id blocks with key == T.  Two CTA prefix
// sums in block-id order give each chosen block its rank j; every block but
// the row's last holds exactly B cells, so chosen block j fills ids[j*B ..],
// written coalesced by the whole CTA.
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

// Exclusive CTA-wide prefix sum of one int per thread; `tot` receives the total.
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
  int base = 0, total = 0;
  for (int w = 0; w < n_warps; ++w) {   // every thread reads the (few) warp totals
    const int x = warp_tot[w];
    base += (w < warp) ? x : 0;
    total += x;
  }
  __syncthreads();
  tot = total;
  return base + inc - v;
}

__global__ void __launch_bounds__(kMaxThreads) topk_kernel(const TopkParams p) {
  extern __shared__ int smem[];          // per-warp histograms [n_warps][256], then chosen list [kb]
  __shared__ int warp_tot[32];
  __shared__ int bin_tot[8];
  __shared__ int s_digit, s_gt;
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_threads = blockDim.x, n_warps = n_threads >> 5;
  const int B = p.block_cells;
  const int n_filled = p.n_filled[t];
  const int nb = (n_filled + B - 1) / B;
  const int kb = min(p.k_cells / B, nb);
  int32_t* ids = p.ids + (size_t)t * p.k_cells;
  if (kb == 0) {
    if (tid == 0) p.n_sel[t] = 0;
    return;
  }
  int* whist = smem;
  int* sel = smem + n_warps * 256;
  const int K = (nb + n_threads - 1) / n_threads;   // <= kMaxKeys
  const int b0 = tid * K;
  const float* sc = p.scores + (size_t)t * p.max_blocks;
  uint32_t key[kMaxKeys];
#pragma unroll
  for (int i = 0; i < kMaxKeys; ++i) key[i] = (i < K && b0 + i < nb) ? score_key(__ldg(sc + b0 + i)) : 0u;

  uint32_t T = 0;
  int need = 0;
  const bool take_all = (kb == nb);
  if (!take_all) {
    uint32_t prefix = 0, mask = 0;
    int rem = kb;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      int* wh = whist + warp * 256;
#pragma unroll
      for (int i = 0; i < 8; ++i) wh[lane * 8 + i] = 0;
      __syncwarp();
#pragma unroll
      for (int i = 0; i < kMaxKeys; ++i) {
        if (i < K) {   // uniform
          const bool live = b0 + i < nb && (key[i] & mask) == prefix;
          const int digit = live ? (int)((key[i] >> shift) & 0xFF) : -1;
          const unsigned peers = __match_any_sync(0xffffffffu, digit);
          if (live && (__ffs(peers) - 1) == lane) atomicAdd(&wh[digit], __popc(peers));
        }
      }
      __syncthreads();
      // Threads 0..255: digit d = 255 - tid; count over warps, then a descending scan.
      if (tid < 256) {
        const int d = 255 - tid;
        int c = 0;
        for (int w = 0; w < n_warps; ++w) c += whist[w * 256 + d];
        int inc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += n;
        }
        if (lane == 31) bin_tot[warp] = inc;
        __syncwarp();
        asm volatile("bar.sync 1, 256;" ::: "memory");
        int before = 0;
        for (int w = 0; w < warp; ++w) before += bin_tot[w];
        const int lo = before + inc - c, hi = before + inc;   // keys above d, and up to d
        if (lo < rem && rem <= hi) {
          s_digit = d;
          s_gt = lo;
        }
      }
      __syncthreads();
      rem -= s_gt;
      prefix |= (uint32_t)s_digit << shift;
      mask |= 0xFFu << shift;
      __syncthreads();
    }
    T = prefix;
    need = rem;   // keys equal to T to take, lowest ids first
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
  for (int idx = tid; idx < kb * B; idx += n_threads) {
    const int cell = sel[idx / B] * B + idx % B;
    if (cell < n_filled) ids[idx] = cell;
  }
  if (tid == 0) {
    const int n_last = n_filled - (nb - 1) * B;
    p.n_sel[t] = kb * B - (sel[kb - 1] == nb - 1 ? (B - n_last) : 0);
  }
}

int topk_threads(int max_nb) {
  // about four keys per thread, 256..1024 threads (256 threads scan the bins)
  int th = ((max_nb + 3) / 4 + 31) / 32 * 32;
  th = th < 256 ? 256 : (th > kMaxThreads ? kMaxThreads : th);
  return th;
}

}  // namespace

size_t topk_smem_bytes(int max_nb) {
  const int th = topk_threads(max_nb);
  return sizeof(int) * ((size_t)(th / 32) * 256 + (size_t)max_nb);
}

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
