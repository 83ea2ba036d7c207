// Block top-k selection (qsa_topk).
//
// Per row: the k_cells / B highest-scoring blocks, emitted as their filled
// cells in ascending cell id.  Scores become order-preserving uint32 keys
// (-0.0 -> +0.0, NaN -> 0, below -inf), so the selection is integer work and
// its ids are exact ("#2806 sycl: decode QSA selection and attention in
// fewer, shorter launches", Summary: the wide top-k's radix passes find each
// digit with a work-group scan; integers only, so the same ids).
//
// One CTA per row holds all of the row's keys in shared memory.  Four radix
// passes of 8 bits (most significant first) find the threshold key T: each
// pass histograms the digit of the keys still matching the prefix (integer
// shared atomics, aggregated per warp over lanes with equal digits, since
// scores of one row share their leading bits; the counts do not depend on
// their order) and one warp scans the 256 bins from the top to find the digit
// holding the k-th key.  Blocks
// with key > T are taken, then the lowest-id blocks with key == T.  Two
// CTA-wide prefix sums over blocks in id order give each chosen block its
// rank j and a slot in a shared list; every block but the row's last holds
// exactly B cells, so the CTA then writes the ids coalesced: chosen block j
// fills ids[j*B ..].
#include "kernels.h"

namespace qsa {

namespace {

constexpr int kMaxThreads = 1024;

__device__ __forceinline__ uint32_t score_key(float x) {
  if (x != x) return 0u;                 // NaN ranks below every number
  if (x == 0.0f) x = 0.0f;               // -0.0 == +0.0
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive CTA-wide prefix sum of one int per thread; also returns the total.
__device__ __forceinline__ int cta_exclusive_scan(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, n_warps = blockDim.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = lane < n_warps ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    warp_tot[lane] = wi - w;              // exclusive base of each warp
    if (lane == 31) warp_tot[32] = wi;    // grand total
  }
  __syncthreads();
  const int base = warp_tot[warp] + inc - v;
  total = warp_tot[32];
  __syncthreads();
  return base;
}

__global__ void __launch_bounds__(kMaxThreads) topk_kernel(const TopkParams p) {
  const int kThreads = blockDim.x;
  extern __shared__ uint32_t keys[];
  __shared__ int hist[256];
  __shared__ int warp_tot[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_rem;

  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  const int B = p.block_cells;
  const int n_filled = p.n_filled[t];
  const int nb = (n_filled + B - 1) / B;
  const int kb = min(p.k_cells / B, nb);
  int32_t* ids = p.ids + (size_t)t * p.k_cells;

  if (kb == 0) {
    if (tid == 0) p.n_sel[t] = 0;
    return;
  }
  const float* sc = p.scores + (size_t)t * p.max_blocks;
  for (int b = tid; b < nb; b += kThreads) keys[b] = score_key(__ldg(sc + b));
  __syncthreads();

  uint32_t T = 0;
  int need = 0;
  const bool take_all = (kb == nb);
  if (!take_all) {
    uint32_t prefix = 0, mask = 0;
    int rem = kb;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
      __syncthreads();
      for (int b0 = 0; b0 < nb; b0 += kThreads) {   // warp-uniform trip count
        const int b = b0 + tid;
        const uint32_t k = b < nb ? keys[b] : 0u;
        const bool live = b < nb && (k & mask) == prefix;
        const unsigned lm = __ballot_sync(0xffffffffu, live);
        const int digit = live ? (int)((k >> shift) & 0xFF) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, digit) & lm;
        if (live && (__ffs(peers) - 1) == (tid & 31)) atomicAdd(&hist[digit], __popc(peers));
      }
      __syncthreads();
      if (tid < 32) {
        // lane l owns bins 255-8l .. 248-8l (descending digit order)
        int cnt[8];
        int s = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) { cnt[i] = hist[255 - 8 * tid - i]; s += cnt[i]; }
        int inc = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(0xffffffffu, inc, o);
          if (tid >= o) inc += n;
        }
        const int before = inc - s;
        const unsigned hit = __ballot_sync(0xffffffffu, inc >= rem);
        const int first = __ffs(hit) - 1;   // rem <= total, so some lane hits
        if (tid == first) {
          int c = before;
          int digit = 0, gt = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (c + cnt[i] >= rem) { digit = 255 - 8 * tid - i; gt = c; break; }
            c += cnt[i];
          }
          s_rem = rem - gt;
          s_prefix = prefix | ((uint32_t)digit << shift);
        }
      }
      __syncthreads();
      prefix = s_prefix;
      rem = s_rem;
      mask |= 0xFFu << shift;
      __syncthreads();
    }
    T = prefix;
    need = rem;   // keys equal to T to take, lowest ids first
  }

  // Each thread owns a contiguous range of blocks, so ranks follow block ids.
  const int per = (nb + kThreads - 1) / kThreads;
  const int b0 = min(nb, tid * per), b1 = min(nb, b0 + per);
  int total;
  int eq_base = 0;
  if (!take_all) {
    int eq = 0;
    for (int b = b0; b < b1; ++b) eq += (keys[b] == T);
    eq_base = cta_exclusive_scan(eq, warp_tot, total);
  }
  int chosen = 0;
  {
    int e = eq_base;
    for (int b = b0; b < b1; ++b) {
      const uint32_t k = keys[b];
      bool c = take_all || k > T;
      if (!take_all && k == T) { c = e < need; ++e; }
      chosen += c;
    }
  }
  const int rank0 = cta_exclusive_scan(chosen, warp_tot, total);
  int* sel = reinterpret_cast<int*>(keys + nb);   // chosen block ids in ascending order
  {
    int e = eq_base, j = rank0;
    for (int b = b0; b < b1; ++b) {
      const uint32_t k = keys[b];
      bool c = take_all || k > T;
      if (!take_all && k == T) { c = e < need; ++e; }
      if (c) sel[j++] = b;
    }
  }
  __syncthreads();
  // Every block but the row's last holds B cells, so chosen block j fills ids[j*B ..].
  for (int idx = tid; idx < kb * B; idx += kThreads) {
    const int cell = sel[idx / B] * B + idx % B;
    if (cell < n_filled) ids[idx] = cell;
  }
  if (tid == 0) {
    const int n_last = n_filled - (nb - 1) * B;
    p.n_sel[t] = kb * B - (sel[kb - 1] == nb - 1 ? (B - n_last) : 0);
  }
}

}  // namespace

size_t topk_smem_bytes(int max_nb) { return 2 * sizeof(uint32_t) * (size_t)max_nb; }

cudaError_t launch_topk(const TopkParams& p, int max_nb, cudaStream_t stream) {
  const size_t smem = topk_smem_bytes(max_nb);
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(topk_kernel), (size_t)smem);
  if (e != cudaSuccess) return e;
  // About two keys per thread, 128..1024 threads.
  const int threads = min(kMaxThreads, max(128, ((max_nb + 1) / 2 + 31) / 32 * 32));
  topk_kernel<<<p.n_rows, threads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace qsa
