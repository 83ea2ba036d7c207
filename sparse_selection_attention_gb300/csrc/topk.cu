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
// registers.  The threshold T (the kb-th largest key) is found one 8-bit digit
// at a time from the most significant byte in which the largest and the
// smallest key differ (the bytes above it are common to every key): for the
// keys that share the digits found so far, a 256-bin shared-memory histogram
// of the next digit is scanned from the top by one warp, which picks the digit
// where the running count reaches the number still needed.  Blocks with key > T
// are taken, then the lowest-id blocks with key == T.  Two CTA prefix sums in
// block-id order give each chosen block its rank j; every block but the row's
// last holds exactly B cells, so chosen block j fills ids[j*B ..], written
// coalesced by the whole CTA.
#include "kernels.h"
#include "mma_sync.cuh"

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

// Adds, for every key of this thread whose bits under `mask` equal `prefix`, one count to the
// bin of its digit (key >> shift) & 255; lanes with the same digit add once, together.
template <int KK>
__device__ __forceinline__ void add_digits(const uint32_t (&key)[KK], int b0, int nb, uint32_t mask, uint32_t prefix,
                                           int shift, unsigned* hist) {
#pragma unroll
  for (int i = 0; i < KK; ++i)
    if (b0 + i < nb && (key[i] & mask) == prefix) atomicAdd(hist + ((key[i] >> shift) & 255u), 1u);
}

// Warp 0: the largest digit d whose count of keys with digit >= d reaches `need`; returns (d, need
// minus the keys with digit > d) through s_out.  Lane l scans bins 8l .. 8l+7.
__device__ __forceinline__ void pick_digit(const unsigned* hist, int need, int* s_out) {
  const int lane = threadIdx.x & 31;
  unsigned c[8], own = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = hist[8 * lane + j];
    own += c[j];
  }
  unsigned incl = own;   // keys in bins of lanes >= this lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned n = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += n;
  }
  const unsigned above = incl - own;
  if (above < (unsigned)need && (unsigned)need <= incl) {   // exactly one lane
    unsigned cum = above;
    int d = 8 * lane;
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      if (cum + c[j] >= (unsigned)need) {
        d = 8 * lane + j;
        break;
      }
      cum += c[j];
    }
    s_out[0] = d;
    s_out[1] = need - (int)cum;
  }
}

// KK keys per thread: thread i holds blocks [i KK, (i + 1) KK).
template <int KK>
__global__ void __launch_bounds__(kMaxThreads) topk_kernel(const TopkParams p) {
  extern __shared__ int smem[];          // chosen list [kb]
  __shared__ int warp_tot[32];
  __shared__ unsigned hist[4][256];
  __shared__ int s_pick[2];
  __shared__ uint32_t s_mm[2][32];
  const int t = blockIdx.x, tid = threadIdx.x;
  for (int i = tid; i < 4 * 256; i += blockDim.x) (&hist[0][0])[i] = 0u;
  // Scores come from the preceding launch of the stream (a no-op without that dependency); the next
  // launch may start its CTAs now (they wait for this grid before reading ids).
  ms::pdl_trigger();
  ms::pdl_wait();
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
  const int b0 = tid * KK;
  const float* sc = p.scores + (size_t)t * p.max_blocks;
  uint32_t key[KK];
#pragma unroll
  for (int i = 0; i < KK; ++i) key[i] = (b0 + i < nb) ? score_key(__ldg(sc + b0 + i)) : 0u;

  const bool take_all = (kb == nb);
  uint32_t T = 0;
  int need = 0;
  if (!take_all) {
    // The leading bytes that the largest and the smallest key share are common to every key: the
    // passes start at the first byte where they differ.
    uint32_t mn = 0xFFFFFFFFu, mx = 0u;
#pragma unroll
    for (int i = 0; i < KK; ++i)
      if (b0 + i < nb) {
        mn = min(mn, key[i]);
        mx = max(mx, key[i]);
      }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    if ((tid & 31) == 0) {
      s_mm[0][tid >> 5] = mn;
      s_mm[1][tid >> 5] = mx;
    }
    __syncthreads();   // also: histograms zeroed
    {
      const int lane = tid & 31, n_warps = blockDim.x >> 5;
      mn = __reduce_min_sync(0xffffffffu, lane < n_warps ? s_mm[0][lane] : 0xFFFFFFFFu);
      mx = __reduce_max_sync(0xffffffffu, lane < n_warps ? s_mm[1][lane] : 0u);
    }
    const int first = (mn == mx) ? 4 : __clz(mn ^ mx) >> 3;   // leading bytes shared by every key
    uint32_t mask = first == 0 ? 0u : (first >= 4 ? 0xFFFFFFFFu : ~(0xFFFFFFFFu >> (8 * first)));
    T = mx & mask;
    need = kb;
    for (int pass = first; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      add_digits<KK>(key, b0, nb, mask, T, shift, hist[pass]);
      __syncthreads();
      if (tid < 32) pick_digit(hist[pass], need, s_pick);
      __syncthreads();
      T |= (uint32_t)s_pick[0] << shift;
      need = s_pick[1];
      mask |= 255u << shift;
      // s_pick is rewritten in the next pass only after its histogram barrier
    }
    // need = the keys equal to T that are taken (lowest block ids first)
  }

  int tot = 0;
  int eq = 0;
  if (!take_all) {
#pragma unroll
    for (int i = 0; i < KK; ++i) eq += (b0 + i < nb && key[i] == T);
  }
  int e = take_all ? 0 : cta_exclusive_scan(eq, warp_tot, tot);
  int chosen = 0;
  uint32_t chosen_bits = 0;
#pragma unroll
  for (int i = 0; i < KK; ++i) {
    if (b0 + i < nb) {
      bool c = take_all || key[i] > T;
      if (!take_all && key[i] == T) { c = e < need; ++e; }
      if (c) { ++chosen; chosen_bits |= 1u << i; }
    }
  }
  int j = cta_exclusive_scan(chosen, warp_tot, tot);
#pragma unroll
  for (int i = 0; i < KK; ++i)
    if (chosen_bits & (1u << i)) sel[j++] = b0 + i;
  __syncthreads();
  // ids[j*B + i] = sel[j]*B + i, four at a time when the row's ids start 16-byte aligned (ids aligned,
  // k_cells and B multiples of 4); cells past n_filled (the row's last block) are not written.
  if ((B & 3) == 0 && (p.k_cells & 3) == 0 && (reinterpret_cast<uintptr_t>(p.ids) & 15) == 0) {
    for (int i4 = tid; i4 < kb * B / 4; i4 += blockDim.x) {
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
    for (int idx = tid; idx < kb * B; idx += blockDim.x) {
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

cudaError_t launch_topk_ex(const TopkParams& p, int max_nb, cudaStream_t stream, bool pdl) {
  const int th = topk_threads(max_nb);
  const int need = (max_nb + th - 1) / th;
  if (need > kMaxKeys) return cudaErrorInvalidValue;
  const int kk = need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : need <= 8 ? 8 : 16;
  const size_t smem = topk_smem_bytes(max_nb);
  void (*kern)(TopkParams) = kk == 1 ? topk_kernel<1> : kk == 2 ? topk_kernel<2> : kk == 4 ? topk_kernel<4>
                                : kk == 8 ? topk_kernel<8> : topk_kernel<16>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_rows);
  cfg.blockDim = dim3(th);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_topk(const TopkParams& p, int max_nb, cudaStream_t stream) {
  return launch_topk_ex(p, max_nb, stream, false);
}

}  // namespace qsa
