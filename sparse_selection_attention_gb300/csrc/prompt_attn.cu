// Causal prompt attention on the tcgen05 tensor cores (qsa_prompt_attn).
//
// Method ("#1367 prompt attention: STRATA_PROMPT_ATTN_IMMA=1", What it does):
// both products run on the tensor cores directly on the stored K/V codes; the
// other operand (q, and p times the V scale) is split into exact parts whose
// partial sums are combined in fp32, and softmax is online over K/V tiles.
// On this GPU the 16-bit tensor path is the fast one, so the split is into two
// fp16 parts (hi + lo, 22 significant bits) instead of three 8-bit parts; int8
// and 4-bit codes are exact in fp16.
//
// One CTA = 128 rows x one KV head, row r = (query q0 + r / G, q head
// kvh*G + r % G): the G q heads of a KV head share every K/V tile.  Per
// 64-cell tile:
//   1. TMA bulk copies (prefetched one tile ahead) bring the tile's int8 K,
//      V codes and their scales into a staging buffer;
//   2. threads convert K to fp16 (K-major, 128-byte swizzle) and V to fp16
//      transposed (dims x cells, K-major for the second product);
//   3. S_g = (Qhi + Qlo) . Kcode over the 64 dims of K-scale group g,
//      accumulated in tensor memory (one fp32 column per cell);
//   4. thread r (row r): logit = (S_0 ks_0 + S_1 ks_1) / (f sqrt(D)),
//      causal mask, running max (rescaled lazily, only when it grows by more
//      than 2^8), p = 2^(y - m), W_g = p * vscale_g * 2^k (k a per-tile power
//      of two), W split into fp16 hi + lo;
//   5. P[:, group g] = (Whi_g + Wlo_g) . Vcode[:, group g], a fresh tensor-
//      memory accumulator per tile (8 MMA steps), folded into the running
//      output O (also in tensor memory) with fp32 FMAs on the CUDA cores:
//      O = O * factor + P, factor = the tile's change of running max and of
//      the V-scale power of two.  Keeping the long sum over thousands of
//      tiles out of the tensor-core accumulator keeps its rounding at fp32
//      round-to-nearest level.
// Waits are bounded: a wait that runs out sets the device error word, drains
// the CTA's copies and exits.
#include <cuda_fp16.h>

#include "kernels.h"
#include "tc.cuh"

namespace qsa {

__device__ int g_device_error = 0;

namespace {

constexpr int kThreads = 128;
constexpr int kM = 128;
constexpr int kTileN = 64;

// Shared memory map (offsets from a 1024-byte aligned base).
constexpr int kQhiOff = 0;          // 2 K-blocks x [128 rows][128 B]
constexpr int kQloOff = 32768;
constexpr int kKfOff = 65536;       // 2 K-blocks x [64 cells][128 B]
constexpr int kVfOff = 81920;       // [128 dims][64 cells x 2 B]
constexpr int kWOff = 98304;        // 2 slots x (hi [128][128 B] + lo [128][128 B])
constexpr int kWSlot = 32768;
constexpr int kStageOff = 163840;   // 2 stages
constexpr int kStK = 0, kStV = 8192, kStKs = 16384, kStVs = 16896, kStBytes = 17920;
constexpr int kVspOff = kStageOff + 2 * kStBytes;   // float [4][64]
constexpr int kBarOff = kVspOff + 1024;
constexpr int kSmemBytes = kBarOff + 128 + 1024;    // + alignment slack

constexpr uint32_t kTmemCols = 512;  // S: [0,128), tile P.V: [128,256), O: [256,384)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kDrainLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Four int8 codes (w) -> two fp16 pairs, exact: bias to unsigned, place the
// byte in the mantissa of 1024 (0x6400), subtract 1152.
__device__ __forceinline__ void s8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const __half2 bias = bits_h2(0x64806480u);  // 1152, 1152
  lo = h2_bits(__hsub2(bits_h2(__byte_perm(u, 0x64646464u, 0x4140)), bias));
  hi = h2_bits(__hsub2(bits_h2(__byte_perm(u, 0x64646464u, 0x4342)), bias));
}

// Two bytes (b0, b1) of an already-biased word -> fp16 pair 1024 + b, minus `bias`.
__device__ __forceinline__ uint32_t bytes_to_h2(uint32_t u, uint32_t sel, uint32_t bias) {
  return h2_bits(__hsub2(bits_h2(__byte_perm(u, 0x64646464u, sel)), bits_h2(bias)));
}

// x -> (hi, lo) fp16 with hi + lo = x to ~2^-22 relative.
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 back = __half22float2(h);
  hi = h2_bits(h);
  lo = h2_bits(__floats2half2_rn(a - back.x, b - back.y));
}

__device__ __forceinline__ int sw128(int row, int chunk) {
  return (row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4);
}

template <int N>
__device__ __forceinline__ uint4 pick(const uint4 (&v)[N], int j) {
  uint4 r = v[0];
#pragma unroll
  for (int i = 1; i < N; ++i)
    if (j == i) r = v[i];
  return r;
}

__device__ __forceinline__ void raise_device_error(int code) { atomicCAS(&g_device_error, 0, code); }

__global__ void __launch_bounds__(kThreads, 1) prompt_attn_kernel(const PromptParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = tc::smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = p.n_kv_heads;
  const int G = p.n_q_heads / Hkv;
  const int QPC = kM / G;
  const int kvh = blockIdx.y;
  const int q_begin = blockIdx.x * QPC;
  const int q_end = min(p.n_q, q_begin + QPC);
  const PoolDev& pool = p.pool;
  const int n_vg = pool.v_bits == 8 ? 2 : 4;
  const int vg_dims = kD / n_vg;
  const int v_row_bytes = pool.v_bits == 8 ? 128 : 64;

  const int r = tid;
  const int qi = q_begin + r / G;
  const bool row_valid = (r < QPC * G) && (qi < q_end);
  const int head = kvh * G + (r % G);
  const int pos = row_valid ? p.q_pos0 + qi : p.q_pos0;
  const int pos_first = p.q_pos0 + q_begin;
  const int pos_last = p.q_pos0 + q_end - 1;
  const int n_tiles = pos_last / kTileN + 1;

  const uint32_t bar_st0 = sbase + kBarOff, bar_mma = sbase + kBarOff + 16;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kBarOff + 32);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kBarOff + 40);
  volatile int* s_rho = reinterpret_cast<volatile int*>(smem + kBarOff + 44);
  volatile int* s_kref = reinterpret_cast<volatile int*>(smem + kBarOff + 48);
  float* vsp = reinterpret_cast<float*>(smem + kVspOff);

  if (tid == 0) {
    tc::mbar_init(bar_st0, 1);
    tc::mbar_init(bar_st0 + 8, 1);
    tc::mbar_init(bar_mma, 1);
    tc::mbar_fence_init();
    *s_abort = 0;
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(tmem_holder), kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_holder;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t tS = tmem + lane_base;
  const uint32_t tP = tmem + lane_base + 128;
  const uint32_t tO = tmem + lane_base + 256;

  // ---- Q: scale row by a power of two f (max |q f| in [64, 128)), split hi/lo.
  float lambda;
  {
    const float4* q4 = reinterpret_cast<const float4*>(p.q + ((size_t)qi * p.n_q_heads + head) * kD);
    float amax = 0.f;
    if (row_valid) {
      for (int k = 0; k < 32; ++k) {
        const float4 v = __ldg(q4 + k);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
      }
    }
    int e = 0;
    if (amax > 0.f) frexpf(amax, &e);
    const int fexp = amax > 0.f ? 7 - e : 0;
    for (int c = 0; c < 16; ++c) {
      float x[8];
      if (row_valid) {
        const float4 a = __ldg(q4 + 2 * c), b = __ldg(q4 + 2 * c + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = 0.f;
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) split2(ldexpf(x[2 * k], fexp), ldexpf(x[2 * k + 1], fexp), hi[k], lo[k]);
      const int off = (c >> 3) * 16384 + sw128(r, c & 7);
      *reinterpret_cast<uint4*>(smem + kQhiOff + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(smem + kQloOff + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    lambda = ldexpf(kLog2e * kInvSqrtD, -fexp);
  }
  tc::fence_proxy_async_smem();

  // Thread 0 owns the copy / MMA issue and tracks what is in flight.
  uint32_t st_par[2] = {0u, 0u};
  uint32_t mma_par = 0u;
  bool st_busy[2] = {false, false};
  bool mma_busy = false;
  auto issue_tile = [&](int tile, int stage) {
    const int cell0 = tile * kTileN;
    const int page = __ldg(pool.page_table + cell0 / pool.page_cells);
    const long long slot0 = ((long long)page * Hkv + kvh) * pool.page_cells + (cell0 % pool.page_cells);
    const uint32_t st = sbase + kStageOff + stage * kStBytes;
    const uint32_t vbytes = kTileN * v_row_bytes, vsbytes = kTileN * n_vg * 4;
    const uint32_t bar = bar_st0 + 8 * stage;
    tc::mbar_expect_tx(bar, 8192 + vbytes + 512 + vsbytes);
    tc::bulk_g2s(st + kStK, pool.k_codes + slot0 * kD, 8192, bar);
    tc::bulk_g2s(st + kStV, pool.v_codes + slot0 * v_row_bytes, vbytes, bar);
    tc::bulk_g2s(st + kStKs, pool.k_scales + slot0 * 2, 512, bar);
    tc::bulk_g2s(st + kStVs, pool.v_scales + slot0 * n_vg, vsbytes, bar);
    st_busy[stage] = true;
  };
  if (tid == 0) issue_tile(0, 0);
  __syncthreads();

  // Every thread waits; the CTA then agrees on whether any wait ran out.
  auto cta_wait = [&](uint32_t bar, uint32_t parity) -> bool {
    const bool ok = tc::mbar_wait(bar, parity, p.wait_limit_ns);
    if (!ok) *s_abort = 1;
    __syncthreads();
    const bool go = (*s_abort == 0);
    __syncthreads();
    return go;
  };

  float m_ref = -INFINITY, l_run = 0.f;
  int k_ref = 0;   // V-scale exponent (warp 0 keeps it; the CTA sees s_rho)
  bool aborted = false;
  const uint32_t idesc_s = tc::idesc_f16_f32(kM, kTileN);
  const uint32_t idesc_o = tc::idesc_f16_f32(kM, vg_dims);

  for (int i = 0; i < n_tiles; ++i) {
    const int stage = i & 1;
    const int cell0 = i * kTileN;
    if (tid == 0 && i + 1 < n_tiles) issue_tile(i + 1, stage ^ 1);
    if (!cta_wait(bar_st0 + 8 * stage, st_par[stage])) { aborted = true; break; }
    st_par[stage] ^= 1u;
    if (tid == 0) st_busy[stage] = false;
    const uint8_t* st = smem + kStageOff + stage * kStBytes;

    // ---- K codes -> fp16, K-major [cell][dim] in two 64-dim blocks.
    {
      const int c = tid >> 1, hf = tid & 1;
      const uint8_t* src = st + kStK + c * 128 + hf * 64;
      uint8_t* dst = smem + kKfOff + hf * 8192;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int i4 = (s + c) & 3;
        const uint4 v = *reinterpret_cast<const uint4*>(src + i4 * 16);
        uint32_t h[8];
        s8x4_to_h2x2(v.x, h[0], h[1]);
        s8x4_to_h2x2(v.y, h[2], h[3]);
        s8x4_to_h2x2(v.z, h[4], h[5]);
        s8x4_to_h2x2(v.w, h[6], h[7]);
        *reinterpret_cast<uint4*>(dst + sw128(c, 2 * i4)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(dst + sw128(c, 2 * i4 + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
      }
    }
    // ---- V codes -> fp16 transposed [dim][cell] (K-major for p.V).
    if (pool.v_bits == 8) {
      const int dq = tid & 31, co = tid >> 5;
#pragma unroll
      for (int oi = 0; oi < 2; ++oi) {
        const int oct = co + 4 * oi;
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          w[k] = *reinterpret_cast<const uint32_t*>(st + kStV + (8 * oct + k) * 128 + 4 * dq) ^ 0x80808080u;
        uint4 out[4];
        uint32_t a[4], b[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          a[kk] = __byte_perm(w[2 * kk], w[2 * kk + 1], 0x5140);  // dims 0,1 of cells 2kk, 2kk+1
          b[kk] = __byte_perm(w[2 * kk], w[2 * kk + 1], 0x7362);  // dims 2,3
        }
        out[0] = make_uint4(bytes_to_h2(a[0], 0x4140, 0x64806480u), bytes_to_h2(a[1], 0x4140, 0x64806480u),
                            bytes_to_h2(a[2], 0x4140, 0x64806480u), bytes_to_h2(a[3], 0x4140, 0x64806480u));
        out[1] = make_uint4(bytes_to_h2(a[0], 0x4342, 0x64806480u), bytes_to_h2(a[1], 0x4342, 0x64806480u),
                            bytes_to_h2(a[2], 0x4342, 0x64806480u), bytes_to_h2(a[3], 0x4342, 0x64806480u));
        out[2] = make_uint4(bytes_to_h2(b[0], 0x4140, 0x64806480u), bytes_to_h2(b[1], 0x4140, 0x64806480u),
                            bytes_to_h2(b[2], 0x4140, 0x64806480u), bytes_to_h2(b[3], 0x4140, 0x64806480u));
        out[3] = make_uint4(bytes_to_h2(b[0], 0x4342, 0x64806480u), bytes_to_h2(b[1], 0x4342, 0x64806480u),
                            bytes_to_h2(b[2], 0x4342, 0x64806480u), bytes_to_h2(b[3], 0x4342, 0x64806480u));
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const int j = (s + (dq >> 1)) & 3;
          const int d = 4 * dq + j;
          *reinterpret_cast<uint4*>(smem + kVfOff + sw128(d, oct)) = pick(out, j);
        }
      }
    } else {
      const int dq = tid & 15, oct = tid >> 4;
      uint32_t e[8], o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(st + kStV + (8 * oct + k) * 64 + 4 * dq);
        e[k] = w & 0x0F0F0F0Fu;          // even dims 8dq + 0,2,4,6 as nibble values
        o[k] = (w >> 4) & 0x0F0F0F0Fu;   // odd dims 8dq + 1,3,5,7
      }
      uint4 out[8];
#pragma unroll
      for (int par = 0; par < 2; ++par) {
        const uint32_t* src = par ? o : e;
        uint32_t a[4], b[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          a[kk] = __byte_perm(src[2 * kk], src[2 * kk + 1], 0x5140);
          b[kk] = __byte_perm(src[2 * kk], src[2 * kk + 1], 0x7362);
        }
        // byte j of the word -> dim 8dq + 2j + par; nibble n -> 1024 + n - 1032
        out[0 + par] = make_uint4(bytes_to_h2(a[0], 0x4140, 0x64086408u), bytes_to_h2(a[1], 0x4140, 0x64086408u),
                                  bytes_to_h2(a[2], 0x4140, 0x64086408u), bytes_to_h2(a[3], 0x4140, 0x64086408u));
        out[2 + par] = make_uint4(bytes_to_h2(a[0], 0x4342, 0x64086408u), bytes_to_h2(a[1], 0x4342, 0x64086408u),
                                  bytes_to_h2(a[2], 0x4342, 0x64086408u), bytes_to_h2(a[3], 0x4342, 0x64086408u));
        out[4 + par] = make_uint4(bytes_to_h2(b[0], 0x4140, 0x64086408u), bytes_to_h2(b[1], 0x4140, 0x64086408u),
                                  bytes_to_h2(b[2], 0x4140, 0x64086408u), bytes_to_h2(b[3], 0x4140, 0x64086408u));
        out[6 + par] = make_uint4(bytes_to_h2(b[0], 0x4342, 0x64086408u), bytes_to_h2(b[1], 0x4342, 0x64086408u),
                                  bytes_to_h2(b[2], 0x4342, 0x64086408u), bytes_to_h2(b[3], 0x4342, 0x64086408u));
      }
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int j = (s + dq) & 7;
        const int d = 8 * dq + j;
        *reinterpret_cast<uint4*>(smem + kVfOff + sw128(d, oct)) = pick(out, j);
      }
    }
    // ---- V scales of this tile times a power of two 2^k_ref (warp 0).
    if (warp == 0) {
      const float* vs = reinterpret_cast<const float*>(st + kStVs);
      float mx = 0.f;
      for (int idx = lane; idx < kTileN * n_vg; idx += 32)
        if (cell0 + idx / n_vg < pool.n_filled) mx = fmaxf(mx, fabsf(vs[idx]));
      mx = warp_max(mx);
      int e = 0;
      if (mx > 0.f) frexpf(mx, &e);
      const int k = mx > 0.f ? 4 - e : k_ref;   // max |vs| 2^k in [8, 16)
      int rho = 0;
      if (i == 0) k_ref = k;
      else if (k < k_ref) { rho = k - k_ref; k_ref = k; }
      for (int idx = lane; idx < kTileN * n_vg; idx += 32) {
        const int c = idx / n_vg, g = idx % n_vg;
        vsp[g * kTileN + c] = (cell0 + c < pool.n_filled) ? ldexpf(vs[idx], k_ref) : 0.f;
      }
      if (lane == 0) {
        *s_rho = rho;
        *s_kref = k_ref;
      }
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();

    // ---- S_g = (Qhi + Qlo) . K over 64-dim group g.
    if (tid == 0) {
      tc::fence_after_sync();
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const uint64_t ah = tc::sw128_desc(sbase + kQhiOff + g * 16384);
        const uint64_t al = tc::sw128_desc(sbase + kQloOff + g * 16384);
        const uint64_t bk = tc::sw128_desc(sbase + kKfOff + g * 8192);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          tc::mma_f16(tmem + g * kTileN, ah + 2 * kk, bk + 2 * kk, idesc_s, kk > 0);
          tc::mma_f16(tmem + g * kTileN, al + 2 * kk, bk + 2 * kk, idesc_s, 1);
        }
      }
      tc::mma_commit(bar_mma);
      mma_busy = true;
    }
    if (!cta_wait(bar_mma, mma_par)) { aborted = true; break; }
    mma_par ^= 1u;
    if (tid == 0) mma_busy = false;
    tc::fence_after_sync();

    // ---- softmax of row r over the tile.
    float X[kTileN];
    {
      const float2* ks = reinterpret_cast<const float2*>(st + kStKs);
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float s0[32], s1[32];
        tc::tmem_ld32(tS + 32 * h2, s0);
        tc::tmem_ld32(tS + kTileN + 32 * h2, s1);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float2 kk = ks[32 * h2 + j];
          X[32 * h2 + j] = fmaf(s1[j], kk.y, s0[j] * kk.x);
        }
      }
    }
    const bool full = (cell0 + kTileN - 1 <= pos_first);
    float ymax = -INFINITY;
#pragma unroll
    for (int c = 0; c < kTileN; ++c) {
      float y = X[c] * lambda;
      if (!full && cell0 + c > pos) y = -INFINITY;
      X[c] = y;
      ymax = fmaxf(ymax, y);
    }
    const float m_new = (ymax > m_ref + 8.0f) ? ymax : m_ref;
    const float alpha = (m_new == m_ref) ? 1.f : exp2f(m_ref - m_new);
    const int rho = *s_rho;
    const float factor = ldexpf(alpha, rho);
    m_ref = m_new;
    float psum = 0.f;
#pragma unroll
    for (int c = 0; c < kTileN; ++c) {
      const float pc = (X[c] == -INFINITY) ? 0.f : exp2f(X[c] - m_ref);
      X[c] = pc;
      psum += pc;
    }
    l_run = fmaf(l_run, alpha, psum);

    // ---- W_g = p * vscale_g * 2^k, fp16 hi/lo, then O += W . V per V group.
    bool pv_ok = true;
    for (int round = 0; round * 2 < n_vg; ++round) {
      if (round > 0) {
        if (!cta_wait(bar_mma, mma_par)) { pv_ok = false; break; }
        mma_par ^= 1u;
        if (tid == 0) mma_busy = false;
        tc::fence_after_sync();
      }
#pragma unroll
      for (int slot = 0; slot < 2; ++slot) {
        const float* vg = vsp + (round * 2 + slot) * kTileN;
        uint8_t* whi = smem + kWOff + slot * kWSlot;
        uint8_t* wlo = whi + 16384;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            split2(X[8 * ch + 2 * k] * vg[8 * ch + 2 * k], X[8 * ch + 2 * k + 1] * vg[8 * ch + 2 * k + 1], hi[k],
                   lo[k]);
          *reinterpret_cast<uint4*>(whi + sw128(r, ch)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(wlo + sw128(r, ch)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncthreads();
      if (tid == 0) {
        tc::fence_after_sync();
#pragma unroll
        for (int slot = 0; slot < 2; ++slot) {
          const int g = round * 2 + slot;
          const uint64_t ah = tc::sw128_desc(sbase + kWOff + slot * kWSlot);
          const uint64_t al = tc::sw128_desc(sbase + kWOff + slot * kWSlot + 16384);
          const uint64_t bv = tc::sw128_desc(sbase + kVfOff + g * vg_dims * 128);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            tc::mma_f16(tmem + 128 + g * vg_dims, ah + 2 * kk, bv + 2 * kk, idesc_o, kk > 0);
            tc::mma_f16(tmem + 128 + g * vg_dims, al + 2 * kk, bv + 2 * kk, idesc_o, 1);
          }
        }
        tc::mma_commit(bar_mma);
        mma_busy = true;
      }
    }
    if (!pv_ok) { aborted = true; break; }
    if (!cta_wait(bar_mma, mma_par)) { aborted = true; break; }
    mma_par ^= 1u;
    if (tid == 0) mma_busy = false;
    tc::fence_after_sync();
    // ---- O = O * factor + P (row r, 128 dims), fp32 round-to-nearest.
#pragma unroll
    for (int h4 = 0; h4 < 4; ++h4) {
      float pv[32], o[32];
      tc::tmem_ld32(tP + 32 * h4, pv);
      if (i > 0) tc::tmem_ld32(tO + 32 * h4, o);
      tc::tmem_wait_ld();
      if (i > 0) {
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = fmaf(o[j], factor, pv[j]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = pv[j];
      }
      tc::tmem_st32(tO + 32 * h4, o);
    }
    tc::tmem_wait_st();
    tc::fence_before_sync();
    tc::fence_proxy_async_smem();
  }

  if (aborted) {
    if (tid == 0) {
      raise_device_error(1);
      for (int s = 0; s < 2; ++s)
        if (st_busy[s]) tc::mbar_wait(bar_st0 + 8 * s, st_par[s], kDrainLimitNs);
      if (mma_busy) tc::mbar_wait(bar_mma, mma_par, kDrainLimitNs);
    }
    __syncthreads();
  } else {
    // ---- out = O 2^-k / l, lse = (m + log2 l) ln 2.
    const float scale = ldexpf(1.f / l_run, -*s_kref);
    float* orow = p.out + ((size_t)qi * p.n_q_heads + head) * kD;
#pragma unroll
    for (int h4 = 0; h4 < 4; ++h4) {
      float o[32];
      tc::tmem_ld32(tO + 32 * h4, o);
      tc::tmem_wait_ld();
      if (row_valid) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(orow + 32 * h4 + j) =
              make_float4(o[j] * scale, o[j + 1] * scale, o[j + 2] * scale, o[j + 3] * scale);
      }
    }
    if (row_valid && p.lse) p.lse[(size_t)qi * p.n_q_heads + head] = (m_ref + log2f(l_run)) * kLn2;
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

namespace ws {

// Warp-specialised prompt attention for int8 V (see the file comment for the
// arithmetic).  Roles of the 16 warps of a CTA:
//   warp 0      one thread issues the bulk copies of each 64-cell K/V tile into
//               a 3-stage ring of raw staging buffers;
//   warp 1      one thread issues every tcgen05.mma: S(i) = Q K(i)^T into one
//               of two tensor-memory S slots, then P += W(i-1) V(i-1) with W
//               read from tensor memory;
//   warps 4-7   convert raw tiles into fp16 operands (2-stage ring): K (K-major)
//               and V transposed, plus the per-cell scales and the tile's
//               V-scale power of two;
//   warps 8-15  softmax, two threads per row (32 cells each): logits, running
//               max (lazy, threshold 2^8), p, and W = p * vscale * 2^k split
//               into fp16 hi/lo, written back over S(i) in tensor memory.
// QK of tile i+1 overlaps the softmax of tile i and P.V of tile i-1.  P
// accumulates at most kFoldEvery tiles in tensor memory; it is then folded
// into O with fp32 FMAs (O = O * factor + P), and also whenever a row's
// running max or the V-scale exponent changes, so that P always holds tiles
// of one reference.  Every mbarrier wait is bounded; a wait that runs out
// sets the device error word and every role stops at its next wait.
constexpr int kThreads = 512;
constexpr int kM = 128;
constexpr int kN = 64;
constexpr int kRawStages = 3;
constexpr int kFoldEvery = 8;
constexpr int kQhi = 0, kQlo = 32768;                     // 2 K-blocks x [128 rows][128 B] each
constexpr int kOp0 = 65536, kOpBytes = 32768;             // per op stage: K [2][64][128 B], V^T [128][128 B]
constexpr int kOpK = 0, kOpV = 16384;
constexpr int kRaw0 = kOp0 + 2 * kOpBytes, kRawBytes = 17408;   // raw K 8 KB, V 8 KB, ks 512 B, vs 512 B
constexpr int kRK = 0, kRV = 8192, kRKs = 16384, kRVs = 16896;
constexpr int kAux0 = kRaw0 + kRawStages * kRawBytes, kAuxBytes = 1088;   // per op stage: ks, vsp, info
constexpr int kAuxKs = 0, kAuxVs = 512, kAuxInfo = 1024;
constexpr int kRed = kAux0 + 2 * kAuxBytes;               // tile maxima [2 halves][128], l [2][128]
constexpr int kCtl = kRed + 2048;                         // barriers and control words
constexpr int kSmemBytes = kCtl + 512 + 1024;             // + alignment slack

// Barrier indices.
constexpr int RAW_FULL = 0, RAW_EMPTY = 3, OP_FULL = 6, OP_EMPTY = 8, S_FULL = 10, S_EMPTY = 12, W_FULL = 14,
              PV_DONE = 16, N_BARS = 17;
// Control words (ints) after the barriers.
constexpr int C_ABORT = 0, C_TMEM = 1, C_PVACC = 2 /* [2] */, C_FOLD = 4 /* [2] */, C_GO_SM = 6 /* [2] */,
              C_GO_CV = 8 /* [2] */, C_GO_FD = 10 /* [2] */, C_GO_EP = 12, C_ISSUED = 13, C_LAST_BAR = 14,
              C_LAST_PAR = 15, N_CTL = 16;

struct Ctl {
  uint32_t bars;
  volatile int* w;
};

// Bounded wait that gives up at once once the CTA has aborted.
__device__ __forceinline__ bool wait_b(const Ctl& c, int bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t b = c.bars + 8 * bar;
  if (limit_ns == 0) {
    c.w[C_ABORT] = 1;
    raise_device_error(1);
    return false;
  }
  if (tc::mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = tc::globaltimer_ns();
  while (true) {
    if (tc::mbar_try_wait(b, parity)) return true;
    if (c.w[C_ABORT]) return false;
    if (tc::globaltimer_ns() - t0 > limit_ns) {
      c.w[C_ABORT] = 1;
      raise_device_error(1);
      return false;
    }
  }
}

// Acquire side of a phase that another thread of the role has already seen complete.
__device__ __forceinline__ void acquire(const Ctl& c, int bar, uint32_t parity) {
  tc::mbar_wait(c.bars + 8 * bar, parity, 2000000000ull);
}

__device__ __forceinline__ void arrive(const Ctl& c, int bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(c.bars + 8 * bar) : "memory");
}

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + max(-126, min(127, e))) << 23); }

__global__ void __launch_bounds__(kThreads, 1) prompt_attn_ws_kernel(const PromptParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = tc::smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = p.n_kv_heads;
  const int G = p.n_q_heads / Hkv;
  const int QPC = kM / G;
  const int kvh = blockIdx.y;
  const int q_begin = blockIdx.x * QPC;
  const int q_end = min(p.n_q, q_begin + QPC);
  const PoolDev& pool = p.pool;
  const int pos_first = p.q_pos0 + q_begin;
  const int pos_last = p.q_pos0 + q_end - 1;
  const int n_tiles = pos_last / kN + 1;
  const uint64_t limit = p.wait_limit_ns;

  Ctl c;
  c.bars = sbase + kCtl;
  c.w = reinterpret_cast<volatile int*>(smem + kCtl + 8 * N_BARS);
  float* red = reinterpret_cast<float*>(smem + kRed);

  if (tid == 0) {
    for (int s = 0; s < kRawStages; ++s) {
      tc::mbar_init(c.bars + 8 * (RAW_FULL + s), 1);
      tc::mbar_init(c.bars + 8 * (RAW_EMPTY + s), 4);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(c.bars + 8 * (OP_FULL + s), 4);
      tc::mbar_init(c.bars + 8 * (OP_EMPTY + s), 1);
      tc::mbar_init(c.bars + 8 * (S_FULL + s), 1);
      tc::mbar_init(c.bars + 8 * (S_EMPTY + s), 1);
      tc::mbar_init(c.bars + 8 * (W_FULL + s), 8);
    }
    tc::mbar_init(c.bars + 8 * PV_DONE, 1);
    tc::mbar_fence_init();
    for (int i = 0; i < N_CTL; ++i) c.w[i] = 0;
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(const_cast<int*>(c.w) + C_TMEM), 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = static_cast<uint32_t>(c.w[C_TMEM]);

  // ---- softmax threads: row r (lane quarter of the warp), half h (32 cells, 64 dims).
  const bool is_sm = warp >= 8;
  const int r = 32 * (warp & 3) + lane;
  const int half = (warp - 8) >> 2;
  const int qi = q_begin + r / G;
  const bool row_valid = (r < QPC * G) && (qi < q_end);
  const int head = kvh * G + (r % G);
  const int pos = row_valid ? p.q_pos0 + qi : p.q_pos0;
  float lambda = 0.f;
  if (is_sm) {
    // Q row scaled by a power of two (max |q 2^f| in [64, 128)), this half's 64 dims split hi/lo.
    const float4* q4 = reinterpret_cast<const float4*>(p.q + ((size_t)qi * p.n_q_heads + head) * kD);
    float amax = 0.f;
    if (row_valid) {
      for (int k = 0; k < 32; ++k) {
        const float4 v = __ldg(q4 + k);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
      }
    }
    int e = 0;
    if (amax > 0.f) frexpf(amax, &e);
    const int fexp = amax > 0.f ? max(-126, min(127, 7 - e)) : 0;
    const float f = pow2f(fexp);
    for (int cch = 0; cch < 8; ++cch) {
      float x[8];
      if (row_valid) {
        const float4 a = __ldg(q4 + 16 * half + 2 * cch), b = __ldg(q4 + 16 * half + 2 * cch + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = 0.f;
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) split2(x[2 * k] * f, x[2 * k + 1] * f, hi[k], lo[k]);
      const int off = half * 16384 + sw128(r, cch);
      *reinterpret_cast<uint4*>(smem + kQhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(smem + kQlo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    lambda = kLog2e * kInvSqrtD * pow2f(-fexp);
  }
  tc::fence_proxy_async_smem();
  __syncthreads();

  // =========================================================== producer
  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % kRawStages;
        if (i >= kRawStages && !wait_b(c, RAW_EMPTY + st, ((i / kRawStages) - 1) & 1, limit)) break;
        const int cell0 = i * kN;
        const int page = __ldg(pool.page_table + cell0 / pool.page_cells);
        const long long slot0 = ((long long)page * Hkv + kvh) * pool.page_cells + (cell0 % pool.page_cells);
        const uint32_t dst = sbase + kRaw0 + st * kRawBytes;
        const uint32_t bar = c.bars + 8 * (RAW_FULL + st);
        tc::mbar_expect_tx(bar, 8192 + 8192 + 512 + 512);
        tc::bulk_g2s(dst + kRK, pool.k_codes + slot0 * kD, 8192, bar);
        tc::bulk_g2s(dst + kRV, pool.v_codes + slot0 * kD, 8192, bar);
        tc::bulk_g2s(dst + kRKs, pool.k_scales + slot0 * 2, 512, bar);
        tc::bulk_g2s(dst + kRVs, pool.v_scales + slot0 * 2, 512, bar);
        issued = i + 1;
      }
      c.w[C_ISSUED] = issued;
    }
  }
  // =========================================================== MMA issuer
  else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc_s = tc::idesc_f16_f32(kM, kN);
      const uint32_t idesc_o = tc::idesc_f16_f32(kM, 64);
      int last_bar = -1;
      uint32_t last_par = 0;
      bool ok = true;
      for (int i = 0; i <= n_tiles && ok; ++i) {
        if (i < n_tiles) {
          const int sl = i & 1;
          ok = wait_b(c, OP_FULL + sl, (i >> 1) & 1, limit);
          if (ok && i >= 2) ok = wait_b(c, S_EMPTY + sl, ((i - 2) >> 1) & 1, limit);
          if (!ok) break;
          tc::fence_after_sync();
          const uint32_t kop = sbase + kOp0 + sl * kOpBytes + kOpK;
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const uint64_t ah = tc::sw128_desc(sbase + kQhi + g * 16384);
            const uint64_t al = tc::sw128_desc(sbase + kQlo + g * 16384);
            const uint64_t bk = tc::sw128_desc(kop + g * 8192);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              tc::mma_f16(tmem + sl * 128 + g * kN, ah + 2 * kk, bk + 2 * kk, idesc_s, kk > 0);
              tc::mma_f16(tmem + sl * 128 + g * kN, al + 2 * kk, bk + 2 * kk, idesc_s, 1);
            }
          }
          tc::mma_commit(c.bars + 8 * (S_FULL + sl));
          last_bar = S_FULL + sl;
          last_par = (i >> 1) & 1;
        }
        if (i >= 1) {
          const int j = i - 1, sj = j & 1;
          if (!wait_b(c, W_FULL + sj, (j >> 1) & 1, limit)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t acc = c.w[C_PVACC + sj];
          const uint32_t vop = sbase + kOp0 + sj * kOpBytes + kOpV;
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const uint64_t bv = tc::sw128_desc(vop + g * 64 * 128);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t aw = tmem + sj * 128 + (2 * g) * 32 + 8 * kk;
              tc::mma_f16_tmem_a(tmem + 256 + g * 64, aw, bv + 2 * kk, idesc_o, (kk > 0 || acc) ? 1u : 0u);
              tc::mma_f16_tmem_a(tmem + 256 + g * 64, aw + 32, bv + 2 * kk, idesc_o, 1u);
            }
          }
          tc::mma_commit(c.bars + 8 * (S_EMPTY + sj));
          tc::mma_commit(c.bars + 8 * (OP_EMPTY + sj));
          tc::mma_commit(c.bars + 8 * PV_DONE);
          last_bar = PV_DONE;
          last_par = j & 1;
        }
      }
      c.w[C_LAST_BAR] = last_bar;
      c.w[C_LAST_PAR] = (int)last_par;
    }
  }
  // =========================================================== converters
  else if (warp >= 4 && warp < 8) {
    const int ct = tid - 128;   // 0..127
    int k_ref = 0;              // V-scale exponent reference (identical in the 4 warps)
    for (int i = 0; i < n_tiles; ++i) {
      const int rs = i % kRawStages, os = i & 1;
      if (ct == 0) {
        bool ok = wait_b(c, RAW_FULL + rs, (i / kRawStages) & 1, limit);
        if (ok && i >= 2) ok = wait_b(c, OP_EMPTY + os, ((i - 2) >> 1) & 1, limit);
        c.w[C_GO_CV + (i & 1)] = ok && !c.w[C_ABORT];
      }
      tc::named_barrier(2, 128);
      if (!c.w[C_GO_CV + (i & 1)]) break;
      if (ct != 0) {
        acquire(c, RAW_FULL + rs, (i / kRawStages) & 1);
        if (i >= 2) acquire(c, OP_EMPTY + os, ((i - 2) >> 1) & 1);
      }
      const uint8_t* raw = smem + kRaw0 + rs * kRawBytes;
      uint8_t* op = smem + kOp0 + os * kOpBytes;
      uint8_t* aux = smem + kAux0 + os * kAuxBytes;
      const int cell0 = i * kN;
      // K codes -> fp16, K-major [cell][dim] in two 64-dim blocks.
      {
        const int cc = ct >> 1, hf = ct & 1;
        const uint8_t* src = raw + kRK + cc * 128 + hf * 64;
        uint8_t* dst = op + kOpK + hf * 8192;
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
          const int i4 = (s4 + cc) & 3;
          const uint4 v = *reinterpret_cast<const uint4*>(src + i4 * 16);
          uint32_t hh[8];
          s8x4_to_h2x2(v.x, hh[0], hh[1]);
          s8x4_to_h2x2(v.y, hh[2], hh[3]);
          s8x4_to_h2x2(v.z, hh[4], hh[5]);
          s8x4_to_h2x2(v.w, hh[6], hh[7]);
          *reinterpret_cast<uint4*>(dst + sw128(cc, 2 * i4)) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
          *reinterpret_cast<uint4*>(dst + sw128(cc, 2 * i4 + 1)) = make_uint4(hh[4], hh[5], hh[6], hh[7]);
        }
      }
      // V codes -> fp16 transposed [dim][cell].
      {
        const int dq = ct & 31, co = ct >> 5;
#pragma unroll
        for (int oi = 0; oi < 2; ++oi) {
          const int oct = co + 4 * oi;
          uint32_t w[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            w[k] = *reinterpret_cast<const uint32_t*>(raw + kRV + (8 * oct + k) * 128 + 4 * dq) ^ 0x80808080u;
          uint4 out[4];
          uint32_t a[4], b[4];
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            a[kk] = __byte_perm(w[2 * kk], w[2 * kk + 1], 0x5140);
            b[kk] = __byte_perm(w[2 * kk], w[2 * kk + 1], 0x7362);
          }
          out[0] = make_uint4(bytes_to_h2(a[0], 0x4140, 0x64806480u), bytes_to_h2(a[1], 0x4140, 0x64806480u),
                              bytes_to_h2(a[2], 0x4140, 0x64806480u), bytes_to_h2(a[3], 0x4140, 0x64806480u));
          out[1] = make_uint4(bytes_to_h2(a[0], 0x4342, 0x64806480u), bytes_to_h2(a[1], 0x4342, 0x64806480u),
                              bytes_to_h2(a[2], 0x4342, 0x64806480u), bytes_to_h2(a[3], 0x4342, 0x64806480u));
          out[2] = make_uint4(bytes_to_h2(b[0], 0x4140, 0x64806480u), bytes_to_h2(b[1], 0x4140, 0x64806480u),
                              bytes_to_h2(b[2], 0x4140, 0x64806480u), bytes_to_h2(b[3], 0x4140, 0x64806480u));
          out[3] = make_uint4(bytes_to_h2(b[0], 0x4342, 0x64806480u), bytes_to_h2(b[1], 0x4342, 0x64806480u),
                              bytes_to_h2(b[2], 0x4342, 0x64806480u), bytes_to_h2(b[3], 0x4342, 0x64806480u));
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4) {
            const int jj = (s4 + (dq >> 1)) & 3;
            const int d = 4 * dq + jj;
            *reinterpret_cast<uint4*>(op + kOpV + sw128(d, oct)) = pick(out, jj);
          }
        }
      }
      // K scales (as staged) and V scales times 2^k_ref; k_ref only decreases, tile by tile.
      {
        const float* ksr = reinterpret_cast<const float*>(raw + kRKs);
        const float* vsr = reinterpret_cast<const float*>(raw + kRVs);
        float* ksa = reinterpret_cast<float*>(aux + kAuxKs);
        float* vsa = reinterpret_cast<float*>(aux + kAuxVs);
        ksa[ct] = ksr[ct];   // 128 floats = [64 cells][2]
        float mx = 0.f;
        const bool v0 = cell0 + (ct >> 1) < pool.n_filled;
        if (v0) mx = fabsf(vsr[ct]);
        mx = warp_max(mx);
        // combine the 4 warps' maxima through the aux info words
        volatile float* cm = reinterpret_cast<volatile float*>(aux + kAuxInfo + 8);
        if (lane == 0) cm[ct >> 5] = mx;
        tc::named_barrier(2, 128);
        mx = fmaxf(fmaxf(cm[0], cm[1]), fmaxf(cm[2], cm[3]));
        int e = 0;
        if (mx > 0.f) frexpf(mx, &e);
        const int kt = mx > 0.f ? 4 - e : k_ref;   // max |vs| 2^k in [8, 16)
        int changed = 0;
        if (i == 0) k_ref = kt;
        else if (kt < k_ref) { k_ref = kt; changed = 1; }
        const float up = pow2f(k_ref);
        // vsa[g][cell] from vsr[cell][g]
        vsa[(ct & 1) * 64 + (ct >> 1)] = v0 ? vsr[ct] * up : 0.f;
        if (ct == 0) {
          reinterpret_cast<volatile int*>(aux + kAuxInfo)[0] = k_ref;
          reinterpret_cast<volatile int*>(aux + kAuxInfo)[1] = changed;
        }
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        arrive(c, RAW_EMPTY + rs);
        arrive(c, OP_FULL + os);
      }
    }
  }
  // =========================================================== softmax
  else if (is_sm) {
    const int st_id = tid - 256;   // 0..255
    float m_P = -INFINITY, m_O = -INFINITY, l = 0.f;
    int k_P = 0, k_O = 0;
    bool o_empty = true;
    bool alive = true;
    for (int i = 0; i < n_tiles && alive; ++i) {
      const int sl = i & 1;
      if (st_id == 0) {
        bool ok = wait_b(c, OP_FULL + sl, (i >> 1) & 1, limit);
        if (ok) ok = wait_b(c, S_FULL + sl, (i >> 1) & 1, limit);
        c.w[C_GO_SM + (i & 1)] = ok && !c.w[C_ABORT];
      }
      tc::named_barrier(1, 256);
      if (!c.w[C_GO_SM + (i & 1)]) { alive = false; break; }
      if (st_id != 0) {
        acquire(c, OP_FULL + sl, (i >> 1) & 1);
        acquire(c, S_FULL + sl, (i >> 1) & 1);
      }
      tc::fence_after_sync();
      const uint8_t* aux = smem + kAux0 + sl * kAuxBytes;
      const float2* ks = reinterpret_cast<const float2*>(aux + kAuxKs);
      const float* vsa = reinterpret_cast<const float*>(aux + kAuxVs);
      const int k_tile = reinterpret_cast<const volatile int*>(aux + kAuxInfo)[0];
      const int k_changed = reinterpret_cast<const volatile int*>(aux + kAuxInfo)[1];
      const int cell0 = i * kN;
      // logits (scaled by f) of this half's 32 cells
      float X[32];
      {
        const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + sl * 128 + 32 * half;
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          float s0[16], s1[16];
          tc::tmem_ld16(trow + 16 * q2, s0);
          tc::tmem_ld16(trow + kN + 16 * q2, s1);
          tc::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 kk = ks[32 * half + 16 * q2 + j];
            X[16 * q2 + j] = fmaf(s1[j], kk.y, s0[j] * kk.x);
          }
        }
      }
      const bool full = (cell0 + kN - 1 <= pos_first);
      float xmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (!full && cell0 + 32 * half + j > pos) X[j] = -INFINITY;
        xmax = fmaxf(xmax, X[j]);
      }
      // row maximum over both halves; fold decision for the CTA
      red[half * 128 + r] = xmax;
      if (st_id == 0) c.w[C_FOLD + ((i + 1) & 1)] = 0;
      tc::named_barrier(1, 256);
      xmax = fmaxf(xmax, red[(1 - half) * 128 + r]);
      const float ymax = xmax * lambda;   // lambda > 0
      const float m_new = (ymax > m_P + 8.0f) ? ymax : m_P;
      if (m_new != m_P || (st_id == 0 && (k_changed || (i > 0 && i % kFoldEvery == 0))))
        c.w[C_FOLD + (i & 1)] = 1;
      tc::named_barrier(1, 256);
      const bool fold = c.w[C_FOLD + (i & 1)] != 0 && i > 0;
      if (fold) {
        // P holds tiles since the last fold, referenced to (m_P, k_P): wait for P.V(i-1), then
        // O = O * 2^(m_O - m_P) * 2^(k_P - k_O) + P.
        if (st_id == 0) c.w[C_GO_FD + (i & 1)] = wait_b(c, PV_DONE, (i - 1) & 1, limit) && !c.w[C_ABORT];
        tc::named_barrier(1, 256);
        if (!c.w[C_GO_FD + (i & 1)]) { alive = false; break; }
        if (st_id != 0) acquire(c, PV_DONE, (i - 1) & 1);
        tc::fence_after_sync();
        const float fo = o_empty ? 0.f : exp2f(m_O - m_P) * pow2f(k_P - k_O);
        const uint32_t tp = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 256 + 64 * half;
#pragma unroll 1
        for (int h4 = 0; h4 < 4; ++h4) {
          float pv[16], o[16];
          tc::tmem_ld16(tp + 16 * h4, pv);
          if (!o_empty) tc::tmem_ld16(tp + 128 + 16 * h4, o);
          tc::tmem_wait_ld();
          if (o_empty) {
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] = pv[j];
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] = fmaf(o[j], fo, pv[j]);
          }
          tc::tmem_st16f(tp + 128 + 16 * h4, o);
        }
        tc::tmem_wait_st();
        o_empty = false;
        m_O = m_P;
        k_O = k_P;
      }
      // new references for the tiles from i on
      if (m_new != m_P) {
        if (m_P != -INFINITY) l *= exp2f(m_P - m_new);
        m_P = m_new;
      }
      k_P = k_tile;
      // p, this half's l, and W = p vscale 2^k as fp16 hi/lo, written over S(i)
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float pj = (X[j] == -INFINITY) ? 0.f : exp2f(fmaf(X[j], lambda, -m_P));
        X[j] = pj;
        psum += pj;
      }
      l += psum;
      const uint32_t tw = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + sl * 128;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int c0 = 32 * half + 2 * j;
          split2(X[2 * j] * vsa[g * 64 + c0], X[2 * j + 1] * vsa[g * 64 + c0 + 1], hi[j], lo[j]);
        }
        tc::tmem_st16(tw + (2 * g) * 32 + 16 * half, hi);
        tc::tmem_st16(tw + (2 * g + 1) * 32 + 16 * half, lo);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      // One thread takes every phase of PV_DONE in order (P.V(i-1) here, unless the fold took it),
      // so that each parity wait on it is unambiguous.  A wait that runs out raises the abort.
      if (st_id == 0 && i > 0 && !fold) wait_b(c, PV_DONE, (i - 1) & 1, limit);
      if (st_id == 0) c.w[C_PVACC + sl] = fold ? 0 : (i == 0 ? 0 : 1);
      __syncwarp();
      if (lane == 0) arrive(c, W_FULL + sl);
    }
    // ---- epilogue: last P.V, final fold, normalise, write.
    if (alive) {
      if (st_id == 0) c.w[C_GO_EP] = wait_b(c, PV_DONE, (n_tiles - 1) & 1, limit) && !c.w[C_ABORT];
      tc::named_barrier(1, 256);
      alive = c.w[C_GO_EP] != 0;
    }
    if (alive) {
      if (st_id != 0) acquire(c, PV_DONE, (n_tiles - 1) & 1);
      tc::fence_after_sync();
      red[1024 / 4 + half * 128 + r] = l;   // l area: [2][128] after the maxima
      tc::named_barrier(1, 256);
      const float lt = red[256 + r] + red[256 + 128 + r];
      const float fo = o_empty ? 0.f : exp2f(m_O - m_P) * pow2f(k_P - k_O);
      const float scale = pow2f(-k_P) / lt;
      const uint32_t tp = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 256 + 64 * half;
      float* orow = p.out + ((size_t)qi * p.n_q_heads + head) * kD + 64 * half;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float pv[32], o[32];
        tc::tmem_ld32(tp + 32 * h2, pv);
        tc::tmem_ld32(tp + 128 + 32 * h2, o);
        tc::tmem_wait_ld();
        if (row_valid) {
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = (o_empty ? pv[j + u] : fmaf(o[j + u], fo, pv[j + u])) * scale;
            *reinterpret_cast<float4*>(orow + 32 * h2 + j) = make_float4(v[0], v[1], v[2], v[3]);
          }
        }
      }
      if (row_valid && half == 0 && p.lse) p.lse[(size_t)qi * p.n_q_heads + head] = (m_P + log2f(lt)) * kLn2;
    }
  }

  // After an abort (seen here by every role), nothing may still write this CTA's shared or tensor
  // memory when it exits: wait for the latest fill of every raw stage and the last MMA commit.
  __syncthreads();
  if (c.w[C_ABORT] && lane == 0) {
    const int issued = c.w[C_ISSUED], last_bar = c.w[C_LAST_BAR];
    if (warp == 0) {
      for (int st = 0; st < kRawStages && st < issued; ++st) {
        const int last = st + kRawStages * ((issued - 1 - st) / kRawStages);
        tc::mbar_wait(c.bars + 8 * (RAW_FULL + st), (last / kRawStages) & 1, 2000000000ull);
      }
    } else if (warp == 1 && last_bar >= 0) {
      tc::mbar_wait(c.bars + 8 * last_bar, (uint32_t)c.w[C_LAST_PAR], 2000000000ull);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace ws

cudaError_t launch_prompt_attn(const PromptParams& p, cudaStream_t stream) {
  const int G = p.n_q_heads / p.n_kv_heads;
  const int qpc = kM / G;
  dim3 grid((p.n_q + qpc - 1) / qpc, p.n_kv_heads);
  if (p.pool.v_bits == 8) {
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(ws::prompt_attn_ws_kernel), (size_t)ws::kSmemBytes);
    if (e != cudaSuccess) return e;
    ws::prompt_attn_ws_kernel<<<grid, ws::kThreads, ws::kSmemBytes, stream>>>(p);
    return cudaGetLastError();
  }
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(prompt_attn_kernel), (size_t)kSmemBytes);
  if (e != cudaSuccess) return e;
  prompt_attn_kernel<<<grid, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t read_and_clear_device_error(int32_t* code, cudaStream_t stream) {
  static const int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(code, g_device_error, sizeof(int), 0, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace qsa
