// Causal prompt attention on the tcgen05 tensor cores (qsa_prompt_attn).
//
// Method ("#1367 prompt attention: STRATA_PROMPT_ATTN_IMMA=1", What it does):
// both products run on the tensor cores with the stored codes as one operand
// and an exact split of the other; partial sums are combined in fp32, and the
// softmax is online over K/V tiles.  On this GPU the 16-bit tensor path is the
// fast one, so every operand is an fp16 hi + lo pair (22 significant bits):
// K' = kcode * kscale and V' = vcode * vscale (scaled per KV head by a power
// of two into fp16 range) are split once per tile into operand images, q and
// p inside the kernel; each product is issued as hi.hi + hi.lo + lo.hi.
// int8 and 4-bit codes (4-bit V; 4-bit K of the q4_0 layout) take the same
// path (the images hold K' and V').
#include <cuda_fp16.h>

#include <algorithm>

#include "kernels.h"
#include "tc.cuh"

namespace qsa {

__device__ int g_device_error = 0;

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// x -> (hi, lo) fp16 with hi + lo = x to ~2^-22 relative.
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 back = __half22float2(h);
  hi = h2_bits(h);
  lo = h2_bits(__floats2half2_rn(a - back.x, b - back.y));
}

__device__ __forceinline__ void raise_device_error(int code) { atomicCAS(&g_device_error, 0, code); }

}  // namespace

namespace ws {

// Warp-specialised prompt attention, in three launches (four when the units of a partly empty last
// round are cut into tile ranges).
//
// 1. prompt_vmax_kernel takes each KV head's largest |V scale| and |K scale| over the cells the
//    call reads (atomic max on their bits): exponents kv_h, kk_h with max |scale| 2^k in [8, 16).
// 2. prompt_stage_kernel converts each 64-cell tile of the context once per KV head into the
//    shared-memory image the tensor cores read: K' = kcode * kscale * 2^kk_h and V' = vcode *
//    vscale * 2^kv_h, each split into fp16 hi + lo (22 significant bits), in the stored
//    [cell][dim] order as two 64-dim blocks in the 128-byte swizzle (0 past n_filled).
// 3. prompt_attn_ws_kernel, one CTA per (128 rows, KV head), or per tile range of one, 8 warps:
//      warp 0      one thread copies each tile image (one bulk copy) into a 3-stage ring;
//      warp 1      issues every tcgen05.mma from one elected lane: S(i) = Q K'(i)^T as hi.hi +
//                  hi.lo + lo.hi (Q in tensor memory) into one of two S slots of tensor memory;
//                  then P += P'(i-1) V'(i-1) as hi.hi + hi.lo + lo.hi over all 128 output dims,
//                  with P' read from the S slot it was written over (V' the MN-major B operand);
//      warps 4-7   softmax, one thread per row (TMEM lane = row) over all 64 cells of a tile:
//                  logits, running max (lazy, past 2^8), P' = 2^(y - m + 5) split into fp16
//                  hi + lo, stored over S(i).  The scales live in K' and V', so the softmax reads
//                  one accumulator and does no per-group work.
//    S(i+1) overlaps the softmax of tile i and P.V of tile i-1.  P holds at most kFoldEvery tiles
//    in tensor memory: a warp folds its rows' P into the output O, also in tensor memory, with
//    fp32 FMAs (O = O * factor + P) and zeroes P when one of its rows changes its running max and
//    every kFoldEvery tiles (the tensor core's own accumulation over thousands of steps would not
//    round to nearest).  out = O 2^-(kv_h + 5) / l.  No thread barrier sits in the loop: every
//    hand-off is an mbarrier with a bounded wait.  A wait that runs out sets the device error
//    word; every role then stops at its next wait and the CTA drains its copies and MMAs before
//    it exits.  A tile range writes its rows unnormalised with (m, l) instead.
// 4. prompt_merge_kernel combines the ranges of each cut unit by log-sum-exp, in range order.
constexpr int kThreads = 256;
constexpr int kM = 128;
constexpr int kN = 64;
constexpr int kStages = 3;
constexpr int kFoldEvery = 8;
constexpr int kPShift = 5;   // P' = p 2^5 <= 2^13 (p <= 2^8 under the lazy running max)
// Tile image (global scratch and shared-memory stage alike): K' and V' in fp16 hi + lo, each two
// 64-dim blocks of [64 cells][128 B] in the 128-byte swizzle.
constexpr int kImgKhi = 0, kImgKlo = 16384, kImgVhi = 32768, kImgVlo = 49152, kImgBytes = 65536;
static_assert(kImgVlo - kImgVhi == kImgKlo - kImgKhi, "lo copies sit at one offset from their hi copies");
constexpr int kScratchHeader = 256;   // uint32 max |V scale| bits per KV head, then max |K scale| bits
constexpr int kMaxHeadsHeader = kScratchHeader / 8;
// Tensor memory columns (512 allocated).
constexpr uint32_t kTQ = 0;     // Q of dim group g: hi at 64g, lo at 64g + 32 (fp16 pairs)
constexpr uint32_t kTS = 128;   // S slot s at 128 + 64s (fp32 logits of 64 cells); P' hi at +0, lo at +32
constexpr uint32_t kTP = 256;   // P: output dim d at 256 + d (fp32)
constexpr uint32_t kTO = 384;   // O: output dim d at 384 + d (fp32)
// Shared memory map (offsets from a 1024-byte aligned base).
constexpr int kStage0 = 0;
constexpr int kCtl = kStage0 + kStages * kImgBytes;
constexpr int kSmemBytes = kCtl + 512 + 1024;           // + alignment slack

constexpr int FULL = 0, EMPTY = kStages, S_FULL = 2 * kStages, S_EMPTY = S_FULL + 2, W_FULL = S_EMPTY + 2,
              N_BARS = W_FULL + 2;
constexpr int C_ABORT = 0, C_TMEM = 1, C_ISSUED = 2, C_LAST_BAR = 3, C_LAST_PAR = 4, N_CTL = 5;

struct Ctl {
  uint32_t bars;
  volatile int* w;
};

// Bounded wait on a phase; gives up at once when the CTA has already aborted.
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

__device__ __forceinline__ void arrive(const Ctl& c, int bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(c.bars + 8 * bar) : "memory");
}

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + max(-126, min(127, e))) << 23); }

// Packed fp32 pairs (round to nearest, like the scalar operations).
__device__ __forceinline__ uint64_t pk(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 upk(uint64_t r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// 2^x (hardware approximation; 2^-inf = +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// (a, b) -> fp16 pairs hi, lo with hi + lo = (a, b) to ~2^-21 relative (|a|, |b| < 65504): hi keeps
// the top 11 significant bits (exact in fp16 down to 2^-14), lo = x - hi exactly in fp32, rounded.
__device__ __forceinline__ void split_pair(uint64_t ab, uint32_t& hi, uint32_t& lo) {
  const float2 v = upk(ab);
  const float ha = __uint_as_float(__float_as_uint(v.x) & 0xFFFFE000u);
  const float hb = __uint_as_float(__float_as_uint(v.y) & 0xFFFFE000u);
  const float2 rem = upk(ffma2(pk(ha, hb), pk(-1.f, -1.f), ab));
  hi = h2_bits(__floats2half2_rn(ha, hb));
  lo = h2_bits(__floats2half2_rn(rem.x, rem.y));
}

// One CTA per (64-cell tile, KV head), 64 threads (one per cell): the head's largest |V scale| and
// |K scale| (header words h and kMaxHeadsHeader + h).
__global__ void __launch_bounds__(64) prompt_vmax_kernel(const PoolDev pool, int n_kv_heads, uint8_t* scratch) {
  const int t = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  const int cell = t * kN + c;
  float mv = 0.f, mk = 0.f;
  if (cell < pool.n_filled) {
    const long long slot = cell_slot(pool, n_kv_heads, h, cell);
    if (pool.v_bits == 8) {
      const float2 vs = __ldg(reinterpret_cast<const float2*>(pool.v_scales) + slot);
      mv = fmaxf(fabsf(vs.x), fabsf(vs.y));
    } else {
      const float4 vs = __ldg(reinterpret_cast<const float4*>(pool.v_scales) + slot);
      mv = fmaxf(fmaxf(fabsf(vs.x), fabsf(vs.y)), fmaxf(fabsf(vs.z), fabsf(vs.w)));
    }
    if (pool.k_bits == 8) {
      const float2 ks = __ldg(reinterpret_cast<const float2*>(pool.k_scales) + slot);
      mk = fmaxf(fabsf(ks.x), fabsf(ks.y));
    } else {
      const float4 ks = __ldg(reinterpret_cast<const float4*>(pool.k_scales) + slot);
      mk = fmaxf(fmaxf(fabsf(ks.x), fabsf(ks.y)), fmaxf(fabsf(ks.z), fabsf(ks.w)));
    }
  }
  mv = warp_max(mv);
  mk = warp_max(mk);
  if ((c & 31) == 0) {
    atomicMax(reinterpret_cast<unsigned int*>(scratch) + h, __float_as_uint(mv));
    atomicMax(reinterpret_cast<unsigned int*>(scratch) + kMaxHeadsHeader + h, __float_as_uint(mk));
  }
}

// Exponent k with max |scale| 2^k in [8, 16) for header word w (0 when every scale is 0).
__device__ __forceinline__ int head_scale_exp(const uint8_t* scratch, int w) {
  const float vmax = __uint_as_float(reinterpret_cast<const unsigned int*>(scratch)[w]);
  int e = 0;
  if (vmax > 0.f) frexpf(vmax, &e);
  return vmax > 0.f ? max(-126, min(127, 4 - e)) : 0;
}

// One CTA per (64-cell tile, KV head), 256 threads.  The image is four 8 KB blocks (K dims 0-63,
// K dims 64-127, V dims 0-63, V dims 64-127), each with a hi and a lo copy; a thread makes one
// 16-byte chunk of a block (8 dims of one cell) per step, chunks in image order, so a warp reads
// four cells' rows and writes 512 contiguous bytes of each copy.  Physical chunk p of row r holds
// the dims of logical chunk p ^ (r & 7) (the 128-byte swizzle).
__global__ void __launch_bounds__(256) prompt_stage_kernel(const PoolDev pool, int n_kv_heads, int n_tiles,
                                                           uint8_t* scratch) {
  const int t = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  uint8_t* img = scratch + kScratchHeader + ((size_t)h * n_tiles + t) * kImgBytes;
  const int cell0 = t * kN;
  const int page = __ldg(pool.page_table + cell0 / pool.page_cells);
  const long long slot0 = ((long long)page * n_kv_heads + h) * pool.page_cells + (cell0 % pool.page_cells);
  const float ksh = pow2f(head_scale_exp(scratch, kMaxHeadsHeader + h));   // K' = kcode kscale 2^kk_h
  const float vsh = pow2f(head_scale_exp(scratch, h));                     // V' = vcode vscale 2^kv_h
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int blk = j >> 1, hf = blk & 1;
    const int o16 = (j & 1) * 256 + tid;   // chunk of the 8 KB block, in memory order
    const int row = o16 >> 3, lc = (o16 & 7) ^ (row & 7);
    const int d0 = 64 * hf + 8 * lc;       // first of the chunk's 8 dims
    const bool valid = cell0 + row < pool.n_filled;
    const long long slot = slot0 + row;
    float x[8];
    if ((blk < 2 ? pool.k_bits : pool.v_bits) == 8) {   // int8 codes, one scale per 64 dims
      const int8_t* codes = blk < 2 ? pool.k_codes : reinterpret_cast<const int8_t*>(pool.v_codes);
      const float* scales = blk < 2 ? pool.k_scales : pool.v_scales;
      const uint2 w = valid ? __ldg(reinterpret_cast<const uint2*>(codes + slot * kD + d0)) : make_uint2(0u, 0u);
      const float sc = valid ? __ldg(scales + slot * 2 + hf) * (blk < 2 ? ksh : vsh) : 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = (float)(int8_t)((((k < 4) ? w.x : w.y) >> (8 * (k & 3))) & 0xFFu) * sc;
    } else {   // 4-bit codes (V, or K of the q4_0 layout): byte j = dims 2j (low nibble), 2j + 1; one scale per 32 dims
      const uint8_t* codes = blk < 2 ? reinterpret_cast<const uint8_t*>(pool.k_codes) : pool.v_codes;
      const float* scales = blk < 2 ? pool.k_scales : pool.v_scales;
      const uint32_t w = valid ? __ldg(reinterpret_cast<const uint32_t*>(codes + slot * (kD / 2) + d0 / 2)) : 0u;
      const float sc = valid ? __ldg(scales + slot * 4 + d0 / 32) * (blk < 2 ? ksh : vsh) : 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t b = (w >> (8 * k)) & 0xFFu;
        x[2 * k] = (float)((int)(b & 15u) - 8) * sc;
        x[2 * k + 1] = (float)((int)(b >> 4) - 8) * sc;
      }
    }
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) split2(x[2 * k], x[2 * k + 1], hi[k], lo[k]);
    uint8_t* dst = img + (blk < 2 ? kImgKhi : kImgVhi) + hf * 8192 + o16 * 16;
    *reinterpret_cast<uint4*>(dst) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(dst + (kImgKlo - kImgKhi)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

__global__ void __launch_bounds__(kThreads, 1) prompt_attn_ws_kernel(const PromptParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = tc::smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.n_q_heads / p.n_kv_heads;
  const int QPC = p.qpc;
  // This CTA's work: unit u (query block, KV head) over tiles [t0, t0 + n_tiles); part >= 0 for a
  // unit split across n_split CTAs (part-major order, so concurrent CTAs walk the same tiles).
  int u = blockIdx.x, part = -1;
  if (u >= p.n_whole) {
    const int n_tail = p.n_qb * p.n_kv_heads - p.n_whole;
    part = u - p.n_whole;
    u = p.n_whole + part % n_tail;
  }
  const int kvh = u / p.n_qb;
  const int q_begin = (u % p.n_qb) * QPC;
  const int q_end = min(p.n_q, q_begin + QPC);
  const int pos_first = p.q_pos0 + q_begin;
  const int pos_last = p.q_pos0 + q_end - 1;
  const int unit_tiles = pos_last / kN + 1;
  int t0 = 0, n_tiles = unit_tiles;
  if (part >= 0) {
    const int k = part / (p.n_qb * p.n_kv_heads - p.n_whole);
    t0 = (int)((long long)k * unit_tiles / p.n_split);
    n_tiles = (int)((long long)(k + 1) * unit_tiles / p.n_split) - t0;
  }
  const uint64_t limit = p.wait_limit_ns;

  // The part merge (launched after this grid) may be scheduled once every CTA has started; it
  // waits for this grid to complete before it reads anything.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  Ctl c;
  c.bars = sbase + kCtl;
  c.w = reinterpret_cast<volatile int*>(smem + kCtl + 8 * N_BARS);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(c.bars + 8 * (FULL + s), 1);
      tc::mbar_init(c.bars + 8 * (EMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(c.bars + 8 * (S_FULL + s), 1);
      tc::mbar_init(c.bars + 8 * (S_EMPTY + s), 1);
      tc::mbar_init(c.bars + 8 * (W_FULL + s), 4);
    }
    tc::mbar_fence_init();
    for (int i = 0; i < N_CTL; ++i) c.w[i] = 0;
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(const_cast<int*>(c.w) + C_TMEM), 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  // Softmax threads: row r of the CTA = TMEM lane r.
  const bool is_sm = warp >= 4;
  const int quarter = warp & 3;
  const int r = 32 * quarter + lane;
  const int qi = q_begin + r / G;
  const bool row_valid = is_sm && (r < QPC * G) && (qi < q_end);
  const int head = kvh * G + (r % G);
  const int pos = row_valid ? p.q_pos0 + qi : p.q_pos0;
  float lambda = 0.f;
  if (is_sm) {
    // Q row scaled by a power of two f (max |q f| in [64, 128)), split into fp16 hi + lo and stored
    // in tensor memory as the A operand (element pairs packed two per column).
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
    const uint32_t tq = static_cast<uint32_t>(c.w[C_TMEM]) + ((uint32_t)(32 * quarter) << 16);
#pragma unroll
    for (int part = 0; part < 4; ++part) {   // dims 32 part .. + 31
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row_valid) v = __ldg(q4 + 8 * part + k);
        split2(v.x * f, v.y * f, hi[2 * k], lo[2 * k]);
        split2(v.z * f, v.w * f, hi[2 * k + 1], lo[2 * k + 1]);
      }
      const uint32_t col = kTQ + 64 * (part >> 1) + 16 * (part & 1);
      tc::tmem_st16(tq + col, hi);
      tc::tmem_st16(tq + col + 32, lo);
    }
    tc::tmem_wait_st();
    lambda = kLog2e * kInvSqrtD * pow2f(-fexp);
  }
  tc::fence_before_sync();
  __syncthreads();   // Q is in tensor memory
  tc::fence_after_sync();
  const uint32_t tmem = static_cast<uint32_t>(c.w[C_TMEM]);

  if (warp < 4) {
  // =========================================================== producer
    if (warp == 0) {
      if (lane == 0) {
        const uint8_t* img0 = p.scratch + kScratchHeader + ((size_t)kvh * p.n_tiles + t0) * kImgBytes;
        int issued = 0;
        for (int i = 0; i < n_tiles; ++i) {
          const int st = i % kStages;
          if (i >= kStages && !wait_b(c, EMPTY + st, ((i / kStages) - 1) & 1, limit)) break;
          const uint32_t bar = c.bars + 8 * (FULL + st);
          tc::mbar_expect_tx(bar, kImgBytes);
          tc::bulk_g2s(sbase + kStage0 + st * kImgBytes, img0 + (size_t)i * kImgBytes, kImgBytes, bar);
          issued = i + 1;
        }
        c.w[C_ISSUED] = issued;
      }
    }
  // =========================================================== MMA issuer
    // The whole warp runs the loop and waits; one elected lane issues.
    else if (warp == 1) {
      const uint32_t idesc_s = tc::idesc_f16_f32(kM, kN);
      const uint32_t idesc_v = tc::idesc_f16_f32_bmn(kM, 128);
      const uint32_t d_hi = tc::sw128_desc_hi();
      const uint32_t vhi_lo0 = tc::sw128_desc_lo(sbase + kStage0 + kImgVhi, 8192);
      const uint32_t khi_lo0 = tc::sw128_desc_lo(sbase + kStage0 + kImgKhi, 16);
      const uint32_t klo_lo0 = tc::sw128_desc_lo(sbase + kStage0 + kImgKlo, 16);
      const uint32_t vlo_lo0 = tc::sw128_desc_lo(sbase + kStage0 + kImgVlo, 8192);
      int last_bar = -1;
      uint32_t last_par = 0;
      for (int i = 0; i <= n_tiles; ++i) {
        if (i < n_tiles) {
          const int sl = i & 1, st = i % kStages;
          bool ok = wait_b(c, FULL + st, (i / kStages) & 1, limit);
          if (ok && i >= 2) ok = wait_b(c, S_EMPTY + sl, ((i - 2) >> 1) & 1, limit);
          if (!__all_sync(0xffffffffu, ok)) break;
          tc::fence_after_sync();
          if (tc::elect_one()) {
            const uint32_t d = tmem + kTS + 64 * sl;
            const uint32_t so = (uint32_t)(st * (kImgBytes >> 4));
#pragma unroll
            for (int g = 0; g < 2; ++g) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint32_t bh = khi_lo0 + so + (uint32_t)((g * 8192 + kk * 32) >> 4);
                const uint32_t bl = klo_lo0 + so + (uint32_t)((g * 8192 + kk * 32) >> 4);
                const uint32_t ah = tmem + kTQ + 64 * g + 8 * kk, al = ah + 32;
                tc::mma_f16_tmem_a_w(d, ah, bh, d_hi, idesc_s, (g > 0 || kk > 0) ? 1u : 0u);
                tc::mma_f16_tmem_a_w(d, ah, bl, d_hi, idesc_s, 1u);
                tc::mma_f16_tmem_a_w(d, al, bh, d_hi, idesc_s, 1u);
              }
            }
            tc::mma_commit(c.bars + 8 * (S_FULL + sl));
          }
          __syncwarp();
          last_bar = S_FULL + sl;
          last_par = (i >> 1) & 1;
        }
        if (i >= 1) {
          const int j = i - 1, sj = j & 1, sv = j % kStages;
          if (!__all_sync(0xffffffffu, wait_b(c, W_FULL + sj, (j >> 1) & 1, limit))) break;
          tc::fence_after_sync();
          if (tc::elect_one()) {
            const uint32_t so = (uint32_t)(sv * (kImgBytes >> 4));
            const uint32_t aw = tmem + kTS + 64 * sj;
            const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t bh = vhi_lo0 + so + (uint32_t)((kk * 2048) >> 4);
              const uint32_t bl = vlo_lo0 + so + (uint32_t)((kk * 2048) >> 4);
              tc::mma_f16_tmem_a_w(tmem + kTP, aw + 8 * kk, bh, d_hi, idesc_v, kk > 0 ? 1u : acc0);
              tc::mma_f16_tmem_a_w(tmem + kTP, aw + 8 * kk, bl, d_hi, idesc_v, 1u);
              tc::mma_f16_tmem_a_w(tmem + kTP, aw + 32 + 8 * kk, bh, d_hi, idesc_v, 1u);
            }
            tc::mma_commit(c.bars + 8 * (S_EMPTY + sj));
            tc::mma_commit(c.bars + 8 * (EMPTY + sv));
          }
          __syncwarp();
          last_bar = EMPTY + sv;
          last_par = (j / kStages) & 1;
        }
      }
      if (lane == 0) {
        c.w[C_LAST_BAR] = last_bar;
        c.w[C_LAST_PAR] = (int)last_par;
      }
    }
    // After an abort (seen by every role at the first barrier), nothing may still write this
    // CTA's shared or tensor memory when it exits: wait for the latest fill of every stage and the
    // last MMA commit.  (The softmax warpgroup meets these two barriers at the end of its branch.)
    __syncthreads();
    if (c.w[C_ABORT] && lane == 0) {
      const int issued = c.w[C_ISSUED], last_bar = c.w[C_LAST_BAR];
      if (warp == 0) {
        for (int st = 0; st < kStages && st < issued; ++st) {
          const int last = st + kStages * ((issued - 1 - st) / kStages);
          tc::mbar_wait(c.bars + 8 * (FULL + st), (last / kStages) & 1, 2000000000ull);
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
    return;
  }

  // =========================================================== softmax (warps 4-7)
  {
    const uint32_t tl = tmem + ((uint32_t)(32 * quarter) << 16);
    // K' carries 2^kk_h (folded into lambda), V' 2^kv_h and P' 2^kPShift: out = O 2^-(kv_h + kPShift) / l.
    lambda *= pow2f(-head_scale_exp(p.scratch, kMaxHeadsHeader + kvh));
    const float out_scale = pow2f(-(head_scale_exp(p.scratch, kvh) + kPShift));
    float m_P = -INFINITY, m_O = -INFINITY, l = 0.f;
    bool o_empty = true, alive = true;
    const float zero16[16] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < n_tiles; ++i) {
      const int sl = i & 1, st = i % kStages;
      bool ok = wait_b(c, FULL + st, (i / kStages) & 1, limit);
      if (ok) ok = wait_b(c, S_FULL + sl, (i >> 1) & 1, limit);
      if (!__all_sync(0xffffffffu, ok && !c.w[C_ABORT])) { alive = false; break; }
      tc::fence_after_sync();
      const int cell0 = (t0 + i) * kN;
      const uint32_t ts = tl + kTS + 64 * sl;
      // ---- logits of the tile's 64 cells (scaled by lambda below)
      float X[64];
      tc::tmem_ld64(ts, X);
      tc::tmem_wait_ld();
      if (cell0 + kN - 1 > pos_first) {   // tile reaches past some row's position: causal mask
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (cell0 + j > pos) X[j] = -INFINITY;
      }
      // row maximum by a tree (independent pairs)
      float mx[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) mx[j] = fmaxf(X[2 * j], X[2 * j + 1]);
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) mx[j] = fmaxf(mx[j], mx[j + w]);
      const float xmax = mx[0];
      const float ymax = xmax * lambda;   // lambda > 0
      const float m_new = (ymax > m_P + 8.0f) ? ymax : m_P;
      const bool fold = __any_sync(0xffffffffu, i > 0 && (m_new != m_P || i % kFoldEvery == 0));
      if (fold) {
        // P holds this warp's rows since their last fold, referenced to m_P; after P.V(i-1):
        // O = O 2^(m_O - m_P) + P, then P = 0.  (A wait that runs out only raises the abort: the
        // warp stops at its next wait.)
        wait_b(c, S_EMPTY + ((i - 1) & 1), ((i - 1) >> 1) & 1, limit);
        tc::fence_after_sync();
        const float fo = (o_empty || m_O == -INFINITY) ? 0.f : ex2(m_O - m_P);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          float pv[16], ov[16];
          tc::tmem_ld16(tl + kTP + 16 * c4, pv);
          if (!o_empty) tc::tmem_ld16(tl + kTO + 16 * c4, ov);   // O holds nothing before the first fold
          tc::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) ov[j] = o_empty ? pv[j] : fmaf(ov[j], fo, pv[j]);
          tc::tmem_st16f(tl + kTO + 16 * c4, ov);
          tc::tmem_st16f(tl + kTP + 16 * c4, zero16);
        }
        o_empty = false;
        m_O = m_P;
      }
      if (m_new != m_P) {
        if (m_P != -INFINITY) l *= ex2(m_P - m_new);
        m_P = m_new;
      }
      // ---- P' = 2^(X lambda - m + kPShift) in fp16 hi + lo over S(i) (hi at +0, lo at +32), and the
      // row sum of p = P' 2^-kPShift
      {
        const uint64_t lam2 = pk(lambda, lambda);
        const float nm = m_P == -INFINITY ? 0.f : (float)kPShift - m_P;   // every X is -inf then
        const uint64_t nm2 = pk(nm, nm);
        uint64_t ps[4] = {0ull, 0ull, 0ull, 0ull};   // packed partial sums, four independent chains
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int j2 = 0; j2 < 16; ++j2) {
            const int j = 32 * h2 + 2 * j2;
            const float2 y = upk(ffma2(pk(X[j], X[j + 1]), lam2, nm2));
            const uint64_t e = pk(ex2(y.x), ex2(y.y));
            ps[j2 & 3] = fadd2(ps[j2 & 3], e);
            split_pair(e, hi[j2], lo[j2]);
          }
          tc::tmem_st16(ts + 16 * h2, hi);
          tc::tmem_st16(ts + 32 + 16 * h2, lo);
        }
        const float2 sa = upk(fadd2(fadd2(ps[0], ps[1]), fadd2(ps[2], ps[3])));
        l += (sa.x + sa.y) * (1.f / (float)(1 << kPShift));
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) arrive(c, W_FULL + sl);
    }
    // ---- epilogue: after the last P.V, out = (O 2^(m_O - m) + P) / l, lse = (m + log2 l) ln 2;
    // a part writes (O 2^(m_O - m) + P) unnormalised with (m, l) for prompt_merge_kernel.
    if (alive) {
      wait_b(c, S_EMPTY + ((n_tiles - 1) & 1), ((n_tiles - 1) >> 1) & 1, limit);
      tc::fence_after_sync();
      const float fo = (o_empty || m_O == -INFINITY) ? 0.f : ex2(m_O - m_P);
      const float scale = part >= 0 ? out_scale : out_scale / l;
      float* orow = part >= 0 ? p.part_o + ((size_t)part * kM + r) * kD
                              : p.out + ((size_t)qi * p.n_q_heads + head) * kD;
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        float pv[16], ov[16];
        tc::tmem_ld16(tl + kTP + 16 * c4, pv);
        if (!o_empty) tc::tmem_ld16(tl + kTO + 16 * c4, ov);
        tc::tmem_wait_ld();
        if (row_valid) {
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = (o_empty ? pv[j + u] : fmaf(ov[j + u], fo, pv[j + u])) * scale;
            *reinterpret_cast<float4*>(orow + 16 * c4 + j) = make_float4(v[0], v[1], v[2], v[3]);
          }
        }
      }
      if (row_valid && part >= 0)
        *reinterpret_cast<float2*>(p.part_ml + ((size_t)part * kM + r) * 2) = make_float2(m_P, l);
      else if (row_valid && p.lse)
        p.lse[(size_t)qi * p.n_q_heads + head] = (m_P + log2f(l)) * kLn2;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  __syncthreads();
}

// Combines the n_split parts of each split unit: one warp per row (grid (unit, 8-row group)), lane l
// holding output dims 4l .. 4l + 3, every part's loads in flight together.  With w_k = 2^(m_k - M),
// M = max_k m_k:
//   out = sum_k w_k O_k / sum_k w_k l_k,   lse = (M + log2 sum_k w_k l_k) ln 2,
// summed in part order (the result does not depend on which part finished first).
constexpr int kMaxSplit = 8;
__global__ void __launch_bounds__(256) prompt_merge_kernel(const PromptParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int n_tail = p.n_qb * p.n_kv_heads - p.n_whole;
  const int v = blockIdx.x, u = p.n_whole + v;
  const int G = p.n_q_heads / p.n_kv_heads;
  const int kvh = u / p.n_qb, q_begin = (u % p.n_qb) * p.qpc;
  const int rows = (min(p.n_q, q_begin + p.qpc) - q_begin) * G;
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.y * 8 + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int S = p.n_split;
  float2 ml = make_float2(-INFINITY, 0.f);   // (m, l) of part `lane`
  if (lane < S) ml = *reinterpret_cast<const float2*>(p.part_ml + ((size_t)(lane * n_tail + v) * kM + r) * 2);
  float4 ov[kMaxSplit];
#pragma unroll
  for (int k = 0; k < kMaxSplit; ++k)
    if (k < S) ov[k] = reinterpret_cast<const float4*>(p.part_o + ((size_t)(k * n_tail + v) * kM + r) * kD)[lane];
  const float M = warp_max(ml.x);
  const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - M);
  float L = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kMaxSplit; ++k) {
    if (k < S) {
      const float wk = __shfl_sync(0xffffffffu, w, k), lk = __shfl_sync(0xffffffffu, ml.y, k);
      L = fmaf(wk, lk, L);
      o = make_float4(fmaf(wk, ov[k].x, o.x), fmaf(wk, ov[k].y, o.y), fmaf(wk, ov[k].z, o.z), fmaf(wk, ov[k].w, o.w));
    }
  }
  const float inv = 1.f / L;
  const int qi = q_begin + r / G, head = kvh * G + r % G;
  reinterpret_cast<float4*>(p.out + ((size_t)qi * p.n_q_heads + head) * kD)[lane] =
      make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
  if (p.lse && lane == 0) p.lse[(size_t)qi * p.n_q_heads + head] = (M + log2f(L)) * kLn2;
}

// A split unit's CTA costs this many tiles beyond its share (prologue, pipeline fill and drain).
constexpr int kPartOverheadTiles = 4;
constexpr int kMinPartTiles = 8;

}  // namespace ws

// Units (query block, KV head) run in rounds of n_sm CTAs; when the last round is partly empty,
// its units are each cut into n_split equal tile ranges (the n_split minimising the modelled
// finish time of the tail: rounds of parts x (tiles per part + overhead)), and the parts' rows
// are merged by one more launch.
bool prompt_plan(int v_bits, int n_kv_heads, int n_q_heads, int n_q, int q_pos0, int n_sm, PromptPlan* plan) {
  if ((v_bits != 8 && v_bits != 4) || n_kv_heads < 1 || n_q_heads < 1 || n_q_heads % n_kv_heads != 0 ||
      n_q_heads / n_kv_heads > ws::kM || n_q < 1 || q_pos0 < 0 || n_sm < 1 || !plan)
    return false;
  PromptPlan pl{};
  pl.qpc = ws::kM / (n_q_heads / n_kv_heads);
  pl.n_qb = (n_q + pl.qpc - 1) / pl.qpc;
  pl.n_units = pl.n_qb * n_kv_heads;
  pl.n_whole = pl.n_units;
  pl.n_split = 1;
  const int n_tail = pl.n_units % n_sm;
  if (n_tail > 0) {
    int l_min = 1 << 30;
    double l_sum = 0.0;
    for (int u = pl.n_units - n_tail; u < pl.n_units; ++u) {
      const int qb = u % pl.n_qb;
      const int l = (q_pos0 + std::min(n_q, (qb + 1) * pl.qpc) - 1) / ws::kN + 1;
      l_min = std::min(l_min, l);
      l_sum += l;
    }
    const double l_avg = l_sum / n_tail;
    double best = 0.0;
    for (int s = 1; s <= ws::kMaxSplit && (s == 1 || l_min / s >= ws::kMinPartTiles); ++s) {
      const double cost = (double)((n_tail * s + n_sm - 1) / n_sm) * (l_avg / s + ws::kPartOverheadTiles);
      if (s == 1 || cost < best) {
        best = cost;
        pl.n_split = s;
      }
    }
    if (pl.n_split > 1) {
      pl.n_whole = pl.n_units - n_tail;
      pl.n_parts = n_tail * pl.n_split;
    }
  }
  const int n_tiles = (q_pos0 + n_q - 1) / ws::kN + 1;
  pl.images_offset = ws::kScratchHeader;
  pl.parts_offset = pl.images_offset + (size_t)n_kv_heads * n_tiles * ws::kImgBytes;
  pl.ml_offset = pl.parts_offset + (size_t)pl.n_parts * ws::kM * kD * sizeof(float);
  pl.bytes = pl.ml_offset + (size_t)pl.n_parts * ws::kM * 2 * sizeof(float);
  *plan = pl;
  return true;
}

cudaError_t launch_prompt_attn(const PromptParams& p, cudaStream_t stream) {
  const int n_tail = p.n_qb * p.n_kv_heads - p.n_whole;
  const dim3 grid(p.n_whole + (p.n_split > 1 ? n_tail * p.n_split : 0));
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(ws::prompt_attn_ws_kernel), (size_t)ws::kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p.scratch, 0, ws::kScratchHeader, stream);
  if (e != cudaSuccess) return e;
  ws::prompt_vmax_kernel<<<dim3(p.n_tiles, p.n_kv_heads), 64, 0, stream>>>(p.pool, p.n_kv_heads, p.scratch);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ws::prompt_stage_kernel<<<dim3(p.n_tiles, p.n_kv_heads), 256, 0, stream>>>(p.pool, p.n_kv_heads, p.n_tiles,
                                                                              p.scratch);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ws::prompt_attn_ws_kernel<<<grid, ws::kThreads, ws::kSmemBytes, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.n_split <= 1) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_tail, ws::kM / 8);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ws::prompt_merge_kernel, p);
}

int* device_error_word() {
  static int* ptr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    ptr[dev] = static_cast<int*>(p);
  }
  return ptr[dev];
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
