// Decode block scores (qsa_block_scores).
//
// S[t,b] = sum_h (1/n_b) sum_{c in b} sum_{g in G(h)} q[t,g] . K[c,h] / sqrt(D)
//        = sum_h (1/n_b) sum_{c in b} sum_grp kscale[c,h,grp] (qbar[t,h] . kcode[c,h])_grp / sqrt(D),
// qbar[t,h] = sum_{g in G(h)} q[t,g]: the group's q heads are summed once, and
// a block is read once per window for all of its slot's rows ("#2806 sycl:
// decode QSA selection and attention in fewer, shorter launches", Summary: a
// block's (query, head) sums are reduced together; scores once per slot).
// HBM-bound: every filled K code and scale is read exactly once per call.
//
// The per-(cell, row) dot products run on mma.sync m16n8k16: A = K codes of
// 16 cells (int8 -> fp16, exact), B = qbar 2^f of 8 rows split into fp16
// hi + lo (both accumulate into one fp32 sum), one accumulator per 64-dim
// K-scale group.  A persistent grid of one 512-thread CTA per SM walks the
// (pool, block) units; warp task = (unit, KV head, 16-cell m-tile).  Each
// thread loads the 64 code bytes of its two cells with four 16-byte loads,
// straight into registers, and the next unit's loads are in flight while the
// current one is reduced.  The epilogue weights each cell by its K scales,
// reduces over cells (lane butterfly), then over the unit's m-tiles and heads
// with a fixed butterfly: bitwise reproducible.
#include <cuda_fp16.h>

#include "kernels.h"

namespace qsa {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kTpwMax = 2;   // warp tasks per warp per iteration
constexpr int kNtMax = 4;    // 8-row n-tiles (rows <= 32)

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Two bytes of a biased word (code + 128) -> exact fp16 pair of the codes.
__device__ __forceinline__ uint32_t byte_pair_h2(uint32_t u, uint32_t sel) {
  return h2u(__hsub2(u2h(__byte_perm(u, 0x64646464u, sel)), u2h(0x64806480u)));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + max(-126, min(127, e))) << 23); }

__host__ __device__ inline int round4(int x) { return (x + 3) & ~3; }

// One warp task's operands: codes of cells cb+g and cb+g+8 (dims 64 grp + 16 tq .. +15) and scales.
struct TaskData {
  uint4 c[2][2];   // [cell a/b][K-scale group]
  float2 ks[2];
};

struct TaskRef {
  int u_s, h, mt;   // unit slot, KV head, m-tile
  bool live;
};

__device__ __forceinline__ int pool_of(const ScoresParams& p, int unit) {
  int pi = 0;
  while (pi + 1 < p.n_pools && unit >= p.unit_begin[pi + 1]) ++pi;
  return pi;
}

__device__ __forceinline__ void load_task(const ScoresParams& p, int unit, const TaskRef& r, TaskData& d) {
  const int lane = threadIdx.x & 31, g = lane >> 2, tq = lane & 3;
  const int B = p.block_cells;
  const int pi = pool_of(p, unit);
  const PoolDev& pool = p.pools[pi];
  const int b = unit - p.unit_begin[pi];
  const int cell0 = b * B;
  const int n_b = min(B, pool.n_filled - cell0);
  const int page = __ldg(pool.page_table + cell0 / pool.page_cells);
  const long long slot0 = ((long long)page * p.n_kv_heads + r.h) * pool.page_cells + cell0 % pool.page_cells;
#pragma unroll
  for (int ab = 0; ab < 2; ++ab) {
    const int c = 16 * r.mt + g + 8 * ab;
    if (c < n_b) {
      const uint4* src = reinterpret_cast<const uint4*>(pool.k_codes + (slot0 + c) * kD);
      d.c[ab][0] = __ldg(src + tq);
      d.c[ab][1] = __ldg(src + 4 + tq);
      d.ks[ab] = __ldg(reinterpret_cast<const float2*>(pool.k_scales) + slot0 + c);
    } else {
      d.c[ab][0] = d.c[ab][1] = make_uint4(0u, 0u, 0u, 0u);
      d.ks[ab] = make_float2(0.f, 0.f);
    }
  }
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int w) {
  return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
}

template <int kMaxNt, int kMaxTpw>
__global__ void __launch_bounds__(kThreads, 1) block_scores_kernel(const ScoresParams p) {
  extern __shared__ __align__(16) float smem[];
  const int Hkv = p.n_kv_heads, G = p.n_q_heads / Hkv, B = p.block_cells;
  const int R = p.n_rows, NT = (R + 7) / 8;
  const int tpu = Hkv * (B / 16);                 // warp tasks per unit (<= 32)
  const int upi = max(1, kWarps / tpu);           // units per iteration
  const int tpw = (upi * tpu + kWarps - 1) / kWarps;
  // smem: B fragments [Hkv][NT][8 k-steps][32 lanes] uint4, 1/f [R][Hkv] (padded to 4), partial sums
  // [upi][tpu][NT*8], then the staging area for q rows.
  uint4* bfrag = reinterpret_cast<uint4*>(smem);
  float* inv_f = reinterpret_cast<float*>(bfrag + Hkv * NT * 8 * 32);
  float* part = inv_f + round4(R * Hkv);
  float* qstage = part + upi * tpu * NT * 8;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tq = lane & 3;
  const int n_super = (p.total_units + upi - 1) / upi;
  if ((int)blockIdx.x >= n_super) return;

  TaskRef ref[kMaxTpw];
#pragma unroll
  for (int k = 0; k < kMaxTpw; ++k) {
    const int ti = warp + kWarps * k;
    ref[k].live = k < tpw && ti < upi * tpu;
    ref[k].u_s = ti / tpu;
    ref[k].h = (ti % tpu) / (B / 16);
    ref[k].mt = ti % (B / 16);
  }
  TaskData cur[kMaxTpw], nxt[kMaxTpw];
#pragma unroll
  for (int k = 0; k < kMaxTpw; ++k) {
    const int unit = blockIdx.x * upi + ref[k].u_s;
    if (ref[k].live && unit < p.total_units) load_task(p, unit, ref[k], cur[k]);
  }

  // ---- qbar 2^f per (row, head), split fp16 hi/lo, laid out as this kernel's B fragments.
  {
    const int row_floats = p.n_q_heads * kD;
    for (int r0 = 0; r0 < R; r0 += p.q_rows_per_batch) {
      const int nr = min(p.q_rows_per_batch, R - r0);
      const float4* q4 = reinterpret_cast<const float4*>(p.q + (size_t)r0 * row_floats);
      for (int k = tid; k < nr * row_floats / 4; k += kThreads) reinterpret_cast<float4*>(qstage)[k] = __ldg(q4 + k);
      __syncthreads();
      // One warp per (row, head): qbar in registers (4 dims per lane), max |qbar| -> 2^f.
      for (int rh = warp; rh < nr * Hkv; rh += kWarps) {
        const int tr = rh / Hkv, h = rh % Hkv, t = r0 + tr;
        const float* qg = qstage + (size_t)tr * row_floats + h * G * kD;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float s = 0.f;
          for (int gg = 0; gg < G; ++gg) s += qg[gg * kD + 4 * lane + i];
          v[i] = s;
        }
        float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
        amax = warp_max(amax);
        int e = 0;
        if (amax > 0.f) frexpf(amax, &e);
        const int fe = amax > 0.f ? max(-126, min(127, 7 - e)) : 0;
        const float f = pow2i(fe);
        if (lane == 0) inv_f[t * Hkv + h] = pow2i(-fe);
        // dims 4 lane .. +3 = 64 grp + 16 tq' + 4 s' .. : k-step 4 grp + s', fragment lane (row % 8, tq')
        const int d0 = 4 * lane, grp = d0 >> 6, tqp = (d0 >> 4) & 3, sp = (d0 >> 2) & 3;
        const int s = 4 * grp + sp, nt = t >> 3, gp = t & 7;
        const __half2 h01 = __floats2half2_rn(v[0] * f, v[1] * f), h23 = __floats2half2_rn(v[2] * f, v[3] * f);
        const float2 b01 = __half22float2(h01), b23 = __half22float2(h23);
        const __half2 l01 = __floats2half2_rn(v[0] * f - b01.x, v[1] * f - b01.y);
        const __half2 l23 = __floats2half2_rn(v[2] * f - b23.x, v[3] * f - b23.y);
        bfrag[((h * NT + nt) * 8 + s) * 32 + gp * 4 + tqp] = make_uint4(h2u(h01), h2u(h23), h2u(l01), h2u(l23));
      }
      __syncthreads();
    }
    for (int k = tid; k < Hkv * 8 * 32; k += kThreads) {   // rows R .. NT*8-1: zero fragments
      const int h = k / 256, s = (k / 32) % 8, ln = k % 32, row = (NT - 1) * 8 + (ln >> 2);
      if (row >= R) bfrag[((h * NT + NT - 1) * 8 + s) * 32 + ln] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
  }

  for (int su = blockIdx.x; su < n_super; su += gridDim.x) {
    const bool more = su + (int)gridDim.x < n_super;
#pragma unroll
    for (int k = 0; k < kMaxTpw; ++k) {
      const int unit = (su + gridDim.x) * upi + ref[k].u_s;
      if (more && ref[k].live && unit < p.total_units) load_task(p, unit, ref[k], nxt[k]);
    }
#pragma unroll
    for (int k = 0; k < kMaxTpw; ++k) {
      const int unit = su * upi + ref[k].u_s;
      if (!ref[k].live || unit >= p.total_units) continue;   // warp-uniform
      const int h = ref[k].h;
      float d[kMaxNt][2][4];
#pragma unroll
      for (int nt = 0; nt < kMaxNt; ++nt)
#pragma unroll
        for (int gr = 0; gr < 2; ++gr)
#pragma unroll
          for (int i = 0; i < 4; ++i) d[nt][gr][i] = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int gr = s >> 2, w = s & 3;
        const uint32_t wa = word_of(cur[k].c[0][gr], w) ^ 0x80808080u;
        const uint32_t wb = word_of(cur[k].c[1][gr], w) ^ 0x80808080u;
        uint32_t a[4];
        a[0] = byte_pair_h2(wa, 0x4140);
        a[2] = byte_pair_h2(wa, 0x4342);
        a[1] = byte_pair_h2(wb, 0x4140);
        a[3] = byte_pair_h2(wb, 0x4342);
#pragma unroll
        for (int nt = 0; nt < kMaxNt; ++nt) {
          if (nt < NT) {
            const uint4 bf = bfrag[((h * NT + nt) * 8 + s) * 32 + lane];
            mma16816(d[nt][gr], a, bf.x, bf.y);
            mma16816(d[nt][gr], a, bf.z, bf.w);
          }
        }
      }
      // Weight each cell by its K scales, sum the two cells, reduce over the 8 cell pairs.
      const float2 ka = cur[k].ks[0], kb = cur[k].ks[1];
      const int ti = ref[k].u_s * tpu + h * (B / 16) + ref[k].mt;
#pragma unroll
      for (int nt = 0; nt < kMaxNt; ++nt) {
        if (nt < NT) {
          float e0 = fmaf(ka.y, d[nt][1][0], ka.x * d[nt][0][0]);
          e0 += fmaf(kb.y, d[nt][1][2], kb.x * d[nt][0][2]);
          float e1 = fmaf(ka.y, d[nt][1][1], ka.x * d[nt][0][1]);
          e1 += fmaf(kb.y, d[nt][1][3], kb.x * d[nt][0][3]);
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            e0 += __shfl_xor_sync(0xffffffffu, e0, o);
            e1 += __shfl_xor_sync(0xffffffffu, e1, o);
          }
          if (g == 0) {
            const int row = nt * 8 + 2 * tq;
            part[ti * NT * 8 + row] = row < R ? e0 * inv_f[row * Hkv + h] : 0.f;
            part[ti * NT * 8 + row + 1] = row + 1 < R ? e1 * inv_f[(row + 1) * Hkv + h] : 0.f;
          }
        }
      }
    }
    __syncthreads();
    // S[t, b]: one warp per (unit slot, row); lane l holds the unit's task l (<= 32 tasks), then a
    // fixed butterfly over the lanes.
    for (int pr = warp; pr < upi * R; pr += kWarps) {
      const int u_s = pr / R, t = pr % R;
      const int unit = su * upi + u_s;
      if (unit >= p.total_units) continue;
      const int pi = pool_of(p, unit);
      if (p.row_pool[t] != pi) continue;
      float s = lane < tpu ? part[(u_s * tpu + lane) * NT * 8 + t] : 0.f;
      s = warp_sum(s);
      if (lane == 0) {
        const int b = unit - p.unit_begin[pi];
        const int n_b = min(B, p.pools[pi].n_filled - b * B);
        p.scores[(size_t)t * p.max_blocks + b] = s * (kInvSqrtD / (float)n_b);
      }
    }
    if (more) {
#pragma unroll
      for (int k = 0; k < kMaxTpw; ++k) cur[k] = nxt[k];
    }
    __syncthreads();
  }
}

// Floats of the q staging area: up to 16K floats (64 KB), at least one row of q.
size_t q_stage_floats(int n_rows, int n_q_heads) {
  const size_t row = (size_t)n_q_heads * kD, all = row * n_rows;
  return all < 16384 ? all : (row > 16384 ? row : 16384);
}

// ---------------------------------------------------------------------------------------------
// Staged variant (used when a whole unit's K fits a shared-memory stage): the same per-task
// arithmetic, fed by bulk copies.  A persistent CTA owns a contiguous range of units; its
// producer warp looks up the units' pages in parallel (one lane per unit) and issues every copy of
// the range up front into a ring of up to kMaxStages unit stages, so the whole range's K reads are
// in flight together instead of one unit at a time.  Stage layout: K codes [head][B][128 B], then
// K scales [head][B][2] floats.  Sixteen compute warps take the units' (head, m-tile) tasks as the
// stages arrive, keeping each task's sum in shared memory; one barrier at the end precedes the
// fixed-order reduction of every unit's task sums.  Waits are bounded: a
// wait that runs out sets the device error word and the CTA runs to its end without further copies
// (its scores are then not valid); before exiting it waits for every copy it issued.
namespace staged {

constexpr int kComputeWarps = 16;
constexpr int kMaxUnitsPerCta = 64;   // task sums kept for the whole range
constexpr int kThreads = 32 * (kComputeWarps + 1);
constexpr int kMaxStages = 6;

__host__ __device__ inline int stage_bytes(int n_kv_heads, int B) { return n_kv_heads * B * (kD + 8); }

struct Layout {
  int bfrag, inv_f, part, stage0, bars, ctl, total;
};
// upc: units per CTA (task sums are kept for all of them).
__host__ __device__ inline Layout layout(int R, int Hkv, int B, int n_stages, int upc) {
  const int NT = (R + 7) / 8, tpu = Hkv * (B / 16);
  Layout L;
  L.bfrag = 0;
  L.inv_f = L.bfrag + 16 * Hkv * NT * 8 * 32;
  L.part = L.inv_f + 4 * round4(R * Hkv);
  L.stage0 = (L.part + 4 * upc * tpu * NT * 8 + 127) & ~127;
  L.bars = L.stage0 + n_stages * stage_bytes(Hkv, B);
  L.ctl = L.bars + 16 * kMaxStages;
  L.total = L.ctl + 16;
  return L;
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait; false (and the abort flag set) when it runs out or the CTA has aborted.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err,
                                           uint64_t limit_ns) {
  if (mbar_try(bar, parity)) return true;
  if (limit_ns == 0 || *abort_flag) {
    *abort_flag = 1;
    atomicCAS(err, 0, 2);
    return false;
  }
  const uint64_t t0 = gtimer();
  while (!mbar_try(bar, parity)) {
    if (*abort_flag || gtimer() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicCAS(err, 0, 2);
      return false;
    }
  }
  return true;
}

template <int kMaxNt>
__global__ void __launch_bounds__(kThreads, 1) block_scores_staged_kernel(const ScoresParams p, int n_stages, int upc) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int Hkv = p.n_kv_heads, G = p.n_q_heads / Hkv, B = p.block_cells;
  const int R = p.n_rows, NT = (R + 7) / 8;
  const int tpu = Hkv * (B / 16);
  const Layout L = layout(R, Hkv, B, n_stages, upc);
  uint4* bfrag = reinterpret_cast<uint4*>(smem + L.bfrag);
  float* inv_f = reinterpret_cast<float*>(smem + L.inv_f);
  float* part = reinterpret_cast<float*>(smem + L.part);
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  const uint32_t full0 = sbase + L.bars, empty0 = full0 + 8 * kMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.ctl);
  volatile int* issued_w = abort_flag + 1;
  const int SB = stage_bytes(Hkv, B);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, tq = lane & 3;
  // Contiguous unit range of this CTA.
  const int per = p.total_units / gridDim.x, extra = p.total_units % gridDim.x;
  const int u0 = blockIdx.x * per + min((int)blockIdx.x, extra);
  const int n_units = per + ((int)blockIdx.x < extra ? 1 : 0);

  if (tid == 0) {
    for (int s = 0; s < n_stages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(full0 + 8 * s) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(empty0 + 8 * s), "r"(kComputeWarps) : "memory");
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *abort_flag = 0;
    *issued_w = 0;
  }
  __syncthreads();

  if (warp == kComputeWarps) {
    // ================================================= producer
    int issued = 0;
    for (int base = 0; base < n_units; base += 32) {
      const int n = min(32, n_units - base);
      int pg = 0;
      if (lane < n) {
        const int unit = u0 + base + lane;
        const int pi = pool_of(p, unit);
        const int b = unit - p.unit_begin[pi];
        pg = __ldg(p.pools[pi].page_table + (b * B) / p.pools[pi].page_cells);
      }
      for (int k = 0; k < n; ++k) {
        const int page = __shfl_sync(0xffffffffu, pg, k);
        if (lane == 0 && !*abort_flag) {
          const int i = base + k, st = i % n_stages;
          bool ok = true;
          if (i >= n_stages) ok = wait_phase(empty0 + 8 * st, ((i / n_stages) - 1) & 1, abort_flag, p.err, p.wait_limit_ns);
          if (ok) {
            const int unit = u0 + i;
            const int pi = pool_of(p, unit);
            const PoolDev& pool = p.pools[pi];
            const int cell0 = (unit - p.unit_begin[pi]) * B;
            const uint32_t dst = sbase + L.stage0 + st * SB, bar = full0 + 8 * st;
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(SB) : "memory");
            for (int h = 0; h < Hkv; ++h) {
              const long long slot0 = ((long long)page * Hkv + h) * pool.page_cells + cell0 % pool.page_cells;
              asm volatile(
                  "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                      dst + h * B * kD),
                  "l"(pool.k_codes + slot0 * kD), "r"(B * kD), "r"(bar)
                  : "memory");
              asm volatile(
                  "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                      dst + Hkv * B * kD + h * B * 8),
                  "l"(pool.k_scales + slot0 * 2), "r"(B * 8), "r"(bar)
                  : "memory");
            }
            issued = i + 1;
          }
        }
        __syncwarp();
      }
    }
    if (lane == 0) *issued_w = issued;
  } else {
    // ================================================= compute warps
    // qbar 2^f per (row, head) from q in global memory, split fp16 hi/lo, as B fragments.
    for (int rh = warp; rh < R * Hkv; rh += kComputeWarps) {
      const int t = rh / Hkv, h = rh % Hkv;
      const float* qg = p.q + ((size_t)t * p.n_q_heads + h * G) * kD + 4 * lane;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
      for (int gg = 0; gg < G; ++gg) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(qg + gg * kD));
        v[0] += x.x; v[1] += x.y; v[2] += x.z; v[3] += x.w;
      }
      float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
      amax = warp_max(amax);
      int e = 0;
      if (amax > 0.f) frexpf(amax, &e);
      const int fe = amax > 0.f ? max(-126, min(127, 7 - e)) : 0;
      const float f = pow2i(fe);
      if (lane == 0) inv_f[t * Hkv + h] = pow2i(-fe);
      const int d0 = 4 * lane, grp = d0 >> 6, tqp = (d0 >> 4) & 3, sp = (d0 >> 2) & 3;
      const int s = 4 * grp + sp, nt = t >> 3, gp = t & 7;
      const __half2 h01 = __floats2half2_rn(v[0] * f, v[1] * f), h23 = __floats2half2_rn(v[2] * f, v[3] * f);
      const float2 b01 = __half22float2(h01), b23 = __half22float2(h23);
      const __half2 l01 = __floats2half2_rn(v[0] * f - b01.x, v[1] * f - b01.y);
      const __half2 l23 = __floats2half2_rn(v[2] * f - b23.x, v[3] * f - b23.y);
      bfrag[((h * NT + nt) * 8 + s) * 32 + gp * 4 + tqp] = make_uint4(h2u(h01), h2u(h23), h2u(l01), h2u(l23));
    }
    for (int k = tid; k < Hkv * 8 * 32; k += 32 * kComputeWarps) {   // rows R .. NT*8-1: zero fragments
      const int h = k / 256, s = (k / 32) % 8, ln = k % 32, row = (NT - 1) * 8 + (ln >> 2);
      if (row >= R) bfrag[((h * NT + NT - 1) * 8 + s) * 32 + ln] = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kComputeWarps) : "memory");

    for (int i = 0; i < n_units; ++i) {
      const int st = i % n_stages;
      wait_phase(full0 + 8 * st, (i / n_stages) & 1, abort_flag, p.err, p.wait_limit_ns);
      const int unit = u0 + i;
      const int pi = pool_of(p, unit);
      const int b = unit - p.unit_begin[pi];
      const int n_b = min(B, p.pools[pi].n_filled - b * B);
      const uint8_t* stg = smem + L.stage0 + st * SB;
      float* pu = part + i * tpu * NT * 8;
      for (int task = warp; task < tpu; task += kComputeWarps) {   // warp-uniform
        const int h = task / (B / 16), mt = task % (B / 16);
        const uint8_t* codes = stg + h * B * kD;
        const float* kscale = reinterpret_cast<const float*>(stg + Hkv * B * kD + h * B * 8);
        uint4 c[2][2];
        float2 ks[2];
#pragma unroll
        for (int ab = 0; ab < 2; ++ab) {
          const int cell = 16 * mt + g + 8 * ab;
          if (cell < n_b) {
            c[ab][0] = *reinterpret_cast<const uint4*>(codes + cell * kD + 16 * tq);
            c[ab][1] = *reinterpret_cast<const uint4*>(codes + cell * kD + 64 + 16 * tq);
            ks[ab] = *reinterpret_cast<const float2*>(kscale + 2 * cell);
          } else {
            c[ab][0] = c[ab][1] = make_uint4(0u, 0u, 0u, 0u);
            ks[ab] = make_float2(0.f, 0.f);
          }
        }
        // hi and lo parts of q accumulate in separate chains (half the dependent MMA chain), summed after
        float d[kMaxNt][2][4], dl[kMaxNt][2][4];
#pragma unroll
        for (int nt = 0; nt < kMaxNt; ++nt)
#pragma unroll
          for (int gr = 0; gr < 2; ++gr)
#pragma unroll
            for (int q = 0; q < 4; ++q) d[nt][gr][q] = dl[nt][gr][q] = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const int gr = s >> 2, w = s & 3;
          const uint32_t wa = word_of(c[0][gr], w) ^ 0x80808080u;
          const uint32_t wb = word_of(c[1][gr], w) ^ 0x80808080u;
          uint32_t a[4];
          a[0] = byte_pair_h2(wa, 0x4140);
          a[2] = byte_pair_h2(wa, 0x4342);
          a[1] = byte_pair_h2(wb, 0x4140);
          a[3] = byte_pair_h2(wb, 0x4342);
#pragma unroll
          for (int nt = 0; nt < kMaxNt; ++nt) {
            if (nt < NT) {
              const uint4 bf = bfrag[((h * NT + nt) * 8 + s) * 32 + lane];
              mma16816(d[nt][gr], a, bf.x, bf.y);
              mma16816(dl[nt][gr], a, bf.z, bf.w);
            }
          }
        }
#pragma unroll
        for (int nt = 0; nt < kMaxNt; ++nt)
#pragma unroll
          for (int gr = 0; gr < 2; ++gr)
#pragma unroll
            for (int q = 0; q < 4; ++q) d[nt][gr][q] += dl[nt][gr][q];
#pragma unroll
        for (int nt = 0; nt < kMaxNt; ++nt) {
          if (nt < NT) {
            float e0 = fmaf(ks[0].y, d[nt][1][0], ks[0].x * d[nt][0][0]);
            e0 += fmaf(ks[1].y, d[nt][1][2], ks[1].x * d[nt][0][2]);
            float e1 = fmaf(ks[0].y, d[nt][1][1], ks[0].x * d[nt][0][1]);
            e1 += fmaf(ks[1].y, d[nt][1][3], ks[1].x * d[nt][0][3]);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
              e0 += __shfl_xor_sync(0xffffffffu, e0, o);
              e1 += __shfl_xor_sync(0xffffffffu, e1, o);
            }
            if (g == 0) {
              const int row = nt * 8 + 2 * tq;
              pu[task * NT * 8 + row] = row < R ? e0 * inv_f[row * Hkv + h] : 0.f;
              pu[task * NT * 8 + row + 1] = row + 1 < R ? e1 * inv_f[(row + 1) * Hkv + h] : 0.f;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empty0 + 8 * st) : "memory");
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kComputeWarps) : "memory");
    // S[t, b]: one warp per (unit, row); lane l holds task l (<= 32 tasks), then a fixed butterfly.
    for (int ut = warp; ut < n_units * R; ut += kComputeWarps) {
      const int i = ut / R, t = ut % R;
      const int unit = u0 + i;
      const int pi = pool_of(p, unit);
      if (p.row_pool[t] != pi) continue;
      const int b = unit - p.unit_begin[pi];
      const int n_b = min(B, p.pools[pi].n_filled - b * B);
      float s = lane < tpu ? part[(i * tpu + lane) * NT * 8 + t] : 0.f;
      s = warp_sum(s);
      if (lane == 0) p.scores[(size_t)t * p.max_blocks + b] = s * (kInvSqrtD / (float)n_b);
    }
  }

  // Nothing may still write this CTA's shared memory when it exits: after an abort, wait for the
  // latest fill of every stage that was issued.
  __syncthreads();
  if (*abort_flag && tid == 0) {
    const int issued = *issued_w;
    for (int st = 0; st < n_stages && st < issued; ++st) {
      const int last = st + n_stages * ((issued - 1 - st) / n_stages);
      const uint64_t t0 = gtimer();
      while (!mbar_try(full0 + 8 * st, (last / n_stages) & 1) && gtimer() - t0 < 2000000000ull) {
      }
    }
  }
  __syncthreads();
}

// Stages that fit next to the fragment table (0: the staged kernel does not apply).
int n_stages_for(int R, int Hkv, int B, int total_units, int grid, int smem_max) {
  const int units_per_cta = (total_units + grid - 1) / grid;
  if (units_per_cta > kMaxUnitsPerCta || R > 16) return 0;
  const int SB = stage_bytes(Hkv, B);
  if (SB > 72 * 1024) return 0;
  int s = min(kMaxStages, units_per_cta);
  while (s >= 2 && layout(R, Hkv, B, s, units_per_cta).total + 128 > smem_max) --s;
  if (s < 2 && units_per_cta >= 2) return 0;
  if (s < 1 || layout(R, Hkv, B, s, units_per_cta).total + 128 > smem_max) return 0;
  return s;
}

}  // namespace staged

// 4-bit K (the q4_0 layout: 64-byte rows, low nibble = even dim, code = nibble - 8, one scale per
// 32 dims).  One 256-thread CTA per (pool, block); per KV head, qbar of every row is formed in
// shared memory, then thread (cell tid / 4 + 64 m, 32-dim group tid % 4) takes the dot products of
// its group with each row's qbar, weighted by the group's scale; sums over lanes, warps and KV heads
// run in a fixed order.  fp32 arithmetic.
constexpr int kK4Threads = 256;

__global__ void __launch_bounds__(kK4Threads) block_scores_k4_kernel(const ScoresParams p) {
  __shared__ float qb[QSA_MAX_DECODE_ROWS * kD];   // qbar of one KV head, [row][dim]
  __shared__ float red[kK4Threads / 32][QSA_MAX_DECODE_ROWS];
  __shared__ float acc_s[QSA_MAX_DECODE_ROWS];
  const int unit = blockIdx.x;
  int pi = 0;
  while (pi + 1 < p.n_pools && unit >= p.unit_begin[pi + 1]) ++pi;
  const PoolDev& pool = p.pools[pi];
  const int B = p.block_cells, Hkv = p.n_kv_heads, R = p.n_rows, G = p.n_q_heads / Hkv;
  const int b = unit - p.unit_begin[pi];
  const int cell0 = b * B;
  const int n_b = min(B, pool.n_filled - cell0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = tid & 3;
  if (tid < QSA_MAX_DECODE_ROWS) acc_s[tid] = 0.f;
  const int page = __ldg(pool.page_table + cell0 / pool.page_cells);
  const long long slot0 = (long long)page * Hkv * pool.page_cells + cell0 % pool.page_cells;
  for (int h = 0; h < Hkv; ++h) {
    __syncthreads();   // qb and red of the previous head fully read
    for (int i = tid; i < R * kD; i += kK4Threads) {
      const int t = i / kD, d = i - t * kD;
      const float* qg = p.q + ((size_t)t * p.n_q_heads + (size_t)h * G) * kD + d;
      float s = 0.f;
      for (int g = 0; g < G; ++g) s += __ldg(qg + (size_t)g * kD);
      qb[i] = s;
    }
    __syncthreads();
    float part[QSA_MAX_DECODE_ROWS];
#pragma unroll
    for (int t = 0; t < QSA_MAX_DECODE_ROWS; ++t) part[t] = 0.f;
    for (int c = tid >> 2; c < n_b; c += kK4Threads / 4) {
      const long long slot = slot0 + (long long)h * pool.page_cells + c;
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(pool.k_codes + slot * (kD / 2)) + grp);
      const float scale = __ldg(pool.k_scales + slot * 4 + grp);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
      float code[32];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t byte = (ws[j >> 2] >> (8 * (j & 3))) & 0xFFu;
        code[2 * j] = (float)((int)(byte & 15u) - 8);
        code[2 * j + 1] = (float)((int)(byte >> 4) - 8);
      }
#pragma unroll
      for (int t = 0; t < QSA_MAX_DECODE_ROWS; ++t) {
        if (t < R && p.row_pool[t] == pi) {
          const float* qr = qb + t * kD + 32 * grp;
          float dot = 0.f;
#pragma unroll
          for (int d = 0; d < 32; ++d) dot = fmaf(code[d], qr[d], dot);
          part[t] = fmaf(scale, dot, part[t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < QSA_MAX_DECODE_ROWS; ++t) {
      if (t < R) {
        const float v = warp_sum(part[t]);
        if (lane == 0) red[warp][t] = v;
      }
    }
    __syncthreads();
    if (tid < R) {
      float s = 0.f;
      for (int w = 0; w < kK4Threads / 32; ++w) s += red[w][tid];
      acc_s[tid] += s;
    }
  }
  __syncthreads();
  if (tid < R && p.row_pool[tid] == pi)
    p.scores[(size_t)tid * p.max_blocks + b] = acc_s[tid] * (kInvSqrtD / (float)n_b);
}

}  // namespace

int block_scores_q_rows_per_batch(int n_rows, int n_q_heads, int n_kv_heads, int block_cells) {
  (void)n_kv_heads;
  (void)block_cells;
  const int rb = (int)(q_stage_floats(n_rows, n_q_heads) / ((size_t)n_q_heads * kD));
  return rb < 1 ? 1 : (rb > n_rows ? n_rows : rb);
}

size_t block_scores_smem_bytes(int n_rows, int n_q_heads, int n_kv_heads, int block_cells) {
  const int NT = (n_rows + 7) / 8;
  const int tpu = n_kv_heads * (block_cells / 16);
  const int upi = tpu >= kWarps ? 1 : kWarps / tpu;
  return 16 * (size_t)n_kv_heads * NT * 8 * 32 +
         4 * ((size_t)round4(n_rows * n_kv_heads) + (size_t)upi * tpu * NT * 8) + 4 * q_stage_floats(n_rows, n_q_heads);
}

bool block_scores_supported(int n_kv_heads, int block_cells) {
  const int tpu = n_kv_heads * (block_cells / 16);
  const int upi = tpu >= kWarps ? 1 : kWarps / tpu;
  return block_cells % 16 == 0 && tpu <= 32 && (upi * tpu + kWarps - 1) / kWarps <= kTpwMax;
}

template <int NT, int TPW>
static cudaError_t launch_variant(const ScoresParams& p, size_t smem, int grid, cudaStream_t stream) {
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(block_scores_kernel<NT, TPW>), smem);
  if (e != cudaSuccess) return e;
  block_scores_kernel<NT, TPW><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int NT>
static cudaError_t launch_staged(const ScoresParams& p, int grid, int n_stages, cudaStream_t stream) {
  const int upc = (p.total_units + grid - 1) / grid;
  const size_t smem = staged::layout(p.n_rows, p.n_kv_heads, p.block_cells, n_stages, upc).total + 128;
  const void* k = reinterpret_cast<const void*>(staged::block_scores_staged_kernel<NT>);
  cudaError_t e = ensure_dynamic_smem(k, smem);
  if (e != cudaSuccess) return e;
  staged::block_scores_staged_kernel<NT><<<grid, staged::kThreads, smem, stream>>>(p, n_stages, upc);
  return cudaGetLastError();
}

cudaError_t launch_block_scores(const ScoresParams& p, cudaStream_t stream) {
  if (p.total_units == 0) return cudaSuccess;
  if (p.pools[0].k_bits == 4) {   // the pools of one call share k_bits
    block_scores_k4_kernel<<<p.total_units, kK4Threads, 0, stream>>>(p);
    return cudaGetLastError();
  }
  const int nt = (p.n_rows + 7) / 8;
  if (nt > kNtMax) return cudaErrorInvalidValue;
  {
    const int grid = min(p.total_units, device_sm_count());
    const int ns = staged::n_stages_for(p.n_rows, p.n_kv_heads, p.block_cells, p.total_units, grid,
                                        device_max_smem_optin());
    if (ns > 0 && p.n_kv_heads * (p.block_cells / 16) <= 32) {
      if (nt == 1) return launch_staged<1>(p, grid, ns, stream);
      return launch_staged<2>(p, grid, ns, stream);
    }
  }
  const size_t smem = block_scores_smem_bytes(p.n_rows, p.n_q_heads, p.n_kv_heads, p.block_cells);
  const int tpu = p.n_kv_heads * (p.block_cells / 16);
  const int upi = max(1, kWarps / tpu);
  const int tpw = (upi * tpu + kWarps - 1) / kWarps;
  const int n_super = (p.total_units + upi - 1) / upi;
  const int grid = min(n_super, device_sm_count());
  const int ntv = nt == 1 ? 1 : (nt == 2 ? 2 : 4);
  if (tpw == 1) {
    if (ntv == 1) return launch_variant<1, 1>(p, smem, grid, stream);
    if (ntv == 2) return launch_variant<2, 1>(p, smem, grid, stream);
    return launch_variant<4, 1>(p, smem, grid, stream);
  }
  if (ntv == 1) return launch_variant<1, 2>(p, smem, grid, stream);
  if (ntv == 2) return launch_variant<2, 2>(p, smem, grid, stream);
  return launch_variant<4, 2>(p, smem, grid, stream);
}

}  // namespace qsa
