// Quantise-on-append of new K/V cells into a paged pool (qsa_kv_append).
//
// The pages store the cache as int8 codes (4-bit for the V of the K8V4 format, and for K and V of
// the q4_0 format) with one fp32 scale per (cell, KV head, group) ("#1367 prompt attention", Operands; "#2075 QSA decode
// attention", Bit for bit) and append the new cells of each row to it ("#2806 sycl: decode QSA
// selection and attention in fewer, shorter launches", What it leaves alone).  They give no
// quantiser; this one is symmetric by the group's largest magnitude:
//   scale = amax / 127 (int8) or amax / 7 (4-bit),
//   code  = x / scale rounded to nearest, ties to even, clamped to +-127 (+-7),
// with amax = 0 giving scale 0 and codes 0.  The division and the rounding are IEEE fp32
// (round to nearest; the library is built without fast-math), so the codes are exact integers.
#include "kernels.h"

namespace qsa {
namespace {

constexpr int kAppendWarps = 8;

__device__ __forceinline__ float group_scale(float amax, float qmax) { return amax > 0.f ? __fdiv_rn(amax, qmax) : 0.f; }

// code = rint(x / scale) with the quotient rounded to fp32 first (IEEE division), clamped.  y = x *
// (1 / scale), both rounded to nearest, is within 2^-16 of the exact quotient while |x / scale| <=
// 127 (ulp 2^-17 at most), and the rounded quotient within 2^-17: unless y lies within 2^-14 of a
// half-integer, both round to the same integer, so the division is taken only there (and for
// scales below 2^-120, whose reciprocals leave the range this bound assumes).
__device__ __forceinline__ int quant_code(float x, float scale, float inv, float qmax) {
  if (scale == 0.f) return 0;
  const float y = x * inv;
  const bool exact = !(inv <= 0x1p120f) || fabsf(y - floorf(y) - 0.5f) <= 0x1p-14f;
  const float r = exact ? rintf(__fdiv_rn(x, scale)) : rintf(y);
  return (int)fminf(fmaxf(r, -qmax), qmax);
}

__device__ __forceinline__ float max_abs4(float4 x) {
  return fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
}

// Largest magnitude over the `width` lanes of the lane's aligned group (width a power of two <= 32).
__device__ __forceinline__ float group_max(float m, int width) {
  for (int o = width >> 1; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

__device__ __forceinline__ uint32_t pack_s8(int a, int b, int c, int d) {
  return (uint32_t)(a & 0xFF) | ((uint32_t)(b & 0xFF) << 8) | ((uint32_t)(c & 0xFF) << 16) | ((uint32_t)(d & 0xFF) << 24);
}

// Quantises one row (lane l: dims 4l .. 4l + 3) into a code row and its scales at `slot`: int8 with
// one scale per 64 dims (16 lanes), or 4-bit (nibble = code + 8, the even dim in the low nibble)
// with one scale per 32 dims (8 lanes).
__device__ __forceinline__ void store_row(float4 x, int bits, uint8_t* codes, float* scales, long long slot, int lane) {
  if (bits == 8) {
    const float sc = group_scale(group_max(max_abs4(x), 16), 127.f), inv = __frcp_rn(sc);
    reinterpret_cast<uint32_t*>(codes + slot * kD)[lane] =
        pack_s8(quant_code(x.x, sc, inv, 127.f), quant_code(x.y, sc, inv, 127.f), quant_code(x.z, sc, inv, 127.f),
                quant_code(x.w, sc, inv, 127.f));
    if ((lane & 15) == 0) scales[slot * 2 + (lane >> 4)] = sc;
  } else {
    const float sc = group_scale(group_max(max_abs4(x), 8), 7.f), inv = __frcp_rn(sc);
    const uint32_t n0 = (uint32_t)(quant_code(x.x, sc, inv, 7.f) + 8), n1 = (uint32_t)(quant_code(x.y, sc, inv, 7.f) + 8);
    const uint32_t n2 = (uint32_t)(quant_code(x.z, sc, inv, 7.f) + 8), n3 = (uint32_t)(quant_code(x.w, sc, inv, 7.f) + 8);
    reinterpret_cast<uint16_t*>(codes + slot * (kD / 2))[lane] = (uint16_t)(n0 | (n1 << 4) | (n2 << 8) | (n3 << 12));
    if ((lane & 7) == 0) scales[slot * 4 + (lane >> 3)] = sc;
  }
}

// Quantises one (cell, KV head) whose K and V rows this warp holds.
__device__ __forceinline__ void append_item(const AppendParams& p, int item, float4 xk, float4 xv, int lane) {
  const int Hkv = p.n_kv_heads;
  const int i = item / Hkv, h = item % Hkv;
  const long long slot = cell_slot(p.pool, Hkv, h, p.first_cell + i);
  store_row(xk, p.pool.k_bits, reinterpret_cast<uint8_t*>(p.k_codes), p.k_scales, slot, lane);
  store_row(xv, p.pool.v_bits, p.v_codes, p.v_scales, slot, lane);
}

// One (cell, KV head) item per warp, items cell-major (rows of k and v read in order).
constexpr int kItemsPerWarp = 1;
__global__ void __launch_bounds__(32 * kAppendWarps) kv_append_kernel(const AppendParams p) {
  const int n_items = p.n_new * p.n_kv_heads;
  const int item0 = (blockIdx.x * kAppendWarps + (threadIdx.x >> 5)) * kItemsPerWarp;
  const int lane = threadIdx.x & 31;
  float4 xk[kItemsPerWarp], xv[kItemsPerWarp];
#pragma unroll
  for (int j = 0; j < kItemsPerWarp; ++j) {
    if (item0 + j < n_items) {
      xk[j] = __ldg(reinterpret_cast<const float4*>(p.k + (size_t)(item0 + j) * kD) + lane);
      xv[j] = __ldg(reinterpret_cast<const float4*>(p.v + (size_t)(item0 + j) * kD) + lane);
    }
  }
#pragma unroll
  for (int j = 0; j < kItemsPerWarp; ++j)
    if (item0 + j < n_items) append_item(p, item0 + j, xk[j], xv[j], lane);
}

}  // namespace

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream) {
  const long long items = (long long)p.n_new * p.n_kv_heads;
  if (items == 0) return cudaSuccess;
  const long long per_cta = (long long)kAppendWarps * kItemsPerWarp;
  kv_append_kernel<<<(unsigned)((items + per_cta - 1) / per_cta), 32 * kAppendWarps, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace qsa
