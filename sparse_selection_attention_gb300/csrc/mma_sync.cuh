// Register-level helpers of the decode kernels: exact int8 / 4-bit code -> fp16
// conversion, fp16 hi + lo splits, mma.sync m16n8k16, cp.async copies and the
// programmatic-dependent-launch controls.  Written from the public PTX ISA.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace qsa {
namespace ms {

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Two bytes of u (chosen by the byte_perm selector `sel`, each placed in the mantissa of the fp16
// 1024) minus `bias`: for a byte b, 1024 + b - bias.  With b = code + 128 and bias 1152 (0x6480)
// this is the int8 code exactly; with b = nibble and bias 1032 (0x6408) the 4-bit code.
__device__ __forceinline__ uint32_t byte_pair_h2(uint32_t u, uint32_t sel, uint32_t bias) {
  return h2u(__hsub2(u2h(__byte_perm(u, 0x64646464u, sel)), u2h(bias)));
}
constexpr uint32_t kBiasS8 = 0x64806480u;
constexpr uint32_t kBiasNibble = 0x64086408u;

// (a, b) -> fp16 pairs hi, lo with hi + lo = (a, b) to ~2^-22 relative.
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 back = __half22float2(h);
  hi = h2u(h);
  lo = h2u(__floats2half2_rn(a - back.x, b - back.y));
}

// 2^e as a float (e clamped to the normal range), for exact power-of-two scaling.
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + max(-126, min(127, e))) << 23); }

// Exponent fe with max |x 2^fe| in [64, 128) for amax = max |x| > 0 (0 when amax == 0).
__device__ __forceinline__ int scale_exp_128(float amax) {
  int e = 0;
  if (amax > 0.f) frexpf(amax, &e);
  return amax > 0.f ? max(-126, min(127, 7 - e)) : 0;
}

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

// Programmatic dependent launch.  pdl_wait() returns once the grid this launch depends on has
// completed and its memory is visible (a no-op without such a dependency); pdl_trigger() lets
// the next launch of the stream start its CTAs before this grid has finished.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace ms
}  // namespace qsa
