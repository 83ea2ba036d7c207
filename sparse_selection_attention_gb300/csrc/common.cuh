// Shared device-side definitions of the QSA library (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qsa.h"

namespace qsa {

constexpr int kD = QSA_HEAD_DIM;           // head_dim
constexpr float kInvSqrtD = 0.08838834764831845f;  // 1 / sqrt(128)

// One pool as the kernels see it.  Geometry shared by all pools of a launch
// (n_kv_heads, head_dim) travels separately.
struct PoolDev {
  const int8_t* k_codes;
  const uint8_t* v_codes;
  const float* k_scales;
  const float* v_scales;
  const int32_t* page_table;
  int n_filled;
  int page_cells;
  int page_shift;   // log2(page_cells) when page_cells is a power of two, else -1
  int v_bits;
  int k_bits;
  const float* k_sums;   // per (64-cell summary block, KV head) sums of dequantised K, or nullptr
};

// Linear (page, head, cell) slot of logical cell c of KV head h.
__device__ __forceinline__ long long cell_slot(const PoolDev& p, int n_kv_heads, int h, int c) {
  int pg, off;
  if (p.page_shift >= 0) {
    pg = c >> p.page_shift;
    off = c & (p.page_cells - 1);
  } else {
    pg = c / p.page_cells;
    off = c - pg * p.page_cells;
  }
  const int page = __ldg(p.page_table + pg);
  return ((long long)page * n_kv_heads + h) * p.page_cells + off;
}

// int8 code packed in byte j of w -> exact float.
__device__ __forceinline__ float s8_to_f32(uint32_t w, int j) {
  return (float)(int8_t)((w >> (8 * j)) & 0xFF);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Host-side helpers shared by the launchers.
int device_sm_count();
int device_max_smem_optin();
// Raises a kernel's dynamic shared memory limit to at least `bytes` on the
// current device; the attribute call is made only when the limit grows.
cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes);

}  // namespace qsa
