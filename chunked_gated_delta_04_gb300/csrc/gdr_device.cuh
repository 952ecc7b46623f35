// gdr_device.cuh -- small device helpers shared by the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#if defined(__CUDA_ARCH__) && !defined(__CUDA_ARCH_FEAT_SM103_ALL)
#error "libgdr must be compiled for sm_103a only (-gencode arch=compute_103a,code=sm_103a)"
#endif

namespace gdr {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

template <typename T>
__device__ __forceinline__ float ldf(const T* p) { return to_f32(p[0]); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Index of state element (a = dk, b = dv) inside one [DK, DV] ("KV") or
// [DV, DK] ("VK") state matrix.
__device__ __forceinline__ size_t state_idx(int layout, int dk, int dv, int DK, int DV) {
  return layout == 0 ? (size_t)dk * DV + dv : (size_t)dv * DK + dk;
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit) { atomicOr(status, bit); }

}  // namespace gdr
