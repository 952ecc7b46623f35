// tc_common.cuh -- device helpers shared by the tensor-core kernels: 128-byte-swizzled
// row stores/loads of bf16 tiles, TMEM row loads, and the in-chunk gate cumsum.
#pragma once

#include <cuda_bf16.h>

#include "gdr_instrument.cuh"
#include "tc_primitives.cuh"

namespace gdr {
namespace tcx {

using bf16 = __nv_bfloat16;
constexpr int kTcThreads = 128;
constexpr uint32_t kSlab = 64 * 128;  // bytes of one 64-row x 128-byte slab

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return (unsigned char*)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

// Store 64 fp32 values as bf16 into row `row` of a 64-column swizzled slab.
__device__ __forceinline__ void st_row_bf16(unsigned char* slab, int row, const float* v) {
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    uint4 w;
    uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 b = __floats2bfloat162_rn(v[ch * 8 + 2 * e], v[ch * 8 + 2 * e + 1]);
      wp[e] = *reinterpret_cast<uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(slab + row * 128 + (((ch ^ (row & 7)) & 7) << 4)) = w;
  }
}

// Load row `row` (64 bf16) of a 64-column swizzled slab as fp32.
__device__ __forceinline__ void ld_row_bf16(const unsigned char* slab, int row, float* v) {
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    const uint4 w = *reinterpret_cast<const uint4*>(slab + row * 128 + (((ch ^ (row & 7)) & 7) << 4));
    const uint32_t* wp = reinterpret_cast<const uint32_t*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&wp[e]);
      const float2 f = __bfloat1622float2(b);
      v[ch * 8 + 2 * e] = f.x;
      v[ch * 8 + 2 * e + 1] = f.y;
    }
  }
}

// 64 fp32 -> 64 bf16 in global memory (128 bytes, 16-byte aligned).
__device__ __forceinline__ void st_global_bf16x64(bf16* dst, const float* v) {
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    uint4 w;
    uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 b = __floats2bfloat162_rn(v[ch * 8 + 2 * e], v[ch * 8 + 2 * e + 1]);
      wp[e] = *reinterpret_cast<uint32_t*>(&b);
    }
    reinterpret_cast<uint4*>(dst)[ch] = w;
  }
}

// Store 32 fp32 values as bf16 into columns [32 * half, 32 * half + 32) of row `row`
// of a 64-column swizzled slab.
__device__ __forceinline__ void st_halfrow_bf16(unsigned char* slab, int row, int half, const float* v) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int ch = 4 * half + c;
    uint4 w;
    uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 b = __floats2bfloat162_rn(v[c * 8 + 2 * e], v[c * 8 + 2 * e + 1]);
      wp[e] = *reinterpret_cast<uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(slab + row * 128 + (((ch ^ (row & 7)) & 7) << 4)) = w;
  }
}

// Load columns [32 * half, 32 * half + 32) of row `row` (bf16) of a 64-column swizzled slab.
__device__ __forceinline__ void ld_halfrow_bf16(const unsigned char* slab, int row, int half, float* v) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int ch = 4 * half + c;
    const uint4 w = *reinterpret_cast<const uint4*>(slab + row * 128 + (((ch ^ (row & 7)) & 7) << 4));
    const uint32_t* wp = reinterpret_cast<const uint32_t*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wp[e]));
      v[c * 8 + 2 * e] = f.x;
      v[c * 8 + 2 * e + 1] = f.y;
    }
  }
}

// Loads 32 TMEM columns [col, col + 32) of this thread's lane.
__device__ __forceinline__ void tmem_ld32w(uint32_t tbase, int warp, int col, float* v) {
  tc::tmem_ld32(tc::tmem_lane_addr(tbase, warp, col), v);
  tc::tmem_wait_ld();
}

// Loads 64 TMEM columns [col, col + 64) of this thread's lane.
__device__ __forceinline__ void tmem_ld64(uint32_t tbase, int warp, int col, float* v) {
  tc::tmem_ld32(tc::tmem_lane_addr(tbase, warp, col), v);
  tc::tmem_ld32(tc::tmem_lane_addr(tbase, warp, col + 32), v + 32);
  tc::tmem_wait_ld();
}

// In-chunk inclusive cumsum of g over 64 rows (threads 0-63 hold row tid);
// returns gamma_r for r = tid < 64.  `scratch` holds 1 float.
__device__ __forceinline__ float chunk_cumsum64(float x, int tid, float* scratch) {
  const int lane = tid & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (tid == 31) *scratch = x;
  __syncthreads();
  if (tid >= 32 && tid < 64) x += *scratch;
  return x;
}

// e^x as 2^(x log2 e) on the hardware exp2 unit (about 2 ulp; results below 2^-126
// flush to zero).  In the epilogue loops it is several times faster than __expf.
__device__ __forceinline__ float fexp(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
  return y;
}

// Store 32 fp32 values into row `row` of a 128-byte-swizzled fp32 slab (32 columns).
__device__ __forceinline__ void st_row_f32x32(unsigned char* slab, int row, const float* v) {
#pragma unroll
  for (int ch = 0; ch < 8; ++ch)
    *reinterpret_cast<float4*>(slab + row * 128 + (((ch ^ (row & 7)) & 7) << 4)) =
        make_float4(v[4 * ch], v[4 * ch + 1], v[4 * ch + 2], v[4 * ch + 3]);
}

}  // namespace tcx
}  // namespace gdr
