// gdr_prologue.cu -- the fused input prologue of the operator and its backward.
//
// Callers of the gated delta rule usually prepare its inputs the same way: q and k
// L2-normalised per token and head, the log decay g = logsigmoid(a) of a raw gate logit,
// beta = sigmoid(b) of a raw logit.  With gdr_problem.prologue bits set, the operator
// takes the raw tensors and applies these maps itself (forward: into workspace regions
// that the operator's kernels then read in place of q, k, g, beta), and maps the
// gradients back (backward: in place on dq, dk, dg, dbeta, after everything else):
//
//   q_hat = q s,  s = (sum q^2 + 1e-6)^(-1/2)      dq = s (dq_hat - q_hat <q_hat, dq_hat>)
//   g = logsigmoid(a)                               da = dg * sigmoid(-a)
//   beta = sigmoid(b)                               db = dbeta * beta (1 - beta)
//
// Memory-bound elementwise work: one warp per q/k row (one vector access per lane),
// grid-stride loops.
// Sums run in a fixed order (xor butterfly, then lane 0's value is broadcast), so every
// element of a row uses the same scale and results are bitwise reproducible.
#include <cuda_bf16.h>

#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr float kNormEps = 1e-6f;
constexpr int kThreads = 256;

__device__ __forceinline__ float ldv(const float* p) { return *p; }
__device__ __forceinline__ float ldv(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stv(float* p, float x) { *p = x; }
__device__ __forceinline__ void stv(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float row_sum(float x) {  // same value in every lane
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return __shfl_sync(0xffffffffu, x, 0);
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.f / (1.f + expf(-x)); }
__device__ __forceinline__ float logsigmoidf_(float x) { return fminf(x, 0.f) - log1pf(expf(-fabsf(x))); }

// Four consecutive elements (one vector access: 8 bytes of bf16, 16 of fp32).
__device__ __forceinline__ void ld4(const float* p, float* v) {
  const float4 x = *reinterpret_cast<const float4*>(p);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
__device__ __forceinline__ void ld4(const __nv_bfloat16* p, float* v) {
  const uint2 x = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
__device__ __forceinline__ void st4(float* p, const float* v) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void st4(__nv_bfloat16* p, const float* v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
  uint2 x;
  x.x = *reinterpret_cast<uint32_t*>(&a);
  x.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = x;
}

// Rows per warp per step: their loads are all issued before the first reduction, so
// enough bytes are in flight to cover the memory latency.
constexpr int kRows = 4;

// x, y: [rows][D] with D a multiple of 16, at most 128: lane l holds columns 4l .. 4l + 3
// (one vector access per lane per row).  blockIdx.y selects the tensor (q or k).
template <typename IT>
__global__ void __launch_bounds__(kThreads) l2norm_fwd_kernel(const IT* __restrict__ x0, IT* __restrict__ y0,
                                                              const IT* __restrict__ x1, IT* __restrict__ y1,
                                                              long long rows, int D) {
  const IT* x = blockIdx.y ? x1 : x0;
  IT* y = blockIdx.y ? y1 : y0;
  const int lane = threadIdx.x & 31, c = 4 * lane;
  const long long step = (((long long)gridDim.x * blockDim.x) >> 5) * kRows;
  for (long long r0 = (((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * kRows; r0 < rows; r0 += step) {
    float v[kRows][4];
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      v[j][0] = v[j][1] = v[j][2] = v[j][3] = 0.f;
      if (r0 + j < rows && c < D) ld4(x + (r0 + j) * D + c, v[j]);
    }
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      const float s =
          1.f / sqrtf(row_sum(v[j][0] * v[j][0] + v[j][1] * v[j][1] + v[j][2] * v[j][2] + v[j][3] * v[j][3]) +
                      kNormEps);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[j][i] *= s;
      if (r0 + j < rows && c < D) st4(y + (r0 + j) * D + c, v[j]);
    }
  }
}

// dx holds dL/dx_hat on entry and dL/dx on exit; x is the raw input.
template <typename IT>
__global__ void __launch_bounds__(kThreads) l2norm_bwd_kernel(const IT* __restrict__ x0, IT* __restrict__ dx0,
                                                              const IT* __restrict__ x1, IT* __restrict__ dx1,
                                                              long long rows, int D) {
  const IT* x = blockIdx.y ? x1 : x0;
  IT* dx = blockIdx.y ? dx1 : dx0;
  const int lane = threadIdx.x & 31, c = 4 * lane;
  const long long step = (((long long)gridDim.x * blockDim.x) >> 5) * kRows;
  for (long long r0 = (((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * kRows; r0 < rows; r0 += step) {
    float v[kRows][4], dv[kRows][4];
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      v[j][0] = v[j][1] = v[j][2] = v[j][3] = 0.f;
      dv[j][0] = dv[j][1] = dv[j][2] = dv[j][3] = 0.f;
      if (r0 + j < rows && c < D) {
        ld4(x + (r0 + j) * D + c, v[j]);
        ld4(dx + (r0 + j) * D + c, dv[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      const float s =
          1.f / sqrtf(row_sum(v[j][0] * v[j][0] + v[j][1] * v[j][1] + v[j][2] * v[j][2] + v[j][3] * v[j][3]) +
                      kNormEps);
      const float dot =
          row_sum(s * (v[j][0] * dv[j][0] + v[j][1] * dv[j][1] + v[j][2] * dv[j][2] + v[j][3] * dv[j][3]));
#pragma unroll
      for (int i = 0; i < 4; ++i) dv[j][i] = s * (dv[j][i] - v[j][i] * s * dot);
      if (r0 + j < rows && c < D) st4(dx + (r0 + j) * D + c, dv[j]);
    }
  }
}

template <typename IT>
__global__ void __launch_bounds__(kThreads) gates_fwd_kernel(const float* __restrict__ a, const IT* __restrict__ b,
                                                             float* __restrict__ gn, IT* __restrict__ bn,
                                                             long long n, int flags) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    if (flags & GDR_PROLOGUE_G_LOGSIGMOID) gn[i] = logsigmoidf_(a[i]);
    if (flags & GDR_PROLOGUE_BETA_SIGMOID) stv(bn + i, sigmoidf_(ldv(b + i)));
  }
}

template <typename IT>
__global__ void __launch_bounds__(kThreads) gates_bwd_kernel(const float* __restrict__ a, const IT* __restrict__ b,
                                                             float* __restrict__ dg, IT* __restrict__ dbeta,
                                                             long long n, int flags) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    if (flags & GDR_PROLOGUE_G_LOGSIGMOID) dg[i] *= sigmoidf_(-a[i]);
    if (flags & GDR_PROLOGUE_BETA_SIGMOID) {
      const float bt = sigmoidf_(ldv(b + i));
      stv(dbeta + i, ldv(dbeta + i) * bt * (1.f - bt));
    }
  }
}

// One warp per row (or per element group) while that stays under 2^20 blocks; the
// kernels' grid-stride loops cover anything larger.
unsigned grid_for(long long work, int per_block) {
  const long long g = (work + per_block - 1) / per_block;
  return (unsigned)(g < 1 ? 1 : (g > (1ll << 20) ? (1ll << 20) : g));
}

template <typename IT>
cudaError_t prologue_fwd_t(const Dims& d, const void* q, const void* k, const float* g, const void* beta,
                           const Workspace& ws, cudaStream_t s) {
  const long long qk_rows = d.T_total * d.Hk, n = d.T_total * d.Hv;
  if (d.prologue & GDR_PROLOGUE_QK_L2NORM) {
    const dim3 grid(grid_for(qk_rows, kThreads / 32 * kRows), 2);  // y: q, k
    l2norm_fwd_kernel<IT><<<grid, kThreads, 0, s>>>((const IT*)q, (IT*)ws.qn, (const IT*)k, (IT*)ws.kn, qk_rows,
                                                    d.DK);
    stage_mark(s, "prologue");
  }
  if (d.prologue & (GDR_PROLOGUE_G_LOGSIGMOID | GDR_PROLOGUE_BETA_SIGMOID)) {
    gates_fwd_kernel<IT><<<grid_for(n, kThreads), kThreads, 0, s>>>(g, (const IT*)beta, ws.gn, (IT*)ws.bn, n,
                                                                     d.prologue);
    stage_mark(s, "prologue");
  }
  return cudaGetLastError();
}

template <typename IT>
cudaError_t prologue_bwd_t(const Dims& d, const void* q, const void* k, const float* g, const void* beta, void* dq,
                           void* dk, float* dg, void* dbeta, cudaStream_t s) {
  const long long qk_rows = d.T_total * d.Hk, n = d.T_total * d.Hv;
  if (d.prologue & GDR_PROLOGUE_QK_L2NORM) {
    const dim3 grid(grid_for(qk_rows, kThreads / 32 * kRows), 2);  // y: q, k
    l2norm_bwd_kernel<IT><<<grid, kThreads, 0, s>>>((const IT*)q, (IT*)dq, (const IT*)k, (IT*)dk, qk_rows, d.DK);
    stage_mark(s, "prologue_bwd");
  }
  if (d.prologue & (GDR_PROLOGUE_G_LOGSIGMOID | GDR_PROLOGUE_BETA_SIGMOID)) {
    gates_bwd_kernel<IT><<<grid_for(n, kThreads), kThreads, 0, s>>>(g, (const IT*)beta, dg, (IT*)dbeta, n,
                                                                     d.prologue);
    stage_mark(s, "prologue_bwd");
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prologue_fwd(const Dims& d, const void* q, const void* k, const float* g, const void* beta,
                                const Workspace& ws, cudaStream_t s) {
  if (!d.prologue || d.T_total == 0) return cudaSuccess;
  return d.dtype == GDR_DTYPE_BF16 ? prologue_fwd_t<__nv_bfloat16>(d, q, k, g, beta, ws, s)
                                   : prologue_fwd_t<float>(d, q, k, g, beta, ws, s);
}

cudaError_t launch_prologue_bwd(const Dims& d, const void* q, const void* k, const float* g, const void* beta,
                                void* dq, void* dk, float* dg, void* dbeta, cudaStream_t s) {
  if (!d.prologue || d.T_total == 0) return cudaSuccess;
  return d.dtype == GDR_DTYPE_BF16 ? prologue_bwd_t<__nv_bfloat16>(d, q, k, g, beta, dq, dk, dg, dbeta, s)
                                   : prologue_bwd_t<float>(d, q, k, g, beta, dq, dk, dg, dbeta, s);
}

}  // namespace gdr
