// gdr_tc_selftest.cu -- a one-tile tcgen05 GEMM used to check, on the device, the
// operand layouts and descriptors (K-major / MN-major, 128-byte swizzle) and the
// TMEM read-back that the tensor-core kernels rely on.
//
//   D[m][n] = sum_k Amat[m][k] * Bmat[k][n],  M = 128, N in {64, 128}, K in {64, 128}
//   Amat[m][k] = A[m][k] (a_mn = 0, A given [128][K]) or A[k][m] (a_mn = 1, A given [K][128])
//   Bmat[k][n] = B[n][k] (b_mn = 0, B given [N][K])   or B[k][n] (b_mn = 1, B given [K][N])
#include "../../include/gdr_debug.h"
#include "gdr_internal.h"
#include "tc_primitives.cuh"

namespace gdr {
namespace {

__global__ void __launch_bounds__(128) tc_selftest_kernel(const __nv_bfloat16* __restrict__ A,
                                                          const __nv_bfloat16* __restrict__ B,
                                                          float* __restrict__ D, int N, int K, int a_mn, int b_mn,
                                                          uint32_t* status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* sA = smem;              // 32 KB
  unsigned char* sB = smem + 32768;      // 32 KB
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int M = 128;
  // stage A and B into the swizzled layouts
  for (int e = tid; e < M * K; e += 128) {
    int row, col;
    if (!a_mn) { row = e / K; col = e % K; }        // A[m][k]: rows m, cols k
    else { row = e / M; col = e % M; }             // A[k][m]: rows k, cols m
    const int rows = a_mn ? K : M;
    *(__nv_bfloat16*)(sA + tc::sw128_off(row, col, rows)) = A[e];
  }
  for (int e = tid; e < N * K; e += 128) {
    int row, col;
    if (!b_mn) { row = e / K; col = e % K; }        // B[n][k]
    else { row = e / N; col = e % N; }             // B[k][n]
    const int rows = b_mn ? K : N;
    *(__nv_bfloat16*)(sB + tc::sw128_off(row, col, rows)) = B[e];
  }
  tc::fence_proxy_async_smem();
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_barrier_init();
  }
  if (warp == 0) tc::tmem_alloc<128>(&tmem_slot);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tbase = tmem_slot;
  if (tid == 0) {
    const uint32_t idesc = tc::idesc_bf16(M, N, a_mn, b_mn);
    const uint32_t a_s = tc::smem_u32(sA), b_s = tc::smem_u32(sB);
    for (int kk = 0; kk < K / 16; ++kk) {
      const uint64_t ad = a_mn ? tc::mnmajor_step_desc(a_s, (uint32_t)K * 128u, kk)
                               : tc::kmajor_step_desc(a_s, (uint32_t)M * 128u, kk);
      const uint64_t bd = b_mn ? tc::mnmajor_step_desc(b_s, (uint32_t)K * 128u, kk)
                               : tc::kmajor_step_desc(b_s, (uint32_t)N * 128u, kk);
      tc::mma_bf16(tbase, ad, bd, idesc, kk > 0);
    }
    tc::mma_commit(&bar);
  }
  const bool ok = tc::mbar_wait(&bar, 0, status, kDevErrTimeoutFwd);
  tc::tc_fence_after();
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 32) {
      float v[32];
      tc::tmem_ld32(tc::tmem_lane_addr(tbase, warp, c0), v);
      tc::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) D[(size_t)tid * N + c0 + i] = v[i];
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, 128);
}

}  // namespace
}  // namespace gdr

extern "C" int gdr_debug_tc_gemm(const void* A, const void* B, float* D, int N, int K, int a_mn, int b_mn,
                                 unsigned int* status, void* stream) {
  if ((N != 64 && N != 128) || (K != 64 && K != 128)) return 1;
  const size_t smem = 65536 + 1024;
  cudaFuncSetAttribute(gdr::tc_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  gdr::tc_selftest_kernel<<<1, 128, smem, (cudaStream_t)stream>>>((const __nv_bfloat16*)A,
                                                                  (const __nv_bfloat16*)B, D, N, K, a_mn, b_mn,
                                                                  (uint32_t*)status);
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

namespace gdr {
namespace {

// A wait that can never complete (the mbarrier expects one arrival that nobody makes),
// bounded by limit_ns: the kernel must give up, record the timeout bit and return.
__global__ void tc_timeout_selftest_kernel(uint32_t* status, unsigned long long limit_ns,
                                           unsigned long long* waited_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  const uint64_t t0 = tc::globaltimer_ns();
  bool done = false;
  while (!(done = tc::mbar_try_wait(&bar, 0))) {
    if (tc::globaltimer_ns() - t0 > limit_ns) break;
  }
  if (!done && threadIdx.x == 0) {
    atomicOr(status, kDevErrTimeoutFwd);
    *waited_ns = tc::globaltimer_ns() - t0;
  }
}

}  // namespace
}  // namespace gdr

extern "C" int gdr_debug_timeout_selftest(unsigned int* status, unsigned long long limit_ns,
                                          unsigned long long* waited_ns, void* stream) {
  if (limit_ns > 1000000000ull) return 1;  // at most 1 s
  gdr::tc_timeout_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint32_t*)status, limit_ns, waited_ns);
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}
