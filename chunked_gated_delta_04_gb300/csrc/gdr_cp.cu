// gdr_cp.cu -- the scan between the two passes of intra-card context parallelism.
//
// FlashQLA PR #34 ("Current status") lists intra-card CP for the chunked gated delta rule.
// A sequence is cut at chunk boundaries into segments; every chunk maps the state affinely,
// h' = A_c h + b_c with A_c = e^{gamma_C} I - K~^T W, so a segment s maps its start state by
// h_end = Phi_s h_start + R_s (Phi_s the product of its A_c, R_s its end state from a zero
// start), and the reverse walk maps the state gradient by dh_start = Phi_s^T dh_end + E_s.
// The first pass of the state kernel (or of the walk) writes M[s] = Phi_s (or Phi_s^T, both
// stored transposed) and R[s] for every middle segment and the first boundary X; this kernel
// chains the boundaries
//   forward:  X[s + 1] = M[s] X[s] + R[s],  s = 1 .. nseg - 2   (X[s] = state at segment s's start)
//   backward: X[s - 1] = M[s] X[s] + R[s],  s = nseg - 2 .. 1   (X[s] = gradient at segment s's end)
// in fp32, and the second pass starts every segment from its X.
#include "gdr_device.cuh"
#include "gdr_internal.h"
#include "gdr_chunks.cuh"
#include "gdr_instrument.cuh"
#include "tc_primitives.cuh"

namespace gdr {

namespace {

constexpr int kScanThreads = 128;  // four warps, each over a quarter of the contraction
constexpr int kScanCols = 4;       // columns of X per CTA: the columns evolve independently
// shared memory: M of two segments (bulk copies, one segment ahead), the 128 x 4 slice of X, and
// the four warps' partial products
constexpr uint32_t kScanMBytes = 128 * 128 * 4;
constexpr uint32_t kScanSmem = 2 * kScanMBytes + 128 * kScanCols * 4 + 4 * 128 * kScanCols * 4;

// One CTA per (sequence, v-head, 4 columns of X).  The first pass stores M transposed
// (M^T[k][r] at k * 128 + r), so lane l of warp w reads rows 4 l .. 4 l + 3 of column k as one
// float4 (a warp reads 512 contiguous bytes per k) and X[k][0..3] as one broadcast float4, for
// k in [32 w, 32 w + 32); the four partial sums meet in shared memory, added in a fixed order
// (deterministic).  M of the next segment streams in (bulk copies completing on an mbarrier,
// bounded waits) while the current one is applied.
__global__ void __launch_bounds__(kScanThreads) cp_scan_kernel(Dims d, Workspace ws, int P, int backward) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  float* mbuf = reinterpret_cast<float*>(smem_raw);
  float* xs = reinterpret_cast<float*>(smem_raw + 2 * kScanMBytes);  // [128][4]
  float* part = xs + 128 * kScanCols;                                 // [4 warps][128][4]
  __shared__ uint64_t bar[2];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slice = (int)blockIdx.x % (128 / kScanCols), chain = (int)blockIdx.x / (128 / kScanCols);
  const int j = chain % d.Hv, n = chain / d.Hv;
  const int nseg = cp_segment(idx_seq_off(d, ws, n), idx_seq_off(d, ws, n + 1), P, 0).z;
  if (nseg < 3) return;  // at most one boundary: the first pass wrote it
  const int n_steps = nseg - 2;
  const uint32_t bit = backward ? kDevErrTimeoutBwd : kDevErrTimeoutFwd;
  const size_t base = ((size_t)n * d.Hv + j) * P * 16384;
  const int col0 = slice * kScanCols;
  const int s_first = backward ? nseg - 2 : 1, dir = backward ? -1 : 1;
  if (tid == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](int step) {  // M^T of step `step` into buffer step & 1 (thread 0)
    GDR_DELAY(30);
    const float* src = ws.cp_M + base + (size_t)(s_first + dir * step) * 16384;
    float* dst = mbuf + (step & 1) * 16384;
    tc::mbar_arrive_expect_tx(&bar[step & 1], kScanMBytes);
#pragma unroll
    for (int q = 0; q < 4; ++q) tc::bulk_load(dst + q * 4096, src + q * 4096, kScanMBytes / 4, &bar[step & 1]);
  };
  if (tid == 0) {
    issue(0);
    if (n_steps > 1) issue(1);
  }
  // the first boundary's slice: row tid
  *reinterpret_cast<float4*>(xs + tid * kScanCols) =
      *reinterpret_cast<const float4*>(ws.cp_X + base + (size_t)s_first * 16384 + (size_t)tid * 128 + col0);
  __syncthreads();
  int s = s_first;
  for (int step = 0; step < n_steps; ++step) {
    const float4 rv = __ldg(reinterpret_cast<const float4*>(ws.cp_R + base + (size_t)s * 16384 +
                                                            (size_t)tid * 128 + col0));
    if (!__syncthreads_and(tc::mbar_wait(&bar[step & 1], (step >> 1) & 1, ws.status, bit))) {
      // the status bit is set; the copies issued so far (steps `step` and `step + 1`) are given
      // another bounded wait before the block leaves, so none lands in freed shared memory
      if (tid == 0)
        for (int st2 = step; st2 < n_steps && st2 <= step + 1; ++st2)
          (void)tc::mbar_wait(&bar[st2 & 1], (st2 >> 1) & 1, ws.status, bit);
      __syncthreads();
      return;
    }
    const float* mt = mbuf + (step & 1) * 16384 + 4 * lane;
    float acc[4][4] = {};
#pragma unroll 8
    for (int k = 32 * warp; k < 32 * warp + 32; ++k) {
      const float4 m = *reinterpret_cast<const float4*>(mt + k * 128);  // rows 4 lane .. + 3 of column k
      const float4 x = *reinterpret_cast<const float4*>(xs + k * kScanCols);
      const float mr[4] = {m.x, m.y, m.z, m.w}, xr[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(mr[a], xr[c], acc[a][c]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
      *reinterpret_cast<float4*>(part + (warp * 128 + 4 * lane + a) * kScanCols) =
          make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    s += dir;
    tc::fence_proxy_async_smem();
    __syncthreads();  // every warp has read this M buffer and X, and written its partial sums
    if (tid == 0 && step + 2 < n_steps) issue(step + 2);
    float4 v = rv;  // row tid: R + the four quarters in order
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float4 p4 = *reinterpret_cast<const float4*>(part + (w * 128 + tid) * kScanCols);
      v.x += p4.x;
      v.y += p4.y;
      v.z += p4.z;
      v.w += p4.w;
    }
    if (warp == 1) GDR_DELAY(31);  // one warp's part of the next X late
    *reinterpret_cast<float4*>(xs + tid * kScanCols) = v;
    *reinterpret_cast<float4*>(ws.cp_X + base + (size_t)s * 16384 + (size_t)tid * 128 + col0) = v;
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_cp_scan(const Dims& d, const Workspace& ws, int P, bool backward, cudaStream_t s) {
  const long long ctas = (long long)d.num_seqs * d.Hv * (128 / kScanCols);
  if (ctas <= 0 || P < 3) return cudaSuccess;
  cudaError_t e = set_smem_once((const void*)cp_scan_kernel, kScanSmem);
  if (e != cudaSuccess) return e;
  cp_scan_kernel<<<(unsigned)ctas, kScanThreads, kScanSmem, s>>>(d, ws, P, backward ? 1 : 0);
  stage_mark(s, backward ? "bwd_cp_scan" : "fwd_cp_scan");
  return cudaGetLastError();
}

}  // namespace gdr
