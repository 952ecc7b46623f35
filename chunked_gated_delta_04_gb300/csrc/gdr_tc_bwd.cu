// gdr_tc_bwd.cu -- tcgen05 backward of the chunked gated delta rule (bf16, DK = DV = 128).
//
// The backward (the fused backward of FlashQLA PR #34, which walks the chunks in
// reverse carrying the state gradient dh) runs as three stages here:
//   prep   (gdr_tc.cu) W, U, P, gamma and T of every chunk, chunk-parallel.
//   walk   one CTA per (sequence, v-head, 64-wide DV slice), chunks in reverse; dh
//          (dL/dh at the chunk end, "dh'") stays in registers:
//            dVn = scale P^T dO + diag(e^{gamma_C - gamma}) K dh'
//            dh  = e^{gamma_C} dh' + scale Q^T diag(e^gamma) dO - W^T dVn
//          writes dh' and dVn of every chunk (bf16) and dS0.
//   grad   one CTA per (chunk, v-head), everything on chip, from Vn = U - W h (left in U's
//          place by the forward with saved chunk factors, else by tc_vn_kernel):
//            dP = scale (dO Vn^T) * Gam,
//            dq = scale diag(e^gamma) dO h^T + dP K,
//            dk = dP^T Q + diag(e^{gamma_C - gamma}) Vn dh'^T + ...,  dW = -dVn h^T,
//          then the WY backward through W = T' K, U = T'' V, T = (I + A)^{-1}:
//            dT = dW B_k^T + dVn B_v^T, dB_v = T^T dVn, dA = -strict-lower(T^T dT T^T),
//            <dB_k[s], k_s> = sum_m T[m][s] (dW K^T)[m][s],
//            dk += T'^T dW + diag(beta)(dA * Gam) K + (dA * Gam)^T diag(beta) K,
//          and dv, dbeta, dg (in-chunk reverse cumsum of d gamma).  dk stays in TMEM
//          from its first term to its last.
// No floating-point atomics anywhere: every reduction has a fixed order, so the
// backward is bitwise deterministic.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>

#include "gdr_internal.h"
#include "tc_common.cuh"
#include "tc_primitives.cuh"

namespace gdr {
namespace {

using namespace tcx;
using tc::kmaj;
using tc::mnmaj;

// 32 fp32 -> 32 bf16 in global memory (64 bytes, 16-byte aligned).
__device__ __forceinline__ void st_global_bf16x32(bf16* dst, const float* v) {
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
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

// ---------------------------------------------------------------------------------
// walk
// ---------------------------------------------------------------------------------
// NC = 64: a walk unit is one half of DV (two units per sequence and v-head, shorter
// epilogues: for chains that are the critical path).  NC = 128: one unit per sequence and
// v-head (half the SM time per chain: for batches whose gradients dominate).
template <int NC>
struct WalkSmem {
  // per stage: KQ 32 KB | W 16 KB | P 8 KB | dO (NC/64 slabs of 8 KB) | gamma 256 B (+pad)
  static constexpr uint32_t KQ = 0, W = 32768, P = 49152, DO = 57344;
  static constexpr uint32_t GAM = DO + (NC / 64) * 8192;
  static constexpr uint32_t STAGE = (GAM + 256 + 1023) / 1024 * 1024;
  static constexpr uint32_t DH = 2 * STAGE;              // dh' as bf16 B operand: NC/64 slabs of 128 rows x 128 B
  static constexpr uint32_t DVN = DH + (NC / 64) * 16384;  // dVn bf16 [64][NC]
  static constexpr uint32_t DOS = DVN + (NC / 64) * 8192;  // diag(e^gamma) dO bf16 [64][NC]
  // NC = 64: a second dVn tile (chunks alternate, so a store has a whole chunk to read its tile)
  static constexpr uint32_t DVN2 = DOS + (NC / 64) * 8192;
  static constexpr uint32_t BYTES = DVN2 + (NC == 64 ? 8192 : 0);
};

constexpr int kWalkThreads = 256;  // two warps per TMEM lane quarter, each on half of the slice's columns

// Counts one finished slice of a chunk: its TMA stores (async proxy) are complete; order them
// before the count (proxy fence) and publish it with a GPU-scope release reduction (pairs with
// the waiter's acquire load).  A full fence (__threadfence) before a relaxed add measured
// ~1.6k cycles per call on the walk's chain.
__device__ __forceinline__ void publish_chunk(uint32_t* flag) {
  asm volatile("fence.proxy.async.global;" ::: "memory");
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(flag) : "memory");
}

// Bounded wait until *flag >= target (acquire at GPU scope), then orders the caller's later
// TMA loads after it.  On expiry sets `bit` in *status and returns false.
__device__ __forceinline__ bool wait_flag(const uint32_t* flag, uint32_t target, uint32_t* status, uint32_t bit) {
  uint32_t v;
  const uint64_t t0 = tc::globaltimer_ns();
  while (true) {
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v >= target) break;
    if (tc::globaltimer_ns() - t0 > tc::kWaitLimitNs) {
      atomicOr(status, bit);
      return false;
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// One walk unit = (sequence, v-head, NC-wide DV slice); `unit` = (seq rank * Hv + v-head) *
// (128 / NC) + slice, sequences longest first.  tb: 4 NC TMEM columns owned by the caller.
// With kPublish the copy thread counts each chunk into ws.walk_flags[chunk * Hv + v-head] once
// its dh' and dVn tiles have fully reached memory (the fused walk + gradient kernel waits on it).
template <int NC, bool kPublish>
__device__ __forceinline__ void walk_body(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_w,
                                          const CUtensorMap& tm_p, const CUtensorMap& tm_do,
                                          const CUtensorMap& tm_dhs, const CUtensorMap& tm_dvs, const Dims& d,
                                          const float* __restrict__ dS_T, float* __restrict__ dS0,
                                          const Workspace& ws, int unit, uint32_t tb, unsigned char* sm) {
  using WS = WalkSmem<NC>;
  constexpr int kSl = 128 / NC;     // walk units per (sequence, v-head)
  constexpr int CPT = NC / 2;       // columns per thread: half hf of the slice
  constexpr int NSL = NC / 64;      // 64-column slabs of the slice
  __shared__ uint64_t bar_load[2], bar_mma;
  const int n = ws.seq_order[unit / (kSl * d.Hv)], j = (unit / kSl) % d.Hv, i = j / d.G;
  const int dv0 = (unit % kSl) * NC;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int hf = warp >> 2;            // column half [CPT hf, CPT hf + CPT) of the slice
  const int dk = tid & 127;            // TMEM lane = row of the dh' slice
  const int r = tid & 63;              // token row for the 64-row products (lanes 0-63)
  const bool lo = (warp & 3) < 2;      // warps on TMEM lanes 0-63
  // thread 0 issues the MMAs; thread 64 (the "copy thread", in a warp that has no part in
  // the dVn rows) issues every TMA load and store and waits on their bulk groups
  constexpr int kCopyTid = 64;
  const int Hv = d.Hv;
  const int c_begin = ws.seq_chunk_off[n], c_end = ws.seq_chunk_off[n + 1];
  const int t_seq = d.cu ? d.cu[n] : n * d.T;
  const int L = d.cu ? d.cu[n + 1] - t_seq : d.T;

  if (tid == 0) {
    tc::mbar_init(&bar_load[0], 1);
    tc::mbar_init(&bar_load[1], 1);
    tc::mbar_init(&bar_mma, 1);
    tc::fence_barrier_init();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  // TMEM: K dh' (0), P^T dO (NC), W^T dVn (2 NC), Q^T diag(e^gamma) dO (3 NC)
  const uint32_t Da = tb, Db = tb + NC, Dc = tb + 2 * NC, Dd = tb + 3 * NC;

  float dh[CPT];  // dL/dh at the end of the current chunk: row dk, columns dv0 + CPT hf + (0..CPT-1)
  {
    const size_t sb = ((size_t)n * Hv + j) * 128 * 128;
    const int c0 = dv0 + CPT * hf;
#pragma unroll
    for (int b = 0; b < CPT; ++b)
      dh[b] = dS_T ? dS_T[sb + (d.layout == 0 ? (size_t)dk * 128 + c0 + b : (size_t)(c0 + b) * 128 + dk)] : 0.f;
  }
  auto issue_loads = [&](int c, int st) {
    const int tc0 = t_seq + (c - c_begin) * 64;
    const size_t chh = (size_t)c * Hv + j;
    unsigned char* base = sm + st * WS::STAGE;
    uint64_t* bar = &bar_load[st];
    tc::mbar_arrive_expect_tx(bar, (7 + NSL) * kSlab + 256);
    tc::bulk_load(base + WS::GAM, ws.gam + chh * 64, 256, bar);
    tc::tma_load_3d(base + WS::KQ, &tm_k, bar, 0, i, tc0);
    tc::tma_load_3d(base + WS::KQ + 2 * kSlab, &tm_k, bar, 64, i, tc0);
    tc::tma_load_3d(base + WS::KQ + kSlab, &tm_q, bar, 0, i, tc0);
    tc::tma_load_3d(base + WS::KQ + 3 * kSlab, &tm_q, bar, 64, i, tc0);
    tc::tma_load_2d(base + WS::W, &tm_w, bar, 0, (int)(chh * 64));
    tc::tma_load_2d(base + WS::W + kSlab, &tm_w, bar, 64, (int)(chh * 64));
    tc::tma_load_2d(base + WS::P, &tm_p, bar, 0, (int)(chh * 64));
#pragma unroll
    for (int sl = 0; sl < NSL; ++sl) tc::tma_load_3d(base + WS::DO + sl * kSlab, &tm_do, bar, dv0 + 64 * sl, j, tc0);
  };
  if (tid == kCopyTid && c_begin < c_end) issue_loads(c_end - 1, 0);

  bool ok = true;
  uint32_t mma_phase = 0;
  int prev1 = -1, prev2 = -1;  // kPublish: the last two chunks, whose stores may be in flight
  GDR_TRACE_INIT();
  // dh' as the B operand: slab CPT hf / 64 holds columns [64 s, 64 s + 64) of the slice; written
  // here for the first chunk and at the end of each chunk for the next
  auto stage_dh = [&]() {
    if constexpr (NC == 64)
      st_halfrow_bf16(sm + WS::DH, dk, hf, dh);
    else
      st_row_bf16(sm + WS::DH + hf * 16384, dk, dh);
    tc::fence_proxy_async_smem();
  };
  stage_dh();
  tc::tc_fence_before();
  __syncthreads();
  for (int it = 0; c_end - 1 - it >= c_begin && ok; ++it) {
    const int c = c_end - 1 - it, st = it & 1;
    const uint32_t ld_phase = (it >> 1) & 1;
    const int len = min(64, L - (c - c_begin) * 64);
    const size_t chh = (size_t)c * Hv + j;
    if (tid == kCopyTid) {  // dh' of this chunk -> workspace, straight from the operand tile
#pragma unroll
      for (int sl = 0; sl < NSL; ++sl) tc::tma_store_2d(&tm_dhs, sm + WS::DH + sl * 16384, dv0 + 64 * sl, (int)(chh * 128));
      tc::bulk_commit();
    }
    GDR_TRACE_MARK(3, 0);
    ok = __syncthreads_and(tc::mbar_wait(&bar_load[st], ld_phase, ws.status, kDevErrTimeoutBwd));
    GDR_TRACE_MARK(3, 1);
    unsigned char* stg = sm + st * WS::STAGE;
    const float* sgam = reinterpret_cast<const float*>(stg + WS::GAM);
    const float gC = sgam[len - 1], gr = sgam[r];
    // the dh'-dependent products first; Q^T diag(e^gamma) dO waits for its scaled operand
    if (ok && tid == 0) {
      tc::tc_fence_after();
      tc::gemm(Da, kmaj(stg + WS::KQ, 2 * kSlab), mnmaj(sm + WS::DH, 16384), NC, 8, false);  // K dh'
      tc::gemm(Db, mnmaj(stg + WS::P, kSlab), mnmaj(stg + WS::DO, kSlab), NC, 4, false);     // P^T dO
      tc::mma_commit(&bar_mma);
    }
    GDR_TRACE_MARK(3, 7);
    if (tid == kCopyTid && c - 1 >= c_begin) {  // overlaps the MMAs
      GDR_DELAY(10);
      issue_loads(c - 1, st ^ 1);
    }
    GDR_TRACE_MARK(3, 8);
    // NC = 64: this chunk's dVn tile was last stored two chunks ago (groups since: dh', dVn,
    // dh'); NC = 128: one tile, stored one chunk ago (group since: this chunk's dh')
    unsigned char* dvn_t = sm + ((NC == 64 && (it & 1)) ? WS::DVN2 : WS::DVN);
    if (tid == kCopyTid) {
      GDR_TRACE_CLK(tdv);
      if constexpr (NC == 64)
        tc::bulk_wait_read<3>();
      else
        tc::bulk_wait_read<1>();
      GDR_TRACE_SINCE(3, 20, tdv);
    }
    GDR_TRACE_MARK(3, 9);
    if (ok && warp >= 4) {  // diag(e^gamma) dO, zero past the chunk end: row r, half (tid >> 6) & 1
      const int h2 = (tid >> 6) & 1;
      const float e = r < len ? fexp(gr) : 0.f;
      if constexpr (NC == 64) {
        float x[32];
        ld_halfrow_bf16(stg + WS::DO, r, h2, x);
#pragma unroll
        for (int b = 0; b < 32; ++b) x[b] *= e;
        st_halfrow_bf16(sm + WS::DOS, r, h2, x);
      } else {
        float x[64];
        ld_row_bf16(stg + WS::DO + h2 * kSlab, r, x);
#pragma unroll
        for (int b = 0; b < 64; ++b) x[b] *= e;
        st_row_bf16(sm + WS::DOS + h2 * kSlab, r, x);
      }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (ok && tid == 0) {  // committed together with W^T dVn below
      tc::tc_fence_after();
      tc::gemm(Dd, mnmaj(stg + WS::KQ + kSlab, 2 * kSlab), mnmaj(sm + WS::DOS, kSlab), NC, 4,
               false);  // Q^T diag(e^gamma) dO
    }
    GDR_TRACE_MARK(3, 2);
    ok = __syncthreads_and(ok && tc::mbar_wait(&bar_mma, mma_phase, ws.status, kDevErrTimeoutBwd));
    mma_phase ^= 1;
    tc::tc_fence_after();
    GDR_TRACE_MARK(3, 3);
    // kPublish: the copy thread's warp has no part in the dVn rows, so it counts chunk c + 2 (the
    // stores of two chunks ago; bulk groups since: dh', dVn, dh') here, where most of the
    // ~1k-cycle GPU-scope release overlaps the epilogue instead of delaying the chunk's last
    // barrier.  (A standalone acq_rel fence in the earlier MMA-issue window, with only a relaxed
    // count here, measured ~1.9k cycles: slower.)
    if (kPublish && tid == kCopyTid && prev2 >= 0) {
      GDR_TRACE_CLK(tpw);
      tc::bulk_wait<3>();
      GDR_TRACE_SINCE(3, 22, tpw);
      GDR_TRACE_CLK(tpp);
      GDR_DELAY(11);
      publish_chunk(ws.walk_flags + (size_t)prev2 * Hv + j);
      GDR_TRACE_SINCE(3, 23, tpp);
    }
    if (ok && lo) {  // dVn = scale P^T dO + diag(e^{gamma_C - gamma}) K dh', row r, half hf
      if (warp == 1) GDR_DELAY(12);
      const float dec = fexp(gC - gr);
#pragma unroll 1
      for (int q = 0; q < CPT / 32; ++q) {  // 32 columns at a time: [CPT hf + 32 q, +32)
        float x[32], y[32];
        tc::tmem_ld32(tc::tmem_lane_addr(tb, warp, CPT * hf + 32 * q), x);
        tc::tmem_ld32(tc::tmem_lane_addr(tb, warp, NC + CPT * hf + 32 * q), y);
        tc::tmem_wait_ld();
#pragma unroll
        for (int b = 0; b < 32; ++b) y[b] = r < len ? d.scale * y[b] + dec * x[b] : 0.f;
        if constexpr (NC == 64)
          st_halfrow_bf16(dvn_t, r, hf, y);
        else
          st_halfrow_bf16(dvn_t + hf * kSlab, r, q, y);
      }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (ok && tid == 0) {
      GDR_DELAY(13);
      tc::tc_fence_after();
      tc::gemm(Dc, mnmaj(stg + WS::W, kSlab), mnmaj(dvn_t, kSlab), NC, 4, false);  // W^T dVn
      tc::mma_commit(&bar_mma);
    }
    if (ok && tid == kCopyTid) {
#pragma unroll
      for (int sl = 0; sl < NSL; ++sl) tc::tma_store_2d(&tm_dvs, dvn_t + sl * kSlab, dv0 + 64 * sl, (int)(chh * 64));
      tc::bulk_commit();
    }
    GDR_TRACE_MARK(3, 4);
    // this chunk's dh' store has left the operand tile (only the dVn group may still read):
    // the tile takes the next chunk's dh' right after the update below
    if (tid == kCopyTid) {
      GDR_TRACE_CLK(tdr);
      tc::bulk_wait_read<1>();
      GDR_TRACE_SINCE(3, 21, tdr);
    }
    ok = __syncthreads_and(ok && tc::mbar_wait(&bar_mma, mma_phase, ws.status, kDevErrTimeoutBwd));
    mma_phase ^= 1;
    tc::tc_fence_after();
    GDR_TRACE_MARK(3, 5);
    if (ok) {
      const float eC = fexp(gC);
#pragma unroll
      for (int q = 0; q < CPT / 32; ++q) {
        float x[32], y[32];
        tc::tmem_ld32(tc::tmem_lane_addr(tb, warp, 2 * NC + CPT * hf + 32 * q), x);
        tc::tmem_ld32(tc::tmem_lane_addr(tb, warp, 3 * NC + CPT * hf + 32 * q), y);
        tc::tmem_wait_ld();
#pragma unroll
        for (int b = 0; b < 32; ++b) dh[32 * q + b] = eC * dh[32 * q + b] + d.scale * y[b] - x[b];
      }
      stage_dh();  // the next chunk's dh' operand (one barrier for both)
    }
    if (tid == kCopyTid && kPublish) {
      prev2 = prev1;
      prev1 = c;
    }
    tc::tc_fence_before();
    __syncthreads();
    GDR_TRACE_MARK(3, 6);
  }
  if (tid == kCopyTid) {
    tc::bulk_wait_read<0>();  // smem sources read before exit
    if (kPublish && prev1 >= 0) {
      tc::bulk_wait<0>();
      if (prev2 >= 0) publish_chunk(ws.walk_flags + (size_t)prev2 * Hv + j);
      publish_chunk(ws.walk_flags + (size_t)prev1 * Hv + j);
    }
  }
  if (ok && dS0) {
    const size_t sb = ((size_t)n * Hv + j) * 128 * 128;
    const int c0 = dv0 + CPT * hf;
#pragma unroll
    for (int b = 0; b < CPT; ++b)
      dS0[sb + (d.layout == 0 ? (size_t)dk * 128 + c0 + b : (size_t)(c0 + b) * 128 + dk)] = dh[b];
  }
  tc::tc_fence_before();
  __syncthreads();
  if (tid == 0) {  // the next unit of this CTA initialises them again
    tc::mbar_inval(&bar_load[0]);
    tc::mbar_inval(&bar_load[1]);
    tc::mbar_inval(&bar_mma);
  }
}

template <int NC>
__global__ void __launch_bounds__(kWalkThreads) tc_bwd_walk_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_p,
    const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_dhs,
    const __grid_constant__ CUtensorMap tm_dvs, Dims d, const float* __restrict__ dS_T, float* __restrict__ dS0,
    Workspace ws) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = align1024(smem_raw);
  __shared__ uint32_t tmem_slot;
  if (threadIdx.x < 32) tc::tmem_alloc<4 * NC>(&tmem_slot);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  walk_body<NC, false>(tm_q, tm_k, tm_w, tm_p, tm_do, tm_dhs, tm_dvs, d, dS_T, dS0, ws, (int)blockIdx.x, tmem_slot,
                       sm);
  if (threadIdx.x < 32) tc::tmem_dealloc(tmem_slot, 4 * NC);
}

// ---------------------------------------------------------------------------------
// vn: Vn = U - W h of every (chunk, v-head), written over U.  The gradient kernels read Vn
// from U's place; with saved chunk factors the forward's state kernel leaves it there, with
// recomputed factors this kernel does, after the chunk prep.  Persistent, one CTA per SM.
// ---------------------------------------------------------------------------------
struct VnSmem {
  static constexpr uint32_t W = 0;       // W, two 64-column slabs; the M = 128 operand's unused
                                          // rows read the next 16 KB (U)
  static constexpr uint32_t U = 16384;   // U, two slabs
  static constexpr uint32_t H = 32768;   // h bf16: two slabs of [128 dk][64 dv]
  static constexpr uint32_t HF = 65536;  // h fp32 as landed: four slabs of [128][32]
  static constexpr uint32_t BYTES = HF + 65536;
};

__global__ void __launch_bounds__(kTcThreads) tc_vn_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                          const __grid_constant__ CUtensorMap tm_u,
                                                          const __grid_constant__ CUtensorMap tm_h, Dims d,
                                                          Workspace ws) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = align1024(smem_raw);
  using S = VnSmem;
  __shared__ uint64_t bar_tma, bar_mma;
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    tc::mbar_init(&bar_tma, 1);
    tc::mbar_init(&bar_mma, 1);
    tc::fence_barrier_init();
  }
  if (warp == 0) tc::tmem_alloc<128>(&tmem_slot);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tb = tmem_slot;
  const int Hv = d.Hv, n_items = d.max_chunks * Hv;
  bool ok = true;
  uint32_t par = 0;
  for (int w = (int)blockIdx.x; w < n_items && ok; w += (int)gridDim.x) {
    const int c = w / Hv, j = w % Hv;
    const int len = ws.chunks[c].z;
    if (len <= 0) continue;  // an empty chunk slot (uniform across the CTA)
    const size_t ch = (size_t)c * Hv + j;
    if (tid == 0) {
      tc::mbar_arrive_expect_tx(&bar_tma, (d.h_bf16 ? 8 : 12) * kSlab);
      tc::tma_load_2d(sm + S::W, &tm_w, &bar_tma, 0, (int)(ch * 64));
      tc::tma_load_2d(sm + S::W + kSlab, &tm_w, &bar_tma, 64, (int)(ch * 64));
      tc::tma_load_2d(sm + S::U, &tm_u, &bar_tma, 0, (int)(ch * 64));
      tc::tma_load_2d(sm + S::U + kSlab, &tm_u, &bar_tma, 64, (int)(ch * 64));
      for (int q4 = 0; q4 < 4; ++q4) {
        if (d.h_bf16)  // straight into the operand tile: rows (q4 & 1) * 64.., columns (q4 >> 1) * 64..
          tc::tma_load_2d(sm + S::H + (q4 >> 1) * 16384 + (q4 & 1) * kSlab, &tm_h, &bar_tma, (q4 >> 1) * 64,
                          (int)(ch * 128 + (q4 & 1) * 64));
        else  // 32 fp32 columns of all 128 rows
          tc::tma_load_2d(sm + S::HF + q4 * 16384, &tm_h, &bar_tma, q4 * 32, (int)(ch * 128));
      }
    }
    ok = __syncthreads_and(tc::mbar_wait(&bar_tma, par, ws.status, kDevErrTimeoutBwd));
    if (ok && !d.h_bf16) {  // h fp32 -> bf16 operand, row tid (128-byte-swizzled 32-column slabs)
      float hv[64];
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const unsigned char* src = sm + S::HF + (2 * hh + q) * 16384 + tid * 128;
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 f = *reinterpret_cast<const float4*>(src + (((c4 ^ (tid & 7)) & 7) << 4));
            hv[q * 32 + 4 * c4] = f.x;
            hv[q * 32 + 4 * c4 + 1] = f.y;
            hv[q * 32 + 4 * c4 + 2] = f.z;
            hv[q * 32 + 4 * c4 + 3] = f.w;
          }
        }
        st_row_bf16(sm + S::H + hh * 16384, tid, hv);
      }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (ok && tid == 0) {  // W h: rows 0-63 (lanes 0-63)
      tc::tc_fence_after();
      tc::gemm(tb, kmaj(sm + S::W, kSlab), mnmaj(sm + S::H, 16384), 128, 8, false);
      tc::mma_commit(&bar_mma);
    }
    ok = __syncthreads_and(ok && tc::mbar_wait(&bar_mma, par, ws.status, kDevErrTimeoutBwd));
    tc::tc_fence_after();
    if (ok && warp < 2) {  // row r = tid: Vn = U - W h, zero past the chunk end, over U's row
      const int r = tid;
      bf16* dst = reinterpret_cast<bf16*>(ws.U) + (ch * 64 + r) * 128;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        float x[64], u[64];
        tmem_ld64(tb, warp, 64 * hh, x);
        ld_row_bf16(sm + S::U + hh * kSlab, r, u);
#pragma unroll
        for (int b = 0; b < 64; ++b) u[b] = r < len ? u[b] - x[b] : 0.f;
        st_global_bf16x32(dst + 64 * hh, u);
        st_global_bf16x32(dst + 64 * hh + 32, u + 32);
      }
    }
    par ^= 1;
    tc::tc_fence_before();
    __syncthreads();  // the tiles and the accumulator are free for the next item
    tc::tc_fence_after();
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, 128);
}

// ---------------------------------------------------------------------------------
// grad: all gradients of one (chunk, v-head)
// ---------------------------------------------------------------------------------
// Shared memory (1024-aligned tiles; later users of a tile noted after the arrow).
struct GradSmem {
  static constexpr uint32_t KQ = 0;             // [K | Q] x 2 slabs (32 KB), to the end
  static constexpr uint32_t DO = 32768;         // dO (16 KB) -> dk staging
  // O-hat = scale diag(e^gamma) dO and dVn interleaved by 64-column slab (slab s of O-hat at
  // OD + 16 KB s, of dVn 8 KB after it), so [O-hat; dVn] is one 128-row K-major operand
  // (32 KB); O-hat -> V after the first product, dVn to the WY backward
  static constexpr uint32_t OD = 49152;
  static constexpr uint32_t DH = 81920;         // dh' (32 KB) -> dq staging
  static constexpr uint32_t H = 114688;         // h bf16 (32 KB) -> dP | dT | X | dAGb (8 KB each);
                                                //   h fp32 lands in H, H + 16 KB, VN and SCR
  static constexpr uint32_t VN = 147456;        // Vn~ (16 KB) -> T'
  static constexpr uint32_t W = 163840;         // Vn as loaded (16 KB) -> dv staging
  static constexpr uint32_t UT = 180224;        // dW (16 KB)
  static constexpr uint32_t SCR = 196608;       // fp32 [64][65] scratch for row/column sums
  static constexpr uint32_t GAM = SCR + 16640;  // gamma (256 B)
  static constexpr uint32_t BYTES = GAM + 256;
  static constexpr uint32_t OD_SLAB = 16384;    // slab stride of O-hat, dVn and V
  // V and T are fetched right after P2 into the O-hat slabs and the last 8 KB of H (T is
  // last read by the X T^T product, before dAGb is written there)
  static constexpr uint32_t OH = OD, DVN = OD + 8192, V = OD;
  static constexpr uint32_t T = H + 24576, DP = H, DT = H + 8192, XT = H + 16384, DAG = H + 24576;
  // fp32 h slab k (32 columns of 128 rows, 16 KB)
  static constexpr uint32_t hf32(int k) { return k < 3 ? H + (uint32_t)k * 16384 : SCR; }
  static constexpr uint32_t TP = VN, DQS = DH, DVS = W, DKS = DO, DW = UT;
};

constexpr int kGradThreads = 256;  // two warps per TMEM lane quarter, each on half the columns

// kGroup: Hv > Hk; dq, dk are summed over the v-heads of a q/k head.  kPair (Hv = 2 Hk,
// launched as clusters of two CTAs): the two CTAs of a cluster take the two v-heads of one
// q/k head on the same chunk, and each finalises half of the dq and dk columns, adding the
// partner's partial sent through distributed shared memory (no fp32 partials in HBM and
// no separate reduction).  Otherwise (kGroup alone) fp32 partials go to the workspace and
// launch_group_reduce sums them.
// kDyn (fused walk + gradient kernel): items are claimed from ws.grad_queue in the order the
// walk finishes them (last chunk of every sequence first), and a chunk's dh' and dVn
// tiles are loaded only once both walk slices have counted it in ws.walk_flags.
// tb: 512 TMEM columns owned by the caller.
template <bool kGroup, bool kPair, bool kDyn>
__device__ __forceinline__ void grad_body(
    const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v, const CUtensorMap& tm_do,
    const CUtensorMap& tm_w, const CUtensorMap& tm_u, const CUtensorMap& tm_dvn, const CUtensorMap& tm_dh,
    const CUtensorMap& tm_h, const CUtensorMap& tm_t, const CUtensorMap& tm_dq, const CUtensorMap& tm_dk,
    const CUtensorMap& tm_dv, const Dims& d, const bf16* __restrict__ beta, bf16* __restrict__ dq,
    bf16* __restrict__ dk, bf16* __restrict__ dv, float* __restrict__ dg, bf16* __restrict__ dbeta,
    const Workspace& ws, uint32_t tb, unsigned char* sm) {
  __shared__ uint64_t bar_tma, bar_tma2, bar_mma;
  __shared__ uint64_t bar_qfree, bar_qdata, bar_kfree, bar_kdata;  // pair exchange (kPair)
  __shared__ int s_claim, s_claim_c;                               // kDyn: the next item, its chunk
  __shared__ float s_beta[64], s_eg[64], s_dgam[64], s_red[8];
  // column sums of 64 x 64 fp32 products in scratch, as four partial sums over 16 rows each
  // (all 256 threads: column tid & 63, rows 16 (tid >> 6) ..), added where they are used
  __shared__ float s_colpp[4][64], s_colbk[4][64], s_colaa[4][64];
  // per-row partial sums of the two column halves: [half][row]
  __shared__ float s_qh[2][64], s_rowpp[2][64], s_kdv[2][64], s_dbv[2][64], s_akk[2][64], s_rowaa[2][64];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, hf = warp >> 2;  // TMEM lane quarter, column half
  const bool lo = quarter < 2;                    // lanes 0-63 (rows of the 64-row products)
  const int r = (quarter & 1) * 32 + lane;        // row within the lane half
  // thread 0 issues the MMAs; thread 64 (the "copy thread", in warp 2, which has no part
  // in the 64-row epilogues) issues every TMA load and store and waits on the bulk groups
  constexpr int kCopyTid = 64;
  const int Hv = d.Hv;
  using S = GradSmem;

  const uint32_t rank = kPair ? tc::cluster_ctarank() : 0u, peer = rank ^ 1u;
  if (tid == 0) {
    tc::mbar_init(&bar_tma, 1);
    tc::mbar_init(&bar_tma2, 1);
    tc::mbar_init(&bar_mma, 1);
    if (kPair) {
      tc::mbar_init(&bar_qfree, 1);
      tc::mbar_init(&bar_qdata, 1);
      tc::mbar_init(&bar_kfree, 1);
      tc::mbar_init(&bar_kdata, 1);
    }
    tc::fence_barrier_init();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (kPair) tc::cluster_sync();  // the partner's barriers exist before anyone arrives on them
  // TMEM columns: [K K^T ; Q K^T] 0-63 (K K^T kept to the end); dq 256-383; dk 384-511.
  const uint32_t C_KK = tb, C_DQ = tb + 256, C_DK = tb + 384;
  GDR_TRACE_INIT();
  // Persistent: each CTA walks the (chunk, v-head) items w = blockIdx.x + k * gridDim.x,
  // keeping its barriers, TMEM and (warm) instruction cache across items.  The next
  // item's tiles are fetched as soon as the current item is done with their buffers
  // (dh' and dVn after R2, W after R3, K/Q, U, h and gamma after R4, dO after the dk
  // store), all on the next phase of bar_tma, so the loads overlap the current item.
  bool ok = true;
  uint32_t item_par = 0;  // phase parity of bar_tma / bar_tma2 for the current item
  uint32_t mma_par = 0;   // phase parity of bar_mma (five commits per item: it alternates)
  // items: (chunk, v-head), or with kPair (chunk, q/k head) shared by the cluster, whose
  // CTA `rank` takes v-head 2 i + rank; with kDyn every real chunk's v-heads, in walk order
  const int n_steps = kDyn ? ws.step_off[d.max_chunks + 1] : 0;
  const int n_items = kDyn ? ws.step_off[n_steps] * Hv : (kPair ? d.max_chunks * d.Hk : d.max_chunks * Hv);
  const int item0 = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int istep = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  // kDyn: item w = q * Hv + v-head, queue position q in walk order (the index kernel lists
  // each position's chunk)
  auto chunk_of = [&](int w) {
    if (kDyn) return ws.grad_chunk[w / Hv];
    return kPair ? w / d.Hk : w / Hv;
  };
  auto vhead_of = [&](int w) { return kPair ? (w % d.Hk) * 2 + (int)rank : w % Hv; };
  auto next_item = [&](int w) {  // next non-empty item of this CTA after w (or n_items)
    for (w += istep; w < n_items && ws.chunks[chunk_of(w)].z <= 0; w += istep) {
    }
    return w < n_items ? w : n_items;
  };
  int cur_len = 0, cur_t0 = 0, cur_i = 0;  // the current item (for pair_reduce)
  enum : int { kLdDhDvn = 1, kLdW = 2, kLdRest = 4, kLdDo = 8, kLdAll = 15 };
  auto issue_loads = [&](int w, int c2, int groups) {  // copy thread only; c2 = chunk_of(w)
    GDR_DELAY(20);
    const int j2 = vhead_of(w), i2 = j2 / d.G, tt = ws.chunks[c2].y;
    const size_t ch2 = (size_t)c2 * Hv + j2;
    uint64_t* bar = &bar_tma;
    if (groups & kLdDhDvn) {  // the first group of an item sets the whole item's byte count
      // kDyn: dh' and dVn of this chunk come from the walk running in the same kernel; on a
      // timeout the loads are left out and the item's own bounded wait ends the walk
      GDR_TRACE_CLK(tw0);
      const unsigned long long tf0_ = GDR_TRACE_NOW();
      if (kDyn && !wait_flag(ws.walk_flags + ch2, (uint32_t)d.walk_units, ws.status, kDevErrTimeoutBwd)) return;
      GDR_TRACE_INFO_ADD(4, GDR_TRACE_NOW() - tf0_);
      GDR_TRACE_SINCE(2, 20, tw0);
      tc::mbar_arrive_expect_tx(bar, (d.h_bf16 ? 18 : 22) * kSlab + 256);
      for (int q4 = 0; q4 < 4; ++q4)  // dh' rows (q4 & 1) * 64.., columns (q4 >> 1) * 64..
        tc::tma_load_2d(sm + S::DH + (q4 >> 1) * 16384 + (q4 & 1) * kSlab, &tm_dh, bar, (q4 >> 1) * 64,
                        (int)(ch2 * 128 + (q4 & 1) * 64));
      tc::tma_load_2d(sm + S::DVN, &tm_dvn, bar, 0, (int)(ch2 * 64));
      tc::tma_load_2d(sm + S::DVN + S::OD_SLAB, &tm_dvn, bar, 64, (int)(ch2 * 64));
    }
    if (groups & kLdW) {  // Vn (in U's place in memory) into W's tile, once the dv store has read it
      tc::tma_load_2d(sm + S::W, &tm_u, bar, 0, (int)(ch2 * 64));
      tc::tma_load_2d(sm + S::W + kSlab, &tm_u, bar, 64, (int)(ch2 * 64));
    }
    if (groups & kLdRest) {
      tc::bulk_load(sm + S::GAM, ws.gam + ch2 * 64, 256, bar);
      tc::tma_load_3d(sm + S::KQ, &tm_k, bar, 0, i2, tt);
      tc::tma_load_3d(sm + S::KQ + 2 * kSlab, &tm_k, bar, 64, i2, tt);
      tc::tma_load_3d(sm + S::KQ + kSlab, &tm_q, bar, 0, i2, tt);
      tc::tma_load_3d(sm + S::KQ + 3 * kSlab, &tm_q, bar, 64, i2, tt);
      if (d.h_bf16) {  // h (bf16) straight into its operand tile, laid out like dh'
        for (int q4 = 0; q4 < 4; ++q4)
          tc::tma_load_2d(sm + S::H + (q4 >> 1) * 16384 + (q4 & 1) * kSlab, &tm_h, bar, (q4 >> 1) * 64,
                          (int)(ch2 * 128 + (q4 & 1) * 64));
      } else {  // h (fp32) as four 32-column slabs of 128 rows, converted into H
        for (int q4 = 0; q4 < 4; ++q4)
          tc::tma_load_2d(sm + S::hf32(q4), &tm_h, bar, q4 * 32, (int)(ch2 * 128));
      }
    }
    if (groups & kLdDo) {
      tc::tma_load_3d(sm + S::DO, &tm_do, bar, 0, j2, tt);
      tc::tma_load_3d(sm + S::DO + kSlab, &tm_do, bar, 64, j2, tt);
    }
  };
  // kPair: combine one 64 x 128 fp32 result (dq or dk, TMEM columns col..col+127) of the two
  // CTAs.  This CTA finalises columns [64 rank, +64): the lo threads of the other half (hf !=
  // rank) stream their 64 columns of row r into the partner's receive tile `buf` with st.async
  // (each 16-byte piece completes 16 bytes on the partner's bar_data), once the partner has
  // said the tile is free; the lo threads of this half wait for the partner's 16 KB, add and
  // write bf16.  buf is [64][64] fp32 with the 16-byte pieces of row r rotated by (r & 15).
  // Every thread calls it; all waits are bounded (and made warp-uniform: the loops hold
  // warp-collective TMEM loads).
  auto pair_reduce = [&](uint32_t col, uint32_t buf_off, uint64_t* bar_free, uint64_t* bar_data, bf16* out,
                         bool okin) {
    bool okw = true;
    if (tid == 0) tc::mbar_arrive_expect_tx(bar_data, 64 * 256);  // the partner's half for this item
    if (okin && lo && hf != (int)rank) {
      if (rank == 1u) GDR_DELAY(23);
      okw = __all_sync(0xffffffffu, tc::mbar_wait_cluster(bar_free, item_par, ws.status, kDevErrTimeoutBwd));
      const uint32_t dst = tc::mapa(tc::smem_u32(sm + buf_off), peer) + (uint32_t)r * 256u;
      const uint32_t cbar = tc::mapa(tc::smem_u32(bar_data), peer);
#pragma unroll 1
      for (int q2 = 0; q2 < 2 && okw; ++q2) {
        float x[32];
        tmem_ld32w(tb, warp, col + hf * 64 + 32 * q2, x);
#pragma unroll
        for (int p4 = 0; p4 < 8; ++p4)
          tc::st_async_cluster_f32x4(dst + (uint32_t)(((8 * q2 + p4) ^ (r & 15)) << 4), x[4 * p4], x[4 * p4 + 1],
                                     x[4 * p4 + 2], x[4 * p4 + 3], cbar);
      }
    }
    if (okin && lo && hf == (int)rank) {
      okw = __all_sync(0xffffffffu, tc::mbar_wait_cluster(bar_data, item_par, ws.status, kDevErrTimeoutBwd));
      const unsigned char* src = sm + buf_off + r * 256;
#pragma unroll 1
      for (int q2 = 0; q2 < 2 && okw; ++q2) {
        float x[32];
        tmem_ld32w(tb, warp, col + hf * 64 + 32 * q2, x);
#pragma unroll
        for (int p4 = 0; p4 < 8; ++p4) {
          const float4 t = *reinterpret_cast<const float4*>(src + (((8 * q2 + p4) ^ (r & 15)) << 4));
          x[4 * p4] += t.x;
          x[4 * p4 + 1] += t.y;
          x[4 * p4 + 2] += t.z;
          x[4 * p4 + 3] += t.w;
        }
        if (r < cur_len) st_global_bf16x32(out + ((size_t)(cur_t0 + r) * d.Hk + cur_i) * 128 + rank * 64 + 32 * q2, x);
      }
    }
    return (bool)__syncthreads_and(okin && okw);
  };
  // kDyn: the copy thread claims an item and decodes its chunk once; the other threads read
  // both from shared memory after a barrier.  Inside the item loop the claim is split so its
  // two dependent global round trips stay off the critical path: the counter is bumped at the
  // start of an item, the chunk fetched after P4, and the item published after R2.
  auto claim = [&]() {
    const int w = (int)atomicAdd(ws.grad_queue, 1u);
    s_claim = w;
    s_claim_c = w < n_items ? chunk_of(w) : 0;
  };
  int pre_w = n_items, pre_c = 0;  // kDyn, copy thread: the next item, claimed ahead
  int witem, cur_c = 0;
  if (kDyn) {
    if (tid == kCopyTid) claim();
    __syncthreads();
    witem = s_claim;
    cur_c = s_claim_c;
    __syncthreads();
  } else {
    witem = item0 < n_items && ws.chunks[chunk_of(item0)].z <= 0 ? next_item(item0) : item0;
  }
  if (tid == kCopyTid && witem < n_items) issue_loads(witem, kDyn ? cur_c : chunk_of(witem), kLdAll);
  int pending = witem < n_items ? 0 : -1;  // groups of the next item issued so far (-1: none expected)
  int cl_w = n_items, cl_c = 0;            // kDyn, copy thread: the claimed next item and its chunk
  while (witem < n_items && ok) {
  // the next item (kDyn: claimed at the first prefetch point, known to all after the item)
  const int wnext = kDyn ? n_items : next_item(witem);
  const int cnext = kDyn ? 0 : (wnext < n_items ? chunk_of(wnext) : 0);
  const int c = kDyn ? cur_c : chunk_of(witem), j = vhead_of(witem), i = j / d.G;
  const int4 ci = ws.chunks[c];
  const int len = ci.z, t0 = ci.y;
  cur_len = len;
  cur_t0 = t0;
  cur_i = i;
  const size_t ch = (size_t)c * Hv + j;
  if (kDyn && tid == kCopyTid) pre_w = (int)atomicAdd(ws.grad_queue, 1u);  // used after R2
  if (tid < 64) s_beta[tid] = tid < len ? __bfloat162float(beta[(size_t)(t0 + tid) * Hv + j]) : 0.f;
  ok = __syncthreads_and(tc::mbar_wait(&bar_tma, item_par, ws.status, kDevErrTimeoutBwd));
  pending = (kDyn || wnext < n_items) ? 0 : -1;  // kDyn: decided when the next item is claimed
  const float* sgam = reinterpret_cast<const float*>(sm + S::GAM);
  if (tid < 64) s_eg[tid] = fexp(sgam[tid]);
  const float gC = sgam[len - 1], gr = sgam[r];
  const float dec = fexp(gC - gr);
  GDR_TRACE_MARK(2, 0);

  // h: fp32 slabs (32 columns) -> bf16 operand slabs (64 columns) in place; thread = (row
  // tid & 127, column half tid >> 7).  bf16 slab s overwrites fp32 slab s, which only the
  // half-0 threads read before the barrier.  <dh', h> is accumulated on the way.
  // dot products below keep four partial sums (a quarter of one running sum's dependent adds)
  float hdh4[4] = {0.f, 0.f, 0.f, 0.f};
  if (d.h_bf16) {  // h arrived as bf16 operand slabs: only <dh', h>
    const int hrow = tid & 127, hh = tid >> 7;
    float hv[64], dv_[64];
    if (ok) {
      ld_row_bf16(sm + S::H + hh * 16384, hrow, hv);
      ld_row_bf16(sm + S::DH + hh * 16384, hrow, dv_);
#pragma unroll
      for (int b = 0; b < 64; ++b) hdh4[b & 3] += hv[b] * dv_[b];
    }
  } else {
    const int hrow = tid & 127, hh = tid >> 7;
    float hv[64], dv_[64];
    if (ok) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const unsigned char* src = sm + S::hf32(2 * hh + q) + hrow * 128;
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 f = *reinterpret_cast<const float4*>(src + (((c4 ^ (hrow & 7)) & 7) << 4));
          hv[q * 32 + 4 * c4] = f.x; hv[q * 32 + 4 * c4 + 1] = f.y;
          hv[q * 32 + 4 * c4 + 2] = f.z; hv[q * 32 + 4 * c4 + 3] = f.w;
        }
      }
      ld_row_bf16(sm + S::DH + hh * 16384, hrow, dv_);
#pragma unroll
      for (int b = 0; b < 64; ++b) hdh4[b & 3] += hv[b] * dv_[b];
    }
    __syncthreads();
    if (ok) st_row_bf16(sm + S::H + hh * 16384, hrow, hv);
  }
  float hdh = warp_sum((hdh4[0] + hdh4[1]) + (hdh4[2] + hdh4[3]));
  if (lane == 0) s_red[warp] = hdh;
  if (ok && lo) {  // half hf of row r
    float x[64];
    // O-hat = scale diag(e^gamma) dO, zero past the chunk end
    const float e = r < len ? d.scale * s_eg[r] : 0.f;
    ld_row_bf16(sm + S::DO + hf * kSlab, r, x);
#pragma unroll
    for (int b = 0; b < 64; ++b) x[b] *= e;
    st_row_bf16(sm + S::OH + hf * S::OD_SLAB, r, x);
    // Vn~ = diag(e^{gamma_C - gamma}) Vn (Vn arrives in W's tile) into VN's tile, which the fp32
    // h no longer occupies past the conversion's barrier
    ld_row_bf16(sm + S::W + hf * kSlab, r, x);
#pragma unroll
    for (int b = 0; b < 64; ++b) x[b] *= dec;
    st_row_bf16(sm + S::VN + hf * kSlab, r, x);
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  hdh = ((s_red[0] + s_red[1]) + (s_red[2] + s_red[3])) + ((s_red[4] + s_red[5]) + (s_red[6] + s_red[7]));
  GDR_TRACE_MARK(2, 1);
  // P2: [K;Q] K^T (0-63: K K^T on lanes 0-63, Q K^T on lanes 64-127), [O-hat; dVn] h^T
  // (256-383: lanes 0-63 start dq, lanes 64-127 are dVn h^T = -dW), dO Vn^T (64-127, lanes
  // 64-127: the operand's rows start one slab early) and dk = Vn~ dh'^T (384-511)
  if (ok && tid == 0) {
    tc::tc_fence_after();
    tc::gemm(C_KK, kmaj(sm + S::KQ, 2 * kSlab), kmaj(sm + S::KQ, 2 * kSlab), 64, 8, false);
    tc::gemm(C_DQ, kmaj(sm + S::OD, S::OD_SLAB), kmaj(sm + S::H, 16384), 128, 8, false);
    GDR_DELAY(22);
    tc::gemm(tb + 64, kmaj(sm + S::DO - kSlab, kSlab), kmaj(sm + S::W, kSlab), 64, 8, false);
    tc::gemm(C_DK, kmaj(sm + S::VN, kSlab), kmaj(sm + S::DH, 16384), 128, 8, false);
    tc::mma_commit(&bar_mma);
  }
  ok = __syncthreads_and(ok && tc::mbar_wait(&bar_mma, mma_par, ws.status, kDevErrTimeoutBwd));
  mma_par ^= 1;
  tc::tc_fence_after();
  GDR_TRACE_MARK(2, 2);
  if (ok && tid == kCopyTid) {  // O-hat and h are consumed: fetch V and T for the WY backward
    tc::mbar_arrive_expect_tx(&bar_tma2, 3 * kSlab);
    tc::tma_load_3d(sm + S::V, &tm_v, &bar_tma2, 0, j, t0);
    tc::tma_load_3d(sm + S::V + S::OD_SLAB, &tm_v, &bar_tma2, 64, j, t0);
    tc::tma_load_2d(sm + S::T, &tm_t, &bar_tma2, 0, (int)(ch * 64));
  }
  if (kDyn && tid == kCopyTid) pre_c = pre_w < n_items ? chunk_of(pre_w) : 0;  // used after R2
  if (kPair && tid == 0) {  // P2 was the last reader of DH and DO: the partner may fill them
    tc::mbar_arrive_cluster(tc::mapa(tc::smem_u32(&bar_qfree), peer));
    tc::mbar_arrive_cluster(tc::mapa(tc::smem_u32(&bar_kfree), peer));
  }
  float* scr = reinterpret_cast<float*>(sm + S::SCR);
  auto col_partial = [&](float (*dst)[64]) {
    const int cc = tid & 63, g = tid >> 6;
    const float* src = scr + g * 16 * 65 + cc;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int rr = 0; rr < 16; rr += 4) {
      a0 += src[rr * 65];
      a1 += src[(rr + 1) * 65];
      a2 += src[(rr + 2) * 65];
      a3 += src[(rr + 3) * 65];
    }
    dst[g][cc] = (a0 + a1) + (a2 + a3);
  };
  if (ok) {
    if (lo) {  // row r, columns [64 hf, +64): q_r . (O-hat h^T)[r] and k_r . (Vn~ dh'^T)[r]
      float x[64], u[64];
      tmem_ld64(tb, warp, 256 + hf * 64, x);                    // (O-hat h^T)[r]
      ld_row_bf16(sm + S::KQ + kSlab + hf * 2 * kSlab, r, u);  // q_r
      float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int b = 0; b < 64; ++b) a4[b & 3] += x[b] * u[b];
      s_qh[hf][r] = (a4[0] + a4[1]) + (a4[2] + a4[3]);
      tmem_ld64(tb, warp, 384 + hf * 64, x);                    // (Vn~ dh'^T)[r]
      ld_row_bf16(sm + S::KQ + hf * 2 * kSlab, r, u);           // k_r
      float k4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int b = 0; b < 64; ++b) k4[b & 3] += x[b] * u[b];
      s_kdv[hf][r] = (k4[0] + k4[1]) + (k4[2] + k4[3]);        // e^{gamma_C - gamma_r} k_r^T dh' vn_r
    } else {  // lanes 64-127, row r
      {         // -dW, columns [64 hf, +64), into U's tile (not loaded: Vn comes ready)
        float x[64];
        tmem_ld64(tb, warp, 256 + hf * 64, x);
#pragma unroll
        for (int b = 0; b < 64; ++b) x[b] = -x[b];
        st_row_bf16(sm + S::DW + hf * kSlab, r, x);
      }
      if (warp == 7) GDR_DELAY(21);
      // dP and dP * QK, columns [32 hf, +32)
      float x[32], qk[32];
      tmem_ld32w(tb, warp, 64 + 32 * hf, x);  // (dO Vn^T)[r]
      tmem_ld32w(tb, warp, 32 * hf, qk);      // (Q K^T)[r]
      float rowpp4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < 32; ++s) {
        const int sc = 32 * hf + s;
        const float dp = (sc <= r && r < len) ? d.scale * x[s] * fexp(gr - sgam[sc]) : 0.f;
        x[s] = dp;
        qk[s] *= dp;
        rowpp4[s & 3] += qk[s];
      }
#pragma unroll
      for (int s = 0; s < 32; ++s) scr[r * 65 + 32 * hf + s] = qk[s];
      st_halfrow_bf16(sm + S::DP, r, hf, x);  // dP (h no longer needed)
      s_rowpp[hf][r] = (rowpp4[0] + rowpp4[1]) + (rowpp4[2] + rowpp4[3]);
    }
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  GDR_TRACE_MARK(2, 3);
  if (ok) col_partial(s_colpp);  // column sums of dP * QK
  if (ok && tid < 64) {  // sum_s e^{gC - g_s} k_s^T dh' vn_s
    const float kdv = tid < len ? s_kdv[0][tid] + s_kdv[1][tid] : 0.f;
    s_kdv[0][tid] = kdv;
    const float part = warp_sum(kdv);
    if (lane == 0) s_red[warp] = part;
  }
  ok = __syncthreads_and(ok && tc::mbar_wait(&bar_tma2, item_par, ws.status, kDevErrTimeoutBwd));
  GDR_TRACE_MARK(2, 5);
  // P6: dq += dP K, dk += dP^T Q; on lanes 64-127 (operand rows shifted by one slab: [.; dW]
  // and [V; dVn]) dW K^T (64-127) and dVn V^T (128-191)
  if (ok && tid == 0) {
    tc::tc_fence_after();
    tc::gemm(C_DQ, kmaj(sm + S::DP, kSlab), mnmaj(sm + S::KQ, 2 * kSlab), 128, 4, true);
    tc::gemm(C_DK, mnmaj(sm + S::DP, kSlab), mnmaj(sm + S::KQ + kSlab, 2 * kSlab), 128, 4, true);
    tc::gemm(tb + 64, kmaj(sm + S::DW - kSlab, kSlab), kmaj(sm + S::KQ, 2 * kSlab), 64, 8, false);
    tc::gemm(tb + 128, kmaj(sm + S::OD, S::OD_SLAB), kmaj(sm + S::V, S::OD_SLAB), 64, 8, false);
    tc::mma_commit(&bar_mma);
  }
  ok = __syncthreads_and(ok && tc::mbar_wait(&bar_mma, mma_par, ws.status, kDevErrTimeoutBwd));
  mma_par ^= 1;
  tc::tc_fence_after();
  GDR_TRACE_MARK(2, 6);
  if (ok && !lo) {
    // lanes 64-127, row r: dT = dW B_k^T + dVn B_v^T = (dW K^T) diag(beta e^gamma) + (dVn V^T)
    // diag(beta); T * (dW K^T) for <dB_k[s], k_s> = sum_m T[m][s] (dW K^T)[m][s]; columns [32 hf, +32)
    float x[32], y[32], tr[32];
    tmem_ld32w(tb, warp, 64 + 32 * hf, x);
    tmem_ld32w(tb, warp, 128 + 32 * hf, y);
    ld_halfrow_bf16(sm + S::T, r, hf, tr);
#pragma unroll
    for (int s = 0; s < 32; ++s) {
      const int sc = 32 * hf + s;
      const float be = s_beta[sc] * s_eg[sc];
      scr[r * 65 + sc] = tr[s] * x[s];
      y[s] = (r < len && sc < len) ? be * x[s] + s_beta[sc] * y[s] : 0.f;
      tr[s] *= be;  // T' = T diag(beta e^gamma)
    }
    st_halfrow_bf16(sm + S::DT, r, hf, y);
    st_halfrow_bf16(sm + S::TP, r, hf, tr);
  }
  if (kPair) ok = pair_reduce(256, S::DH, &bar_qfree, &bar_qdata, dq, ok);  // dq; DH receives
  if (ok && lo) {
    if (!kPair) {  // dq columns [64 hf, +64) (final for one v-head per q/k head)
      float x[64];
      tmem_ld64(tb, warp, 256 + hf * 64, x);
      if (kGroup) {
        if (r < len) {
          float* dst = ws.dq_part + ((size_t)(t0 + r) * Hv + j) * 128 + hf * 64;
#pragma unroll
          for (int b = 0; b < 64; b += 4) *reinterpret_cast<float4*>(dst + b) = make_float4(x[b], x[b + 1], x[b + 2], x[b + 3]);
        }
      } else if (len == 64) {
        st_row_bf16(sm + S::DQS + hf * kSlab, r, x);
      } else if (r < len) {
        st_global_bf16x64(dq + ((size_t)(t0 + r) * d.Hk + i) * 128 + hf * 64, x);
      }
    }
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  if (ok) col_partial(s_colbk);
  GDR_TRACE_MARK(2, 7);
  // R2: T^T dVn = dB_v (128-255), X = T^T dT (64-127, lanes 64-127: T^T's M atoms start one
  // slab early)
  if (ok && tid == kCopyTid && !kGroup && len == 64) {
    tc::tma_store_3d(&tm_dq, sm + S::DQS, 0, i, t0);
    tc::tma_store_3d(&tm_dq, sm + S::DQS + kSlab, 64, i, t0);
    tc::bulk_commit();
  }
  if (ok && tid == 0) {
    tc::tc_fence_after();
    tc::gemm(tb + 128, mnmaj(sm + S::T, kSlab), mnmaj(sm + S::DVN, S::OD_SLAB), 128, 4, false);
    tc::gemm(tb + 64, mnmaj(sm + S::T - kSlab, kSlab), mnmaj(sm + S::DT, kSlab), 64, 4, false);
    tc::mma_commit(&bar_mma);
  }
  ok = __syncthreads_and(ok && tc::mbar_wait(&bar_mma, mma_par, ws.status, kDevErrTimeoutBwd));
  mma_par ^= 1;
  tc::tc_fence_after();
  if (ok && tid == kCopyTid && pending >= 0) {  // dVn is consumed, dq has left its staging tile
    GDR_TRACE_CLK(tb21);
    tc::bulk_wait_read<0>();
    GDR_TRACE_SINCE(2, 21, tb21);
    if (kDyn) {  // publish the item claimed ahead
      GDR_TRACE_CLK(tc24);
      s_claim = cl_w = pre_w;
      s_claim_c = cl_c = pre_c;
      GDR_TRACE_SINCE(2, 24, tc24);
      if (cl_w >= n_items) pending = -1;
    }
    if (pending >= 0) {
      issue_loads(kDyn ? cl_w : wnext, kDyn ? cl_c : cnext, kLdDhDvn);
      pending |= kLdDhDvn;
    }
  }
  GDR_TRACE_MARK(2, 8);
  if (ok && lo) {
    {  // dv = diag(beta) dB_v, columns [64 hf, +64)
      float x[64], y[64];
      const float br = s_beta[r];
      float dbv4[4] = {0.f, 0.f, 0.f, 0.f};
      tmem_ld64(tb, warp, 128 + hf * 64, x);  // dB_v[r]
      ld_row_bf16(sm + S::V + hf * S::OD_SLAB, r, y);
#pragma unroll
      for (int b = 0; b < 64; ++b) {
        dbv4[b & 3] += x[b] * y[b];
        x[b] *= br;
      }
      s_dbv[hf][r] = (dbv4[0] + dbv4[1]) + (dbv4[2] + dbv4[3]);
      if (len == 64)
        st_row_bf16(sm + S::DVS + hf * kSlab, r, x);
      else if (r < len)
        st_global_bf16x64(dv + ((size_t)(t0 + r) * Hv + j) * 128 + hf * 64, x);
    }
  }
  if (ok && !lo) {  // lanes 64-127 meanwhile: X = T^T dT, row r, columns [32 hf, +32)
    float x[32];
    tmem_ld32w(tb, warp, 64 + 32 * hf, x);
    st_halfrow_bf16(sm + S::XT, r, hf, x);
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  GDR_TRACE_MARK(2, 9);
  // R3: X T^T (64-127)
  if (ok && tid == kCopyTid && len == 64) {
    tc::tma_store_3d(&tm_dv, sm + S::DVS, 0, j, t0);
    tc::tma_store_3d(&tm_dv, sm + S::DVS + kSlab, 64, j, t0);
    tc::bulk_commit();
  }
  if (ok && tid == 0) {
    tc::tc_fence_after();
    tc::gemm(tb + 64, kmaj(sm + S::XT, kSlab), kmaj(sm + S::T, kSlab), 64, 4, false);
    tc::mma_commit(&bar_mma);
  }
  ok = __syncthreads_and(ok && tc::mbar_wait(&bar_mma, mma_par, ws.status, kDevErrTimeoutBwd));
  mma_par ^= 1;
  tc::tc_fence_after();
  if (ok && tid == kCopyTid && pending >= 0) {  // dv has left its staging tile (W)
    GDR_TRACE_CLK(tb22);
    tc::bulk_wait_read<0>();
    GDR_TRACE_SINCE(2, 22, tb22);
    issue_loads(kDyn ? cl_w : wnext, kDyn ? cl_c : cnext, kLdW);
    pending |= kLdW;
  }
  GDR_TRACE_MARK(2, 10);
  if (ok && lo) {  // columns [32 hf, +32)
    const float br = s_beta[r];
    float x[32], gs[32], kk[32], akk4[4] = {0.f, 0.f, 0.f, 0.f}, rowaa4[4] = {0.f, 0.f, 0.f, 0.f};
    tmem_ld32w(tb, warp, 64 + 32 * hf, x);   // (T^T dT T^T)[r]
    tmem_ld32w(tb, warp, 32 * hf, kk);       // K K^T row r
#pragma unroll
    for (int s = 0; s < 32; ++s) gs[s] = sgam[32 * hf + s];
#pragma unroll
    for (int s = 0; s < 32; ++s) {
      const int sc = 32 * hf + s;
      // exp(gamma_r - gamma_s) only below the diagonal: above it the exponent is
      // positive and can overflow, and 0 * inf would give NaN
      const float dag = (sc < r && r < len) ? -x[s] * fexp(gr - gs[s]) : 0.f;
      akk4[s & 3] += dag * kk[s];
      x[s] = br * dag;
      kk[s] *= x[s];  // dA * A with A = beta_r Gam K K^T
      rowaa4[s & 3] += kk[s];
    }
#pragma unroll
    for (int s = 0; s < 32; ++s) scr[r * 65 + 32 * hf + s] = kk[s];
    st_halfrow_bf16(sm + S::DAG, r, hf, x);
    s_akk[hf][r] = (akk4[0] + akk4[1]) + (akk4[2] + akk4[3]);
    s_rowaa[hf][r] = (rowaa4[0] + rowaa4[1]) + (rowaa4[2] + rowaa4[3]);
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  if (ok) col_partial(s_colaa);
  GDR_TRACE_MARK(2, 11);
  // R4: dk += T'^T dW + dAGb K + dAGb^T K
  if (ok && tid == 0) {
    tc::tc_fence_after();
    tc::gemm(C_DK, mnmaj(sm + S::TP, kSlab), mnmaj(sm + S::DW, kSlab), 128, 4, true);
    tc::gemm(C_DK, kmaj(sm + S::DAG, kSlab), mnmaj(sm + S::KQ, 2 * kSlab), 128, 4, true);
    tc::gemm(C_DK, mnmaj(sm + S::DAG, kSlab), mnmaj(sm + S::KQ, 2 * kSlab), 128, 4, true);
    tc::mma_commit(&bar_mma);
  }
  ok = __syncthreads_and(ok && tc::mbar_wait(&bar_mma, mma_par, ws.status, kDevErrTimeoutBwd));
  mma_par ^= 1;
  tc::tc_fence_after();
  if (ok && tid == kCopyTid && pending >= 0) {  // every operand tile but dO (dk staging) is free
    issue_loads(kDyn ? cl_w : wnext, kDyn ? cl_c : cnext, kLdRest);
    pending |= kLdRest;
  }
  GDR_TRACE_MARK(2, 12);
  if (kPair) ok = pair_reduce(384, S::DO, &bar_kfree, &bar_kdata, dk, ok);  // dk; DO receives
  if (ok && lo) {
    float x[64];
    if (!kPair) tmem_ld64(tb, warp, 384 + hf * 64, x);  // dk columns [64 hf, +64)
    if (kPair) {
    } else if (kGroup) {
      if (r < len) {
        float* dst = ws.dk_part + ((size_t)(t0 + r) * Hv + j) * 128 + hf * 64;
#pragma unroll
        for (int b = 0; b < 64; b += 4) *reinterpret_cast<float4*>(dst + b) = make_float4(x[b], x[b + 1], x[b + 2], x[b + 3]);
      }
    } else if (len == 64) {
      st_row_bf16(sm + S::DKS + hf * kSlab, r, x);
    } else if (r < len) {
      st_global_bf16x64(dk + ((size_t)(t0 + r) * d.Hk + i) * 128 + hf * 64, x);
    }
    if (hf == 0) {  // per-row scalars: dbeta and d gamma
      const float br = s_beta[r], eg = s_eg[r];
      const float akk = s_akk[0][r] + s_akk[1][r], dbv = s_dbv[0][r] + s_dbv[1][r];
      const float colbk = (s_colbk[0][r] + s_colbk[1][r]) + (s_colbk[2][r] + s_colbk[3][r]);
      const float colpp = (s_colpp[0][r] + s_colpp[1][r]) + (s_colpp[2][r] + s_colpp[3][r]);
      const float colaa = (s_colaa[0][r] + s_colaa[1][r]) + (s_colaa[2][r] + s_colaa[3][r]);
      if (r < len) dbeta[(size_t)(t0 + r) * Hv + j] = __float2bfloat16_rn(eg * colbk + dbv + akk);
      float dgm = 0.f;
      if (r < len) {
        dgm = (s_rowpp[0][r] + s_rowpp[1][r]) - colpp + (s_qh[0][r] + s_qh[1][r]) - s_kdv[0][r] +
              br * eg * colbk + (s_rowaa[0][r] + s_rowaa[1][r]) - colaa;
        if (r == len - 1) dgm += fexp(gC) * hdh + (s_red[0] + s_red[1]);
      }
      s_dgam[r] = dgm;
    }
  }
  tc::fence_proxy_async_smem();
  __syncthreads();
  if (ok && tid == kCopyTid && !kGroup && len == 64) {
    tc::tma_store_3d(&tm_dk, sm + S::DKS, 0, i, t0);
    tc::tma_store_3d(&tm_dk, sm + S::DKS + kSlab, 64, i, t0);
    tc::bulk_commit();
  }
  if (ok && tid < 64) {  // dg = in-chunk reverse cumsum of d gamma (rows >= len hold 0)
    float x = s_dgam[63 - tid];  // reversed order: prefix sums become suffix sums
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    s_colaa[0][tid] = x;  // s_colaa is free again: reuse it for the warp totals
  }
  __syncthreads();
  if (ok && tid < 64) {
    const int rr = 63 - tid;
    const float v = s_colaa[0][tid] + (tid >= 32 ? s_colaa[0][31] : 0.f);
    if (rr < len) dg[(size_t)(t0 + rr) * Hv + j] = v;
  }
  if (tid == kCopyTid) {
    GDR_TRACE_CLK(tb23);
    tc::bulk_wait_read<0>();  // staging tiles read before the next item's loads
    GDR_TRACE_SINCE(2, 23, tb23);
    if (ok && pending >= 0) {
      issue_loads(kDyn ? cl_w : wnext, kDyn ? cl_c : cnext, kLdDo);
      pending |= kLdDo;
    }
  }
  GDR_TRACE_MARK(2, 13);
  GDR_TRACE_COUNT(2, 31);
  if (tid == 0) GDR_TRACE_INFO_ADD(3, 1);
  item_par ^= 1;
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (kDyn) {  // claimed at this item's first prefetch point (if that ran: else ok is false)
    witem = ok ? s_claim : n_items;
    cur_c = s_claim_c;
  } else {
    witem = wnext;
  }
  }  // items
  // A failed wait ends the walk early: let the next item's loads that are already in
  // flight land (bounded) before the CTA gives up its shared memory.
  if (tid == kCopyTid && !ok && pending > 0) (void)tc::mbar_wait(&bar_tma, item_par, ws.status, kDevErrTimeoutBwd);
  tc::tc_fence_before();
  __syncthreads();
}

template <bool kGroup, bool kPair = false>
__global__ void __launch_bounds__(kGradThreads) tc_bwd_grad_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_u,
    const __grid_constant__ CUtensorMap tm_dvn, const __grid_constant__ CUtensorMap tm_dh,
    const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_t,
    const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
    const __grid_constant__ CUtensorMap tm_dv, Dims d, const bf16* __restrict__ beta, bf16* __restrict__ dq,
    bf16* __restrict__ dk, bf16* __restrict__ dv, float* __restrict__ dg, bf16* __restrict__ dbeta,
    Workspace ws) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = align1024(smem_raw);
  __shared__ uint32_t tmem_slot;
  if (threadIdx.x < 32) tc::tmem_alloc<512>(&tmem_slot);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  grad_body<kGroup, kPair, false>(tm_q, tm_k, tm_v, tm_do, tm_w, tm_u, tm_dvn, tm_dh, tm_h, tm_t, tm_dq, tm_dk,
                                  tm_dv, d, beta, dq, dk, dv, dg, dbeta, ws, tmem_slot, sm);
  if (threadIdx.x < 32) tc::tmem_dealloc(tmem_slot, 512);
  // no CTA of a pair leaves while its partner may still write into its shared memory
  if (kPair) tc::cluster_sync();
}

// The backward's reverse walk and its gradient kernel in one cooperative launch (every CTA
// resident, one per SM): CTAs first run walk units (64 at B=2, H=16, leaving the other SMs
// free), then every CTA claims gradient items in the order the walk completes chunks, so the
// gradients of late chunks overlap the walk of early ones.
template <bool kGroup, int NC>
__global__ void __launch_bounds__(kGradThreads) tc_bwd_walkgrad_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_u,
    const __grid_constant__ CUtensorMap tm_p, const __grid_constant__ CUtensorMap tm_dvn,
    const __grid_constant__ CUtensorMap tm_dh, const __grid_constant__ CUtensorMap tm_dhs,
    const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_t,
    const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
    const __grid_constant__ CUtensorMap tm_dv, Dims d, const float* __restrict__ dS_T, float* __restrict__ dS0,
    const bf16* __restrict__ beta, bf16* __restrict__ dq, bf16* __restrict__ dk, bf16* __restrict__ dv,
    float* __restrict__ dg, bf16* __restrict__ dbeta, Workspace ws) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = align1024(smem_raw);
  __shared__ uint32_t tmem_slot;
  if (threadIdx.x < 32) tc::tmem_alloc<512>(&tmem_slot);  // both roles' columns
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const int n_units = d.num_seqs * d.Hv * (128 / NC);
  if (threadIdx.x == 0) GDR_TRACE_INFO_SET(0, GDR_TRACE_NOW());
  for (int u = (int)blockIdx.x; u < n_units; u += (int)gridDim.x)
    walk_body<NC, true>(tm_q, tm_k, tm_w, tm_p, tm_do, tm_dhs, tm_dvn, d, dS_T, dS0, ws, u, tmem_slot, sm);
  if (threadIdx.x == 0) GDR_TRACE_INFO_SET(1, GDR_TRACE_NOW());
  grad_body<kGroup, false, true>(tm_q, tm_k, tm_v, tm_do, tm_w, tm_u, tm_dvn, tm_dh, tm_h, tm_t, tm_dq, tm_dk,
                                 tm_dv, d, beta, dq, dk, dv, dg, dbeta, ws, tmem_slot, sm);
  if (threadIdx.x == 0) GDR_TRACE_INFO_SET(2, GDR_TRACE_NOW());
  if (threadIdx.x < 32) tc::tmem_dealloc(tmem_slot, 512);
}

}  // namespace

// Hv = 2 Hk on the tensor-core path: the gradient kernel runs as clusters of two CTAs that
// sum dq and dk on chip (no fp32 partials in the workspace).
bool grad_pair_mode(const Dims& d) { return d.path == 1 && d.G == 2; }

// Tensor-core backward (not the pair mode; at most kMaxFusedSeqs sequences, whose longest-first
// order the item queue needs): walk and gradients run as one cooperative kernel, see
// tc_bwd_walkgrad_kernel.
bool fused_walk_grad(const Dims& d) {
  return d.path == 1 && !grad_pair_mode(d) && d.num_seqs > 0 && d.num_seqs <= kMaxFusedSeqs && d.T_total > 0;
}

bool tc_bwd_available() { return get_encoder(); }

#ifdef GDR_TRACE
extern "C" int gdr_debug_cta_info_bwd(unsigned long long* out) {
  return cudaMemcpyFromSymbol(out, tcx::g_gdr_cta_info, sizeof(tcx::g_gdr_cta_info)) == cudaSuccess ? 0 : 1;
}
extern "C" int gdr_debug_trace_bwd(unsigned long long* out) {
  return cudaMemcpyFromSymbol(out, tcx::g_gdr_trace, sizeof(tcx::g_gdr_trace)) == cudaSuccess ? 0 : 1;
}
#endif

cudaError_t tc_backward(const Dims& d, const BwdArgs& a, const Workspace& ws, cudaStream_t s) {
  if (!get_encoder()) return cudaErrorNotSupported;
  const uint64_t Tt = (uint64_t)d.T_total;
  const uint64_t rows = (uint64_t)d.max_chunks * d.Hv * 64;
  if (Tt == 0 && d.num_seqs == 0) return cudaSuccess;
  // the chunk factors: recomputed, or (save_wy) kept by the forward in the saved buffer
  cudaError_t e = d.save_wy ? cudaSuccess : tc_launch_prep(d, a.q, a.k, a.v, a.g, a.beta, ws, 1, s, "bwd_prep");
  if (e != cudaSuccess) return e;
  CUtensorMap tq{}, tk{}, tv{}, tdo{}, tw{}, tp{}, tdvn{}, tdh{}, tt{}, tdhs{}, tu{}, tdq{}, tdk{}, tdv{}, thf{};
  if (Tt > 0) {  // with no tokens no kernel reads the maps (see tc_forward)
    if (!map_3d(&tq, a.q, 128, d.Hk, Tt) || !map_3d(&tk, a.k, 128, d.Hk, Tt) || !map_3d(&tv, a.v, 128, d.Hv, Tt) ||
        !map_3d(&tdo, a.dO, 128, d.Hv, Tt) || !map_2d(&tw, ws.W, 128, rows) || !map_2d(&tp, ws.P, 64, rows) ||
        !map_2d(&tdvn, ws.dVn, 128, rows) || !map_2d(&tdh, ws.dhp, 128, rows * 2) || !map_2d(&tt, ws.Tb, 64, rows) ||
        !map_2d_box(&tdhs, ws.dhp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 128, rows * 2, 64, 128) ||
        !map_2d(&tu, ws.U, 128, rows) || !map_3d(&tdq, a.dq, 128, d.Hk, Tt) || !map_3d(&tdk, a.dk, 128, d.Hk, Tt) ||
        !map_3d(&tdv, a.dv, 128, d.Hv, Tt) ||
        !(d.h_bf16 ? map_2d(&thf, a.h_saved, 128, rows * 2)
                   : map_2d_box(&thf, a.h_saved, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 128, rows * 2, 32, 128)))
      return cudaErrorInvalidValue;
  }
  int dev = 0, n_sm = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (!d.save_wy && d.max_chunks > 0 && Tt > 0) {  // recomputed factors: Vn over U (see tc_vn_kernel)
    const long long n_items = (long long)d.max_chunks * d.Hv;
    const size_t smv = VnSmem::BYTES + 1024;
    cudaFuncSetAttribute(tc_vn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smv);
    tc_vn_kernel<<<(unsigned)(n_items < n_sm ? n_items : n_sm), kTcThreads, smv, s>>>(tw, tu, thf, d, ws);
    stage_mark(s, "bwd_vn");
  }
  // Walk units per (sequence, v-head): the two DV halves (shorter epilogues, so a shorter
  // chain) while the walk units fill at most a quarter of the SMs, i.e. when there are so few
  // chains that the walk is the critical path; else one unit over all of DV, which takes half
  // the SM time per chain and leaves the SMs to the gradient items.
  Dims dd = d;
  dd.walk_units = (long long)d.num_seqs * d.Hv * 2 * 4 <= n_sm ? 2 : 1;
  const bool halves = dd.walk_units == 2;
  if (fused_walk_grad(d)) {  // walk and gradients in one cooperative kernel
    int per_sm = 0;
    const size_t smg =
        (halves ? std::max(GradSmem::BYTES, WalkSmem<64>::BYTES) : std::max(GradSmem::BYTES, WalkSmem<128>::BYTES)) +
        1024;
    auto kern = d.G > 1 ? (halves ? tc_bwd_walkgrad_kernel<true, 64> : tc_bwd_walkgrad_kernel<true, 128>)
                        : (halves ? tc_bwd_walkgrad_kernel<false, 64> : tc_bwd_walkgrad_kernel<false, 128>);
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smg);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGradThreads, smg) != cudaSuccess || per_sm < 1)
      return cudaErrorInvalidConfiguration;
    e = cudaMemsetAsync(ws.walk_flags, 0, sizeof(uint32_t) * ((size_t)d.max_chunks * d.Hv + 64), s);
    if (e != cudaSuccess) return e;
    const bf16* beta = (const bf16*)a.beta;
    bf16 *dq = (bf16*)a.dq, *dk = (bf16*)a.dk, *dv = (bf16*)a.dv, *dbeta = (bf16*)a.dbeta;
    const float* dS_T = a.dS_T;
    float *dS0 = a.dS0, *dg = a.dg;
    Workspace w = ws;
    void* args[] = {&tq, &tk, &tv, &tdo, &tw, &tu, &tp, &tdvn, &tdh, &tdhs, &thf, &tt, &tdq, &tdk, &tdv, &dd,
                    (void*)&dS_T, (void*)&dS0, (void*)&beta, (void*)&dq, (void*)&dk, (void*)&dv, (void*)&dg,
                    (void*)&dbeta, &w};
    e = cudaLaunchCooperativeKernel((const void*)kern, dim3((unsigned)(per_sm * n_sm)), dim3(kGradThreads), args, smg, s);
    if (e != cudaSuccess) return e;
    stage_mark(s, "bwd_walkgrad");
    if (d.G > 1) {
      e = launch_group_reduce(d, a.dq, a.dk, ws, s);
      if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
  }
  if (d.num_seqs > 0) {
    const size_t sm = (halves ? WalkSmem<64>::BYTES : WalkSmem<128>::BYTES) + 1024;
    auto kern = halves ? tc_bwd_walk_kernel<64> : tc_bwd_walk_kernel<128>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    kern<<<d.num_seqs * d.Hv * dd.walk_units, kWalkThreads, sm, s>>>(tq, tk, tw, tp, tdo, tdhs, tdvn, dd, a.dS_T,
                                                                    a.dS0, ws);
    stage_mark(s, "bwd_walk");
  }
  if (d.max_chunks > 0 && Tt > 0) {
    const long long n_items = (long long)d.max_chunks * d.Hv;
    const dim3 grid((unsigned)(n_items < n_sm ? n_items : n_sm));  // persistent: one CTA per SM
    const size_t smg = GradSmem::BYTES + 1024;
    if (grad_pair_mode(d)) {  // clusters of two CTAs, one per v-head of a q/k head
      auto kern = tc_bwd_grad_kernel<true, true>;
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smg);
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.blockDim = dim3(kGradThreads);
      cfg.dynamicSmemBytes = smg;
      cfg.stream = s;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      cfg.gridDim = dim3(2);
      int n_clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&n_clusters, kern, &cfg) != cudaSuccess || n_clusters < 1) n_clusters = 1;
      const long long pairs = (long long)d.max_chunks * d.Hk;
      cfg.gridDim = dim3(2u * (unsigned)(pairs < n_clusters ? pairs : n_clusters));  // persistent
#ifdef GDR_TRACE
      fprintf(stderr, "grad pair mode: %d co-resident clusters, grid %u\n", n_clusters, cfg.gridDim.x);
#endif
      e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tdo, tw, tu, tdvn, tdh, thf, tt, tdq, tdk, tdv, d,
                             (const bf16*)a.beta, (bf16*)a.dq, (bf16*)a.dk, (bf16*)a.dv, a.dg, (bf16*)a.dbeta, ws);
      if (e != cudaSuccess) return e;
    } else if (d.G > 1) {
      cudaFuncSetAttribute(tc_bwd_grad_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smg);
      tc_bwd_grad_kernel<true><<<grid, kGradThreads, smg, s>>>(tq, tk, tv, tdo, tw, tu, tdvn, tdh, thf, tt, tdq, tdk,
                                                              tdv, d, (const bf16*)a.beta, (bf16*)a.dq,
                                                              (bf16*)a.dk, (bf16*)a.dv, a.dg, (bf16*)a.dbeta, ws);
    } else {
      cudaFuncSetAttribute(tc_bwd_grad_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smg);
      tc_bwd_grad_kernel<false><<<grid, kGradThreads, smg, s>>>(tq, tk, tv, tdo, tw, tu, tdvn, tdh, thf, tt, tdq, tdk,
                                                               tdv, d, (const bf16*)a.beta, (bf16*)a.dq,
                                                               (bf16*)a.dk, (bf16*)a.dv, a.dg, (bf16*)a.dbeta, ws);
    }
    stage_mark(s, "bwd_grad");
    if (d.G > 1 && !grad_pair_mode(d)) {
      e = launch_group_reduce(d, a.dq, a.dk, ws, s);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaGetLastError();
}

}  // namespace gdr
