// gdr_tc_bwd.cu -- tcgen05 backward of the chunked gated delta rule (bf16, DK = DV = 128).
//
// The backward (the fused backward of FlashQLA PR #34, which walks the chunks in
// reverse carrying the state gradient dh) runs as three stages here:
//   prep   (gdr_tc.cu) W, U, P, gamma and T of every chunk, chunk-parallel.
//   walk   one CTA per (sequence, v-head), all of DK and DV, chunks in reverse; dh
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
#include "gdr_chunks.cuh"
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
// One walk unit = (sequence, v-head), all of DK and DV, chunks in reverse.  dh (dL/dh at the
// end of the current chunk, "dh'") stays in registers, fp32.  Per chunk, with
//   K^ = diag(e^{gamma_C - gamma} / scale) K,   Q^ = diag(scale e^gamma) Q
// formed in place in the chunk's shared-memory tiles (rows past the chunk end zero):
//   accV = P^T dO + K^ dh'             = dVn / scale  (64 tokens on TMEM lanes 0-63)
//   dVn  = scale accV, zero past the chunk end
//   accH = Q^^T dO - W^T dVn           (DK x DV; the minus is the MMA's negate-A bit)
//   dh   = e^{gamma_C} dh' + accH
// Roles (12 warps): warps 0-7 run the epilogues (dVn on the four warps of lanes 0-63, dh on
// all eight) and the four warps of lanes 64-127 form the next chunk's K^ and Q^ while the dVn
// epilogue runs; in the third warpgroup, warp 8 (lane 0) issues every MMA, warp 9 (lane 0)
// stores dh' and dVn of every chunk to the workspace and, with kPublish, counts each chunk
// into ws.walk_flags once its stores have landed, and warp 10 (lane 0) issues the TMA loads
// and L2 prefetches.  The roles hand off through mbarriers only.
// P^T dO and Q^^T dO do not need dh', so they run while the previous chunk's epilogues do: a
// chunk's chain is the 8 MMAs of K^ dh', the dVn epilogue, the 4 MMAs of W^T dVn and the dh
// epilogue.  Tiles are loaded one chunk ahead (two stages) after an L2 prefetch one chunk
// before that.
struct WalkSmem {
  // per stage: [K | Q] interleaved by 64-column slab (K rows 0-63 and, as the unused rows 64-127
  // of the M = 128 operand, Q) 32 KB | W 16 KB | dO 16 KB | P 8 KB | gamma 256 B
  static constexpr uint32_t KQ = 0, W = 32768, DO = 49152, P = 65536, GAM = 73728;
  static constexpr uint32_t STAGE = 74752;
  static constexpr uint32_t DH = 2 * STAGE;    // dh' bf16: two slabs of [128 dk][64 dv]
  static constexpr uint32_t DVN = DH + 32768;  // two dVn tiles (chunks alternate), [64 tokens][128 dv]
  static constexpr uint32_t BYTES = DVN + 2 * 16384;
};
static_assert(WalkSmem::GAM + 256 <= WalkSmem::STAGE && WalkSmem::STAGE % 1024 == 0, "walk stage layout");

// 8 epilogue warps, then one warpgroup of roles: MMA, store, load and a spare (setmaxnreg works
// on whole warpgroups, see tc_bwd_walkgrad_kernel)
constexpr int kWalkThreads = 384;
constexpr int kWalkMmaTid = 256;      // lane 0 of warp 8
constexpr int kWalkCopyTid = 288;     // lane 0 of warp 9
constexpr int kWalkLoadTid = 320;     // lane 0 of warp 10
constexpr uint32_t kWalkTmemCols = 512;  // accV x 2 at 0, accH x 2 at 256 (128 columns each)

// Counts one finished chunk: its TMA stores (async proxy) are complete; order them before the
// count (proxy fence) and publish it with a GPU-scope release reduction (pairs with the
// waiter's acquire load).  A full fence (__threadfence) before a relaxed add measured ~1.6k
// cycles per call.
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

// Bounded wait made uniform across the calling warp (every lane waits on the same barrier).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint32_t* status, uint32_t bit) {
  return __all_sync(0xffffffffu, tc::mbar_wait(bar, parity, status, bit));
}

// What one walk unit computes: a (sequence, v-head) walked backward over a range of its
// chunks, from the state gradient at the range's end to the one at its start.  Without
// segments the range is the whole sequence, from dS_T to dS0, and every chunk's dh' and dVn go
// to the workspace.  The context-parallel passes (CpArgs) cut it into segments:
//   first pass, per (sequence, v-head): the last segment from dS_T with its stores, its start
//     gradient into X[nseg - 2] (or dS0 when it is the only segment); and for each segment
//     s = 1 .. nseg - 2 its walk from a zero end gradient R[s] = E_s and its transposed
//     transition M[s] = Phi_s^T (the walk with dO = 0 from the identity: dh = A_c^T dh'), both
//     without stores;
//   second pass: segments s = 0 .. nseg - 2 from X[s] with their stores, segment 0 into dS0.
struct WalkUnit {
  int n, j;
  int c_begin, c_end;  // chunk range
  int t_seq, L;        // first token of the range, tokens from there to the sequence end
  const float* g0;     // gradient at the range's end (nullptr: zero) ...
  int g0_kv;           // ... stored [DK][DV] (else [DV][DK])
  bool g0_eye;         // the identity instead
  float* g1;           // gradient at the range's start (nullptr: not written), orientation g1_kv
  int g1_kv;
  bool stores;         // dh' and dVn of every chunk to the workspace
  bool zero_do;        // dO taken as zero (transition columns)
  bool skip;           // nothing to compute
};

__device__ __forceinline__ int walk_units_per_chain(const CpArgs& cp) {
  return cp.pass == 1 ? 1 + 2 * (cp.P - 2) : (cp.pass == 3 ? cp.P - 1 : 1);
}

// Unit `unit` of a walk launch: (sequence rank, v-head, unit within the chain), the last fastest.
__device__ __forceinline__ WalkUnit walk_unit(const Dims& d, const Workspace& ws, const CpArgs& cp, int unit,
                                              const float* dS_T, float* dS0) {
  WalkUnit u{};
  const int per = walk_units_per_chain(cp);
  const int k = unit % per, rest = unit / per;
  u.j = rest % d.Hv;
  u.n = idx_seq(d, ws, rest / d.Hv);
  const int s0 = idx_seq_off(d, ws, u.n), s1 = idx_seq_off(d, ws, u.n + 1);
  const int t_seq = d.cu ? d.cu[u.n] : u.n * d.T;
  const int L = d.cu ? d.cu[u.n + 1] - t_seq : d.T;
  const size_t sb = ((size_t)u.n * d.Hv + u.j) * 128 * 128;
  u.c_begin = s0;
  u.c_end = s1;
  u.t_seq = t_seq;
  u.L = L;
  u.g0 = dS_T ? dS_T + sb : nullptr;
  u.g0_kv = d.layout == 0;
  u.g1 = dS0 ? dS0 + sb : nullptr;
  u.g1_kv = d.layout == 0;
  u.stores = true;
  if (cp.pass == 0) return u;
  const int nseg = cp_segment(s0, s1, cp.P, 0).z;
  int seg, mode = 0;  // mode 0: true walk with stores; 1: zero end gradient; 2: transition
  if (cp.pass == 1) {
    seg = k == 0 ? nseg - 1 : 1 + (k - 1) / 2;
    mode = k == 0 ? 0 : 1 + ((k - 1) & 1);
  } else {
    seg = k;
  }
  const int3 sg = cp_segment(s0, s1, cp.P, seg);
  auto mat = [&](float* base, int s2) { return base + (sb * cp.P) + (size_t)s2 * 128 * 128; };
  u.c_begin = sg.x;
  u.c_end = sg.y;
  u.t_seq = t_seq + (sg.x - s0) * kChunk;
  u.L = L - (sg.x - s0) * kChunk;
  if (cp.pass == 1) {
    if (mode == 0) {
      if (nseg > 1) {
        u.g1 = mat(cp.X, nseg - 2);
        u.g1_kv = 1;
      }
    } else {
      u.skip = seg > nseg - 2;
      u.stores = false;
      u.g0 = nullptr;
      u.g0_eye = mode == 2;
      u.zero_do = mode == 2;
      u.g1 = mat(mode == 2 ? cp.M : cp.R, seg);
      u.g1_kv = mode == 2 ? 0 : 1;  // M transposed: the scan reads M^T[k][r] = M[r][k] as rows
    }
  } else {
    u.skip = seg > nseg - 2;
    u.g0 = mat(cp.X, seg);
    u.g0_kv = 1;
    if (seg != 0) u.g1 = nullptr;
  }
  return u;
}

// One walk unit (see WalkUnit).  tb: the caller's 512 TMEM columns.  Every thread of the CTA
// (kWalkThreads) calls it.  kModes: the unit may be a first-pass map (no stores, or dO = 0 from the
// identity); without it those cases are compiled out (true walks only, as the plain chain and
// the second pass run).
template <bool kPublish, bool kModes>
__device__ __forceinline__ void walk_body(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_w,
                                          const CUtensorMap& tm_p, const CUtensorMap& tm_do,
                                          const CUtensorMap& tm_dhs, const CUtensorMap& tm_dvs, const Dims& d,
                                          const Workspace& ws, const WalkUnit& un, uint32_t tb, unsigned char* sm) {
  using WS = WalkSmem;
  __shared__ uint64_t bar_load[2], bar_scaled[2], bar_vfull[2], bar_hfull[2], bar_dvn[2], bar_dvnfree[2];
  __shared__ uint64_t bar_dh, bar_dhfree, bar_drain;
  const int j = un.j, i = j / d.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hv = d.Hv;
  const int c_begin = un.c_begin, c_end = un.c_end;
  const int nch = c_end - c_begin;
  const int t_seq = un.t_seq;
  const int L = un.L;
  const bool stores = !kModes || un.stores, zero_do = kModes && un.zero_do, g0_eye = kModes && un.g0_eye;
  uint32_t* const status = ws.status;
  constexpr uint32_t kBit = kDevErrTimeoutBwd;
  // walk step it = 0, 1, ... is chunk c_end - 1 - it (stage it & 1); its first token, length
  auto chunk_of = [&](int it) { return c_end - 1 - it; };
  auto tok0_of = [&](int it) { return t_seq + (nch - 1 - it) * 64; };
  auto len_of = [&](int it) { return min(64, L - (nch - 1 - it) * 64); };
  const uint32_t accV0 = tb, accH0 = tb + 256;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&bar_load[s], 1);
      tc::mbar_init(&bar_scaled[s], 4);
      tc::mbar_init(&bar_vfull[s], 1);
      tc::mbar_init(&bar_hfull[s], 1);
      tc::mbar_init(&bar_dvn[s], 8);
      tc::mbar_init(&bar_dvnfree[s], 1);
    }
    tc::mbar_init(&bar_dh, 8);
    tc::mbar_init(&bar_dhfree, 1);
    tc::mbar_init(&bar_drain, 1);
    tc::fence_barrier_init();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();

  if (tid == kWalkLoadTid) {
    // ---------------------------------------------------------------- load role
    const uint64_t keep = tc::l2_policy_evict_last();
    const uint64_t keep_kq = d.G == 1 ? keep : tc::l2_policy_evict_normal();
    auto issue_loads = [&](int it) {
      const int st = it & 1, tc0 = tok0_of(it);
      const size_t chh = (size_t)chunk_of(it) * Hv + j;
      unsigned char* base = sm + st * WS::STAGE;
      uint64_t* bar = &bar_load[st];
      GDR_DELAY(14);
      // Q, dO and P feed only the dO products: the transition walk (dO = 0) leaves them out
      // (the scaling of Q's rows and the skipped products then touch stale tiles no one reads)
      const bool dO_tiles = !zero_do;
      tc::mbar_arrive_expect_tx(bar, (dO_tiles ? 9 : 4) * kSlab + 256);
      tc::bulk_load(base + WS::GAM, ws.gam + chh * 64, 256, bar);
      // q, k and dO are read again by the chunk's gradient item: kept in L2 (evict_last), whose
      // load lets them go (evict_first); q and k only with one v-head per q/k head, where that
      // item is their last reader
      tc::tma_load_3d_hint(base + WS::KQ, &tm_k, bar, 0, i, tc0, keep_kq);
      tc::tma_load_3d_hint(base + WS::KQ + 2 * kSlab, &tm_k, bar, 64, i, tc0, keep_kq);
      if (dO_tiles) {
        tc::tma_load_3d_hint(base + WS::KQ + kSlab, &tm_q, bar, 0, i, tc0, keep_kq);
        tc::tma_load_3d_hint(base + WS::KQ + 3 * kSlab, &tm_q, bar, 64, i, tc0, keep_kq);
        tc::tma_load_3d_hint(base + WS::DO, &tm_do, bar, 0, j, tc0, keep);
        tc::tma_load_3d_hint(base + WS::DO + kSlab, &tm_do, bar, 64, j, tc0, keep);
        tc::tma_load_2d(base + WS::P, &tm_p, bar, 0, (int)(chh * 64));
      }
      tc::tma_load_2d(base + WS::W, &tm_w, bar, 0, (int)(chh * 64));
      tc::tma_load_2d(base + WS::W + kSlab, &tm_w, bar, 64, (int)(chh * 64));
    };
    auto prefetch = [&](int it) {  // the same tiles into L2, a chunk before their load
      const int tc0 = tok0_of(it);
      const size_t chh = (size_t)chunk_of(it) * Hv + j;
      tc::bulk_prefetch_l2(ws.gam + chh * 64, 256);
      tc::tma_prefetch_l2_3d(&tm_k, 0, i, tc0);
      tc::tma_prefetch_l2_3d(&tm_k, 64, i, tc0);
      if (!zero_do) {
        tc::tma_prefetch_l2_3d(&tm_q, 0, i, tc0);
        tc::tma_prefetch_l2_3d(&tm_q, 64, i, tc0);
        tc::tma_prefetch_l2_3d(&tm_do, 0, j, tc0);
        tc::tma_prefetch_l2_3d(&tm_do, 64, j, tc0);
        tc::tma_prefetch_l2_2d(&tm_p, 0, (int)(chh * 64));
      }
      tc::tma_prefetch_l2_2d(&tm_w, 0, (int)(chh * 64));
      tc::tma_prefetch_l2_2d(&tm_w, 64, (int)(chh * 64));
    };
    int loaded = -1;  // last walk step whose tiles were requested
    if (nch > 0) {
      issue_loads(0);
      loaded = 0;
    }
    if (nch > 1) {
      issue_loads(1);
      loaded = 1;
    }
    if (nch > 2) prefetch(2);
    // step it + 2 goes into step it's stage once its last MMA (W^T dVn) has completed; the
    // epilogue warps stop reading a stage before that
    for (int it = 0; it + 2 < nch; ++it) {
      if (!tc::mbar_wait(&bar_hfull[it & 1], (it >> 1) & 1, status, kBit)) break;
      GDR_TRACE_CLK(tl0);
      issue_loads(it + 2);
      loaded = it + 2;
      if (it + 3 < nch) prefetch(it + 3);
      GDR_TRACE_SINCE(3, 16, tl0);
    }
    // every load requested has landed (bounded) before the CTA's shared memory serves the
    // next role.  A stage's earlier loads completed before its next was requested (their MMAs
    // had read them), so only the last load of each stage can be pending; waiting on an older
    // phase of a barrier that has moved on two phases would not return.
    for (int it = loaded > 0 ? loaded - 1 : 0; it <= loaded; ++it)
      (void)tc::mbar_wait(&bar_load[it & 1], (it >> 1) & 1, status, kBit);
  } else if (tid == kWalkMmaTid) {
    // ---------------------------------------------------------------- MMA role
    // the products that do not need dh': P^T dO into accV, Q^^T dO into accH
    auto issue_free = [&](int it) -> bool {
      const int st = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      unsigned char* stg = sm + st * WS::STAGE;
      if (!tc::mbar_wait(&bar_load[st], ph, status, kBit)) return false;
      tc::tc_fence_after();
      if (!zero_do)
        tc::gemm(accV0 + 128 * st, tc::mnmaj(stg + WS::P, kSlab), tc::mnmaj(stg + WS::DO, kSlab), 128, 4, false);
      if (!tc::mbar_wait(&bar_scaled[st], ph, status, kBit)) return false;
      tc::tc_fence_after();
      if (!zero_do)
        tc::gemm(accH0 + 128 * st, tc::mnmaj(stg + WS::KQ + kSlab, 2 * kSlab), tc::mnmaj(stg + WS::DO, kSlab), 128,
                 4, false);
      return true;
    };
    bool ok = true;
    if (nch > 0) ok = issue_free(0);
    for (int it = 0; it < nch && ok; ++it) {
      const int st = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      unsigned char* stg = sm + st * WS::STAGE;
      // the chain: K^ dh' once dh' is staged, then W^T dVn once dVn is
      GDR_TRACE_CLK(tw0);
      ok = tc::mbar_wait(&bar_dh, it & 1, status, kBit);
      GDR_TRACE_SINCE(3, 10, tw0);
      if (!ok) break;
      tc::tc_fence_after();
      GDR_DELAY(13);
      GDR_TRACE_CLK(tw1);
      tc::gemm(accV0 + 128 * st, tc::kmaj(stg + WS::KQ, 2 * kSlab), tc::mnmaj(sm + WS::DH, 16384), 128, 8,
               !zero_do);
      tc::mma_commit(&bar_vfull[st]);
      GDR_TRACE_SINCE(3, 11, tw1);
      GDR_TRACE_CLK(tw2);
      ok = tc::mbar_wait(&bar_dvn[st], ph, status, kBit);
      GDR_TRACE_SINCE(3, 12, tw2);
      if (!ok) break;
      tc::tc_fence_after();
      GDR_TRACE_CLK(tw3);
      tc::gemm(accH0 + 128 * st, tc::mnmaj(stg + WS::W, kSlab), tc::mnmaj(sm + WS::DVN + st * 16384, kSlab), 128,
               4, !zero_do, true);
      tc::mma_commit(&bar_hfull[st]);
      GDR_TRACE_SINCE(3, 13, tw3);
      // the next chunk's dh'-free products
      GDR_TRACE_CLK(tw4);
      if (it + 1 < nch) ok = issue_free(it + 1);
      GDR_TRACE_SINCE(3, 14, tw4);
    }
    // drain: every MMA issued has completed before the CTA's tensor memory serves the next role
    tc::mma_commit(&bar_drain);
    (void)tc::mbar_wait(&bar_drain, 0, status, kBit);
  } else if (tid == kWalkCopyTid) {
    // ---------------------------------------------------------------- store + publish role
    // kPublish: chunks stored whose counts are still due: the previous step's (pub) and, every
    // other step, the one before (held).  The counts go out in pairs, so the GPU-scope release
    // that orders each count after its chunk's stores is paid back to back every second step
    // instead of once a step on the copy thread's path to the next dh' store.
    int pub = -1, held = -1;
    const uint64_t keep = tc::l2_policy_evict_last();
    for (int it = 0; it < nch; ++it) {
      const int st = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      const size_t chh = (size_t)chunk_of(it) * Hv + j;
      GDR_TRACE_CLK(tc0_);
      if (!tc::mbar_wait(&bar_dh, it & 1, status, kBit)) break;
      GDR_TRACE_SINCE(3, 20, tc0_);
      GDR_DELAY(10);
      if (stores) {  // kept in L2 for the gradient item that reads them (evict_last)
        tc::tma_store_2d_hint(&tm_dhs, sm + WS::DH, 0, (int)(chh * 128), keep);
        tc::tma_store_2d_hint(&tm_dhs, sm + WS::DH + 16384, 64, (int)(chh * 128), keep);
        tc::bulk_commit();
        tc::bulk_wait_read<0>();  // the dh' tile has been read: the next dh' may replace it
      }
      tc::mbar_arrive(&bar_dhfree);
      if (!tc::mbar_wait(&bar_dvn[st], ph, status, kBit)) break;
      if (stores) {
        unsigned char* dvn = sm + WS::DVN + st * 16384;
        tc::tma_store_2d_hint(&tm_dvs, dvn, 0, (int)(chh * 64), keep);
        tc::tma_store_2d_hint(&tm_dvs, dvn + kSlab, 64, (int)(chh * 64), keep);
        tc::bulk_commit();
        tc::bulk_wait_read<0>();
      }
      tc::mbar_arrive(&bar_dvnfree[st]);
      GDR_TRACE_CLK(tc1_);
      if (kPublish && stores && pub >= 0) {
        if (held >= 0) {  // the two previous steps' groups have landed: both counts
          tc::bulk_wait<2>();
          GDR_DELAY(11);
          publish_chunk(ws.walk_flags + (size_t)held * Hv + j);
          publish_chunk(ws.walk_flags + (size_t)pub * Hv + j);
          held = -1;
        } else {
          held = pub;
        }
      }
      GDR_TRACE_SINCE(3, 21, tc1_);
      pub = chunk_of(it);
    }
    tc::bulk_wait<0>();
    if (kPublish && stores) {
      if (held >= 0) publish_chunk(ws.walk_flags + (size_t)held * Hv + j);
      if (pub >= 0) publish_chunk(ws.walk_flags + (size_t)pub * Hv + j);
    }
  } else if (tid < 256) {
    // ---------------------------------------------------------------- epilogue warps
    const int ln = (warp & 3) * 32 + lane;  // TMEM lane: token of accV (lanes 0-63), dk of accH
    const int hf = warp >> 2;               // accV: dv [64 hf, +64); accH: dv [64 hf, +64)
    const bool lo = (warp & 3) < 2;         // the dVn rows (lanes 0-63)
    const float scale = d.scale, inv_scale = 1.f / d.scale;
    // lanes 64-127 warps: K^ and Q^ of step it in place, one row of both slabs of K (threads
    // 0-63) or of Q (64-127) per thread
    auto scale_tiles = [&](int it) -> bool {
      const int st = it & 1;
      GDR_TRACE_CLK(ts0);
      if (!warp_wait(&bar_load[st], (it >> 1) & 1, status, kBit)) return false;
      if (tid == 64) GDR_TRACE_SINCE(3, 17, ts0);
      unsigned char* stg = sm + st * WS::STAGE;
      const float* g = reinterpret_cast<const float*>(stg + WS::GAM);
      const int len = len_of(it);
      const int h = ((warp & 3) - 2) * 32 + lane + 64 * hf;  // 0..127
      const int r = h & 63, isq = h >> 6;
      const float f = r < len ? (isq ? scale * fexp(g[r]) : fexp(g[len - 1] - g[r]) * inv_scale) : 0.f;
#pragma unroll 1
      for (int k = 0; k < 2; ++k) {  // slabs: K at 0 and 2 kSlab, Q at kSlab and 3 kSlab
        unsigned char* slab = stg + WS::KQ + (2 * k + isq) * kSlab;
        float x[64];
        ld_row_bf16(slab, r, x);
#pragma unroll
        for (int b = 0; b < 64; ++b) x[b] *= f;
        st_row_bf16(slab, r, x);
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar_scaled[st]);
      return true;
    };
    float dh[64];
#pragma unroll
    for (int b = 0; b < 64; ++b)
      dh[b] = g0_eye ? (ln == 64 * hf + b ? 1.f : 0.f)
              : un.g0   ? un.g0[un.g0_kv ? (size_t)ln * 128 + 64 * hf + b : (size_t)(64 * hf + b) * 128 + ln]
                        : 0.f;
    auto stage_dh = [&]() {  // dh' of the next step as the MMA's bf16 operand
      st_row_bf16(sm + WS::DH + hf * 16384, ln, dh);
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar_dh);
    };
    bool ok = true;
    if (nch > 0) {
      stage_dh();
      if (!lo) ok = scale_tiles(0);
    }
    GDR_TRACE_INIT();
    for (int it = 0; it < nch && ok; ++it) {
      const int st = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      const int len = len_of(it);
      ok = warp_wait(&bar_vfull[st], ph, status, kBit);
      GDR_TRACE_MARK(3, 0);
      if (!ok) break;
      tc::tc_fence_after();
      // gamma_C while the stage still holds this step (it is reloaded after W^T dVn)
      const float gC = reinterpret_cast<const float*>(sm + st * WS::STAGE + WS::GAM)[len - 1];
      if (lo) {  // dVn = scale accV, token row ln, columns [64 hf, +64), zero past the chunk end
        float x[64];
        tmem_ld64(accV0 + 128 * st, warp, 64 * hf, x);
        tc::tc_fence_before();
        GDR_TRACE_MARK(3, 7);
        if (it >= 2) {
          ok = warp_wait(&bar_dvnfree[st], ((it - 2) >> 1) & 1, status, kBit);
          if (!ok) break;
        }
        GDR_TRACE_MARK(3, 8);
        if (warp == 1) GDR_DELAY(12);
        const float f = ln < len ? scale : 0.f;
#pragma unroll
        for (int b = 0; b < 64; ++b) x[b] *= f;
        st_row_bf16(sm + WS::DVN + st * 16384 + hf * kSlab, ln, x);
        GDR_TRACE_MARK(3, 9);
        tc::fence_proxy_async_smem();
      }
      // every epilogue warp counts in (the others have read gamma_C, so the stage may be
      // reloaded once W^T dVn, which waits for this, has run)
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar_dvn[st]);
      // meanwhile the lanes 64-127 warps prepare the next step's K^, Q^
      if (!lo && it + 1 < nch) {
        ok = scale_tiles(it + 1);
        if (!ok) break;
      }
      GDR_TRACE_MARK(3, 2);
      GDR_TRACE_MARK(3, 1);
      // dh = e^{gamma_C} dh' + accH, staged as the next step's dh'
      ok = warp_wait(&bar_hfull[st], ph, status, kBit);
      GDR_TRACE_MARK(3, 3);
      if (!ok) break;
      tc::tc_fence_after();
      {
        float y0[32], y1[32];
        tc::tmem_ld32(tc::tmem_lane_addr(accH0 + 128 * st, warp, 64 * hf), y0);
        tc::tmem_ld32(tc::tmem_lane_addr(accH0 + 128 * st, warp, 64 * hf + 32), y1);
        tc::tmem_wait_ld();
        tc::tc_fence_before();
        const float eC = fexp(gC);
#pragma unroll
        for (int b = 0; b < 32; ++b) {
          dh[b] = eC * dh[b] + y0[b];
          dh[32 + b] = eC * dh[32 + b] + y1[b];
        }
      }
      GDR_TRACE_MARK(3, 4);
      if (it + 1 < nch) {
        ok = warp_wait(&bar_dhfree, it & 1, status, kBit);
        GDR_TRACE_MARK(3, 5);
        if (!ok) break;
        stage_dh();
      }
      GDR_TRACE_MARK(3, 6);
    }
    if (ok && un.g1) {
#pragma unroll
      for (int b = 0; b < 64; ++b)
        un.g1[un.g1_kv ? (size_t)ln * 128 + 64 * hf + b : (size_t)(64 * hf + b) * 128 + ln] = dh[b];
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (tid == 0) {  // the next unit of this CTA (or the next role) initialises them again
    for (int s = 0; s < 2; ++s) {
      tc::mbar_inval(&bar_load[s]);
      tc::mbar_inval(&bar_scaled[s]);
      tc::mbar_inval(&bar_vfull[s]);
      tc::mbar_inval(&bar_hfull[s]);
      tc::mbar_inval(&bar_dvn[s]);
      tc::mbar_inval(&bar_dvnfree[s]);
    }
    tc::mbar_inval(&bar_dh);
    tc::mbar_inval(&bar_dhfree);
    tc::mbar_inval(&bar_drain);
  }
  __syncthreads();
  tc::tc_fence_after();
}

// The reverse walk alone (cluster-pair gradients, more sequences than the fused kernel's order
// table holds, or the first context-parallel pass): one CTA per walk unit.  kPublish: counts
// every stored chunk in ws.walk_flags for a fused kernel launched after it.
template <bool kPublish, bool kModes>
__global__ void __launch_bounds__(kWalkThreads, 1) tc_bwd_walk_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_p,
    const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_dhs,
    const __grid_constant__ CUtensorMap tm_dvs, Dims d, const float* __restrict__ dS_T, float* __restrict__ dS0,
    Workspace ws, CpArgs cp) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = align1024(smem_raw);
  const WalkUnit un = walk_unit(d, ws, cp, (int)blockIdx.x, dS_T, dS0);
  if (un.skip) return;  // uniform over the block, before any barrier or tensor memory
  __shared__ uint32_t tmem_slot;
  if (threadIdx.x < 32) tc::tmem_alloc<kWalkTmemCols>(&tmem_slot);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  walk_body<kPublish, kModes>(tm_q, tm_k, tm_w, tm_p, tm_do, tm_dhs, tm_dvs, d, ws, un, tmem_slot, sm);
  if (threadIdx.x < 32) tc::tmem_dealloc(tmem_slot, kWalkTmemCols);
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
    const int len = idx_chunk(d, ws, c).z;
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
  static constexpr uint32_t DO = 32768;         // dO (16 KB); cluster pairs: -> the partner's dk half
  // O-hat = scale diag(e^gamma) dO and dVn interleaved by 64-column slab (slab s of O-hat at
  // OD + 16 KB s, of dVn 8 KB after it), so [O-hat; dVn] is one 128-row K-major operand
  // (32 KB); O-hat -> V after the first product, dVn to the WY backward
  static constexpr uint32_t OD = 49152;
  static constexpr uint32_t DH = 81920;         // dh' (32 KB) -> dq staging
  static constexpr uint32_t H = 114688;         // h bf16 (32 KB) -> dP | dT | X | dAGb (8 KB each);
                                                //   h fp32 lands in H, H + 16 KB, VN and SCR
  static constexpr uint32_t VN = 147456;        // Vn~ (16 KB) -> T'
  static constexpr uint32_t W = 163840;         // Vn as loaded (16 KB) -> dv staging
  static constexpr uint32_t UT = 180224;        // dW (16 KB) -> dk staging
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
  static constexpr uint32_t TP = VN, DQS = DH, DVS = W, DKS = UT, DW = UT;
};

constexpr int kGradThreads = 256;  // two warps per TMEM lane quarter, each on half the columns

// The gradient role's barriers: named barrier 1 over its kGradThreads threads (warps 0-7), so
// that a kernel may run the role on part of a larger CTA (the fused walk + gradient kernel,
// whose walk role also has an MMA warp and a copy warp).
__device__ __forceinline__ void gsync() { tc::named_sync(1, kGradThreads); }
__device__ __forceinline__ bool gsync_and(bool p) { return tc::named_sync_and(1, kGradThreads, p); }

// kGroup: Hv > Hk; dq, dk are summed over the v-heads of a q/k head.  kPair (Hv = 2 Hk,
// launched as clusters of two CTAs): the two CTAs of a cluster take the two v-heads of one
// q/k head on the same chunk, and each finalises half of the dq and dk columns, adding the
// partner's partial sent through distributed shared memory (no fp32 partials in HBM and
// no separate reduction).  Otherwise (kGroup alone) fp32 partials go to the workspace and
// launch_group_reduce sums them.
// kDyn (fused walk + gradient kernel): items are claimed from ws.grad_queue in the order the
// walk finishes them (last chunk of every sequence first), and a chunk's dh' and dVn
// tiles are loaded only once the walk unit has counted it in ws.walk_flags.
// tb: 512 TMEM columns owned by the caller.
template <bool kGroup, bool kPair, bool kDyn, bool kCpOrder = false>
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
  gsync();
  tc::tc_fence_after();
  if (kPair) tc::cluster_sync();  // the partner's barriers exist before anyone arrives on them
  // TMEM columns: [K K^T ; Q K^T] 0-63 (K K^T kept to the end); dq 256-383; dk 384-511.
  const uint32_t C_KK = tb, C_DQ = tb + 256, C_DK = tb + 384;
  GDR_TRACE_INIT();
  // Persistent: each CTA walks the (chunk, v-head) items w = blockIdx.x + k * gridDim.x,
  // keeping its barriers, TMEM and (warm) instruction cache across items.  The next
  // item's tiles are fetched as soon as the current item is done with their buffers
  // (dh', dVn and dO after R2, W after R3, K/Q, U, h and gamma after R4; with cluster pairs
  // dO after the dk exchange, which receives into its tile), all on the next phase of
  // bar_tma, so the loads overlap the current item.
  bool ok = true;
  uint32_t item_par = 0;  // phase parity of bar_tma / bar_tma2 for the current item
  uint32_t mma_par = 0;   // phase parity of bar_mma (five commits per item: it alternates)
  // items: (chunk, v-head), or with kPair (chunk, q/k head) shared by the cluster, whose
  // CTA `rank` takes v-head 2 i + rank; with kDyn every real chunk's v-heads, in walk order
  const int n_steps = kDyn ? idx_n_steps(d, ws) : 0;
  const int n_items = kDyn ? idx_step_off(d, ws, n_steps) * Hv : (kPair ? d.max_chunks * d.Hk : d.max_chunks * Hv);
  const int item0 = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int istep = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  // kDyn: item w = q * Hv + v-head, queue position q in walk order (the index kernel lists
  // each position's chunk)
  auto chunk_of = [&](int w) {
    if (kDyn) return kCpOrder ? idx_cp_grad_chunk(d, w / Hv) : idx_grad_chunk(d, ws, w / Hv);
    return kPair ? w / d.Hk : w / Hv;
  };
  auto vhead_of = [&](int w) { return kPair ? (w % d.Hk) * 2 + (int)rank : w % Hv; };
  auto next_item = [&](int w) {  // next non-empty item of this CTA after w (or n_items)
    for (w += istep; w < n_items && idx_chunk(d, ws, chunk_of(w)).z <= 0; w += istep) {
    }
    return w < n_items ? w : n_items;
  };
  int cur_len = 0, cur_t0 = 0, cur_i = 0;  // the current item (for pair_reduce)
  enum : int { kLdDhDvn = 1, kLdW = 2, kLdRest = 4, kLdDo = 8, kLdAll = 15 };
  auto issue_loads = [&](int w, int c2, int groups) {  // copy thread only; c2 = chunk_of(w)
    GDR_DELAY(20);
    const int j2 = vhead_of(w), i2 = j2 / d.G, tt = idx_chunk(d, ws, c2).y;
    const size_t ch2 = (size_t)c2 * Hv + j2;
    uint64_t* bar = &bar_tma;
    if (groups & kLdDhDvn) {  // the first group of an item sets the whole item's byte count
      // kDyn: dh' and dVn of this chunk come from the walk running in the same kernel; on a
      // timeout the loads are left out and the item's own bounded wait ends the walk
      GDR_TRACE_CLK(tw0);
      const unsigned long long tf0_ = GDR_TRACE_NOW();
      if (kDyn && !wait_flag(ws.walk_flags + ch2, 1u, ws.status, kDevErrTimeoutBwd)) return;
      GDR_TRACE_INFO_ADD(4, GDR_TRACE_NOW() - tf0_);
      GDR_TRACE_SINCE(2, 20, tw0);
      tc::mbar_arrive_expect_tx(bar, (d.h_bf16 ? 18 : 22) * kSlab + 256);
      const uint64_t once = tc::l2_policy_evict_first();  // read once: released first
      for (int q4 = 0; q4 < 4; ++q4)  // dh' rows (q4 & 1) * 64.., columns (q4 >> 1) * 64..
        tc::tma_load_2d_hint(sm + S::DH + (q4 >> 1) * 16384 + (q4 & 1) * kSlab, &tm_dh, bar, (q4 >> 1) * 64,
                             (int)(ch2 * 128 + (q4 & 1) * 64), once);
      tc::tma_load_2d_hint(sm + S::DVN, &tm_dvn, bar, 0, (int)(ch2 * 64), once);
      tc::tma_load_2d_hint(sm + S::DVN + S::OD_SLAB, &tm_dvn, bar, 64, (int)(ch2 * 64), once);
    }
    if (groups & kLdW) {  // Vn (in U's place in memory) into W's tile, once the dv store has read it
      tc::tma_load_2d(sm + S::W, &tm_u, bar, 0, (int)(ch2 * 64));
      tc::tma_load_2d(sm + S::W + kSlab, &tm_u, bar, 64, (int)(ch2 * 64));
    }
    if (groups & kLdRest) {
      tc::bulk_load(sm + S::GAM, ws.gam + ch2 * 64, 256, bar);
      // K and Q: the walk left them in L2; with one v-head per q/k head this is their last
      // reader (evict_first), else the other v-heads' items read them too (no policy)
      if (d.G == 1) {
        const uint64_t once = tc::l2_policy_evict_first();
        tc::tma_load_3d_hint(sm + S::KQ, &tm_k, bar, 0, i2, tt, once);
        tc::tma_load_3d_hint(sm + S::KQ + 2 * kSlab, &tm_k, bar, 64, i2, tt, once);
        tc::tma_load_3d_hint(sm + S::KQ + kSlab, &tm_q, bar, 0, i2, tt, once);
        tc::tma_load_3d_hint(sm + S::KQ + 3 * kSlab, &tm_q, bar, 64, i2, tt, once);
      } else {
        tc::tma_load_3d(sm + S::KQ, &tm_k, bar, 0, i2, tt);
        tc::tma_load_3d(sm + S::KQ + 2 * kSlab, &tm_k, bar, 64, i2, tt);
        tc::tma_load_3d(sm + S::KQ + kSlab, &tm_q, bar, 0, i2, tt);
        tc::tma_load_3d(sm + S::KQ + 3 * kSlab, &tm_q, bar, 64, i2, tt);
      }
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
      const uint64_t once = tc::l2_policy_evict_first();  // dO: its last reader
      tc::tma_load_3d_hint(sm + S::DO, &tm_do, bar, 0, j2, tt, once);
      tc::tma_load_3d_hint(sm + S::DO + kSlab, &tm_do, bar, 64, j2, tt, once);
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
    return (bool)gsync_and(okin && okw);
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
    gsync();
    witem = s_claim;
    cur_c = s_claim_c;
    gsync();
  } else {
    witem = item0 < n_items && idx_chunk(d, ws, chunk_of(item0)).z <= 0 ? next_item(item0) : item0;
  }
  if (tid == kCopyTid && witem < n_items) issue_loads(witem, kDyn ? cur_c : chunk_of(witem), kLdAll);
  int pending = witem < n_items ? 0 : -1;  // groups of the next item issued so far (-1: none expected)
  int cl_w = n_items, cl_c = 0;            // kDyn, copy thread: the claimed next item and its chunk
  while (witem < n_items && ok) {
  // the next item (kDyn: claimed at the first prefetch point, known to all after the item)
  const int wnext = kDyn ? n_items : next_item(witem);
  const int cnext = kDyn ? 0 : (wnext < n_items ? chunk_of(wnext) : 0);
  const int c = kDyn ? cur_c : chunk_of(witem), j = vhead_of(witem), i = j / d.G;
  const int4 ci = idx_chunk(d, ws, c);
  const int len = ci.z, t0 = ci.y;
  cur_len = len;
  cur_t0 = t0;
  cur_i = i;
  const size_t ch = (size_t)c * Hv + j;
  if (kDyn && tid == kCopyTid) pre_w = (int)atomicAdd(ws.grad_queue, 1u);  // used after R2
  if (tid < 64) s_beta[tid] = tid < len ? __bfloat162float(beta[(size_t)(t0 + tid) * Hv + j]) : 0.f;
  ok = gsync_and(tc::mbar_wait(&bar_tma, item_par, ws.status, kDevErrTimeoutBwd));
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
    gsync();
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
  gsync();
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
  ok = gsync_and(ok && tc::mbar_wait(&bar_mma, mma_par, ws.status, kDevErrTimeoutBwd));
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
  gsync();
  GDR_TRACE_MARK(2, 3);
  if (ok) col_partial(s_colpp);  // column sums of dP * QK
  if (ok && tid < 64) {  // sum_s e^{gC - g_s} k_s^T dh' vn_s
    const float kdv = tid < len ? s_kdv[0][tid] + s_kdv[1][tid] : 0.f;
    s_kdv[0][tid] = kdv;
    const float part = warp_sum(kdv);
    if (lane == 0) s_red[warp] = part;
  }
  ok = gsync_and(ok && tc::mbar_wait(&bar_tma2, item_par, ws.status, kDevErrTimeoutBwd));
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
  ok = gsync_and(ok && tc::mbar_wait(&bar_mma, mma_par, ws.status, kDevErrTimeoutBwd));
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
  gsync();
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
  ok = gsync_and(ok && tc::mbar_wait(&bar_mma, mma_par, ws.status, kDevErrTimeoutBwd));
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
    if (pending >= 0) {  // dO too (last read by P2), unless the dk exchange receives into its tile
      constexpr int groups = kPair ? (int)kLdDhDvn : (int)(kLdDhDvn | kLdDo);
      issue_loads(kDyn ? cl_w : wnext, kDyn ? cl_c : cnext, groups);
      pending |= groups;
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
  gsync();
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
  ok = gsync_and(ok && tc::mbar_wait(&bar_mma, mma_par, ws.status, kDevErrTimeoutBwd));
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
  gsync();
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
  ok = gsync_and(ok && tc::mbar_wait(&bar_mma, mma_par, ws.status, kDevErrTimeoutBwd));
  mma_par ^= 1;
  tc::tc_fence_after();
  if (ok && tid == kCopyTid && pending >= 0) {  // every operand tile but dO (cluster pairs) is free
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
  gsync();
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
  gsync();
  if (ok && tid < 64) {
    const int rr = 63 - tid;
    const float v = s_colaa[0][tid] + (tid >= 32 ? s_colaa[0][31] : 0.f);
    if (rr < len) dg[(size_t)(t0 + rr) * Hv + j] = v;
  }
  if (tid == kCopyTid) {
    GDR_TRACE_CLK(tb23);
    tc::bulk_wait_read<0>();  // staging tiles read before the next item's loads
    GDR_TRACE_SINCE(2, 23, tb23);
    if (kPair && ok && pending >= 0) {  // the dk exchange is done with the dO tile
      issue_loads(kDyn ? cl_w : wnext, kDyn ? cl_c : cnext, kLdDo);
      pending |= kLdDo;
    }
  }
  GDR_TRACE_MARK(2, 13);
  GDR_TRACE_COUNT(2, 31);
  if (tid == 0) GDR_TRACE_INFO_ADD(3, 1);
  item_par ^= 1;
  tc::tc_fence_before();
  gsync();
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
  gsync();
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
// resident, one per SM): CTAs first run walk units (32 at B=2, H=16, leaving the other SMs
// free), then every CTA claims gradient items in the order the walk completes chunks, so the
// gradients of late chunks overlap the walk of early ones.  Launched with kWalkThreads (384)
// threads: three warps of a register-file quarter (warps q, q + 4, q + 8) cap a thread at 168
// registers, enough for the walk.  For the gradient role the third warpgroup (the walk's MMA,
// store and load warps) hands its registers to warps 0-7: setmaxnreg.dec to 40 there and
// setmaxnreg.inc to 232 here, 4 x 32 x 40 + 8 x 32 x 232 = 384 x 168 registers, which is
// exactly the block's allocation (the launcher checks the kernel was built with 168 per
// thread), so the increase never waits for registers that are not there.
constexpr uint32_t kWalkRegs = 168, kGradRegs = 232, kIdleRegs = 40;
static_assert(4 * 32 * kIdleRegs + 8 * 32 * kGradRegs == (uint32_t)kWalkThreads * kWalkRegs, "register split");
template <bool kGroup, bool kCpOrder>
__global__ void __launch_bounds__(kWalkThreads, 1) tc_bwd_walkgrad_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_u,
    const __grid_constant__ CUtensorMap tm_p, const __grid_constant__ CUtensorMap tm_dvn,
    const __grid_constant__ CUtensorMap tm_dh, const __grid_constant__ CUtensorMap tm_dhs,
    const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_t,
    const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
    const __grid_constant__ CUtensorMap tm_dv, Dims d, const float* __restrict__ dS_T, float* __restrict__ dS0,
    const bf16* __restrict__ beta, bf16* __restrict__ dq, bf16* __restrict__ dk, bf16* __restrict__ dv,
    float* __restrict__ dg, bf16* __restrict__ dbeta, Workspace ws, CpArgs cp) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = align1024(smem_raw);
  __shared__ uint32_t tmem_slot;
  if (threadIdx.x < 32) tc::tmem_alloc<512>(&tmem_slot);  // both roles' columns
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  // walk units: one per (sequence, v-head), or the second context-parallel pass's segment walks
  // (the first pass ran before this kernel and counted its chunks in ws.walk_flags)
  const int n_units = d.num_seqs * d.Hv * walk_units_per_chain(cp);
  if (threadIdx.x == 0) GDR_TRACE_INFO_SET(0, GDR_TRACE_NOW());
  for (int u = (int)blockIdx.x; u < n_units; u += (int)gridDim.x) {
    const WalkUnit un = walk_unit(d, ws, cp, u, dS_T, dS0);
    if (!un.skip) walk_body<true, false>(tm_q, tm_k, tm_w, tm_p, tm_do, tm_dhs, tm_dvn, d, ws, un, tmem_slot, sm);
  }
  if (threadIdx.x == 0) GDR_TRACE_INFO_SET(1, GDR_TRACE_NOW());
  if (threadIdx.x >= kGradThreads) {  // the walk's single-thread roles: registers to the gradients
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kIdleRegs) : "memory");
    return;
  }
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kGradRegs) : "memory");
  grad_body<kGroup, false, true, kCpOrder>(tm_q, tm_k, tm_v, tm_do, tm_w, tm_u, tm_dvn, tm_dh, tm_h, tm_t, tm_dq,
                                           tm_dk, tm_dv, d, beta, dq, dk, dv, dg, dbeta, ws, tmem_slot, sm);
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
    set_smem_once((const void*)tc_vn_kernel, smv);
    tc_vn_kernel<<<(unsigned)(n_items < n_sm ? n_items : n_sm), kTcThreads, smv, s>>>(tw, tu, thf, d, ws);
    stage_mark(s, "bwd_vn");
  }
  // One walk unit per (sequence, v-head), over all of DV.
  Dims dd = d;
  const bool cp_on = d.num_seqs > 0 && d.cp_bwd > 1 && Tt > 0;
  // the fused kernel; with context-parallel segments the instantiation whose item queue follows
  // the segment walks
  auto kern = d.G > 1 ? (cp_on ? tc_bwd_walkgrad_kernel<true, true> : tc_bwd_walkgrad_kernel<true, false>)
                      : (cp_on ? tc_bwd_walkgrad_kernel<false, true> : tc_bwd_walkgrad_kernel<false, false>);
  // the fused kernel's register split assumes the block holds exactly kWalkRegs per thread; a
  // build that allocated another count runs the walk and the gradients as two launches
  cudaFuncAttributes fa{};
  const bool regs_ok = cudaFuncGetAttributes(&fa, (const void*)kern) == cudaSuccess && fa.numRegs == (int)kWalkRegs;
  auto walk_launch = [&](bool publish, const CpArgs& cp, long long units, const char* stage) -> cudaError_t {
    if (units <= 0) return cudaSuccess;
    const size_t sm = WalkSmem::BYTES + 1024;
    const bool modes = cp.pass == 1;  // only the first pass has map units
    auto wk = publish ? (modes ? tc_bwd_walk_kernel<true, true> : tc_bwd_walk_kernel<true, false>)
                      : (modes ? tc_bwd_walk_kernel<false, true> : tc_bwd_walk_kernel<false, false>);
    set_smem_once((const void*)wk, sm);
    wk<<<(unsigned)units, kWalkThreads, sm, s>>>(tq, tk, tw, tp, tdo, tdhs, tdvn, dd, a.dS_T, a.dS0, ws, cp);
    stage_mark(s, stage);
    return cudaGetLastError();
  };
  const int P = d.cp_bwd;
  const long long chains = (long long)d.num_seqs * d.Hv;
  // walk and gradients in one cooperative kernel; with context-parallel segments (fixed length)
  // the kernel runs the second pass's walks, after the first pass and the scan
  if (fused_walk_grad(d) && regs_ok && (!cp_on || d.cu == nullptr)) {
    int per_sm = 0;
    const size_t smg = std::max(GradSmem::BYTES, WalkSmem::BYTES) + 1024;
    set_smem_once((const void*)kern, smg);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWalkThreads, smg) != cudaSuccess || per_sm < 1)
      return cudaErrorInvalidConfiguration;
    e = cudaMemsetAsync(ws.walk_flags, 0, sizeof(uint32_t) * ((size_t)d.max_chunks * d.Hv + 64), s);
    if (e != cudaSuccess) return e;
    CpArgs cp{};
    if (cp_on) {
      cp = CpArgs{1, P, ws.cp_X, ws.cp_M, ws.cp_R};
      e = walk_launch(true, cp, chains * (1 + 2 * (P - 2)), "bwd_cp_maps");
      if (e == cudaSuccess && P > 2) e = launch_cp_scan(d, ws, P, true, s);
      if (e != cudaSuccess) return e;
      cp.pass = 3;
    }
    const bf16* beta = (const bf16*)a.beta;
    bf16 *dq = (bf16*)a.dq, *dk = (bf16*)a.dk, *dv = (bf16*)a.dv, *dbeta = (bf16*)a.dbeta;
    const float* dS_T = a.dS_T;
    float *dS0 = a.dS0, *dg = a.dg;
    Workspace w = ws;
    void* args[] = {&tq, &tk, &tv, &tdo, &tw, &tu, &tp, &tdvn, &tdh, &tdhs, &thf, &tt, &tdq, &tdk, &tdv, &dd,
                    (void*)&dS_T, (void*)&dS0, (void*)&beta, (void*)&dq, (void*)&dk, (void*)&dv, (void*)&dg,
                    (void*)&dbeta, &w, &cp};
    e = cudaLaunchCooperativeKernel((const void*)kern, dim3((unsigned)(per_sm * n_sm)), dim3(kWalkThreads), args, smg,
                                    s);
    if (e != cudaSuccess) return e;
    stage_mark(s, "bwd_walkgrad");
    if (d.G > 1) {
      e = launch_group_reduce(d, a.dq, a.dk, ws, s);
      if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
  }
  if (cp_on) {
    // context parallel: the last segment's walk and every middle segment's maps, the scan of the
    // boundary gradients, then segments 0 .. nseg - 2 from their true end gradients (WalkUnit)
    CpArgs cp{1, P, ws.cp_X, ws.cp_M, ws.cp_R};
    e = walk_launch(false, cp, chains * (1 + 2 * (P - 2)), "bwd_cp_maps");
    if (e == cudaSuccess && P > 2) e = launch_cp_scan(d, ws, P, true, s);
    cp.pass = 3;
    if (e == cudaSuccess) e = walk_launch(false, cp, chains * (P - 1), "bwd_cp_walk");
    if (e != cudaSuccess) return e;
  } else if (d.num_seqs > 0) {
    e = walk_launch(false, CpArgs{}, chains, "bwd_walk");
    if (e != cudaSuccess) return e;
  }
  if (d.max_chunks > 0 && Tt > 0) {
    const long long n_items = (long long)d.max_chunks * d.Hv;
    const dim3 grid((unsigned)(n_items < n_sm ? n_items : n_sm));  // persistent: one CTA per SM
    const size_t smg = GradSmem::BYTES + 1024;
    if (grad_pair_mode(d)) {  // clusters of two CTAs, one per v-head of a q/k head
      auto kern = tc_bwd_grad_kernel<true, true>;
      set_smem_once((const void*)kern, smg);
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
      set_smem_once((const void*)tc_bwd_grad_kernel<true>, smg);
      tc_bwd_grad_kernel<true><<<grid, kGradThreads, smg, s>>>(tq, tk, tv, tdo, tw, tu, tdvn, tdh, thf, tt, tdq, tdk,
                                                              tdv, d, (const bf16*)a.beta, (bf16*)a.dq,
                                                              (bf16*)a.dk, (bf16*)a.dv, a.dg, (bf16*)a.dbeta, ws);
    } else {
      set_smem_once((const void*)tc_bwd_grad_kernel<false>, smg);
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
