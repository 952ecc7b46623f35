// gdr_tc.cu -- tcgen05 tensor-core kernels of the chunked gated delta rule
// (bf16 inputs, DK = DV = 128, fp32 state), chunk = 64 tokens.
//
// Notation per chunk (FlashQLA PR #34, Summary: the chunked gated delta rule), with
// h := S^T (DK x DV) the state at the chunk start, gamma the in-chunk cumsum of g,
// Gam[r,s] = exp(gamma_r - gamma_s) for r >= s:
//   A  = strict-lower(diag(beta) K K^T * Gam),  T = (I + A)^{-1}
//   T' = T diag(beta e^gamma),  T'' = T diag(beta),  W = T' K,  U = T'' V
//   P  = (Q K^T) * Gam (lower incl. diagonal)
//   Vn = U - W h
//   O  = scale (diag(e^gamma) Q h + P Vn)
//   h <- e^{gamma_C} h + K^T diag(e^{gamma_C - gamma}) Vn
//
// Kernels
//   tc_prep   one CTA per (chunk, v-head): [K;Q] K^T on the tensor core (one M = 128
//             MMA gives K K^T and Q K^T), the 64 x 64 unit-lower solve on CUDA cores
//             (one thread per column of T, the column in registers), then
//             [T';T''] K and [T';T''] V (two M = 128 MMAs: W lands in TMEM lanes 0-63,
//             U in lanes 64-127).  Writes W, U, P (bf16) and gamma to the workspace.
//   tc_fwd_state  one CTA per (sequence, v-head, 64-column slice of DV), sequential
//             over the chunks: h stays in registers (thread t = row t of h); per
//             chunk [W;Q] h (M = 128), then P Vn and K^T Vn~; TMA prefetches the next
//             chunk's tiles into the other stage while the current chunk computes.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>

#include <mutex>

#include "../../include/gdr_debug.h"
#include "gdr_internal.h"
#include "gdr_chunks.cuh"
#include "tc_common.cuh"
#include "tc_primitives.cuh"

namespace gdr {

namespace {

using namespace tcx;

// ---------------------------------------------------------------------------------
// host: tensor maps
// ---------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

}  // namespace

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  });
  return g_encode != nullptr;
}

// 3D map over a [rows][heads][cols] bf16 tensor, box = 64 columns x 1 head x 64 rows.
bool map_3d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t heads, uint64_t rows) {
  cuuint64_t dims[3] = {cols, heads, rows};
  cuuint64_t strides[2] = {cols * 2, heads * cols * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D map over a [rows][cols] matrix of `dt` (element size esz) with a box of
// box_cols x box_rows, 128-byte swizzle (box_cols * esz must be 128).
bool map_2d_box(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint32_t esz, uint64_t cols,
                uint64_t rows, uint32_t box_cols, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * esz};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D map over a [rows][cols] bf16 matrix, box = 64 columns x 64 rows.
bool map_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D map over a [rows][cols] bf16 matrix with a 32-column (64-byte) x box_rows box and
// 64-byte swizzle: in the shared-memory tile, row r's 16-byte piece c sits at piece
// position c ^ ((r >> 1) & 3).  (Unswizzled 64-byte rows make the TMA engine's
// shared-memory reads much slower.)
static bool map_2d_sw64(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// ---------------------------------------------------------------------------------
// tc_prep: W, U, P, gamma of one (chunk, v-head)
// ---------------------------------------------------------------------------------
struct PrepSmem {
  static constexpr uint32_t KQ = 0;              // [K | Q] x 2 slabs: 32 KB
  static constexpr uint32_t V = 32768;           // 2 slabs: 16 KB
  static constexpr uint32_t TT = V + 16384;      // [T' | T''] bf16: 16 KB
  static constexpr uint32_t A = TT + 16384;      // fp32 A [64][68] (row stride kLdA)
  static constexpr uint32_t TF = A + 17408;      // fp32 T [64][68]
  static constexpr uint32_t Y = TF + 17408;      // fp32 3 x [16][16] block products
  static constexpr uint32_t PS = Y + 4096;       // P (then T) staged for TMA stores: 8 KB
  static constexpr uint32_t BYTES = PS + 8192;   // 110 KB (two CTAs per SM)
};

// Row stride (floats) of the fp32 A and T tiles: rows start 16-byte aligned for vector
// loads, and 68 = 4 (mod 32) keeps 8 rows read at one column on distinct banks.
constexpr int kLdA = 68;

// 4 * N consecutive floats from shared memory (16-byte aligned) into v.
template <int N>
__device__ __forceinline__ void ld_f4(const float* __restrict__ src, float* v) {
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float4 t = reinterpret_cast<const float4*>(src)[i];
    v[4 * i] = t.x;
    v[4 * i + 1] = t.y;
    v[4 * i + 2] = t.z;
    v[4 * i + 3] = t.w;
  }
}

// T = (I + A)^{-1} for strictly lower-triangular A (fp32, row stride kLdA) by recursive
// 2 x 2 block inversion: with L = [[L11, 0], [L21, L22]], L^{-1} = [[L11^{-1}, 0],
// [-L22^{-1} L21 L11^{-1}, L22^{-1}]].  Steps: the four 16 x 16 diagonal inverses by
// forward substitution (one thread per column); the two 16 x 16 off-diagonal blocks
// of the 32 x 32 diagonal halves; the 32 x 32 lower-left block.  Every product is
// register-tiled with vector loads (all loads of a thread before its stores).  Writes the
// full T (zeros above the diagonal) into sT (row stride kLdA).  All 128 threads take part.
__device__ __forceinline__ void solve_unit_lower64(const float* __restrict__ sA, float* __restrict__ sT,
                                                   float* __restrict__ sY, int tid) {
  GDR_TRACE_INIT();
  for (int e = tid; e < 64 * kLdA / 4; e += kTcThreads) reinterpret_cast<float4*>(sT)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  __syncthreads();
  GDR_TRACE_MARK(0, 16 + 0);
  if (tid < 64) {  // diagonal 16 x 16 blocks
    const int b = tid >> 4, c = tid & 15;
    const float* Ab = sA + (16 * b) * kLdA + 16 * b;
    float col[16];
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
      float acc = (rr == c) ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < rr; ++m) acc -= Ab[rr * kLdA + m] * col[m];
      col[rr] = acc;
    }
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) sT[(16 * b + rr) * kLdA + 16 * b + c] = col[rr];
  }
  __syncthreads();
  GDR_TRACE_MARK(0, 16 + 1);
  {  // T_{2b+1,2b} = -T_{2b+1,2b+1} A_{2b+1,2b} T_{2b,2b}, b = 0, 1; thread: 1 row x 4 columns
    const int b = tid >> 6, rr = (tid >> 2) & 15, c4 = (tid & 3) * 4;
    const int r0 = 16 * (2 * b + 1), c0 = 16 * (2 * b);
    float x[16], z[16][4], o[4];
    ld_f4<4>(sA + (r0 + rr) * kLdA + c0, x);
#pragma unroll
    for (int k = 0; k < 16; ++k) ld_f4<1>(sT + (c0 + k) * kLdA + c0 + c4, z[k]);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      o[q] = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) o[q] += x[k] * z[k][q];
    }
    *reinterpret_cast<float4*>(sY + b * 256 + rr * 16 + c4) = make_float4(o[0], o[1], o[2], o[3]);
    __syncthreads();
    ld_f4<4>(sT + (r0 + rr) * kLdA + r0, x);
#pragma unroll
    for (int k = 0; k < 16; ++k) ld_f4<1>(sY + b * 256 + k * 16 + c4, z[k]);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      o[q] = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) o[q] += x[k] * z[k][q];
    }
    *reinterpret_cast<float4*>(sT + (r0 + rr) * kLdA + c0 + c4) = make_float4(-o[0], -o[1], -o[2], -o[3]);
  }
  __syncthreads();
  GDR_TRACE_MARK(0, 16 + 2);
  {  // T_[23][01] = -T_[23][23] A_[23][01] T_[01][01] (32 x 32); thread: 1 row x 8 columns
    const int rr = tid >> 2, c8 = (tid & 3) * 8;
    float o[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) o[q] = 0.f;
#pragma unroll
    for (int kh = 0; kh < 32; kh += 16) {
      float x[16], z[16][8];
      ld_f4<4>(sA + (32 + rr) * kLdA + kh, x);
#pragma unroll
      for (int k = 0; k < 16; ++k) ld_f4<2>(sT + (kh + k) * kLdA + c8, z[k]);
#pragma unroll
      for (int q = 0; q < 8; ++q)
#pragma unroll
        for (int k = 0; k < 16; ++k) o[q] += x[k] * z[k][q];
    }
    *reinterpret_cast<float4*>(sY + rr * 32 + c8) = make_float4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<float4*>(sY + rr * 32 + c8 + 4) = make_float4(o[4], o[5], o[6], o[7]);
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 8; ++q) o[q] = 0.f;
#pragma unroll
    for (int kh = 0; kh < 32; kh += 16) {
      float x[16], z[16][8];
      ld_f4<4>(sT + (32 + rr) * kLdA + 32 + kh, x);
#pragma unroll
      for (int k = 0; k < 16; ++k) ld_f4<2>(sY + (kh + k) * 32 + c8, z[k]);
#pragma unroll
      for (int q = 0; q < 8; ++q)
#pragma unroll
        for (int k = 0; k < 16; ++k) o[q] += x[k] * z[k][q];
    }
    float* dst = sT + (32 + rr) * kLdA + c8;
    *reinterpret_cast<float4*>(dst) = make_float4(-o[0], -o[1], -o[2], -o[3]);
    *reinterpret_cast<float4*>(dst + 4) = make_float4(-o[4], -o[5], -o[6], -o[7]);
  }
  __syncthreads();
  GDR_TRACE_MARK(0, 16 + 3);
}

// Publishes one finished chunk-head of the fused forward: its TMA stores (async proxy) and
// gamma (plain stores before the caller's barrier) are complete; order them before the flag
// (proxy fence) and set it with a GPU-scope release reduction (pairs with the waiter's acquire
// load; cheaper than a full fence).
__device__ __forceinline__ void publish_prep(uint32_t* flag) {
  asm volatile("fence.proxy.async.global;" ::: "memory");
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(flag) : "memory");
}

// Bounded wait until *flag != 0 (acquire at GPU scope), then orders the caller's later TMA
// loads after it.  On expiry sets `bit` in *status and returns false.
__device__ __forceinline__ bool wait_prep(const uint32_t* flag, uint32_t* status, uint32_t bit) {
  uint32_t v;
  const uint64_t t0 = tc::globaltimer_ns();
  while (true) {
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v != 0u) break;
    if (tc::globaltimer_ns() - t0 > tc::kWaitLimitNs) {
      atomicOr(status, bit);
      return false;
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// The chunk prep of a CTA's items (chunk c, v-head j).  kFused = false: the persistent grid's
// items w = blockIdx.x + k * gridDim.x in chunk-major order.  kFused = true (fused forward
// kernel): items claimed from ws.fwd_queue in the forward's step order (queue position q =
// w / Hv holds chunk ws.fwd_chunk[q]); each item's stores are waited for and counted into
// ws.fwd_flags[c * Hv + j], one item late so the wait overlaps the next item's loads.
template <bool kFused>
__device__ __forceinline__ void prep_body(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                          const CUtensorMap& tm_w, const CUtensorMap& tm_u, const CUtensorMap& tm_p,
                                          const CUtensorMap& tm_t, const Dims& d, const float* __restrict__ g,
                                          const bf16* __restrict__ beta, const Workspace& ws, int write_T,
                                          unsigned char* sm) {
  // kFused: one CTA per SM with the state's shared memory, so the q/k/v tiles have two stages
  // (the second after PrepSmem::BYTES, checked at the fused kernel) and the next item's tiles
  // load during this item
  __shared__ uint64_t bar_tma[2], bar_mma;
  __shared__ uint32_t tmem_slot;
  __shared__ float s_gam[64], s_beta[64], s_bexp[64], s_carry;
  __shared__ int s_item[4];  // the current item and its chunk; kFused: the next (claimed ahead)
  const int tid = threadIdx.x, warp = tid >> 5;
  const int Hv = d.Hv;

  if (tid == 0) {
    tc::mbar_init(&bar_tma[0], 1);
    tc::mbar_init(&bar_tma[1], 1);
    tc::mbar_init(&bar_mma, 1);
    tc::fence_barrier_init();
  }
  if (warp == 0) tc::tmem_alloc<256>(&tmem_slot);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tbase = tmem_slot;
  GDR_TRACE_INIT();
  GDR_TRACE_CTA_BEGIN();
  bool ok = true;
  uint32_t item_par = 0;  // phase parity of bar_tma for the current item (bar_mma: 2 per item)
  const int n_items = kFused ? idx_step_off(d, ws, idx_n_steps(d, ws)) * Hv : d.max_chunks * Hv;
  // the next item and its chunk into s_item[slot], s_item[slot + 1] (thread 0 decides; everyone
  // reads them after a barrier)
  auto next_item = [&](int w, int slot) {
    if (kFused) {
      const int q = (int)atomicAdd(ws.fwd_queue, 1u);
      s_item[slot] = q < n_items ? q : n_items;
      s_item[slot + 1] = q < n_items ? idx_fwd_chunk(d, ws, q / Hv) : 0;
    } else {
      w = w < 0 ? (int)blockIdx.x : w + (int)gridDim.x;
      s_item[slot] = w;
      s_item[slot + 1] = w < n_items ? w / Hv : 0;
    }
  };
  // q/k/v tiles of item w (chunk cc) into stage st
  auto issue_loads = [&](int w, int cc, int st) {
    const int j2 = w % Hv, i2 = j2 / d.G, tt = idx_chunk(d, ws, cc).y;
    unsigned char* kq = sm + (st ? PrepSmem::BYTES : PrepSmem::KQ);
    unsigned char* vv = sm + (st ? PrepSmem::BYTES + 2 * 16384 : PrepSmem::V);
    tc::mbar_arrive_expect_tx(&bar_tma[st], 6 * kSlab);
    tc::tma_load_3d(kq, &tm_k, &bar_tma[st], 0, i2, tt);
    tc::tma_load_3d(kq + 2 * kSlab, &tm_k, &bar_tma[st], 64, i2, tt);
    tc::tma_load_3d(kq + kSlab, &tm_q, &bar_tma[st], 0, i2, tt);
    tc::tma_load_3d(kq + 3 * kSlab, &tm_q, &bar_tma[st], 64, i2, tt);
    tc::tma_load_3d(vv, &tm_v, &bar_tma[st], 0, j2, tt);
    tc::tma_load_3d(vv + kSlab, &tm_v, &bar_tma[st], 64, j2, tt);
  };
  if (tid == 0) {
    next_item(-1, 0);
    if (kFused && s_item[0] < n_items) issue_loads(s_item[0], s_item[1], 0);
  }
  __syncthreads();
  int witem = s_item[0], c = s_item[1];
  int pub = -1;  // kFused: the flag index of the previous item, not yet published
  int it = 0;    // kFused: items done (stage it & 1, phase (it >> 1) & 1)
  // !kFused, thread 0: the item whose tiles are already loading (issued once this item's last
  // product had read its K/Q/V tiles)
  int prefetched = -1;
  while (witem < n_items && ok) {
  const int j = witem % Hv, i = j / d.G;
  const int4 ci = idx_chunk(d, ws, c);
  const int len = ci.z, t0 = ci.y;
  const size_t ch = (size_t)c * Hv + j;
  const int st = kFused ? (it & 1) : 0;
  unsigned char* const kq_t = sm + (st ? PrepSmem::BYTES : PrepSmem::KQ);
  unsigned char* const v_t = sm + (st ? PrepSmem::BYTES + 2 * 16384 : PrepSmem::V);
  if (len > 0) {  // (an empty chunk slot: uniform across the CTA)
  if (tid == 0) {
    GDR_DELAY(1);
    if (kFused) {  // claim the next item and load its tiles into the other stage, whose last
                   // reader (two items ago) is done; then publish the previous item
      next_item(witem, 2);
      if (s_item[2] < n_items) issue_loads(s_item[2], s_item[3], st ^ 1);
      if (pub >= 0) {
        tc::bulk_wait<0>();
        GDR_DELAY(2);
        publish_prep(ws.fwd_flags + pub);
        pub = -1;
      }
    } else if (prefetched != witem) {
      issue_loads(witem, c, 0);
    }
  }
  // gamma (in-chunk cumsum of g) and beta, zero past the chunk end
  {
    float x = 0.f, b = 0.f;
    if (tid < 64 && tid < len) {
      x = g[(size_t)(t0 + tid) * Hv + j];
      b = __bfloat162float(beta[(size_t)(t0 + tid) * Hv + j]);
    }
    x = chunk_cumsum64(x, tid, &s_carry);
    if (tid < 64) {
      s_gam[tid] = x;
      s_beta[tid] = b;
      s_bexp[tid] = b * fexp(x);  // beta_s e^{gamma_s}
    }
  }
  ok = __syncthreads_and(tc::mbar_wait(&bar_tma[st], kFused ? (uint32_t)(it >> 1) & 1u : item_par, ws.status,
                                       kDevErrTimeoutPrep));
  GDR_TRACE_MARK(0, 0);
  const uint32_t s_kq = tc::smem_u32(kq_t), s_v = tc::smem_u32(v_t);
  const uint32_t s_tt = tc::smem_u32(sm + PrepSmem::TT);
  if (ok && tid == 0) {
    tc::tc_fence_after();
    const uint32_t id = tc::idesc_bf16(128, 64, 0, 0);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      tc::mma_bf16(tbase, tc::kmajor_step_desc(s_kq, 2 * kSlab, kk), tc::kmajor_step_desc(s_kq, 2 * kSlab, kk), id,
                   kk > 0);
    tc::mma_commit(&bar_mma);
  }
  ok = __syncthreads_and(ok && tc::mbar_wait(&bar_mma, 0, ws.status, kDevErrTimeoutPrep));
  GDR_TRACE_MARK(0, 1);
  tc::tc_fence_after();
  float* sA = reinterpret_cast<float*>(sm + PrepSmem::A);
  if (ok) {
    float row[64];
    tmem_ld64(tbase, warp, 0, row);
    const int r = tid & 63;
    const float gr = s_gam[r];
    if (tid < 64) {  // A row r (all loads before the stores: smem pointers may alias)
      const float br = s_beta[r];
      float gs[64];
#pragma unroll
      for (int s = 0; s < 64; ++s) gs[s] = s_gam[s];
#pragma unroll
      for (int s = 0; s < 64; ++s) row[s] = (s < r && r < len) ? br * fexp(gr - gs[s]) * row[s] : 0.f;
#pragma unroll
      for (int s = 0; s < 64; s += 4)
        *reinterpret_cast<float4*>(sA + r * kLdA + s) = make_float4(row[s], row[s + 1], row[s + 2], row[s + 3]);
    } else {  // P row r
#pragma unroll
      for (int s = 0; s < 64; ++s) row[s] = (s <= r && r < len) ? row[s] * fexp(gr - s_gam[s]) : 0.f;
      st_row_bf16(sm + PrepSmem::PS, r, row);
    }
  }
  tc::fence_proxy_async_smem();
  __syncthreads();
  if (ok && tid == 0) {
    tc::tma_store_2d(&tm_p, sm + PrepSmem::PS, 0, (int)(ch * 64));
    tc::bulk_commit();
  }
  GDR_TRACE_MARK(0, 2);
  // T = (I + A)^{-1}
  if (tid == 0) tc::bulk_wait_read<0>();  // P has left its staging tile (reused for T below)
  GDR_TRACE_MARK(0, 8);
  float* sT = reinterpret_cast<float*>(sm + PrepSmem::TF);
  solve_unit_lower64(sA, sT, reinterpret_cast<float*>(sm + PrepSmem::Y), tid);
  GDR_TRACE_MARK(0, 9);
  if (ok) {  // rows of T' = T diag(beta e^gamma) (threads 0-63), T'' = T diag(beta) (64-127)
    const int r = tid & 63;
    float x[64];
    ld_f4<16>(sT + r * kLdA, x);
#pragma unroll
    for (int s2 = 0; s2 < 64; ++s2) x[s2] *= (tid < 64 ? s_bexp[s2] : s_beta[s2]);
    st_row_bf16(sm + PrepSmem::TT + (tid < 64 ? 0 : kSlab), r, x);
    if (write_T && tid < 64) {  // T itself for the backward
      ld_f4<16>(sT + r * kLdA, x);
      st_row_bf16(sm + PrepSmem::PS, r, x);
    }
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  GDR_TRACE_MARK(0, 3);
  if (ok && tid == 0) {
    if (write_T) {
      tc::tma_store_2d(&tm_t, sm + PrepSmem::PS, 0, (int)(ch * 64));
      tc::bulk_commit();
    }
    tc::tc_fence_after();
    // W = T' K (lanes 0-63 of cols [0,128)), U = T'' V (lanes 64-127 of cols [128,256))
    const uint32_t id = tc::idesc_bf16(128, 128, 0, 1);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t a = tc::kmajor_step_desc(s_tt, kSlab, kk);
      tc::mma_bf16(tbase, a, tc::mnmajor_step_desc(s_kq, 2 * kSlab, kk), id, kk > 0);
      tc::mma_bf16(tbase + 128, a, tc::mnmajor_step_desc(s_v, kSlab, kk), id, kk > 0);
    }
    tc::mma_commit(&bar_mma);
  }
  ok = __syncthreads_and(ok && tc::mbar_wait(&bar_mma, 1, ws.status, kDevErrTimeoutPrep));
  GDR_TRACE_MARK(0, 4);
  tc::tc_fence_after();
  // !kFused: the products are done with this item's K/Q/V tiles, so the next item's tiles load
  // into them now, overlapping the stores below (W and U are staged in the T' and A tiles, free
  // too)
  if (!kFused && ok && tid == 0) {
    const int wn = witem + (int)gridDim.x;
    if (wn < n_items && idx_chunk(d, ws, wn / Hv).z > 0) {
      issue_loads(wn, wn / Hv, 0);
      prefetched = wn;
    }
  }
  if (ok) {  // W rows (threads 0-63) and U rows (threads 64-127) staged in the free T' and A tiles
    const int r = tid & 63;
    const int col = tid < 64 ? 0 : 128;
    unsigned char* stg = sm + (tid < 64 ? PrepSmem::TT : PrepSmem::A);
    float v[64];
    tmem_ld64(tbase, warp, col, v);
    st_row_bf16(stg, r, v);
    tmem_ld64(tbase, warp, col + 64, v);
    st_row_bf16(stg + kSlab, r, v);
    if (tid < 64) ws.gam[ch * 64 + tid] = s_gam[tid];
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  if (ok && tid == 0) {
    tc::tma_store_2d(&tm_w, sm + PrepSmem::TT, 0, (int)(ch * 64));
    tc::tma_store_2d(&tm_w, sm + PrepSmem::TT + kSlab, 64, (int)(ch * 64));
    tc::tma_store_2d(&tm_u, sm + PrepSmem::A, 0, (int)(ch * 64));
    tc::tma_store_2d(&tm_u, sm + PrepSmem::A + kSlab, 64, (int)(ch * 64));
    tc::bulk_commit();
  }
  if (tid == 0) tc::bulk_wait_read<0>();  // staging tiles read before the next item writes them
  GDR_TRACE_MARK(0, 5);
  item_par ^= 1;
  ++it;
  if (kFused && tid == 0) pub = (int)ch;
  }  // len > 0
  if (!kFused && tid == 0) next_item(witem, 0);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  witem = s_item[kFused ? 2 : 0];
  c = s_item[kFused ? 3 : 1];
  __syncthreads();  // s_item is rewritten by the next claim
  }  // items
  if (kFused && tid == 0 && pub >= 0) {  // the last item (its gamma stores are behind the barriers above)
    tc::bulk_wait<0>();
    publish_prep(ws.fwd_flags + pub);
  }
  GDR_TRACE_CTA_END();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, 256);
  if (tid == 0) {  // a later role of this CTA (none today) would initialise them again
    tc::mbar_inval(&bar_tma[0]);
    tc::mbar_inval(&bar_tma[1]);
    tc::mbar_inval(&bar_mma);
  }
}

__global__ void __launch_bounds__(kTcThreads) tc_prep_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                             const __grid_constant__ CUtensorMap tm_k,
                                                             const __grid_constant__ CUtensorMap tm_v,
                                                             const __grid_constant__ CUtensorMap tm_w,
                                                             const __grid_constant__ CUtensorMap tm_u,
                                                             const __grid_constant__ CUtensorMap tm_p,
                                                             const __grid_constant__ CUtensorMap tm_t, Dims d,
                                                             const float* __restrict__ g,
                                                             const bf16* __restrict__ beta, Workspace ws,
                                                             int write_T) {
  extern __shared__ unsigned char smem_raw[];
  prep_body<false>(tm_q, tm_k, tm_v, tm_w, tm_u, tm_p, tm_t, d, g, beta, ws, write_T, align1024(smem_raw));
}

// ---------------------------------------------------------------------------------
// tc_fwd_state: sequential chunk walk of one (sequence, v-head, 32-wide DV slice).
// The recurrence over chunks is serial, so the DV columns of the state are split
// four ways (they evolve independently) to put 4 x sequences x v-heads CTAs on the
// SMs, and each chunk's output rows are finished while the next chunk's first
// product runs.
// ---------------------------------------------------------------------------------
constexpr int kStateSlices = 4;  // DV = 128 as four 32-column slices

// kSingle = false: two stages of the chunk tiles, so all of chunk c + 1's tiles load while
// chunk c runs (~161 KB, one CTA per SM).  kSingle = true: one buffer per tile, each refilled
// for the next chunk as soon as its last reader is done ([W|Q] and gamma after the first
// product, U after the Vn epilogue, K and P once the previous chunk's P Vn has run): ~97 KB,
// two CTAs per SM, for grids larger than the SM count.  A chain is ~20 % slower single-buffered.
template <bool kSingle>
struct StateSmem {
  static constexpr uint32_t NST = kSingle ? 1 : 2;
  // per stage: [W|Q] x 2 slabs (32 KB), K 2 slabs (16 KB), [U | P] (16 KB)
  static constexpr uint32_t STAGE = 65536;
  static constexpr uint32_t WQ = 0, K = 32768, U = 49152, P = 57344;
  static constexpr uint32_t HT = NST * STAGE;     // h^T slice (bf16, K-major B operand): 2 slabs of 32 rows
  static constexpr uint32_t VNT = HT + 8192;      // Vn^T slice: 32 rows x 64 tokens (4 KB)
  static constexpr uint32_t VTT = VNT + 4096;     // (e^{gamma_C - gamma} Vn)^T slice (4 KB)
  static constexpr uint32_t HS = VTT + 4096;      // h slice staged for the h_saved store: fp32 (16 KB) or bf16 (8 KB)
  static constexpr uint32_t GAM = HS + 16384;     // gamma of each stage: 256 B each
  // two stages: chunk c's P tile rotates over three buffers (the stages' P slots and PX), so a
  // chunk's P is loaded where P Vn of chunk c - 3 read, which the previous chunk's first
  // product has waited for; single buffer: the stage's slot
  static constexpr uint32_t PX = (GAM + NST * 256 + 1023) / 1024 * 1024;
  static constexpr uint32_t BYTES = kSingle ? GAM + NST * 256 : PX + 8192;
  __host__ __device__ static constexpr uint32_t pbuf(int c) {
    return c % 3 == 2 ? PX : (uint32_t)(c % 3) * STAGE + P;
  }
};

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

// Column `col` of a K-major operand tile of 32 rows (one row per DV column of the
// slice): v[b] goes to row b.  Within a warp the 32 threads hold 32 consecutive
// columns, so each store instruction touches one 64-byte run of a row.
__device__ __forceinline__ void st_col32_bf16(unsigned char* tile, int col, const float* v) {
#pragma unroll
  for (int b = 0; b < 32; ++b)
    *reinterpret_cast<bf16*>(tile + tc::sw128_off(b, col, 32)) = __float2bfloat16_rn(v[b]);
}

// Row `row` (32 fp32 -> bf16, 64 bytes) of a 64-byte-swizzled [rows][32] bf16 tile: piece
// c at piece position c ^ ((row >> 1) & 3), which also spreads the 32 rows of a warp's
// store instruction over all 32 banks.
__device__ __forceinline__ void st_row_bf16x32_sw64(unsigned char* tile, int row, const float* v) {
  uint4 w[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t* wp = reinterpret_cast<uint32_t*>(&w[c]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 b = __floats2bfloat162_rn(v[c * 8 + 2 * e], v[c * 8 + 2 * e + 1]);
      wp[e] = *reinterpret_cast<uint32_t*>(&b);
    }
  }
  const int sw = (row >> 1) & 3;
#pragma unroll
  for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(tile + row * 64 + ((c ^ sw) << 4)) = w[c];
}

// What one state unit computes: a (sequence, v-head, 32-column DV slice) over a range of its
// chunks, from a start state to an end state.  Without segments the range is the whole
// sequence, from S0 to S_T.  The context-parallel passes (CpArgs) cut it into segments:
//   first pass, per (sequence, v-head): segment 0 from S0 with every output, its end state into
//     X[1] (or S_T when it is the only segment); and for each segment s = 1 .. nseg - 2 its
//     zero-start end state R[s] (no outputs) and its transition M[s] = Phi_s (the same
//     recurrence with U = 0 started from the identity's columns: h' = (e^{gamma_C} I - K~^T W) h);
//   second pass: segments s = 1 .. nseg - 1 from X[s] with every output, the last into S_T.
struct StateUnit {
  int n, j, slice;
  int c_begin, c_end;  // chunk range
  int t_seq, L;        // first token of the range, tokens from there to the sequence end
  const float* h0;     // start state of (n, j) (nullptr: zero) ...
  int h0_kv;           // ... stored [DK][DV] (else [DV][DK])
  bool h0_eye;         // start from the identity's columns instead
  float* h1;           // end state (nullptr: not written), orientation h1_kv
  int h1_kv;
  bool outputs;        // o, h_saved and the saved Vn
  bool zero_u;         // U taken as zero (transition columns)
  bool skip;           // nothing to compute
};

__device__ __forceinline__ int state_units_per_chain(const CpArgs& cp) {
  return cp.pass == 1 ? 4 + 8 * (cp.P - 2) : (cp.pass == 3 ? 4 * (cp.P - 1) : 4);
}

// Unit `cta` of a state launch: (sequence rank, v-head, unit within the chain), the last fastest.
__device__ __forceinline__ StateUnit state_unit(const Dims& d, const Workspace& ws, const CpArgs& cp, int cta,
                                                const float* S0, float* S_T) {
  StateUnit u{};
  const int per = state_units_per_chain(cp);
  const int k = cta % per, rest = cta / per;
  u.j = rest % d.Hv;
  u.n = idx_seq(d, ws, rest / d.Hv);
  int seg = 0, mode = 0;  // mode 0: every output; 1: zero start; 2: transition
  if (cp.pass == 1 && k >= 4) {
    const int e = k - 4;
    seg = 1 + e / 8;
    u.slice = e & 3;
    mode = (e & 7) < 4 ? 1 : 2;
  } else if (cp.pass == 3) {
    seg = 1 + k / 4;
    u.slice = k & 3;
  } else {
    u.slice = k;
  }
  const int s0 = idx_seq_off(d, ws, u.n), s1 = idx_seq_off(d, ws, u.n + 1);
  const int t_seq = d.cu ? d.cu[u.n] : u.n * d.T;
  const int L = d.cu ? d.cu[u.n + 1] - t_seq : d.T;
  const size_t sb = ((size_t)u.n * d.Hv + u.j) * 128 * 128;
  u.c_begin = s0;
  u.c_end = s1;
  u.t_seq = t_seq;
  u.L = L;
  u.h0 = S0 ? S0 + sb : nullptr;
  u.h0_kv = d.layout == 0;
  u.h1 = S_T ? S_T + sb : nullptr;
  u.h1_kv = d.layout == 0;
  u.outputs = true;
  if (cp.pass == 0) return u;
  const int3 sg = cp_segment(s0, s1, cp.P, seg);
  auto mat = [&](float* base, int s2) { return base + (sb * cp.P) + (size_t)s2 * 128 * 128; };
  u.c_begin = sg.x;
  u.c_end = sg.y;
  u.t_seq = t_seq + (sg.x - s0) * kChunk;
  u.L = L - (sg.x - s0) * kChunk;
  if (cp.pass == 1) {
    if (mode == 0) {
      if (sg.z > 1) {
        u.h1 = mat(cp.X, 1);
        u.h1_kv = 1;
      }
    } else {
      u.skip = seg >= sg.z - 1;
      u.outputs = false;
      u.h0 = nullptr;
      u.h0_eye = mode == 2;
      u.zero_u = mode == 2;
      u.h1 = mat(mode == 2 ? cp.M : cp.R, seg);
      u.h1_kv = mode == 2 ? 0 : 1;  // M transposed: the scan reads M^T[k][r] = M[r][k] as rows
    }
  } else {
    u.skip = seg >= sg.z;
    u.h0 = mat(cp.X, seg);
    u.h0_kv = 1;
    if (seg != sg.z - 1) u.h1 = nullptr;
  }
  return u;
}

// One state unit (see StateUnit).  kFused (fused
// forward kernel, double-buffered): chunk c's W, U, P and gamma are loaded only after the prep
// role has counted (c, v-head) in ws.fwd_flags; the copy thread waits for chunk c + 1 while
// chunk c's first product runs, off the chain.
template <bool kSingle, bool kFused, bool kModes>
__device__ __forceinline__ void state_body(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_w,
                                           const CUtensorMap& tm_u, const CUtensorMap& tm_p,
                                           const CUtensorMap& tm_hs, const Dims& d, bf16* __restrict__ o,
                                           const Workspace& ws, const StateUnit& un, unsigned char* sm) {
  using SS = StateSmem<kSingle>;
  // two stages: bar_load[st] per stage; single buffers: bar_load[0] = [W|Q] and gamma,
  // bar_load[1] = U, bar_kp = K and P (one phase per chunk each)
  __shared__ uint64_t bar_load[2], bar_kp, bar_mma, bar_pv;
  __shared__ uint32_t tmem_slot;
  // the slices of one (sequence, head) are adjacent units, so they share its W/Q/K tiles in L2
  const int j = un.j, i = j / d.G;
  const int dv0 = un.slice * 32;
  const int tid = threadIdx.x, warp = tid >> 5;
  // thread 0 issues the MMAs; thread 32 (the "copy thread") issues every TMA load and
  // store and waits on their bulk groups, so neither kind of issue delays the other
  constexpr int kCopyTid = 32;
  const int Hv = d.Hv;
  const int c_begin = un.c_begin, c_end = un.c_end;
  const int t_seq = un.t_seq;  // first token of the range
  const int L = un.L;          // tokens from there to the sequence end
  // kModes: the unit may be a first-pass map (no outputs, or U = 0 from the identity); without
  // it those cases are compiled out (as the plain chain and the second pass run)
  const bool outputs = !kModes || un.outputs, zero_u = kModes && un.zero_u, h0_eye = kModes && un.h0_eye;

  if (tid == 0) {
    tc::mbar_init(&bar_load[0], 1);
    tc::mbar_init(&bar_load[1], 1);
    tc::mbar_init(&bar_kp, 1);
    tc::mbar_init(&bar_mma, 1);
    tc::mbar_init(&bar_pv, 1);
    tc::fence_barrier_init();
  }
  if (warp == 0) tc::tmem_alloc<128>(&tmem_slot);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tbase = tmem_slot;
  // TMEM: [W;Q] h^T (0-31), [U;P] Vn (32-63; lanes 64-127 = P Vn), K^T Vn~ (64-95)
  const uint32_t D1 = tbase, D2 = tbase + 32, D3 = tbase + 64;

  // h row `tid` (dk = tid), columns dv0 .. dv0 + 31
  float h[32];
#pragma unroll
  for (int b = 0; b < 32; ++b)
    h[b] = h0_eye ? (tid == dv0 + b ? 1.f : 0.f)
           : un.h0   ? un.h0[un.h0_kv ? (size_t)tid * 128 + dv0 + b : (size_t)(dv0 + b) * 128 + tid]
                     : 0.f;
  // two stages: every tile of chunk c into stage st, P into its rotating buffer (whose last
  // reader, P Vn of chunk c - 3, completed before chunk c - 2's first product did)
  auto issue_loads = [&](int c, int st) {
    const int tc0 = t_seq + (c - c_begin) * 64;
    const size_t chh = (size_t)c * Hv + j;
    unsigned char* base = sm + st * SS::STAGE;
    // Q and P feed only the output rows: units without outputs leave them out (the products
    // that read those tiles then fill TMEM lanes no one reads)
    tc::mbar_arrive_expect_tx(&bar_load[st], (outputs ? 8 : 5) * kSlab + 256);
    tc::bulk_load(sm + SS::GAM + st * 256, ws.gam + chh * 64, 256, &bar_load[st]);
    tc::tma_load_2d(base + SS::WQ, &tm_w, &bar_load[st], 0, (int)(chh * 64));
    tc::tma_load_2d(base + SS::WQ + 2 * kSlab, &tm_w, &bar_load[st], 64, (int)(chh * 64));
    if (outputs) {
      tc::tma_load_3d(base + SS::WQ + kSlab, &tm_q, &bar_load[st], 0, i, tc0);
      tc::tma_load_3d(base + SS::WQ + 3 * kSlab, &tm_q, &bar_load[st], 64, i, tc0);
    }
    tc::tma_load_3d(base + SS::K, &tm_k, &bar_load[st], 0, i, tc0);
    tc::tma_load_3d(base + SS::K + kSlab, &tm_k, &bar_load[st], 64, i, tc0);
    tc::tma_load_2d(base + SS::U, &tm_u, &bar_load[st], dv0 & 64, (int)(chh * 64));  // 64-col tile
    if (outputs) tc::tma_load_2d(sm + SS::pbuf(c - c_begin), &tm_p, &bar_load[st], 0, (int)(chh * 64));
  };
  auto load_wq = [&](int c) {  // single buffers: [W|Q] and gamma of chunk c
    const int tc0 = t_seq + (c - c_begin) * 64;
    const size_t chh = (size_t)c * Hv + j;
    tc::mbar_arrive_expect_tx(&bar_load[0], (outputs ? 4 : 2) * kSlab + 256);
    tc::bulk_load(sm + SS::GAM, ws.gam + chh * 64, 256, &bar_load[0]);
    tc::tma_load_2d(sm + SS::WQ, &tm_w, &bar_load[0], 0, (int)(chh * 64));
    tc::tma_load_2d(sm + SS::WQ + 2 * kSlab, &tm_w, &bar_load[0], 64, (int)(chh * 64));
    if (outputs) {
      tc::tma_load_3d(sm + SS::WQ + kSlab, &tm_q, &bar_load[0], 0, i, tc0);
      tc::tma_load_3d(sm + SS::WQ + 3 * kSlab, &tm_q, &bar_load[0], 64, i, tc0);
    }
  };
  auto load_u = [&](int c) {  // single buffers: U of chunk c
    const size_t chh = (size_t)c * Hv + j;
    tc::mbar_arrive_expect_tx(&bar_load[1], kSlab);
    tc::tma_load_2d(sm + SS::U, &tm_u, &bar_load[1], dv0 & 64, (int)(chh * 64));
  };
  auto load_kp = [&](int c) {  // single buffers: K and P of chunk c
    const int tc0 = t_seq + (c - c_begin) * 64;
    const size_t chh = (size_t)c * Hv + j;
    tc::mbar_arrive_expect_tx(&bar_kp, (outputs ? 3 : 2) * kSlab);
    tc::tma_load_3d(sm + SS::K, &tm_k, &bar_kp, 0, i, tc0);
    tc::tma_load_3d(sm + SS::K + kSlab, &tm_k, &bar_kp, 64, i, tc0);
    if (outputs) tc::tma_load_2d(sm + SS::P, &tm_p, &bar_kp, 0, (int)(chh * 64));
  };
  // kFused: the prep role's flag of chunk c (bounded wait; on expiry the loads are left out
  // and the consumer's own bounded wait ends the chain).  (Reading the next chunk's flag a
  // chunk early with a relaxed load and an acquire fence when it was set measured slower: the
  // fence costs more than the poll it replaces.)
  // A thread of warp 3 (kPollTid) reads chunk c + 2's flag (acquire) while chunk c's
  // recurrence product runs and leaves what it saw in s_seen; the copy thread then skips its own
  // poll of that chunk when the flag was already set (ordered through the CTA barriers between).
  constexpr int kPollTid = 96;
  __shared__ uint32_t s_seen[2];
  if (tid == 0) s_seen[0] = s_seen[1] = 0u;
  auto prep_ready = [&](int c) {
    if (!kFused) return true;
    if (c - c_begin >= 2 && s_seen[c & 1] != 0u) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      return true;
    }
    return wait_prep(ws.fwd_flags + (size_t)c * Hv + j, ws.status, kDevErrTimeoutFwd);
  };
  if (tid == kCopyTid && c_begin < c_end && prep_ready(c_begin)) {
    if (kSingle) {
      load_wq(c_begin);
      load_u(c_begin);
      load_kp(c_begin);
    } else {
      issue_loads(c_begin, 0);
    }
  }
  static_assert(!(kSingle && kFused), "the fused forward runs the double-buffered state");
  st_col32_bf16(sm + SS::HT, tid, h);

  bool ok = true;
  uint32_t mma_phase = 0;
  GDR_TRACE_INIT();
  const uint32_t s_ht = tc::smem_u32(sm + SS::HT), s_vnt = tc::smem_u32(sm + SS::VNT);
  const uint32_t s_vtt = tc::smem_u32(sm + SS::VTT);
  const int r = tid & 63;
  // output rows of the previous chunk, finished during this chunk's first product
  // (warps 2-3: row r = tid - 64): (Q h)[r] slice, e^{gamma_r}, chunk start and length
  float xq[32];
  float p_eg = 0.f;
  int p_t0 = 0, p_len = 0;
  auto finish_o = [&](uint32_t pv_phase) {  // o[r] = scale (e^{gamma_r} (Q h)[r] + (P Vn)[r]) of the previous chunk
    float y[32];
    if (!tc::mbar_wait(&bar_pv, pv_phase, ws.status, kDevErrTimeoutFwd)) return;
    tc::tc_fence_after();
    tmem_ld32w(tbase, warp, 32, y);
    if (r < p_len && outputs) {
#pragma unroll
      for (int b = 0; b < 32; ++b) y[b] = d.scale * (p_eg * xq[b] + y[b]);
      st_global_bf16x32(o + ((size_t)(p_t0 + r) * Hv + j) * 128 + dv0, y);
    }
  };
  for (int c = c_begin; c < c_end && ok; ++c) {
    const int it = c - c_begin, st = kSingle ? 0 : it & 1;
    const uint32_t ld_phase = kSingle ? it & 1 : (it >> 1) & 1;  // phase of this chunk's tile barriers
    const int t0 = t_seq + it * 64;
    const int len = min(64, L - it * 64);
    const size_t chh = (size_t)c * Hv + j;
    // h^T (bf16 B operand) was written at the end of the previous chunk / before the loop; one
    // barrier publishes it and this chunk's tiles
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    GDR_TRACE_MARK(1, 0);
    ok = __syncthreads_and(tc::mbar_wait(&bar_load[st], ld_phase, ws.status, kDevErrTimeoutFwd));
    GDR_TRACE_MARK(1, 1);
    const float* sgam = reinterpret_cast<const float*>(sm + SS::GAM + st * 256);
    const float gC = sgam[len - 1];
    const float gr = sgam[r];
    unsigned char* stg = sm + st * SS::STAGE;
    const uint32_t s_wq = tc::smem_u32(stg + SS::WQ), s_k = tc::smem_u32(stg + SS::K);
    // A operand of P Vn: P as rows 64-127; rows 0-63 (the 8 KB before it) give unused lanes
    const uint32_t s_up = kSingle ? tc::smem_u32(stg + SS::U) : tc::smem_u32(sm + SS::pbuf(it)) - 8192u;
    if (ok && tid == 0) {
      tc::tc_fence_after();
      const uint32_t id = tc::idesc_bf16(128, 32, 0, 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // [W;Q] h
        tc::mma_bf16(D1, tc::kmajor_step_desc(s_wq, 2 * kSlab, kk), tc::kmajor_step_desc(s_ht, 4096, kk), id, kk > 0);
      tc::mma_commit(&bar_mma);
    }
    GDR_TRACE_MARK(1, 7);
    // two stages: chunk c + 1's tiles go where chunk c - 1's were
    if (tid == kCopyTid) GDR_DELAY(3);
    if (!kSingle && tid == kCopyTid && c + 1 < c_end && prep_ready(c + 1)) issue_loads(c + 1, st ^ 1);
    // single buffers: this chunk's K and P, once the previous chunk's P Vn (their last
    // reader) has run
    if (kSingle && ok && tid == kCopyTid && it > 0 &&
        tc::mbar_wait(&bar_pv, (it - 1) & 1, ws.status, kDevErrTimeoutFwd))
      load_kp(c);
    GDR_TRACE_MARK(1, 8);
    // while [W;Q] h runs: stage the chunk-start state (fp32) for its h_saved store, and
    // finish the previous chunk's output rows (P Vn is still in TMEM)
    if (d.h_bf16)  // bf16 saved states: a 64-byte-swizzled [128][32] bf16 tile
      st_row_bf16x32_sw64(sm + SS::HS, tid, h);
    else
      st_row_f32x32(sm + SS::HS, tid, h);
    if (ok && warp >= 2 && it > 0) finish_o((it - 1) & 1);
    tc::fence_proxy_async_smem();
    GDR_TRACE_MARK(1, 6);
    ok = __syncthreads_and(ok && tc::mbar_wait(&bar_mma, mma_phase, ws.status, kDevErrTimeoutFwd));
    mma_phase ^= 1;
    tc::tc_fence_after();
    if (ok && tid == kCopyTid) {  // h_saved[chunk] rows 0..127, columns dv0..dv0+31
      if (outputs) {
        tc::tma_store_2d(&tm_hs, sm + SS::HS, dv0, (int)(chh * 128));
        tc::bulk_commit();
      }
      if (kSingle && c + 1 < c_end) load_wq(c + 1);  // [W|Q] and gamma were last read by [W;Q] h
    }
    GDR_TRACE_MARK(1, 2);
    float vn_keep[32];  // saved factors: this thread's Vn row slice, stored once the chain has moved on
    if (ok) {
      if (warp < 2) {  // Vn = U - W h (rows >= len are zero: W and U are zero there)
        if (warp == 1) GDR_DELAY(4);
        float x[32], u[32];
        const bool uok = !kSingle || __all_sync(0xffffffffu, tc::mbar_wait(&bar_load[1], ld_phase, ws.status,
                                                                            kDevErrTimeoutFwd));
        tmem_ld32w(tbase, warp, 0, x);
        if (uok) ld_halfrow_bf16(stg + SS::U, r, (dv0 >> 5) & 1, u);
#pragma unroll
        for (int b = 0; b < 32; ++b) u[b] = uok ? (zero_u ? -x[b] : u[b] - x[b]) : 0.f;
        st_col32_bf16(sm + SS::VNT, r, u);
#pragma unroll
        for (int b = 0; b < 32; ++b) vn_keep[b] = u[b];
        const float dec = fexp(gC - gr);
#pragma unroll
        for (int b = 0; b < 32; ++b) u[b] *= dec;
        st_col32_bf16(sm + SS::VTT, r, u);
      } else {  // keep (Q h)[r] for the output rows
        tmem_ld32w(tbase, warp, 0, xq);
        p_eg = fexp(gr);
        p_t0 = t0;
        p_len = len;
      }
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    GDR_TRACE_MARK(1, 3);
    if (kFused && tid == kPollTid && c + 2 < c_end) {
      GDR_DELAY(6);
      uint32_t v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ws.fwd_flags + (size_t)(c + 2) * Hv + j)
                   : "memory");
      s_seen[(c + 2) & 1] = v;
    }
    if (kSingle && ok && tid == kCopyTid && c + 1 < c_end) load_u(c + 1);  // U was last read just above
    if (ok && tid == 0 && (!kSingle || tc::mbar_wait(&bar_kp, ld_phase, ws.status, kDevErrTimeoutFwd))) {
      GDR_DELAY(5);
      tc::tc_fence_after();
      const uint32_t id = tc::idesc_bf16(128, 32, 0, 0);
      const uint32_t idt = tc::idesc_bf16(128, 32, 1, 0);
      // K^T Vn~ (A = K^T, the MN-major view of the K tile) feeds the recurrence: first,
      // with its own commit
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_bf16(D3, tc::mnmajor_step_desc(s_k, kSlab, kk), tc::kmajor_step_desc(s_vtt, 4096, kk), idt, kk > 0);
      tc::mma_commit(&bar_mma);
      // P Vn for the output rows: rows 64-127 of this A operand are P (rows 0-63: unused lanes)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_bf16(D2, tc::kmajor_step_desc(s_up, kSlab, kk), tc::kmajor_step_desc(s_vnt, 4096, kk), id, kk > 0);
      tc::mma_commit(&bar_pv);
    }
    // saved factors: Vn replaces U in the saved buffer (the backward reads Vn; each slice writes
    // only its own columns, which no other CTA reads), off the chain: after the MMA issue
    if (ok && d.save_wy && warp < 2 && outputs)
      st_global_bf16x32(reinterpret_cast<bf16*>(ws.U) + (chh * 64 + r) * 128 + dv0, vn_keep);
    ok = __syncthreads_and(ok && tc::mbar_wait(&bar_mma, mma_phase, ws.status, kDevErrTimeoutFwd));
    mma_phase ^= 1;
    tc::tc_fence_after();
    GDR_TRACE_MARK(1, 4);
    if (ok) {
      float y[32];
      tmem_ld32w(tbase, warp, 64, y);  // h <- e^{gamma_C} h + K^T Vn~, then stage it for the next chunk
      const float eC = fexp(gC);
#pragma unroll
      for (int b = 0; b < 32; ++b) h[b] = eC * h[b] + y[b];
      st_col32_bf16(sm + SS::HT, tid, h);
    }
    if (tid == kCopyTid) tc::bulk_wait_read<0>();  // h staging free for the next chunk
    GDR_TRACE_MARK(1, 5);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (ok && warp >= 2 && c_begin < c_end) finish_o((c_end - c_begin - 1) & 1);  // the last chunk's output rows
  if (tid == kCopyTid) tc::bulk_wait_read<0>();  // smem sources read before exit
  if (ok && un.h1) {
#pragma unroll
    for (int b = 0; b < 32; ++b)
      un.h1[un.h1_kv ? (size_t)tid * 128 + dv0 + b : (size_t)(dv0 + b) * 128 + tid] = h[b];
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, 128);
}

template <bool kSingle, bool kModes>
__global__ void __launch_bounds__(kTcThreads) tc_fwd_state_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_u,
    const __grid_constant__ CUtensorMap tm_p, const __grid_constant__ CUtensorMap tm_hs, Dims d,
    const float* __restrict__ S0, float* __restrict__ S_T, bf16* __restrict__ o, Workspace ws, CpArgs cp) {
  extern __shared__ unsigned char smem_raw[];
  const StateUnit un = state_unit(d, ws, cp, (int)blockIdx.x, S0, S_T);
  if (un.skip) return;  // uniform over the block, before any barrier or tensor memory
  state_body<kSingle, false, kModes>(tm_q, tm_k, tm_w, tm_u, tm_p, tm_hs, d, o, ws, un, align1024(smem_raw));
}

// The forward's prep and state recurrence in one cooperative launch (every CTA resident, one
// per SM): the first n_state CTAs to start (a counter) run the state units, double-buffered;
// every other CTA runs the prep role, whose items are claimed in the forward's step order, so
// chunk c of every chain is prepared before chunk c + 1 of any.  State units wait only for prep
// items, which never wait: every wait ends.
static_assert(PrepSmem::BYTES + 3 * 16384 <= StateSmem<false>::BYTES, "the fused prep role's second tile stage");
__global__ void __launch_bounds__(kTcThreads) tc_fwd_fused_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_w,
    const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_p,
    const __grid_constant__ CUtensorMap tm_t, const __grid_constant__ CUtensorMap tm_hs, Dims d,
    const float* __restrict__ g, const bf16* __restrict__ beta, const float* __restrict__ S0,
    float* __restrict__ S_T, bf16* __restrict__ o, Workspace ws, int write_T, int n_state) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ int s_role;
  if (threadIdx.x == 0) {
    const int u = (int)atomicAdd(ws.fwd_queue + 1, 1u);
    s_role = u < n_state ? u : -1;  // -1: prep
  }
  __syncthreads();
  const int role = s_role;
  if (role >= 0)
    state_body<false, true, false>(tm_q, tm_k, tm_w, tm_u, tm_p, tm_hs, d, o, ws,
                            state_unit(d, ws, CpArgs{}, role, S0, S_T), align1024(smem_raw));
  else
    prep_body<true>(tm_q, tm_k, tm_v, tm_w, tm_u, tm_p, tm_t, d, g, beta, ws, write_T, align1024(smem_raw));
}

}  // namespace

bool tc_available() { return get_encoder(); }

// The forward's prep and state can share one cooperative kernel when the step table exists
// (sorted order: at most kMaxFusedSeqs sequences); tc_forward decides per launch whether the
// state units fit (see tc_fwd_fused_kernel).
bool fused_fwd_possible(const Dims& d) {
  return d.path == 1 && d.num_seqs > 0 && d.num_seqs <= kMaxFusedSeqs && d.T_total > 0 && d.max_chunks > 0;
}

// Persistent grid of the chunk-prep kernel: two CTAs per SM (shared memory allows two).
static dim3 prep_grid(const Dims& d) {
  int dev = 0, n_sm = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  const long long n_items = (long long)d.max_chunks * d.Hv, cap = 2ll * n_sm;
  return dim3((unsigned)(n_items < cap ? n_items : cap));
}

#ifdef GDR_TRACE
extern "C" int gdr_debug_trace_fwd(unsigned long long* out) {
  return cudaMemcpyFromSymbol(out, tcx::g_gdr_trace, sizeof(tcx::g_gdr_trace)) == cudaSuccess ? 0 : 1;
}
extern "C" int gdr_debug_cta_span_fwd(unsigned long long* out) {
  return cudaMemcpyFromSymbol(out, tcx::g_gdr_cta_span, sizeof(tcx::g_gdr_cta_span)) == cudaSuccess ? 0 : 1;
}
#endif

cudaError_t tc_forward(const Dims& d, const FwdArgs& a, const Workspace& ws, cudaStream_t s) {
  if (!get_encoder()) return cudaErrorNotSupported;
  // Maps are built only when there are tokens; with none, no kernel reads them (every
  // chunk slot is empty and the state kernel only copies S0 to S_T).
  CUtensorMap tq{}, tk{}, tv{}, tw{}, tu{}, tp{}, ths{}, tt{};
  const uint64_t Tt = (uint64_t)d.T_total;
  const uint64_t rows = (uint64_t)d.max_chunks * d.Hv * 64;
  if (Tt == 0 && d.num_seqs == 0) return cudaSuccess;
  if (Tt > 0) {
    if (!map_3d(&tq, a.q, 128, d.Hk, Tt) || !map_3d(&tk, a.k, 128, d.Hk, Tt) || !map_3d(&tv, a.v, 128, d.Hv, Tt) ||
        !map_2d(&tw, ws.W, 128, rows) || !map_2d(&tu, ws.U, 128, rows) ||
        !map_2d(&tp, ws.P, 64, rows) ||
        !(d.h_bf16 ? map_2d_sw64(&ths, a.h_saved, 128, rows * 2, 128)
                   : map_2d_box(&ths, a.h_saved, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 128, rows * 2, 32, 128)))
      return cudaErrorInvalidValue;
    // saved factors: T is kept for the backward too
    if (d.save_wy && !map_2d(&tt, ws.Tb, 64, rows)) return cudaErrorInvalidValue;
  }
  int dev = 0, n_sm = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  const long long n_cta = (long long)d.num_seqs * d.Hv * kStateSlices;
  // Prep and state in one cooperative kernel when there are at most half as many state units as
  // SMs (few long chains): one CTA per SM, the state units double-buffered, the other SMs
  // preparing chunks in step order.  (Two CTAs per SM, a state unit beside a prep CTA, would
  // serve more chains, but the occupancy calculation of a cooperative launch admits one CTA per
  // SM for kernels that allocate tensor memory.)  Otherwise the two launches below.
  if (fused_fwd_possible(d) && n_cta * 2 <= n_sm && d.cp_fwd <= 1) {
    const size_t smf = std::max<size_t>(PrepSmem::BYTES, StateSmem<false>::BYTES) + 1024;
    auto kern = tc_fwd_fused_kernel;
    set_smem_once((const void*)kern, smf);
    int per_sm = 0;
    const cudaError_t qe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTcThreads, smf);
    if (qe != cudaSuccess) (void)cudaGetLastError();  // our own query's error: fall back below
    if (qe == cudaSuccess && per_sm == 1) {
      cudaError_t e = cudaMemsetAsync(ws.fwd_flags, 0,
                                      sizeof(uint32_t) * ((size_t)d.max_chunks * d.Hv + 64), s);
      if (e != cudaSuccess) return e;
      Dims dd = d;
      Workspace w = ws;
      const float* g = a.g;
      const bf16* beta = (const bf16*)a.beta;
      const float* S0 = a.S0;
      float* S_T = a.S_T;
      bf16* o = (bf16*)a.o;
      int write_T = d.save_wy;
      int n_state = (int)n_cta;
      CUtensorMap& tt_arg = d.save_wy ? tt : tp;
      void* args[] = {&tq, &tk, &tv, &tw, &tu, &tp, &tt_arg, &ths, &dd, (void*)&g, (void*)&beta, (void*)&S0,
                      (void*)&S_T, (void*)&o, &w, &write_T, &n_state};
      e = cudaLaunchCooperativeKernel((const void*)kern, dim3((unsigned)n_sm), dim3(kTcThreads), args, smf, s);
      if (e != cudaSuccess) return e;
      stage_mark(s, "fwd_fused");
      return cudaGetLastError();
    }
  }
  if (d.max_chunks > 0 && Tt > 0) {
    const size_t smp = PrepSmem::BYTES + 1024;
    set_smem_once((const void*)tc_prep_kernel, smp);
    tc_prep_kernel<<<prep_grid(d), kTcThreads, smp, s>>>(tq, tk, tv, tw, tu, tp, d.save_wy ? tt : tp, d, a.g,
                                                                      (const bf16*)a.beta, ws, d.save_wy);
    stage_mark(s, "fwd_prep");
  }
  auto state_launch = [&](const CpArgs& cp, long long units, const char* stage) -> cudaError_t {
    if (units <= 0) return cudaSuccess;
    // more CTAs than SMs: the single-buffered variant, two CTAs per SM, so they all run at once
    const bool single = units > n_sm;
    const size_t sms = (single ? StateSmem<true>::BYTES : StateSmem<false>::BYTES) + 1024;
    const bool modes = cp.pass == 1;  // only the first pass has map units
    auto kern = single ? (modes ? tc_fwd_state_kernel<true, true> : tc_fwd_state_kernel<true, false>)
                       : (modes ? tc_fwd_state_kernel<false, true> : tc_fwd_state_kernel<false, false>);
    set_smem_once((const void*)kern, sms);
    kern<<<(unsigned)units, kTcThreads, sms, s>>>(tq, tk, tw, tu, tp, ths, d, a.S0, a.S_T, (bf16*)a.o, ws, cp);
    stage_mark(s, stage);
    return cudaGetLastError();
  };
  if (d.num_seqs > 0 && d.cp_fwd > 1 && Tt > 0) {
    // context parallel: segment 0 and every middle segment's maps, the scan of the boundary
    // states, then segments 1 .. nseg - 1 from their true start states (see StateUnit)
    const int P = d.cp_fwd;
    const long long chains = (long long)d.num_seqs * d.Hv;
    CpArgs cp{1, P, ws.cp_X, ws.cp_M, ws.cp_R};
    cudaError_t e = state_launch(cp, chains * (4 + 8 * (P - 2)), "fwd_cp_maps");
    if (e == cudaSuccess && P > 2) e = launch_cp_scan(d, ws, P, false, s);
    cp.pass = 3;
    if (e == cudaSuccess) e = state_launch(cp, chains * 4 * (P - 1), "fwd_cp_state");
    return e;
  }
  if (d.num_seqs > 0) return state_launch(CpArgs{}, n_cta, "fwd_state");
  return cudaGetLastError();
}

cudaError_t tc_launch_prep(const Dims& d, const void* q, const void* k, const void* v, const float* g,
                           const void* beta, const Workspace& ws, int write_T, cudaStream_t s, const char* stage) {
  if (d.max_chunks == 0 || d.T_total == 0) return cudaSuccess;
  CUtensorMap tq, tk, tv, tw, tu, tp, tt{};
  const uint64_t Tt = (uint64_t)d.T_total;
  const uint64_t rows = (uint64_t)d.max_chunks * d.Hv * 64;
  if (!map_3d(&tq, q, 128, d.Hk, Tt) || !map_3d(&tk, k, 128, d.Hk, Tt) || !map_3d(&tv, v, 128, d.Hv, Tt) ||
      !map_2d(&tw, ws.W, 128, rows) || !map_2d(&tu, ws.U, 128, rows) || !map_2d(&tp, ws.P, 64, rows))
    return cudaErrorInvalidValue;
  if (write_T && !map_2d(&tt, ws.Tb, 64, rows)) return cudaErrorInvalidValue;
  const size_t smp = PrepSmem::BYTES + 1024;
  set_smem_once((const void*)tc_prep_kernel, smp);
  tc_prep_kernel<<<prep_grid(d), kTcThreads, smp, s>>>(tq, tk, tv, tw, tu, tp, tt, d, g,
                                                                    (const bf16*)beta, ws, write_T);
  stage_mark(s, stage);
  return cudaGetLastError();
}

}  // namespace gdr
