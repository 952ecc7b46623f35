// gdr_simt_small.cu -- fp32 SIMT kernels for heads of at most 64 features (DK, DV <= 64).
//
// The same chunked steps as gdr_simt.cu (chunked gated delta rule, FlashQLA PR #34, Summary;
// chunk = 64 tokens; h := S^T is DK x DV, gamma the in-chunk cumsum of g, Gam[r][s] =
// exp(gamma_r - gamma_s)), organised around one primitive: a 64 x 64 output tile accumulated
// from two shared-memory operands that are stored with the contraction index leading,
//     C[m][n] += sum_k At[k][m] * B[k][n].
// Each of the 256 threads owns a 4 x 4 block of C (rows 4 ty .. 4 ty + 3, columns 4 tx ..
// 4 tx + 3, ty = tid / 16, tx = tid % 16), so one step of k reads one float4 of each operand
// for 16 FMAs; rows are padded to 68 floats (16-byte aligned, 4 banks apart), which keeps
// those reads free of bank conflicts.  A 64 x 64 x 64 product is FMA-bound at about 2k cycles
// on one SM.  Features past DK / DV and tokens past the chunk end are zero in every tile, so
// each product runs over the padded sizes without masks.
//
// Kernels (256 threads each):
//   prep   per (chunk, v-head): gamma; A = strict-lower(diag(beta) K K^T * Gam);
//          T = (I + A)^{-1} (blocked by 16: diagonal blocks by forward substitution, then
//          the blocks below them by small products);
//          W = T diag(beta e^gamma) K, U = T diag(beta) V.  The backward's variant also forms
//          Vn = U - W h (h as saved by the forward), P = Q K^T * Gam (lower, with the
//          diagonal) and K K^T * Gam (strictly lower), and keeps T.
//   state  per (sequence, v-head), chunks in order: Vn = U - W h,
//          h <- e^{gamma_C} h + K^T diag(e^{gamma_C - gamma}) Vn.
//   out    per (chunk, v-head): O = scale (diag(e^gamma) Q h + P Vn).
//   walk   per (sequence, v-head), chunks in reverse:
//          dVn = scale P^T dO + diag(e^{gamma_C - gamma}) K dh',
//          dh  = e^{gamma_C} dh' + scale (diag(e^gamma) Q)^T dO - W^T dVn.
//   grad   per (chunk, v-head): dq, dk, dv, dbeta, dg of the chunk (the terms of gdr_simt.cu's
//          gradient kernel, regrouped as tile products).
// Chunk records come from gdr_chunks.cuh (computed for fixed-length batches).
#include <type_traits>

#include "gdr_chunks.cuh"
#include "gdr_device.cuh"
#include "gdr_instrument.cuh"
#include "gdr_internal.h"

namespace gdr {

bool simt_small(const Dims& d) { return d.path == 0 && d.DK <= 64 && d.DV <= 64; }

namespace {

using namespace tcx;  // trace marks (-DGDR_TRACE only)

constexpr int kT = 256;                       // threads per CTA
constexpr int kTS = 68;                       // row stride of a tile (floats)
constexpr int kTileF = 64 * kTS;              // floats per tile
constexpr size_t kTileB = sizeof(float) * kTileF;

typedef float Blk[4][4];

__device__ __forceinline__ int ty_() { return threadIdx.x >> 4; }
__device__ __forceinline__ int tx_() { return threadIdx.x & 15; }

__device__ __forceinline__ void blk_zero(Blk& a) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) a[i][j] = 0.f;
}

// acc[i][j] += sum_{k < K} At[k][4 ty + i] * B[k][4 tx + j]   (kNeg: -=)
template <bool kNeg = false>
__device__ __forceinline__ void mm(Blk& acc, const float* __restrict__ At, const float* __restrict__ B, int K) {
  const float* a = At + 4 * ty_();
  const float* b = B + 4 * tx_();
#pragma unroll 8
  for (int k = 0; k < K; ++k) {
    const float4 av = *reinterpret_cast<const float4*>(a + k * kTS);
    const float4 bv = *reinterpret_cast<const float4*>(b + k * kTS);
    const float ar[4] = {av.x, av.y, av.z, av.w};
    const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(kNeg ? -ar[i] : ar[i], br[j], acc[i][j]);
  }
}

// tile[4 ty + i][4 tx + j] = v[i][j]
__device__ __forceinline__ void put_rows(float* t, const Blk& v) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<float4*>(t + (4 * ty_() + i) * kTS + 4 * tx_()) = make_float4(v[i][0], v[i][1], v[i][2], v[i][3]);
}

// tile[4 tx + j][4 ty + i] = v[i][j]  (the transpose)
__device__ __forceinline__ void put_cols(float* t, const Blk& v) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<float4*>(t + (4 * tx_() + j) * kTS + 4 * ty_()) = make_float4(v[0][j], v[1][j], v[2][j], v[3][j]);
}

// tile[r][c] = f(r, c) over the whole 64 x 64 tile (lanes walk c: coalesced when f reads a row)
template <class F>
__device__ __forceinline__ void fill_rows(float* t, F f) {
#pragma unroll
  for (int it = 0; it < 64 * 64 / kT; ++it) {
    const int e = threadIdx.x + it * kT, r = e >> 6, c = e & 63;
    t[r * kTS + c] = f(r, c);
  }
}

// tile[c][r] = f(r, c): the transpose of the matrix f describes
template <class F>
__device__ __forceinline__ void fill_cols(float* t, F f) {
#pragma unroll
  for (int it = 0; it < 64 * 64 / kT; ++it) {
    const int e = threadIdx.x + it * kT, r = e >> 6, c = e & 63;
    t[c * kTS + r] = f(r, c);
  }
}

// Asynchronous global -> shared copies (cp.async; with a source size of 0 the destination is
// zero-filled and nothing is read).  A copy is complete after cp_commit, cp_wait<n> (at most
// n newer groups still pending) and a barrier.
__device__ __forceinline__ unsigned smem_u32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void cp_async4(float* dst, const float* src, bool ok) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(ok ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async16(float* dst, const float* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(ok ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// tile[r][c] = row(r)[c] for r < nr and c < nc, else 0.  fp32 sources are copied with cp.async
// (16 bytes; nc is a multiple of 16), bf16 sources converted through registers.  row(0) must
// be a valid address (it stands in for the rows that are not read).
template <typename T, class Row>
__device__ __forceinline__ void load_rows(float* t, Row row, int nr, int nc) {
  if constexpr (std::is_same<T, float>::value) {
#pragma unroll
    for (int it = 0; it < 64 * 16 / kT; ++it) {
      const int e = threadIdx.x + it * kT, r = e >> 4, c = (e & 15) << 2;
      const bool ok = r < nr && c < nc;
      cp_async16(t + r * kTS + c, ok ? row(r) + c : row(0), ok);
    }
  } else {
    fill_rows(t, [&](int r, int c) { return (r < nr && c < nc) ? to_f32(row(r)[c]) : 0.f; });
  }
}

// tile[c][r] = row(r)[c] (the transpose; fp32 sources: 4-byte cp.async, reads stay coalesced)
template <typename T, class Row>
__device__ __forceinline__ void load_cols(float* t, Row row, int nr, int nc) {
  if constexpr (std::is_same<T, float>::value) {
#pragma unroll
    for (int it = 0; it < 64 * 64 / kT; ++it) {
      const int e = threadIdx.x + it * kT, r = e >> 6, c = e & 63;
      const bool ok = r < nr && c < nc;
      cp_async4(t + c * kTS + r, ok ? row(r) + c : row(0), ok);
    }
  } else {
    fill_cols(t, [&](int r, int c) { return (r < nr && c < nc) ? to_f32(row(r)[c]) : 0.f; });
  }
}

// The saved state of chunk-head ch ([DK][DV], fp32 or bf16) as rows or transposed.
__device__ __forceinline__ void load_h(float* t, const void* h_saved, const Dims& d, size_t ch, bool transposed) {
  const size_t off = ch * d.DK * d.DV;
  if (d.h_bf16) {
    const __nv_bfloat16* h = static_cast<const __nv_bfloat16*>(h_saved) + off;
    auto row = [&](int a) { return h + (size_t)a * d.DV; };
    if (transposed) load_cols<__nv_bfloat16>(t, row, d.DK, d.DV); else load_rows<__nv_bfloat16>(t, row, d.DK, d.DV);
  } else {
    const float* h = static_cast<const float*>(h_saved) + off;
    auto row = [&](int a) { return h + (size_t)a * d.DV; };
    if (transposed) load_cols<float>(t, row, d.DK, d.DV); else load_rows<float>(t, row, d.DK, d.DV);
  }
}

// Sum over the 16 threads of a row group (lanes 0-15 or 16-31 of a warp: same ty).
__device__ __forceinline__ float sum16(float x) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// T = (I + A)^{-1} for a strictly lower 64 x 64 A (row-major tile), written transposed into Tt
// (Tt[c][r] = T[r][c]).  Blocked by 16: the four diagonal blocks by forward substitution (one
// thread per column of a block), then the blocks below the diagonal, one block diagonal at a
// time:  T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj  (i > j).  Y is [3][16][17] scratch.  Every
// thread calls it; it ends with a barrier.
__device__ __forceinline__ void solve_unit_lower(const float* __restrict__ A, float* __restrict__ Tt, float* Y) {
  const int tid = threadIdx.x;
  auto T = [&](int r, int c) -> float& { return Tt[c * kTS + r]; };
  for (int e = tid; e < 64 * 64; e += kT) {  // above the diagonal blocks: 0
    const int r = e >> 6, c = e & 63;
    if ((c >> 4) > (r >> 4)) T(r, c) = 0.f;
  }
  if (tid < 64) {  // diagonal block b, column c of the block: x = (I + A_bb)^{-1} e_c
    const int b = tid >> 4, c = tid & 15, o = 16 * b;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc = r == c ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < r; ++m) acc = fmaf(-A[(o + r) * kTS + o + m], x[m], acc);  // x[m] = 0 for m < c
      x[r] = acc;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) T(o + r, o + c) = x[r];
  }
  __syncthreads();
  for (int dd = 1; dd < 4; ++dd) {
    const int nb = 4 - dd;  // blocks (j + dd, j), j < nb
    for (int e = tid; e < nb * 256; e += kT) {  // Y_j = sum_k A_{j+dd,k} T_kj
      const int j = e >> 8, r = (e >> 4) & 15, c = e & 15, i = j + dd;
      float acc = 0.f;
      for (int k = j; k < i; ++k)
#pragma unroll
        for (int m = 0; m < 16; ++m) acc = fmaf(A[(16 * i + r) * kTS + 16 * k + m], T(16 * k + m, 16 * j + c), acc);
      Y[(j * 16 + r) * 17 + c] = acc;
    }
    __syncthreads();
    for (int e = tid; e < nb * 256; e += kT) {  // T_{j+dd,j} = -T_{j+dd,j+dd} Y_j
      const int j = e >> 8, r = (e >> 4) & 15, c = e & 15, i = j + dd;
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) acc = fmaf(T(16 * i + r, 16 * i + m), Y[(j * 16 + m) * 17 + c], acc);
      T(16 * i + r, 16 * j + c) = -acc;
    }
    __syncthreads();
  }
}

// In-chunk inclusive cumsum of g into sg[64] (warp 0; rows past len add 0).
__device__ __forceinline__ void chunk_gamma(const float* __restrict__ g, size_t t0, int len, int Hv, int j, float* sg) {
  const int tid = threadIdx.x;
  if (tid >= 32) return;
  float run = 0.f;
  for (int base = 0; base < kChunk; base += 32) {
    const int r = base + tid;
    float x = r < len ? g[(t0 + r) * Hv + j] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (tid >= o) x += y;
    }
    sg[r] = run + x;
    run += __shfl_sync(0xffffffffu, x, 31);
  }
}

// ---------------------------------------------------------------------------------
// prep
// ---------------------------------------------------------------------------------
template <typename IT, bool kBwd>
__global__ void __launch_bounds__(kT) s64_prep_kernel(Dims d, const IT* __restrict__ q, const IT* __restrict__ k,
                                                      const IT* __restrict__ v, const float* __restrict__ g,
                                                      const IT* __restrict__ beta, const void* __restrict__ h_saved,
                                                      Workspace ws) {
  extern __shared__ __align__(16) float sm[];
  GDR_TRACE_INIT();
  const int c = blockIdx.x, j = blockIdx.y, i = j / d.G;
  const int4 ci = idx_chunk(d, ws, c);
  const int len = ci.z;
  const size_t t0 = (size_t)ci.y;
  if (len <= 0) return;
  const int DK = d.DK, DV = d.DV, Hv = d.Hv, Hk = d.Hk, tid = threadIdx.x;
  const size_t ch = (size_t)c * Hv + j;
  float* sKt = sm;              // K^T [dk][tok]
  float* sKs = sKt + kTileF;    // diag(beta e^gamma) K [tok][dk]
  float* sVs = sKs + kTileF;    // diag(beta) V [tok][dv]
  float* sA = sVs + kTileF;     // A [r][m]
  float* sTt = sA + kTileF;     // T^T [s][r]
  float* sQt = sTt + kTileF;    // backward: Q^T [dk][tok]
  float* sH = sQt + kTileF;     // backward: h [dk][dv]
  float* sWt = sH + kTileF;     // backward: W^T [dk][tok]
  float* sg = kBwd ? sWt + kTileF : sQt;
  float* sb = sg + kChunk;
  float* sY = sb + kChunk;      // [3][16][17] solve scratch
  auto krow = [&](int r) { return k + ((t0 + r) * Hk + i) * DK; };
  load_cols<IT>(sKt, krow, len, DK);
  load_rows<IT>(sKs, krow, len, DK);
  load_rows<IT>(sVs, [&](int r) { return v + ((t0 + r) * Hv + j) * DV; }, len, DV);
  if (kBwd) {
    load_cols<IT>(sQt, [&](int r) { return q + ((t0 + r) * Hk + i) * DK; }, len, DK);
    load_h(sH, h_saved, d, ch, false);
  }
  cp_commit();
  chunk_gamma(g, t0, len, Hv, j, sg);
  if (tid < kChunk) sb[tid] = tid < len ? ldf(beta + (t0 + tid) * Hv + j) : 0.f;
  cp_wait<0>();
  __syncthreads();
  GDR_TRACE_MARK(kBwd ? 1 : 0, 0);
  for (int e = tid; e < 64 * 64; e += kT) {  // row scales of the W and U operands
    const int r = e >> 6, x = e & 63;
    const float br = sb[r];
    sKs[r * kTS + x] *= br * __expf(sg[r]);
    sVs[r * kTS + x] *= br;
  }
  const int ty = ty_(), tx = tx_();
  {  // A = strict-lower(diag(beta) K K^T * Gam); the backward keeps K K^T * Gam (strictly lower)
    Blk acc;
    blk_zero(acc);
    mm(acc, sKt, sKt, DK);
    Blk ak;
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int r = 4 * ty + a, s = 4 * tx + b;
        const float gm = (s < r && r < len) ? __expf(sg[r] - sg[s]) * acc[a][b] : 0.f;
        ak[a][b] = gm;
        acc[a][b] = sb[r] * gm;
      }
    put_rows(sA, acc);
    if (kBwd) {
      float* Ak = ws.Ak + ch * 64 * 64;
#pragma unroll
      for (int a = 0; a < 4; ++a)
        *reinterpret_cast<float4*>(Ak + (4 * ty + a) * 64 + 4 * tx) = make_float4(ak[a][0], ak[a][1], ak[a][2], ak[a][3]);
    }
  }
  __syncthreads();
  GDR_TRACE_MARK(kBwd ? 1 : 0, 1);
  solve_unit_lower(sA, sTt, sY);
  if (kBwd) {  // T row-major for the gradient kernel
    float* Tg = ws.Tm + ch * 64 * 64;
    for (int e = tid; e < 64 * 64; e += kT) Tg[e] = sTt[(e & 63) * kTS + (e >> 6)];
  }
  GDR_TRACE_MARK(kBwd ? 1 : 0, 2);
  Blk w, u;
  blk_zero(w);
  blk_zero(u);
  mm(w, sTt, sKs, 64);  // W = T diag(beta e^gamma) K
  mm(u, sTt, sVs, 64);  // U = T diag(beta) V
  GDR_TRACE_MARK(kBwd ? 1 : 0, 3);
  if (tid < kChunk) ws.gam[ch * kChunk + tid] = sg[tid];
  if (!kBwd) {
    float* Wt = static_cast<float*>(ws.W) + ch * DK * 64;  // [DK][64]: the state kernel's operand
#pragma unroll
    for (int b = 0; b < 4; ++b)
      if (4 * tx + b < DK)
        *reinterpret_cast<float4*>(Wt + (4 * tx + b) * 64 + 4 * ty) = make_float4(w[0][b], w[1][b], w[2][b], w[3][b]);
    float* U = static_cast<float*>(ws.U) + ch * 64 * DV;
    if (4 * tx < DV)
#pragma unroll
      for (int a = 0; a < 4; ++a)
        *reinterpret_cast<float4*>(U + (4 * ty + a) * DV + 4 * tx) = make_float4(u[a][0], u[a][1], u[a][2], u[a][3]);
    return;
  }
  // backward: W row-major [64][DK] (the walk's operand), P, then Vn = U - W h
  float* W = static_cast<float*>(ws.W) + ch * 64 * DK;
  if (4 * tx < DK)
#pragma unroll
    for (int a = 0; a < 4; ++a)
      *reinterpret_cast<float4*>(W + (4 * ty + a) * DK + 4 * tx) = make_float4(w[a][0], w[a][1], w[a][2], w[a][3]);
  put_cols(sWt, w);
  {
    Blk p;
    blk_zero(p);
    mm(p, sQt, sKt, DK);
    float* P = ws.Pf + ch * 64 * 64;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int r = 4 * ty + a;
      float o[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int s = 4 * tx + b;
        o[b] = (s <= r && r < len) ? __expf(sg[r] - sg[s]) * p[a][b] : 0.f;
      }
      *reinterpret_cast<float4*>(P + r * 64 + 4 * tx) = make_float4(o[0], o[1], o[2], o[3]);
    }
  }
  __syncthreads();
  GDR_TRACE_MARK(1, 4);
  Blk wh;
  blk_zero(wh);
  mm(wh, sWt, sH, DK);
  float* Vn = static_cast<float*>(ws.Vn) + ch * 64 * DV;
  if (4 * tx < DV)
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int r = 4 * ty + a;
      const bool in = r < len;
      *reinterpret_cast<float4*>(Vn + r * DV + 4 * tx) =
          make_float4(in ? u[a][0] - wh[a][0] : 0.f, in ? u[a][1] - wh[a][1] : 0.f, in ? u[a][2] - wh[a][2] : 0.f,
                      in ? u[a][3] - wh[a][3] : 0.f);
    }
}

// ---------------------------------------------------------------------------------
// state (forward recurrence), one CTA per (sequence, v-head)
// ---------------------------------------------------------------------------------
template <typename IT>
__global__ void __launch_bounds__(kT) s64_state_kernel(Dims d, const IT* __restrict__ k, const float* __restrict__ S0,
                                                       float* __restrict__ S_T, void* __restrict__ h_saved,
                                                       Workspace ws) {
  extern __shared__ __align__(16) float sm[];
  GDR_TRACE_INIT();
  const int n = idx_seq(d, ws, blockIdx.x);
  const int c_begin = idx_seq_off(d, ws, n), c_end = idx_seq_off(d, ws, n + 1);
  const int j = blockIdx.y, i = j / d.G;
  const int DK = d.DK, DV = d.DV, Hv = d.Hv, Hk = d.Hk, tid = threadIdx.x, ty = ty_(), tx = tx_();
  float* sH = sm;               // h [dk][dv]
  float* sVd = sH + kTileF;     // diag(e^{gamma_C - gamma}) Vn [tok][dv]
  float* st0 = sVd + kTileF;    // two stages of {W^T [dk][tok], K [tok][dk], U [tok][dv], gamma}
  constexpr int kStageF = 3 * kTileF + kChunk;
  auto issue = [&](int c, int b) {  // chunk c's tiles into stage b (one cp.async group)
    const int4 ci = idx_chunk(d, ws, c);
    const size_t t0 = (size_t)ci.y, ch = (size_t)c * Hv + j;
    float* t = st0 + b * kStageF;
    const float* Wt = static_cast<const float*>(ws.W) + ch * DK * 64;
    const float* U = static_cast<const float*>(ws.U) + ch * 64 * DV;
    load_rows<float>(t, [&](int x) { return Wt + x * 64; }, DK, 64);
    load_rows<IT>(t + kTileF, [&](int r) { return k + ((t0 + r) * Hk + i) * DK; }, ci.z, DK);
    load_rows<float>(t + 2 * kTileF, [&](int r) { return U + r * DV; }, ci.z, DV);
    if (tid < 16) cp_async16(t + 3 * kTileF + 4 * tid, ws.gam + ch * kChunk + 4 * tid, true);
    cp_commit();
  };
  Blk h;
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int x = 4 * ty + a, y = 4 * tx + b;
      h[a][b] = (S0 && x < DK && y < DV) ? S0[((size_t)n * Hv + j) * DK * DV + state_idx(d.layout, x, y, DK, DV)] : 0.f;
    }
  put_rows(sH, h);
  if (c_begin < c_end) issue(c_begin, 0);
  for (int c = c_begin; c < c_end; ++c) {
    const int stg = (c - c_begin) & 1;
    __syncthreads();  // the previous chunk's products are done with its stage and sVd; sH is current
    GDR_TRACE_MARK(2, 4);
    if (c + 1 < c_end) {
      issue(c + 1, stg ^ 1);
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();  // this chunk's stage has landed
    GDR_TRACE_MARK(2, 0);
    const int4 ci = idx_chunk(d, ws, c);
    const int len = ci.z;
    const size_t ch = (size_t)c * Hv + j;
    const float* sWt = st0 + stg * kStageF;
    const float* sK = sWt + kTileF;
    const float* sU = sK + kTileF;
    const float* sg = sU + kTileF;
    if (4 * tx < DV)  // the state at the chunk start
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int x = 4 * ty + a;
        if (x >= DK) continue;
        const size_t e = ch * DK * DV + (size_t)x * DV + 4 * tx;
        if (d.h_bf16) {
          __nv_bfloat16* hp = static_cast<__nv_bfloat16*>(h_saved) + e;
#pragma unroll
          for (int b = 0; b < 4; ++b) hp[b] = __float2bfloat16_rn(h[a][b]);
        } else {
          *reinterpret_cast<float4*>(static_cast<float*>(h_saved) + e) = make_float4(h[a][0], h[a][1], h[a][2], h[a][3]);
        }
      }
    Blk vn;
    blk_zero(vn);
    mm(vn, sWt, sH, DK);  // W h
    GDR_TRACE_MARK(2, 1);
    const float gC = sg[len - 1], eC = __expf(gC);
    float* Vn = static_cast<float*>(ws.Vn) + ch * 64 * DV;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int r = 4 * ty + a;
      const bool in = r < len;
      const float dec = in ? __expf(gC - sg[r]) : 0.f;
      const float4 u4 = *reinterpret_cast<const float4*>(sU + r * kTS + 4 * tx);
      const float val[4] = {in ? u4.x - vn[a][0] : 0.f, in ? u4.y - vn[a][1] : 0.f, in ? u4.z - vn[a][2] : 0.f,
                            in ? u4.w - vn[a][3] : 0.f};
      if (4 * tx < DV) *reinterpret_cast<float4*>(Vn + r * DV + 4 * tx) = make_float4(val[0], val[1], val[2], val[3]);
#pragma unroll
      for (int b = 0; b < 4; ++b) vn[a][b] = dec * val[b];
    }
    put_rows(sVd, vn);
    __syncthreads();
    GDR_TRACE_MARK(2, 2);
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) h[a][b] *= eC;
    mm(h, sK, sVd, 64);  // + K^T diag(e^{gamma_C - gamma}) Vn
    GDR_TRACE_MARK(2, 3);
    put_rows(sH, h);
  }
  if (S_T) {
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int x = 4 * ty + a, y = 4 * tx + b;
        if (x < DK && y < DV) S_T[((size_t)n * Hv + j) * DK * DV + state_idx(d.layout, x, y, DK, DV)] = h[a][b];
      }
  }
}

// ---------------------------------------------------------------------------------
// out: O = scale (diag(e^gamma) Q h + P Vn), one CTA per (chunk, v-head)
// ---------------------------------------------------------------------------------
template <typename IT>
__global__ void __launch_bounds__(kT) s64_out_kernel(Dims d, const IT* __restrict__ q, const IT* __restrict__ k,
                                                     const void* __restrict__ h_saved, IT* __restrict__ o,
                                                     Workspace ws) {
  extern __shared__ __align__(16) float sm[];
  GDR_TRACE_INIT();
  const int c = blockIdx.x, j = blockIdx.y, i = j / d.G;
  const int4 ci = idx_chunk(d, ws, c);
  const int len = ci.z;
  const size_t t0 = (size_t)ci.y;
  if (len <= 0) return;
  const int DK = d.DK, DV = d.DV, Hv = d.Hv, Hk = d.Hk, tid = threadIdx.x, ty = ty_(), tx = tx_();
  const size_t ch = (size_t)c * Hv + j;
  float* sQt = sm;              // Q^T [dk][tok]
  float* sKt = sQt + kTileF;    // K^T [dk][tok]
  float* sH = sKt + kTileF;     // h [dk][dv]
  float* sPt = sH + kTileF;     // P^T [s][r]
  float* sVn = sPt + kTileF;    // Vn [tok][dv]
  float* sg = sVn + kTileF;
  load_cols<IT>(sQt, [&](int r) { return q + ((t0 + r) * Hk + i) * DK; }, len, DK);
  load_cols<IT>(sKt, [&](int r) { return k + ((t0 + r) * Hk + i) * DK; }, len, DK);
  load_h(sH, h_saved, d, ch, false);
  const float* Vn = static_cast<const float*>(ws.Vn) + ch * 64 * DV;
  load_rows<float>(sVn, [&](int r) { return Vn + r * DV; }, 64, DV);
  if (tid < 16) cp_async16(sg + 4 * tid, ws.gam + ch * kChunk + 4 * tid, true);
  cp_commit();
  cp_wait<0>();
  __syncthreads();
  GDR_TRACE_MARK(3, 0);
  Blk p;
  blk_zero(p);
  mm(p, sQt, sKt, DK);
  GDR_TRACE_MARK(3, 1);
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int r = 4 * ty + a, s = 4 * tx + b;
      p[a][b] = (s <= r && r < len) ? __expf(sg[r] - sg[s]) * p[a][b] : 0.f;
    }
  put_cols(sPt, p);
  Blk acc;
  blk_zero(acc);
  mm(acc, sQt, sH, DK);  // Q h
  GDR_TRACE_MARK(3, 2);
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const float eg = __expf(sg[4 * ty + a]);
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] *= eg;
  }
  __syncthreads();
  mm(acc, sPt, sVn, 64);  // + P Vn
  GDR_TRACE_MARK(3, 3);
  if (4 * tx < DV)
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int r = 4 * ty + a;
      if (r >= len) continue;
      IT* op = o + ((t0 + r) * Hv + j) * DV + 4 * tx;
#pragma unroll
      for (int b = 0; b < 4; ++b) op[b] = from_f32<IT>(d.scale * acc[a][b]);
    }
}

// ---------------------------------------------------------------------------------
// walk (reverse state-gradient recurrence), one CTA per (sequence, v-head)
// ---------------------------------------------------------------------------------
template <typename IT>
__global__ void __launch_bounds__(kT) s64_walk_kernel(Dims d, const IT* __restrict__ q, const IT* __restrict__ k,
                                                      const IT* __restrict__ dO, const float* __restrict__ dS_T,
                                                      float* __restrict__ dS0, Workspace ws) {
  extern __shared__ __align__(16) float sm[];
  GDR_TRACE_INIT();
  const int n = idx_seq(d, ws, blockIdx.x);
  const int c_begin = idx_seq_off(d, ws, n), c_end = idx_seq_off(d, ws, n + 1);
  const int j = blockIdx.y, i = j / d.G;
  const int DK = d.DK, DV = d.DV, Hv = d.Hv, Hk = d.Hk, tid = threadIdx.x, ty = ty_(), tx = tx_();
  float* sDh = sm;              // dh' [dk][dv]
  float* sDvn = sDh + kTileF;   // dVn [tok][dv]
  float* st0 = sDvn + kTileF;   // two stages of {P [r][s], dO [tok][dv], K^T [dk][tok], Q [tok][dk], W [tok][dk], gamma}
  constexpr int kStageF = 5 * kTileF + kChunk;
  auto issue = [&](int c, int b) {  // chunk c's tiles into stage b (one cp.async group)
    const int4 ci = idx_chunk(d, ws, c);
    const size_t t0 = (size_t)ci.y, ch = (size_t)c * Hv + j;
    float* t = st0 + b * kStageF;
    const float* P = ws.Pf + ch * 64 * 64;
    const float* W = static_cast<const float*>(ws.W) + ch * 64 * DK;
    load_rows<float>(t, [&](int r) { return P + r * 64; }, 64, 64);
    load_rows<IT>(t + kTileF, [&](int r) { return dO + ((t0 + r) * Hv + j) * DV; }, ci.z, DV);
    load_cols<IT>(t + 2 * kTileF, [&](int r) { return k + ((t0 + r) * Hk + i) * DK; }, ci.z, DK);
    load_rows<IT>(t + 3 * kTileF, [&](int r) { return q + ((t0 + r) * Hk + i) * DK; }, ci.z, DK);
    load_rows<float>(t + 4 * kTileF, [&](int r) { return W + r * DK; }, 64, DK);
    if (tid < 16) cp_async16(t + 5 * kTileF + 4 * tid, ws.gam + ch * kChunk + 4 * tid, true);
    cp_commit();
  };
  Blk dh;
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int x = 4 * ty + a, y = 4 * tx + b;
      dh[a][b] = (dS_T && x < DK && y < DV) ? dS_T[((size_t)n * Hv + j) * DK * DV + state_idx(d.layout, x, y, DK, DV)] : 0.f;
    }
  put_rows(sDh, dh);
  if (c_begin < c_end) issue(c_end - 1, 0);
  for (int c = c_end - 1; c >= c_begin; --c) {
    const int stg = (c_end - 1 - c) & 1;
    __syncthreads();  // the previous chunk's products are done with its stage and sDvn; sDh is current
    GDR_TRACE_MARK(4, 4);
    if (c > c_begin) {
      issue(c - 1, stg ^ 1);
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();  // this chunk's stage has landed
    GDR_TRACE_MARK(4, 0);
    const int4 ci = idx_chunk(d, ws, c);
    const int len = ci.z;
    const size_t ch = (size_t)c * Hv + j;
    float* sP = st0 + stg * kStageF;
    float* sdO = sP + kTileF;
    float* sKt = sdO + kTileF;
    float* sQ = sKt + kTileF;
    float* sW = sQ + kTileF;
    const float* sg = sW + kTileF;
    float* dhp = static_cast<float*>(ws.dhp) + ch * DK * DV;
    if (4 * tx < DV)
#pragma unroll
      for (int a = 0; a < 4; ++a)
        if (4 * ty + a < DK)
          *reinterpret_cast<float4*>(dhp + (4 * ty + a) * DV + 4 * tx) = make_float4(dh[a][0], dh[a][1], dh[a][2], dh[a][3]);
    Blk a1, a2;
    blk_zero(a1);
    blk_zero(a2);
    mm(a1, sP, sdO, 64);   // P^T dO
    mm(a2, sKt, sDh, DK);  // K dh'
    GDR_TRACE_MARK(4, 1);
    const float gC = sg[len - 1], eC = __expf(gC);
    float* dVn = static_cast<float*>(ws.dVn) + ch * 64 * DV;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int s = 4 * ty + a;
      const bool in = s < len;
      const float dec = in ? __expf(gC - sg[s]) : 0.f;
#pragma unroll
      for (int b = 0; b < 4; ++b) a1[a][b] = in ? d.scale * a1[a][b] + dec * a2[a][b] : 0.f;
      if (4 * tx < DV) *reinterpret_cast<float4*>(dVn + s * DV + 4 * tx) = make_float4(a1[a][0], a1[a][1], a1[a][2], a1[a][3]);
    }
    put_rows(sDvn, a1);
#pragma unroll
    for (int it = 0; it < 64 * 16 / kT; ++it) {  // Q rows -> scale e^gamma Q (read after the barrier)
      const int e = tid + it * kT, r = e >> 4, x = (e & 15) << 2;
      float4* p4 = reinterpret_cast<float4*>(sQ + r * kTS + x);
      const float f = d.scale * __expf(sg[r]);
      const float4 v4 = *p4;
      *p4 = make_float4(f * v4.x, f * v4.y, f * v4.z, f * v4.w);
    }
    __syncthreads();
    GDR_TRACE_MARK(4, 2);
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) dh[a][b] *= eC;
    mm(dh, sQ, sdO, 64);        // + scale (diag(e^gamma) Q)^T dO
    mm<true>(dh, sW, sDvn, 64);  // - W^T dVn
    GDR_TRACE_MARK(4, 3);
    put_rows(sDh, dh);
  }
  if (dS0) {
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int x = 4 * ty + a, y = 4 * tx + b;
        if (x < DK && y < DV) dS0[((size_t)n * Hv + j) * DK * DV + state_idx(d.layout, x, y, DK, DV)] = dh[a][b];
      }
  }
}

// ---------------------------------------------------------------------------------
// grad: every gradient of one (chunk, v-head)
// ---------------------------------------------------------------------------------
// The WY backward is regrouped around one identity: with B_k = diag(beta e^gamma) K and
// B_v = diag(beta) V, Vn = U - W h = T (B_v - B_k h), so B_v - B_k h = (I + A) Vn and
//   dT = dW B_k^T + dVn B_v^T = dVn ((I + A) Vn)^T        (dW = -dVn h^T),
//   dB_k = T^T dW = -(T^T dVn) h^T = -dB_v h^T,
// which needs neither dW nor K^T / V^T tiles.  Twelve tile slots, reused as their contents
// die (each step names its operands):
//   phase 1: S0 dO^T, S1 Vn^T, S2 dh'^T, S3 Q, S4 h^T, S5 K, S8 Vn, S9 dVn^T, S10 V, S11 T
//   A  dP = scale (dO Vn^T) * Gam * M          (S0, S1)        -> S6 dP, S7 dP^T
//   A2 Vn dh'^T (registers)                     (S1, S2)
//   phase 2: S1 (K K^T * Gam)^T, S2 dVn
//   A3 dk  = dP^T Q                             (S6, S3)
//   B  dq  = scale diag(e^gamma) dO h^T + dP K  (S0, S4; S7, S5)
//   Z  (I + A) Vn = Vn + diag(beta) (K K^T * Gam) Vn   (S1, S8)  -> S3 transposed; S0 T^T
//   D  dT  = dVn ((I + A) Vn)^T                 (S9, S3)        -> S6
//   E  X   = T^T dT                             (S11, S6)       -> S8 X^T
//   F  dA  = -strict-lower(X T^T)               (S8, S0)        -> S6 L = diag(beta)(dA * Gam)
//      S3 = L + L^T
//   G  dB_v = T^T dVn -> dv                     (S11, S2)       -> S0 dB_v^T
//   H  dB_k = -dB_v h^T; dk += diag(beta e^gamma) dB_k  (S0, S4)
//   I  dk += (L + L^T) K  [= diag(beta)(dA * Gam) K + (dA * Gam)^T diag(beta) K]  (S3, S5)
template <typename IT>
__global__ void __launch_bounds__(kT) s64_grad_kernel(Dims d, const IT* __restrict__ q, const IT* __restrict__ k,
                                                      const IT* __restrict__ v, const IT* __restrict__ beta,
                                                      const void* __restrict__ h_saved, const IT* __restrict__ dO,
                                                      IT* __restrict__ dq, IT* __restrict__ dk, IT* __restrict__ dv,
                                                      float* __restrict__ dg, IT* __restrict__ dbeta, Workspace ws) {
  extern __shared__ __align__(16) float sm[];
  GDR_TRACE_INIT();
  const int c = blockIdx.x, j = blockIdx.y, i = j / d.G;
  const int4 ci = idx_chunk(d, ws, c);
  const int len = ci.z;
  const size_t t0 = (size_t)ci.y;
  if (len <= 0) return;
  const int DK = d.DK, DV = d.DV, Hv = d.Hv, Hk = d.Hk, tid = threadIdx.x, ty = ty_(), tx = tx_();
  const int lane = tid & 31, warp = tid >> 5;
  const size_t ch = (size_t)c * Hv + j;
  float* S[12];
#pragma unroll
  for (int x = 0; x < 12; ++x) S[x] = sm + x * kTileF;
  float* sg = sm + 12 * kTileF;
  float* sb = sg + kChunk;
  float* rows = sb + kChunk;    // [7][64] per-row sums
  float* sred = rows + 7 * 64;  // [8] block reduction
  float* colA = S[7];           // [16][64] column partials of dP * (Q K^T) (S7 is free after step B)
  float* colB = S[9];           // [16][64] column partials of dA * A (S9 is free after step D)
  const float* Vn = static_cast<const float*>(ws.Vn) + ch * 64 * DV;
  const float* dVn = static_cast<const float*>(ws.dVn) + ch * 64 * DV;
  const float* dhp = static_cast<const float*>(ws.dhp) + ch * DK * DV;
  const float* Tg = ws.Tm + ch * 64 * 64;
  const float* Pg = ws.Pf + ch * 64 * 64;
  const float* Akg = ws.Ak + ch * 64 * 64;
  auto qrow = [&](int r) { return q + ((t0 + r) * Hk + i) * DK; };
  auto krow = [&](int r) { return k + ((t0 + r) * Hk + i) * DK; };
  // phase 1
  load_cols<IT>(S[0], [&](int r) { return dO + ((t0 + r) * Hv + j) * DV; }, len, DV);
  load_cols<float>(S[1], [&](int r) { return Vn + r * DV; }, 64, DV);
  load_cols<float>(S[2], [&](int a) { return dhp + a * DV; }, DK, DV);
  load_rows<IT>(S[3], qrow, len, DK);
  load_h(S[4], h_saved, d, ch, true);
  load_rows<IT>(S[5], krow, len, DK);
  load_rows<float>(S[8], [&](int r) { return Vn + r * DV; }, 64, DV);
  load_cols<float>(S[9], [&](int r) { return dVn + r * DV; }, 64, DV);
  load_rows<IT>(S[10], [&](int r) { return v + ((t0 + r) * Hv + j) * DV; }, len, DV);
  load_rows<float>(S[11], [&](int r) { return Tg + r * 64; }, 64, 64);
  if (tid < 16) cp_async16(sg + 4 * tid, ws.gam + ch * kChunk + 4 * tid, true);
  cp_commit();
  if (tid < kChunk) sb[tid] = tid < len ? ldf(beta + (t0 + tid) * Hv + j) : 0.f;
  cp_wait<0>();
  __syncthreads();
  GDR_TRACE_MARK(5, 0);
  {  // <dh', h> (both tiles transposed alike; padding is zero)
    float hdh = 0.f;
#pragma unroll 4
    for (int e = tid; e < 64 * 64; e += kT) {
      const int x = (e >> 6) * kTS + (e & 63);
      hdh = fmaf(S[2][x], S[4][x], hdh);
    }
    hdh = warp_sum(hdh);
    if (lane == 0) sred[warp] = hdh;
  }
  const float gC = sg[len - 1];
  float eg[4], dec[4], br[4];
  int rr[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    rr[a] = 4 * ty + a;
    eg[a] = __expf(sg[rr[a]]);
    dec[a] = rr[a] < len ? __expf(gC - sg[rr[a]]) : 0.f;
    br[a] = sb[rr[a]];
  }
  float pp_r[4], pp_c[4], kdv_r[4], qh_r[4];
  // A: dP
  {
    Blk acc;
    blk_zero(acc);
    mm(acc, S[0], S[1], DV);
#pragma unroll
    for (int b = 0; b < 4; ++b) pp_c[b] = 0.f;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float4 p4 = *reinterpret_cast<const float4*>(Pg + rr[a] * 64 + 4 * tx);
      const float pr[4] = {p4.x, p4.y, p4.z, p4.w};
      pp_r[a] = 0.f;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int s = 4 * tx + b;
        const float raw = d.scale * acc[a][b];
        const float pp = raw * pr[b];  // dP * (Q K^T): P holds Q K^T * Gam on and below the diagonal
        pp_r[a] += pp;
        pp_c[b] += pp;
        acc[a][b] = (s <= rr[a] && rr[a] < len) ? raw * __expf(sg[rr[a]] - sg[s]) : 0.f;
      }
    }
    put_rows(S[6], acc);
    put_cols(S[7], acc);
  }
  // A2: Vn dh'^T
  Blk vd;
  blk_zero(vd);
  mm(vd, S[1], S[2], DV);
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const float4 k4 = *reinterpret_cast<const float4*>(S[5] + rr[a] * kTS + 4 * tx);
    kdv_r[a] = k4.x * vd[a][0] + k4.y * vd[a][1] + k4.z * vd[a][2] + k4.w * vd[a][3];
  }
  GDR_TRACE_MARK(5, 1);
  __syncthreads();
  // phase 2 (S1 and S2 are free)
  load_cols<float>(S[1], [&](int r) { return Akg + r * 64; }, 64, 64);
  load_rows<float>(S[2], [&](int r) { return dVn + r * DV; }, 64, DV);
  cp_commit();
  // A3: dk = dP^T Q
  Blk dkb;
  blk_zero(dkb);
  mm(dkb, S[6], S[3], 64);
  GDR_TRACE_MARK(5, 2);
  // B: dq
  {
    Blk acc;
    blk_zero(acc);
    mm(acc, S[0], S[4], DV);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float4 q4 = *reinterpret_cast<const float4*>(S[3] + rr[a] * kTS + 4 * tx);
      qh_r[a] = q4.x * acc[a][0] + q4.y * acc[a][1] + q4.z * acc[a][2] + q4.w * acc[a][3];
      const float sc = d.scale * eg[a];
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] *= sc;
    }
    mm(acc, S[7], S[5], 64);
    if (4 * tx < DK)
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        if (rr[a] >= len) continue;
        const size_t t = t0 + rr[a];
        if (d.G == 1) {
          IT* p = dq + (t * Hk + i) * DK + 4 * tx;
#pragma unroll
          for (int b = 0; b < 4; ++b) p[b] = from_f32<IT>(acc[a][b]);
        } else {
          *reinterpret_cast<float4*>(ws.dq_part + (t * Hv + j) * DK + 4 * tx) = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        }
      }
  }
  GDR_TRACE_MARK(5, 3);
  cp_wait<0>();
  __syncthreads();  // phase 2 has landed; S0, S3, S6, S7 are free
#pragma unroll
  for (int b = 0; b < 4; ++b) colA[ty * 64 + 4 * tx + b] = pp_c[b];
  for (int e = tid; e < 64 * 64; e += kT) {  // S0 = T^T
    const int r = e >> 6, s = e & 63;
    S[0][s * kTS + r] = S[11][r * kTS + s];
  }
  // Z: (I + A) Vn
  {
    Blk acc;
    blk_zero(acc);
    mm(acc, S[1], S[8], 64);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float4 v4 = *reinterpret_cast<const float4*>(S[8] + rr[a] * kTS + 4 * tx);
      const float vr[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(br[a], acc[a][b], vr[b]);
    }
    put_cols(S[3], acc);
  }
  __syncthreads();
  GDR_TRACE_MARK(5, 4);
  // D: dT = dVn ((I + A) Vn)^T
  {
    Blk acc;
    blk_zero(acc);
    mm(acc, S[9], S[3], DV);
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (!(rr[a] < len && 4 * tx + b < len)) acc[a][b] = 0.f;
    put_rows(S[6], acc);
  }
  __syncthreads();
  GDR_TRACE_MARK(5, 5);
  // E: X = T^T dT
  {
    Blk acc;
    blk_zero(acc);
    mm(acc, S[11], S[6], 64);
    put_cols(S[8], acc);
  }
  __syncthreads();
  GDR_TRACE_MARK(5, 6);
  // F: dA = -strict-lower(X T^T)
  float aa_r[4], aa_c[4], akk_r[4];
  {
    Blk acc;
    blk_zero(acc);
    mm(acc, S[8], S[0], 64);
#pragma unroll
    for (int b = 0; b < 4; ++b) aa_c[b] = 0.f;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      aa_r[a] = 0.f;
      akk_r[a] = 0.f;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int s = 4 * tx + b;
        const float akr = S[1][s * kTS + rr[a]];  // (K K^T * Gam)[r][s], from the transposed tile
        const bool low = s < rr[a] && rr[a] < len;
        const float dA = low ? -acc[a][b] : 0.f;
        const float aa = dA * br[a] * akr;  // dA * A, A = diag(beta) (K K^T * Gam)
        aa_r[a] += aa;
        aa_c[b] += aa;
        akk_r[a] += dA * akr;
        acc[a][b] = low ? br[a] * dA * __expf(sg[rr[a]] - sg[s]) : 0.f;
      }
    }
    put_rows(S[6], acc);
  }
#pragma unroll
  for (int b = 0; b < 4; ++b) colB[ty * 64 + 4 * tx + b] = aa_c[b];
  __syncthreads();
  GDR_TRACE_MARK(5, 7);
  {  // S3 = L + L^T
    Blk m;
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int s = 4 * tx + b;
        m[a][b] = S[6][rr[a] * kTS + s] + S[6][s * kTS + rr[a]];
      }
    put_rows(S[3], m);
  }
  // G: dB_v = T^T dVn -> dv
  float dbv_r[4], dbk_r[4];
  {
    Blk acc;
    blk_zero(acc);
    mm(acc, S[11], S[2], 64);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float4 v4 = *reinterpret_cast<const float4*>(S[10] + rr[a] * kTS + 4 * tx);
      dbv_r[a] = v4.x * acc[a][0] + v4.y * acc[a][1] + v4.z * acc[a][2] + v4.w * acc[a][3];
    }
    if (4 * tx < DV)
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        if (rr[a] >= len) continue;
        IT* p = dv + ((t0 + rr[a]) * Hv + j) * DV + 4 * tx;
#pragma unroll
        for (int b = 0; b < 4; ++b) p[b] = from_f32<IT>(br[a] * acc[a][b]);
      }
    put_cols(S[0], acc);
  }
  __syncthreads();
  GDR_TRACE_MARK(5, 8);
  // H: dB_k = -dB_v h^T
  {
    Blk acc;
    blk_zero(acc);
    mm<true>(acc, S[0], S[4], DV);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float4 k4 = *reinterpret_cast<const float4*>(S[5] + rr[a] * kTS + 4 * tx);
      dbk_r[a] = k4.x * acc[a][0] + k4.y * acc[a][1] + k4.z * acc[a][2] + k4.w * acc[a][3];
      const float sc = br[a] * eg[a];
#pragma unroll
      for (int b = 0; b < 4; ++b) dkb[a][b] = fmaf(sc, acc[a][b], dkb[a][b]);
    }
  }
  // I: dk += (L + L^T) K, + diag(e^{gamma_C - gamma}) Vn dh'^T
  mm(dkb, S[3], S[5], 64);
  GDR_TRACE_MARK(5, 9);
  if (4 * tx < DK)
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      if (rr[a] >= len) continue;
      const size_t t = t0 + rr[a];
      float o4[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) o4[b] = fmaf(dec[a], vd[a][b], dkb[a][b]);
      if (d.G == 1) {
        IT* p = dk + (t * Hk + i) * DK + 4 * tx;
#pragma unroll
        for (int b = 0; b < 4; ++b) p[b] = from_f32<IT>(o4[b]);
      } else {
        *reinterpret_cast<float4*>(ws.dk_part + (t * Hv + j) * DK + 4 * tx) = make_float4(o4[0], o4[1], o4[2], o4[3]);
      }
    }
  // J: per-row sums -> dbeta, d gamma -> dg
  {
    const float vals[7][4] = {
        {pp_r[0], pp_r[1], pp_r[2], pp_r[3]},     {aa_r[0], aa_r[1], aa_r[2], aa_r[3]},
        {akk_r[0], akk_r[1], akk_r[2], akk_r[3]}, {kdv_r[0], kdv_r[1], kdv_r[2], kdv_r[3]},
        {qh_r[0], qh_r[1], qh_r[2], qh_r[3]},     {dbv_r[0], dbv_r[1], dbv_r[2], dbv_r[3]},
        {dbk_r[0], dbk_r[1], dbk_r[2], dbk_r[3]}};
#pragma unroll
    for (int x = 0; x < 7; ++x)
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const float t = sum16(vals[x][a]);
        if (tx == 0) rows[x * 64 + rr[a]] = t;
      }
  }
  __syncthreads();
  GDR_TRACE_MARK(5, 10);
  float* sdg = S[6];  // d gamma per row (S6 is free once S3 = L + L^T is built)
  if (tid < kChunk) {
    const int r = tid;
    float ppc = 0.f, aac = 0.f;
    for (int y = 0; y < 16; ++y) {
      ppc += colA[y * 64 + r];
      aac += colB[y * 64 + r];
    }
    const float egr = __expf(sg[r]), br0 = sb[r];
    const float pp = rows[0 * 64 + r], aa = rows[1 * 64 + r], akk = rows[2 * 64 + r];
    const float kdv = rows[3 * 64 + r], qh = rows[4 * 64 + r], dbv = rows[5 * 64 + r], dbk = rows[6 * 64 + r];
    const float decr = r < len ? __expf(gC - sg[r]) : 0.f;
    float dgam = 0.f;
    if (r < len) {
      dbeta[(t0 + r) * Hv + j] = from_f32<IT>(egr * dbk + dbv + akk);
      dgam = br0 * egr * dbk + (aa - aac) + d.scale * egr * qh + (pp - ppc) - decr * kdv;
    }
    sdg[r] = dgam;
    sdg[64 + r] = decr * kdv;  // for the chunk-end term
  }
  __syncthreads();
  if (tid == 0) {
    float hd = 0.f;
    for (int w = 0; w < kT / 32; ++w) hd += sred[w];
    float extra = __expf(gC) * hd;
    for (int s = 0; s < len; ++s) extra += sdg[64 + s];
    sdg[len - 1] += extra;
    float run = 0.f;
    for (int r = len - 1; r >= 0; --r) {
      run += sdg[r];
      dg[(t0 + r) * Hv + j] = run;
    }
  }
}

constexpr size_t kPrepFwdSmem = 5 * kTileB + (2 * 64 + 3 * 16 * 17) * sizeof(float);
constexpr size_t kPrepBwdSmem = 8 * kTileB + (2 * 64 + 3 * 16 * 17) * sizeof(float);
constexpr size_t kStateSmem = 8 * kTileB + 2 * 64 * sizeof(float);
constexpr size_t kOutSmem = 5 * kTileB + 64 * sizeof(float);
constexpr size_t kWalkSmem = 12 * kTileB + 2 * 64 * sizeof(float);
constexpr size_t kGradSmem = 12 * kTileB + (2 * 64 + 7 * 64 + 8) * sizeof(float);
static_assert(kGradSmem <= 227 * 1024, "gradient tiles exceed the shared memory of one CTA");

template <typename IT>
cudaError_t forward_t(const Dims& d, const FwdArgs& a, const Workspace& ws, cudaStream_t s) {
  if (d.max_chunks > 0) {
    const dim3 gc(d.max_chunks, d.Hv);
    auto prep = s64_prep_kernel<IT, false>;
    set_smem_once((const void*)prep, kPrepFwdSmem);
    prep<<<gc, kT, kPrepFwdSmem, s>>>(d, (const IT*)a.q, (const IT*)a.k, (const IT*)a.v, a.g, (const IT*)a.beta,
                                      nullptr, ws);
    stage_mark(s, "fwd_prep");
  }
  if (d.num_seqs > 0) {
    set_smem_once((const void*)s64_state_kernel<IT>, kStateSmem);
    s64_state_kernel<IT><<<dim3(d.num_seqs, d.Hv), kT, kStateSmem, s>>>(d, (const IT*)a.k, a.S0, a.S_T, a.h_saved, ws);
    stage_mark(s, "fwd_state");
  }
  if (d.max_chunks > 0) {
    set_smem_once((const void*)s64_out_kernel<IT>, kOutSmem);
    s64_out_kernel<IT><<<dim3(d.max_chunks, d.Hv), kT, kOutSmem, s>>>(d, (const IT*)a.q, (const IT*)a.k, a.h_saved,
                                                                      (IT*)a.o, ws);
    stage_mark(s, "fwd_out");
  }
  return cudaGetLastError();
}

template <typename IT>
cudaError_t backward_t(const Dims& d, const BwdArgs& a, const Workspace& ws, cudaStream_t s) {
  const dim3 gc(d.max_chunks, d.Hv);
  if (d.max_chunks > 0) {
    auto prep = s64_prep_kernel<IT, true>;
    set_smem_once((const void*)prep, kPrepBwdSmem);
    prep<<<gc, kT, kPrepBwdSmem, s>>>(d, (const IT*)a.q, (const IT*)a.k, (const IT*)a.v, a.g, (const IT*)a.beta,
                                      a.h_saved, ws);
    stage_mark(s, "bwd_prep");
  }
  if (d.num_seqs > 0) {
    set_smem_once((const void*)s64_walk_kernel<IT>, kWalkSmem);
    s64_walk_kernel<IT><<<dim3(d.num_seqs, d.Hv), kT, kWalkSmem, s>>>(d, (const IT*)a.q, (const IT*)a.k,
                                                                      (const IT*)a.dO, a.dS_T, a.dS0, ws);
    stage_mark(s, "bwd_walk");
  }
  if (d.max_chunks > 0) {
    set_smem_once((const void*)s64_grad_kernel<IT>, kGradSmem);
    s64_grad_kernel<IT><<<gc, kT, kGradSmem, s>>>(d, (const IT*)a.q, (const IT*)a.k, (const IT*)a.v,
                                                  (const IT*)a.beta, a.h_saved, (const IT*)a.dO, (IT*)a.dq,
                                                  (IT*)a.dk, (IT*)a.dv, a.dg, (IT*)a.dbeta, ws);
    stage_mark(s, "bwd_grad");
  }
  if (d.G > 1 && d.T_total > 0) return launch_group_reduce(d, a.dq, a.dk, ws, s);
  return cudaGetLastError();
}

}  // namespace

#ifdef GDR_TRACE
// Phase cycles of the traced CTA, [kernel][mark]: 0 forward prep, 1 backward prep, 2 state,
// 3 out, 4 walk, 5 grad.
extern "C" int gdr_debug_trace_simt(unsigned long long* out) {
  return cudaMemcpyFromSymbol(out, tcx::g_gdr_trace, sizeof(tcx::g_gdr_trace)) == cudaSuccess ? 0 : 1;
}
#endif

cudaError_t simt_small_forward(const Dims& d, const FwdArgs& a, const Workspace& ws, cudaStream_t s) {
  return d.dtype == GDR_DTYPE_F32 ? forward_t<float>(d, a, ws, s) : forward_t<__nv_bfloat16>(d, a, ws, s);
}

cudaError_t simt_small_backward(const Dims& d, const BwdArgs& a, const Workspace& ws, cudaStream_t s) {
  return d.dtype == GDR_DTYPE_F32 ? backward_t<float>(d, a, ws, s) : backward_t<__nv_bfloat16>(d, a, ws, s);
}

}  // namespace gdr
