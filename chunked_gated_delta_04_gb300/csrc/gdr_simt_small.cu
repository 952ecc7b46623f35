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
//          W = T diag(beta e^gamma) K, U = T diag(beta) V; the forward's also P = Q K^T * Gam
//          (lower, with the diagonal, for the state kernel's output).  The backward's variant forms
//          Vn = U - W h (h as saved by the forward), P = Q K^T * Gam (lower, with the
//          diagonal), K K^T * Gam (strictly lower) and the walk's two dh'-free terms
//          scale P^T dO and scale (diag(e^gamma) Q)^T dO, and keeps T.
//   state  per (sequence, v-head, 32 columns of DV), chunks in order: Vn = U - W h, the
//          output's columns O = scale (diag(e^gamma) Q h + P Vn) (P from the prep), and
//          h <- e^{gamma_C} h + K^T diag(e^{gamma_C - gamma}) Vn.
//   walk   per (sequence, v-head, 32 columns of DV), chunks in reverse (two tile products per chunk):
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
#include "tc_primitives.cuh"

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

// acc[i][j] += sum_{k < K} At[k][4 ty + i] * B[k][TN tx + j]   (kNeg: -=).  TN = 4 covers a
// 64 x 64 output, TN = 2 a 64 x 32 one.
template <bool kNeg = false, int TN = 4>
__device__ __forceinline__ void mm(float (&acc)[4][TN], const float* __restrict__ At, const float* __restrict__ B,
                                   int K) {
  const float* a = At + 4 * ty_();
  const float* b = B + TN * tx_();
#pragma unroll 8
  for (int k = 0; k < K; ++k) {
    const float4 av = *reinterpret_cast<const float4*>(a + k * kTS);
    float br[TN];
    if constexpr (TN == 4) {
      const float4 bv = *reinterpret_cast<const float4*>(b + k * kTS);
      br[0] = bv.x; br[1] = bv.y; br[2] = bv.z; br[3] = bv.w;
    } else {
      const float2 bv = *reinterpret_cast<const float2*>(b + k * kTS);
      br[0] = bv.x; br[1] = bv.y;
    }
    const float ar[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(kNeg ? -ar[i] : ar[i], br[j], acc[i][j]);
  }
}

template <int TN>
__device__ __forceinline__ void blk_zero(float (&a)[4][TN]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) a[i][j] = 0.f;
}

// tile[4 ty + i][TN tx + j] = v[i][j]
template <int TN>
__device__ __forceinline__ void put_rows_n(float* t, const float (&v)[4][TN]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float* p = t + (4 * ty_() + i) * kTS + TN * tx_();
    if constexpr (TN == 4)
      *reinterpret_cast<float4*>(p) = make_float4(v[i][0], v[i][1], v[i][2], v[i][3]);
    else
      *reinterpret_cast<float2*>(p) = make_float2(v[i][0], v[i][1]);
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
      float ar[16];  // row r of A_bb, read ahead of the dependent sum (A[r][m] = 0 for m >= r)
#pragma unroll
      for (int m4 = 0; m4 < 16; m4 += 4) {
        if (m4 < r) {
          const float4 a4 = *reinterpret_cast<const float4*>(A + (o + r) * kTS + o + m4);
          ar[m4] = a4.x; ar[m4 + 1] = a4.y; ar[m4 + 2] = a4.z; ar[m4 + 3] = a4.w;
        }
      }
      float p0 = r == c ? 1.f : 0.f, p1 = 0.f;
#pragma unroll
      for (int m = 0; m < r; ++m) {  // x[m] = 0 for m < c
        if (m & 1)
          p1 = fmaf(-ar[m], x[m], p1);
        else
          p0 = fmaf(-ar[m], x[m], p0);
      }
      x[r] = p0 + p1;
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
__device__ __forceinline__ void prep_body(const Dims& d, const IT* __restrict__ q, const IT* __restrict__ k,
                                          const IT* __restrict__ v, const float* __restrict__ g,
                                          const IT* __restrict__ beta, const void* __restrict__ h_saved,
                                          const Workspace& ws, float* sm) {
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
  float* sH = sTt + kTileF;     // backward: h [dk][dv]; forward: Q^T [dk][tok]
  float* sWt = sH + kTileF;     // backward: W^T [dk][tok]
  float* sg = kBwd ? sWt + kTileF : sH + kTileF;
  float* sb = sg + kChunk;
  float* sY = sb + kChunk;      // [3][16][17] solve scratch
  auto krow = [&](int r) { return k + ((t0 + r) * Hk + i) * DK; };
  load_cols<IT>(sKt, krow, len, DK);
  load_rows<IT>(sKs, krow, len, DK);
  load_rows<IT>(sVs, [&](int r) { return v + ((t0 + r) * Hv + j) * DV; }, len, DV);
  if (kBwd)
    load_h(sH, h_saved, d, ch, false);
  else
    load_cols<IT>(sH, [&](int r) { return q + ((t0 + r) * Hk + i) * DK; }, len, DK);
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
    if (kBwd || d.save_wy) {  // K K^T * Gam for the gradients (the backward's, or saved by the forward)
      float* Ak = ws.Ak + ch * 64 * 64;
#pragma unroll
      for (int a = 0; a < 4; ++a)
        *reinterpret_cast<float4*>(Ak + (4 * ty + a) * 64 + 4 * tx) = make_float4(ak[a][0], ak[a][1], ak[a][2], ak[a][3]);
    }
  }
  __syncthreads();
  GDR_TRACE_MARK(kBwd ? 1 : 0, 1);
  if (!kBwd) {  // P = Q K^T * Gam (lower, with the diagonal), kept transposed for the state kernel
    Blk p;
    blk_zero(p);
    mm(p, sH, sKt, DK);
    float* Pt = ws.Pf + ch * 64 * 64;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int s2 = 4 * tx + b;
      float o[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int r = 4 * ty + a;
        o[a] = (s2 <= r && r < len) ? __expf(sg[r] - sg[s2]) * p[a][b] : 0.f;
      }
      *reinterpret_cast<float4*>(Pt + s2 * 64 + 4 * ty) = make_float4(o[0], o[1], o[2], o[3]);
    }
  }
  solve_unit_lower(sA, sTt, sY);
  if (kBwd || d.save_wy) {  // T row-major for the gradient kernel: block (4 ty.., 4 tx..) of T from T^T
    float* Tg = ws.Tm + ch * 64 * 64;
    const int ty2 = ty_(), tx2 = tx_();
    float tb[4][4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float4 t4 = *reinterpret_cast<const float4*>(sTt + (4 * tx2 + b) * kTS + 4 * ty2);
      tb[0][b] = t4.x; tb[1][b] = t4.y; tb[2][b] = t4.z; tb[3][b] = t4.w;
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
      *reinterpret_cast<float4*>(Tg + (4 * ty2 + a) * 64 + 4 * tx2) = make_float4(tb[a][0], tb[a][1], tb[a][2], tb[a][3]);
  }
  GDR_TRACE_MARK(kBwd ? 1 : 0, 2);
  Blk w, u;
  blk_zero(w);
  blk_zero(u);
  mm(w, sTt, sKs, 64);  // W = T diag(beta e^gamma) K
  mm(u, sTt, sVs, 64);  // U = T diag(beta) V
  GDR_TRACE_MARK(kBwd ? 1 : 0, 3);
  if (tid < kChunk) ws.gam[ch * kChunk + tid] = sg[tid];
  {
    float* Wt = static_cast<float*>(ws.W) + ch * DK * 64;  // W^T [DK][64] (the state kernel's and the walk's)
#pragma unroll
    for (int b = 0; b < 4; ++b)
      if (4 * tx + b < DK)
        *reinterpret_cast<float4*>(Wt + (4 * tx + b) * 64 + 4 * ty) = make_float4(w[0][b], w[1][b], w[2][b], w[3][b]);
  }
  if (!kBwd) {
    float* U = static_cast<float*>(ws.U) + ch * 64 * DV;
    if (4 * tx < DV)
#pragma unroll
      for (int a = 0; a < 4; ++a)
        *reinterpret_cast<float4*>(U + (4 * ty + a) * DV + 4 * tx) = make_float4(u[a][0], u[a][1], u[a][2], u[a][3]);
    return;
  }
  // backward: Vn = U - W h
  put_cols(sWt, w);
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

// The backward's chunk terms that involve dO (independent of the solve): P = Q K^T * Gam (lower,
// with the diagonal), and the walk's dh'-free terms scale P^T dO [tok][dv] and
// (scale diag(e^gamma) Q)^T dO [dk][dv].
template <typename IT>
__device__ __forceinline__ void pdo_body(const Dims& d, const IT* __restrict__ q, const IT* __restrict__ k,
                                         const float* __restrict__ g, const IT* __restrict__ dO,
                                         const Workspace& ws, float* sm) {
  const int c = blockIdx.x, j = blockIdx.y, i = j / d.G;
  const int4 ci = idx_chunk(d, ws, c);
  const int len = ci.z;
  const size_t t0 = (size_t)ci.y;
  if (len <= 0) return;
  const int DK = d.DK, DV = d.DV, Hv = d.Hv, Hk = d.Hk, tid = threadIdx.x, ty = ty_(), tx = tx_();
  const size_t ch = (size_t)c * Hv + j;
  float* sQt = sm;              // Q^T [dk][tok]
  float* sKt = sQt + kTileF;    // K^T [dk][tok]
  float* sQ = sKt + kTileF;     // Q [tok][dk], then scale diag(e^gamma) Q
  float* sdO = sQ + kTileF;     // dO [tok][dv]
  float* sP = sdO + kTileF;     // P [r][s]
  float* sg = sP + kTileF;
  auto qrow = [&](int r) { return q + ((t0 + r) * Hk + i) * DK; };
  float* Pt = ws.Pf + ch * 64 * 64;  // P^T [s][r]
  if (d.save_wy) {  // P saved by the forward (transposed): P row-major into its tile
    load_cols<float>(sP, [&](int s2) { return Pt + s2 * 64; }, 64, 64);
  } else {
    load_cols<IT>(sQt, qrow, len, DK);
    load_cols<IT>(sKt, [&](int r) { return k + ((t0 + r) * Hk + i) * DK; }, len, DK);
  }
  load_rows<IT>(sQ, qrow, len, DK);
  load_rows<IT>(sdO, [&](int r) { return dO + ((t0 + r) * Hv + j) * DV; }, len, DV);
  cp_commit();
  chunk_gamma(g, t0, len, Hv, j, sg);
  cp_wait<0>();
  __syncthreads();
  if (!d.save_wy) {
    Blk p;
    blk_zero(p);
    mm(p, sQt, sKt, DK);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int r = 4 * ty + a;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int s = 4 * tx + b;
        p[a][b] = (s <= r && r < len) ? __expf(sg[r] - sg[s]) * p[a][b] : 0.f;
      }
    }
#pragma unroll
    for (int b = 0; b < 4; ++b)
      *reinterpret_cast<float4*>(Pt + (4 * tx + b) * 64 + 4 * ty) = make_float4(p[0][b], p[1][b], p[2][b], p[3][b]);
    put_rows(sP, p);
  }
  for (int e = tid; e < 64 * 64; e += kT) {  // Q rows -> scale e^gamma Q
    const int r = e >> 6, x = e & 63;
    sQ[r * kTS + x] *= d.scale * __expf(sg[r]);
  }
  __syncthreads();
  Blk a1, a2;
  blk_zero(a1);
  blk_zero(a2);
  mm(a1, sP, sdO, 64);
  mm(a2, sQ, sdO, 64);
  float* PdO = ws.PdO + ch * 64 * DV;
  float* QdO = ws.QdO + ch * DK * DV;
  if (4 * tx < DV)
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int r = 4 * ty + a;
      *reinterpret_cast<float4*>(PdO + r * DV + 4 * tx) =
          make_float4(d.scale * a1[a][0], d.scale * a1[a][1], d.scale * a1[a][2], d.scale * a1[a][3]);
      if (r < DK) *reinterpret_cast<float4*>(QdO + r * DV + 4 * tx) = make_float4(a2[a][0], a2[a][1], a2[a][2], a2[a][3]);
    }
}

// Chunk prep, one CTA per (chunk, v-head); the backward's launch has a second CTA per
// (chunk, v-head) (blockIdx.z = 1) that forms the dO terms beside it.
template <typename IT, bool kBwd>
__global__ void __launch_bounds__(kT) s64_prep_kernel(Dims d, const IT* __restrict__ q, const IT* __restrict__ k,
                                                      const IT* __restrict__ v, const float* __restrict__ g,
                                                      const IT* __restrict__ beta, const void* __restrict__ h_saved,
                                                      const IT* __restrict__ dO, Workspace ws) {
  extern __shared__ __align__(16) float sm[];
  // the first kernel of a fixed-length call (no index kernel ran): a fresh status word (these
  // kernels set no bit; a memset node before it measured ~4 us per fwd+bwd step at B=1, T=128)
  if (d.cu == nullptr && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x < 64)
    ws.status[threadIdx.x] = 0u;
  if (kBwd && (blockIdx.z == 1 || d.save_wy))  // with saved factors only the dO terms remain
    pdo_body<IT>(d, q, k, g, dO, ws, sm);
  else
    prep_body<IT, kBwd>(d, q, k, v, g, beta, h_saved, ws, sm);
}

// ---------------------------------------------------------------------------------
// state (forward recurrence), one CTA per (sequence, v-head, 32-column slice of DV): the DV
// columns of the state evolve independently
// ---------------------------------------------------------------------------------
constexpr int kSlice = 32;  // DV columns per CTA of the sequential kernels
constexpr int kSTN = kSlice / 16;
typedef float SBlk[4][kSTN];

template <typename IT>
__global__ void __launch_bounds__(kT) s64_state_kernel(Dims d, const IT* __restrict__ q, const IT* __restrict__ k,
                                                       const float* __restrict__ S0, float* __restrict__ S_T,
                                                       void* __restrict__ h_saved, IT* __restrict__ o, Workspace ws) {
  extern __shared__ __align__(16) float sm[];
  GDR_TRACE_INIT();
  const int n = idx_seq(d, ws, blockIdx.x);
  const int c_begin = idx_seq_off(d, ws, n), c_end = idx_seq_off(d, ws, n + 1);
  const int j = blockIdx.y, i = j / d.G;
  const int DK = d.DK, DV = d.DV, Hv = d.Hv, Hk = d.Hk, tid = threadIdx.x, ty = ty_(), tx = tx_();
  const int dv0 = blockIdx.z * kSlice, nv = min(kSlice, DV - dv0);  // this CTA's columns
  const bool col_ok = kSTN * tx < nv;
  float* sH = sm;               // h [dk][slice]
  float* sVd = sH + kTileF;     // diag(e^{gamma_C - gamma}) Vn [tok][slice]
  float* sVn = sVd + kTileF;    // Vn [tok][slice]
  // two stages of {W^T [dk][tok], K [tok][dk], U [tok][slice], Q^T [dk][tok], P^T [s][r], gamma}
  float* st0 = sVn + kTileF;
  constexpr int kStageF = 5 * kTileF + kChunk;
  auto issue = [&](int c, int b) {  // chunk c's tiles into stage b (one cp.async group)
    const int4 ci = idx_chunk(d, ws, c);
    const size_t t0 = (size_t)ci.y, ch = (size_t)c * Hv + j;
    float* t = st0 + b * kStageF;
    const float* Wt = static_cast<const float*>(ws.W) + ch * DK * 64;
    const float* U = static_cast<const float*>(ws.U) + ch * 64 * DV + dv0;
    const float* Pt = ws.Pf + ch * 64 * 64;
    load_rows<float>(t, [&](int x) { return Wt + x * 64; }, DK, 64);
    load_rows<IT>(t + kTileF, [&](int r) { return k + ((t0 + r) * Hk + i) * DK; }, ci.z, DK);
    load_rows<float>(t + 2 * kTileF, [&](int r) { return U + r * DV; }, ci.z, nv);
    load_cols<IT>(t + 3 * kTileF, [&](int r) { return q + ((t0 + r) * Hk + i) * DK; }, ci.z, DK);
    load_rows<float>(t + 4 * kTileF, [&](int s2) { return Pt + s2 * 64; }, 64, 64);
    if (tid < 16) cp_async16(t + 5 * kTileF + 4 * tid, ws.gam + ch * kChunk + 4 * tid, true);
    cp_commit();
  };
  SBlk h;
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < kSTN; ++b) {
      const int x = 4 * ty + a, y = kSTN * tx + b;
      h[a][b] = (S0 && x < DK && y < nv) ? S0[((size_t)n * Hv + j) * DK * DV + state_idx(d.layout, x, dv0 + y, DK, DV)]
                                         : 0.f;
    }
  put_rows_n(sH, h);
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
    const float* sQt = sU + kTileF;
    const float* sPt = sQt + kTileF;
    const float* sg = sPt + kTileF;
    const size_t t0 = (size_t)ci.y;
    if (col_ok)  // the state at the chunk start
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int x = 4 * ty + a;
        if (x >= DK) continue;
        const size_t e = ch * DK * DV + (size_t)x * DV + dv0 + kSTN * tx;
        if (d.h_bf16) {
          __nv_bfloat16* hp = static_cast<__nv_bfloat16*>(h_saved) + e;
#pragma unroll
          for (int b = 0; b < kSTN; ++b) hp[b] = __float2bfloat16_rn(h[a][b]);
        } else {
          *reinterpret_cast<float2*>(static_cast<float*>(h_saved) + e) = make_float2(h[a][0], h[a][1]);
        }
      }
    SBlk vn, oo;
    blk_zero(vn);
    blk_zero(oo);
    mm(vn, sWt, sH, DK);  // W h
    mm(oo, sQt, sH, DK);  // Q h (the output's inter-chunk term)
    GDR_TRACE_MARK(2, 1);
    const float gC = sg[len - 1], eC = __expf(gC);
    SBlk vu;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int r = 4 * ty + a;
      const bool in = r < len;
      const float dec = in ? __expf(gC - sg[r]) : 0.f, eg = __expf(sg[r]);
      const float2 u2 = *reinterpret_cast<const float2*>(sU + r * kTS + kSTN * tx);
      vu[a][0] = in ? u2.x - vn[a][0] : 0.f;
      vu[a][1] = in ? u2.y - vn[a][1] : 0.f;
#pragma unroll
      for (int b = 0; b < kSTN; ++b) {
        vn[a][b] = dec * vu[a][b];
        oo[a][b] *= eg;
      }
    }
    put_rows_n(sVn, vu);
    put_rows_n(sVd, vn);
    if (d.save_wy && col_ok) {  // Vn for the backward
      float* Vn = static_cast<float*>(ws.Vn) + ch * 64 * DV + dv0;
#pragma unroll
      for (int a = 0; a < 4; ++a)
        *reinterpret_cast<float2*>(Vn + (4 * ty + a) * DV + kSTN * tx) = make_float2(vu[a][0], vu[a][1]);
    }
    __syncthreads();
    GDR_TRACE_MARK(2, 2);
    mm(oo, sPt, sVn, 64);  // + P Vn: O = scale (diag(e^gamma) Q h + P Vn)
    if (col_ok)
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int r = 4 * ty + a;
        if (r >= len) continue;
        IT* op = o + ((t0 + r) * Hv + j) * DV + dv0 + kSTN * tx;
#pragma unroll
        for (int b = 0; b < kSTN; ++b) op[b] = from_f32<IT>(d.scale * oo[a][b]);
      }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < kSTN; ++b) h[a][b] *= eC;
    mm(h, sK, sVd, 64);  // + K^T diag(e^{gamma_C - gamma}) Vn
    GDR_TRACE_MARK(2, 3);
    put_rows_n(sH, h);
  }
  if (S_T) {
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < kSTN; ++b) {
        const int x = 4 * ty + a, y = kSTN * tx + b;
        if (x < DK && y < nv) S_T[((size_t)n * Hv + j) * DK * DV + state_idx(d.layout, x, dv0 + y, DK, DV)] = h[a][b];
      }
  }
}

// ---------------------------------------------------------------------------------
// walk (reverse state-gradient recurrence), one CTA per (sequence, v-head, 32-column slice)
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
  const int dv0 = blockIdx.z * kSlice, nv = min(kSlice, DV - dv0);  // this CTA's columns
  const bool col_ok = kSTN * tx < nv;
  float* sDh = sm;              // dh' [dk][slice]
  float* sDvn = sDh + kTileF;   // dVn [tok][slice]
  // two stages of {scale P^T dO [tok][slice], K^T [dk][tok], (scale diag(e^gamma) Q)^T dO [dk][slice],
  // W [tok][dk], gamma}: the dh'-free terms come ready from the backward's prep
  float* st0 = sDvn + kTileF;
  constexpr int kStageF = 4 * kTileF + kChunk;
  auto issue = [&](int c, int b) {  // chunk c's tiles into stage b (one cp.async group)
    const int4 ci = idx_chunk(d, ws, c);
    const size_t t0 = (size_t)ci.y, ch = (size_t)c * Hv + j;
    float* t = st0 + b * kStageF;
    const float* PdO = ws.PdO + ch * 64 * DV + dv0;
    const float* QdO = ws.QdO + ch * DK * DV + dv0;
    const float* Wt = static_cast<const float*>(ws.W) + ch * DK * 64;
    load_rows<float>(t, [&](int r) { return PdO + r * DV; }, 64, nv);
    load_cols<IT>(t + kTileF, [&](int r) { return k + ((t0 + r) * Hk + i) * DK; }, ci.z, DK);
    load_rows<float>(t + 2 * kTileF, [&](int a) { return QdO + a * DV; }, DK, nv);
    load_cols<float>(t + 3 * kTileF, [&](int x) { return Wt + x * 64; }, DK, 64);  // W rows from W^T
    if (tid < 16) cp_async16(t + 4 * kTileF + 4 * tid, ws.gam + ch * kChunk + 4 * tid, true);
    cp_commit();
  };
  SBlk dh;
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < kSTN; ++b) {
      const int x = 4 * ty + a, y = kSTN * tx + b;
      dh[a][b] = (dS_T && x < DK && y < nv)
                     ? dS_T[((size_t)n * Hv + j) * DK * DV + state_idx(d.layout, x, dv0 + y, DK, DV)]
                     : 0.f;
    }
  put_rows_n(sDh, dh);
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
    const float* sPdO = st0 + stg * kStageF;
    const float* sKt = sPdO + kTileF;
    const float* sQdO = sKt + kTileF;
    const float* sW = sQdO + kTileF;
    const float* sg = sW + kTileF;
    float* dhp = static_cast<float*>(ws.dhp) + ch * DK * DV + dv0;
    if (col_ok)
#pragma unroll
      for (int a = 0; a < 4; ++a)
        if (4 * ty + a < DK)
          *reinterpret_cast<float2*>(dhp + (4 * ty + a) * DV + kSTN * tx) = make_float2(dh[a][0], dh[a][1]);
    SBlk a2;
    blk_zero(a2);
    mm(a2, sKt, sDh, DK);  // K dh'
    GDR_TRACE_MARK(4, 1);
    const float gC = sg[len - 1], eC = __expf(gC);
    float* dVn = static_cast<float*>(ws.dVn) + ch * 64 * DV + dv0;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int s2 = 4 * ty + a;
      const bool in = s2 < len;
      const float dec = in ? __expf(gC - sg[s2]) : 0.f;
      const float2 p2 = *reinterpret_cast<const float2*>(sPdO + s2 * kTS + kSTN * tx);
      a2[a][0] = in ? fmaf(dec, a2[a][0], p2.x) : 0.f;
      a2[a][1] = in ? fmaf(dec, a2[a][1], p2.y) : 0.f;
      if (col_ok) *reinterpret_cast<float2*>(dVn + s2 * DV + kSTN * tx) = make_float2(a2[a][0], a2[a][1]);
    }
    put_rows_n(sDvn, a2);
    __syncthreads();
    GDR_TRACE_MARK(4, 2);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float2 q2 = *reinterpret_cast<const float2*>(sQdO + (4 * ty + a) * kTS + kSTN * tx);
      dh[a][0] = fmaf(eC, dh[a][0], q2.x);
      dh[a][1] = fmaf(eC, dh[a][1], q2.y);
    }
    mm<true>(dh, sW, sDvn, 64);  // - W^T dVn
    GDR_TRACE_MARK(4, 3);
    put_rows_n(sDh, dh);
  }
  if (dS0) {
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < kSTN; ++b) {
        const int x = 4 * ty + a, y = kSTN * tx + b;
        if (x < DK && y < nv) dS0[((size_t)n * Hv + j) * DK * DV + state_idx(d.layout, x, dv0 + y, DK, DV)] = dh[a][b];
      }
  }
}

// ---------------------------------------------------------------------------------
// grad: every gradient of one (chunk, v-head), on a cluster of four CTAs
// ---------------------------------------------------------------------------------
// The WY backward is regrouped around one identity: with B_k = diag(beta e^gamma) K and
// B_v = diag(beta) V, Vn = U - W h = T (B_v - B_k h), so B_v - B_k h = (I + A) Vn and
//   dT = dW B_k^T + dVn B_v^T = dVn ((I + A) Vn)^T        (dW = -dVn h^T),
//   dB_k = T^T dW = -(T^T dVn) h^T = -dB_v h^T,
// which needs neither dW nor K^T / V^T tiles.  The products split over the four CTAs of a
// cluster so that the longest chain, rank 1's, is five products (S = 64 x 68 tiles; each rank
// names its own slots):
//   rank 0: A  dP = scale (dO Vn^T) * Gam * M       (S0 dO^T, S1 Vn^T)     -> S8 dP
//           A3 dk_0 = dP^T Q                         (S8, S2 Q)
//           G  dB_v = T^T dVn -> dv                  (S5 T, S6 dVn)        -> S9 dB_v^T
//           H  dB_k = -dB_v h^T; dk_0 += diag(beta e^gamma) dB_k  (S9, S3 h^T)
//   rank 2: A again (dP^T into S8), then dq = scale diag(e^gamma) dO h^T + dP K  (S0, S3; S8, S4 K)
//   rank 3: Vn dh'^T (S1 Vn^T, S2 dh'^T): dk_3 = diag(e^{gamma_C - gamma}) Vn dh'^T and the gate
//           term k_r^T dh' vn_r; <dh', h>
//   rank 1: Z  (I + A) Vn = Vn + diag(beta)(K K^T * Gam) Vn  (S3 (K K^T * Gam)^T, S4 Vn) -> S0 transposed
//           D  dT = dVn ((I + A) Vn)^T               (S5 dVn^T, S0)         -> S1
//           E  X = T^T dT                            (S6 T, S1)             -> S0 X^T; S4 T^T
//           F  dA = -strict-lower(X T^T)             (S0, S4)               -> S1 L = diag(beta)(dA * Gam)
//           I  dk_1 = (L + L^T) K  [= diag(beta)(dA * Gam) K + (dA * Gam)^T diag(beta) K]  (S5, S2 K)
// Ranks 0, 2 and 3 store what rank 1 needs (dk blocks, per-row and per-column sums) into rank
// 1's shared memory (distributed shared memory); one cluster barrier later rank 1 writes dk,
// dbeta and dg.  All CTAs of a cluster hold the same chunk, so an empty chunk returns from all
// of them before any cluster barrier.
constexpr int kGradTiles = 10;
constexpr int kGradCluster = 4;
template <typename IT>
__global__ void __launch_bounds__(kT) s64_grad_kernel(Dims d, const IT* __restrict__ q, const IT* __restrict__ k,
                                                      const IT* __restrict__ v, const IT* __restrict__ beta,
                                                      const void* __restrict__ h_saved, const IT* __restrict__ dO,
                                                      IT* __restrict__ dq, IT* __restrict__ dk, IT* __restrict__ dv,
                                                      float* __restrict__ dg, IT* __restrict__ dbeta, Workspace ws) {
  extern __shared__ __align__(16) float sm[];
  GDR_TRACE_INIT();
  const int c = blockIdx.x / kGradCluster, j = blockIdx.y, i = j / d.G;
  const uint32_t rank = tc::cluster_ctarank();
  const int4 ci = idx_chunk(d, ws, c);
  const int len = ci.z;
  const size_t t0 = (size_t)ci.y;
  if (len <= 0) return;  // every CTA of the cluster
  const int DK = d.DK, DV = d.DV, Hv = d.Hv, Hk = d.Hk, tid = threadIdx.x, ty = ty_(), tx = tx_();
  const int lane = tid & 31, warp = tid >> 5;
  const size_t ch = (size_t)c * Hv + j;
  float* S[kGradTiles];
#pragma unroll
  for (int x = 0; x < kGradTiles; ++x) S[x] = sm + x * kTileF;
  float* sg = sm + kGradTiles * kTileF;
  float* sb = sg + kChunk;
  // rank 1's exchange area: per-row sums [7][64] (0 dP*QK, 1 dA*A, 2 dA*(KK^T*Gam), 3 kdv, 4 qh,
  // 5 dB_v.v, 6 dB_k.k), <dh', h> (rank 3's 8 warp partials), rank 0's column partials of dP*QK
  // and its own of dA*A ([16][64] each, in S9), the dk blocks of ranks 0 and 3 (S7, S8)
  float* rows = sb + kChunk;
  float* sred = rows + 7 * 64;
  float* colA = S[9];
  float* colB = S[9] + 16 * 64;
  float* dk0 = S[7];
  float* dk3 = S[8];
  const uint32_t peer_base = tc::mapa(tc::smem_u32(sm), 1);  // rank 1's shared memory
  auto peer = [&](const float* local) { return peer_base + (uint32_t)((local - sm) * sizeof(float)); };
  auto st_peer = [&](const float* local, float x) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(peer(local)), "f"(x) : "memory");
  };
  const float* Vn = static_cast<const float*>(ws.Vn) + ch * 64 * DV;
  const float* dVn = static_cast<const float*>(ws.dVn) + ch * 64 * DV;
  const float* dhp = static_cast<const float*>(ws.dhp) + ch * DK * DV;
  const float* Tg = ws.Tm + ch * 64 * 64;
  auto qrow = [&](int r) { return q + ((t0 + r) * Hk + i) * DK; };
  auto krow = [&](int r) { return k + ((t0 + r) * Hk + i) * DK; };
  auto dorow = [&](int r) { return dO + ((t0 + r) * Hv + j) * DV; };
  auto vnrow = [&](int r) { return Vn + r * DV; };
  if (rank == 0 || rank == 2) {
    load_cols<IT>(S[0], dorow, len, DV);
    load_cols<float>(S[1], vnrow, 64, DV);
    load_h(S[3], h_saved, d, ch, true);
    if (rank == 0) {
      load_rows<IT>(S[2], qrow, len, DK);
      load_rows<float>(S[5], [&](int r) { return Tg + r * 64; }, 64, 64);
      load_rows<float>(S[6], [&](int r) { return dVn + r * DV; }, 64, DV);
      load_rows<IT>(S[7], [&](int r) { return v + ((t0 + r) * Hv + j) * DV; }, len, DV);
    } else {
      load_rows<IT>(S[2], qrow, len, DK);
      load_rows<IT>(S[4], krow, len, DK);
    }
  } else if (rank == 3) {
    load_cols<float>(S[1], vnrow, 64, DV);
    load_cols<float>(S[2], [&](int a) { return dhp + a * DV; }, DK, DV);
    load_rows<IT>(S[3], krow, len, DK);
  } else {
    load_cols<float>(S[3], [&](int r) { return ws.Ak + ch * 64 * 64 + r * 64; }, 64, 64);
    load_rows<float>(S[4], vnrow, 64, DV);
    load_cols<float>(S[5], [&](int r) { return dVn + r * DV; }, 64, DV);
    load_rows<float>(S[6], [&](int r) { return Tg + r * 64; }, 64, 64);
    load_rows<IT>(S[2], krow, len, DK);
  }
  if (tid < 16) cp_async16(sg + 4 * tid, ws.gam + ch * kChunk + 4 * tid, true);
  cp_commit();
  if (tid < kChunk) sb[tid] = tid < len ? ldf(beta + (t0 + tid) * Hv + j) : 0.f;
  tc::cluster_sync();  // every CTA is running before any store into rank 1's shared memory
  cp_wait<0>();
  __syncthreads();
  GDR_TRACE_MARK(5, 0);
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
  // per-row sums over the 16 threads of a row group, into rank 1's row slot
  auto rows_to_peer = [&](int slot, const float (&v4)[4]) {
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float t = sum16(v4[a]);
      if (tx == 0) st_peer(rows + slot * 64 + rr[a], t);
    }
  };
  auto dk_to_peer = [&](float* dst, const Blk& v) {
#pragma unroll
    for (int a = 0; a < 4; ++a)
      tc::st_cluster_f32x4(peer(dst + rr[a] * kTS + 4 * tx), v[a][0], v[a][1], v[a][2], v[a][3]);
  };
  if (rank == 0 || rank == 2) {
    // A: dP (rank 0 also forms the column and row sums of dP * (Q K^T))
    float pp_r[4], pp_c[4];
    {
      Blk acc;
      blk_zero(acc);
      mm(acc, S[0], S[1], DV);
      const float* Pg = ws.Pf + ch * 64 * 64;
#pragma unroll
      for (int b = 0; b < 4; ++b) pp_c[b] = 0.f;
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        float pr[4] = {0.f, 0.f, 0.f, 0.f};
        if (rank == 0) {  // P[r][s] from P^T
#pragma unroll
          for (int b = 0; b < 4; ++b) pr[b] = Pg[(4 * tx + b) * 64 + rr[a]];
        }
        pp_r[a] = 0.f;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int s2 = 4 * tx + b;
          const float raw = d.scale * acc[a][b];
          const float pp = raw * pr[b];  // dP * (Q K^T): P holds Q K^T * Gam on and below the diagonal
          pp_r[a] += pp;
          pp_c[b] += pp;
          acc[a][b] = (s2 <= rr[a] && rr[a] < len) ? raw * __expf(sg[rr[a]] - sg[s2]) : 0.f;
        }
      }
      if (rank == 0)
        put_rows_n(S[8], acc);
      else
        put_cols(S[8], acc);
    }
    __syncthreads();
    GDR_TRACE_MARK(5, 1);
    if (rank == 2) {  // dq
      Blk acc;
      blk_zero(acc);
      mm(acc, S[0], S[3], DV);
      float qh_r[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const float4 q4 = *reinterpret_cast<const float4*>(S[2] + rr[a] * kTS + 4 * tx);
        qh_r[a] = q4.x * acc[a][0] + q4.y * acc[a][1] + q4.z * acc[a][2] + q4.w * acc[a][3];
        const float sc = d.scale * eg[a];
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] *= sc;
      }
      mm(acc, S[8], S[4], 64);
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
            *reinterpret_cast<float4*>(ws.dq_part + (t * Hv + j) * DK + 4 * tx) =
                make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
          }
        }
      rows_to_peer(4, qh_r);
      tc::cluster_sync();
      return;
    }
    // rank 0: A3: dk_0 = dP^T Q
    Blk dkb;
    blk_zero(dkb);
    mm(dkb, S[8], S[2], 64);
    float dbv_r[4], dbk_r[4];
    // G: dB_v = T^T dVn -> dv
    {
      Blk acc;
      blk_zero(acc);
      mm(acc, S[5], S[6], 64);
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const float4 v4 = *reinterpret_cast<const float4*>(S[7] + rr[a] * kTS + 4 * tx);
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
      put_cols(S[9], acc);
    }
    __syncthreads();
    GDR_TRACE_MARK(5, 2);
    // H: dB_k = -dB_v h^T
    {
      Blk acc;
      blk_zero(acc);
      mm<true>(acc, S[9], S[3], DV);
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        dbk_r[a] = 0.f;  // k_r . dB_k[r] needs K: formed from dk's own term below
        const float sc = br[a] * eg[a];
#pragma unroll
        for (int b = 0; b < 4; ++b) dkb[a][b] = fmaf(sc, acc[a][b], dkb[a][b]);
      }
      // k_r . dB_k[r] with K rows read from global memory (rank 0 holds no K tile)
      if (4 * tx < DK)
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          if (rr[a] >= len) continue;
          const IT* kr = krow(rr[a]) + 4 * tx;
          dbk_r[a] = ldf(kr) * acc[a][0] + ldf(kr + 1) * acc[a][1] + ldf(kr + 2) * acc[a][2] + ldf(kr + 3) * acc[a][3];
        }
    }
    GDR_TRACE_MARK(5, 3);
    dk_to_peer(dk0, dkb);
#pragma unroll
    for (int b = 0; b < 4; ++b) st_peer(colA + ty * 64 + 4 * tx + b, pp_c[b]);
    rows_to_peer(0, pp_r);
    rows_to_peer(5, dbv_r);
    rows_to_peer(6, dbk_r);
    tc::cluster_sync();  // rank 1 reads what was stored above after this barrier
    return;
  }
  if (rank == 3) {
    float hdh = 0.f;  // <dh', h>: dh' from its transposed tile, h from the saved states
    for (int e = tid; e < 64 * 64; e += kT) {
      const int a = e >> 6, b = e & 63;
      if (a < DK && b < DV) {
        const size_t he = ch * DK * DV + (size_t)a * DV + b;
        const float hv = d.h_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(h_saved)[he])
                                  : static_cast<const float*>(h_saved)[he];
        hdh = fmaf(S[2][b * kTS + a], hv, hdh);
      }
    }
    hdh = warp_sum(hdh);
    if (lane == 0) st_peer(sred + warp, hdh);
    Blk vd;
    blk_zero(vd);
    mm(vd, S[1], S[2], DV);  // Vn dh'^T
    float kdv_r[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float4 k4 = *reinterpret_cast<const float4*>(S[3] + rr[a] * kTS + 4 * tx);
      kdv_r[a] = k4.x * vd[a][0] + k4.y * vd[a][1] + k4.z * vd[a][2] + k4.w * vd[a][3];
#pragma unroll
      for (int b = 0; b < 4; ++b) vd[a][b] *= dec[a];
    }
    dk_to_peer(dk3, vd);
    rows_to_peer(3, kdv_r);
    tc::cluster_sync();
    return;
  }
  // rank 1
  float aa_r[4], aa_c[4], akk_r[4];
  // Z: (I + A) Vn
  {
    Blk acc;
    blk_zero(acc);
    mm(acc, S[3], S[4], 64);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float4 v4 = *reinterpret_cast<const float4*>(S[4] + rr[a] * kTS + 4 * tx);
      const float vr[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(br[a], acc[a][b], vr[b]);
    }
    put_cols(S[0], acc);
  }
  __syncthreads();
  GDR_TRACE_MARK(5, 4);
  // D: dT = dVn ((I + A) Vn)^T; S4 = T^T (Vn is no longer needed)
  {
    Blk acc;
    blk_zero(acc);
    mm(acc, S[5], S[0], DV);
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (!(rr[a] < len && 4 * tx + b < len)) acc[a][b] = 0.f;
    put_rows_n(S[1], acc);
    for (int e = tid; e < 64 * 64; e += kT) {
      const int r = e >> 6, s2 = e & 63;
      S[4][s2 * kTS + r] = S[6][r * kTS + s2];
    }
  }
  __syncthreads();
  GDR_TRACE_MARK(5, 5);
  // E: X = T^T dT
  {
    Blk acc;
    blk_zero(acc);
    mm(acc, S[6], S[1], 64);
    put_cols(S[0], acc);
  }
  __syncthreads();
  GDR_TRACE_MARK(5, 6);
  // F: dA = -strict-lower(X T^T)
  {
    Blk acc;
    blk_zero(acc);
    mm(acc, S[0], S[4], 64);
#pragma unroll
    for (int b = 0; b < 4; ++b) aa_c[b] = 0.f;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      aa_r[a] = 0.f;
      akk_r[a] = 0.f;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int s2 = 4 * tx + b;
        const float akr = S[3][s2 * kTS + rr[a]];  // (K K^T * Gam)[r][s], from the transposed tile
        const bool low = s2 < rr[a] && rr[a] < len;
        const float dA = low ? -acc[a][b] : 0.f;
        const float aa = dA * br[a] * akr;  // dA * A, A = diag(beta) (K K^T * Gam)
        aa_r[a] += aa;
        aa_c[b] += aa;
        akk_r[a] += dA * akr;
        acc[a][b] = low ? br[a] * dA * __expf(sg[rr[a]] - sg[s2]) : 0.f;
      }
    }
    put_rows_n(S[1], acc);
  }
#pragma unroll
  for (int b = 0; b < 4; ++b) colB[ty * 64 + 4 * tx + b] = aa_c[b];
  __syncthreads();
  GDR_TRACE_MARK(5, 7);
  {  // S5 = L + L^T
    Blk m;
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int s2 = 4 * tx + b;
        m[a][b] = S[1][rr[a] * kTS + s2] + S[1][s2 * kTS + rr[a]];
      }
    put_rows_n(S[5], m);
  }
  __syncthreads();
  // I: dk_1 = (L + L^T) K
  Blk dkb;
  blk_zero(dkb);
  mm(dkb, S[5], S[2], 64);
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const float t1 = sum16(aa_r[a]), t2 = sum16(akk_r[a]);
    if (tx == 0) {
      rows[1 * 64 + rr[a]] = t1;
      rows[2 * 64 + rr[a]] = t2;
    }
  }
  GDR_TRACE_MARK(5, 8);
  tc::cluster_sync();  // the other ranks' dk blocks and sums have arrived
  GDR_TRACE_MARK(5, 9);
  if (4 * tx < DK)
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      if (rr[a] >= len) continue;
      const size_t t = t0 + rr[a];
      const float4 o0 = *reinterpret_cast<const float4*>(dk0 + rr[a] * kTS + 4 * tx);
      const float4 o3 = *reinterpret_cast<const float4*>(dk3 + rr[a] * kTS + 4 * tx);
      const float o4[4] = {o0.x + o3.x + dkb[a][0], o0.y + o3.y + dkb[a][1], o0.z + o3.z + dkb[a][2],
                           o0.w + o3.w + dkb[a][3]};
      if (d.G == 1) {
        IT* p = dk + (t * Hk + i) * DK + 4 * tx;
#pragma unroll
        for (int b = 0; b < 4; ++b) p[b] = from_f32<IT>(o4[b]);
      } else {
        *reinterpret_cast<float4*>(ws.dk_part + (t * Hv + j) * DK + 4 * tx) = make_float4(o4[0], o4[1], o4[2], o4[3]);
      }
    }
  float* sdg = S[0];  // d gamma per row (X^T is no longer needed)
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
  if (warp == 0) {  // dg = in-chunk reverse cumsum of d gamma, the chunk-end term added at len - 1
    float hd = 0.f;
#pragma unroll
    for (int w = 0; w < kT / 32; ++w) hd += sred[w];
    const float extra = __expf(gC) * hd + warp_sum(sdg[64 + lane] + sdg[96 + lane]);
    float lo = sdg[lane], hi = sdg[32 + lane];  // rows past len hold 0
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {  // suffix sums within each half
      const float l2 = __shfl_down_sync(0xffffffffu, lo, o), h2 = __shfl_down_sync(0xffffffffu, hi, o);
      if (lane + o < 32) {
        lo += l2;
        hi += h2;
      }
    }
    lo += __shfl_sync(0xffffffffu, hi, 0);  // the whole upper half follows every lower row
    if (lane < len) dg[(t0 + lane) * Hv + j] = lo + extra;
    if (32 + lane < len) dg[(t0 + 32 + lane) * Hv + j] = hi + extra;
  }
}

constexpr size_t kPrepFwdSmem = 6 * kTileB + (2 * 64 + 3 * 16 * 17) * sizeof(float);
constexpr size_t kPrepBwdSmem = 7 * kTileB + (2 * 64 + 3 * 16 * 17) * sizeof(float);
constexpr size_t kStateSmem = 13 * kTileB + 2 * 64 * sizeof(float);
static_assert(kStateSmem <= 227 * 1024, "state tiles exceed the shared memory of one CTA");
constexpr size_t kWalkSmem = 10 * kTileB + 2 * 64 * sizeof(float);
constexpr size_t kGradSmem = kGradTiles * kTileB + (2 * 64 + 7 * 64 + 8) * sizeof(float);
static_assert(kGradSmem <= 227 * 1024, "gradient tiles exceed the shared memory of one CTA");

// One launch; cluster > 1 = clusters of that many CTAs along x.  (Programmatic dependent launch
// of the later kernels, each letting its successor launch at its start, measured ~25 us slower
// per fwd+bwd step at B=1, T=128, D=64, and no faster without the early trigger: not used.)
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kern)(KArgs...), dim3 grid, size_t smem, cudaStream_t s, unsigned cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  unsigned na = 0;
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename IT>
cudaError_t forward_t(const Dims& d, const FwdArgs& a, const Workspace& ws, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  if (d.max_chunks > 0) {
    auto prep = s64_prep_kernel<IT, false>;
    set_smem_once((const void*)prep, kPrepFwdSmem);
    e = launch(prep, dim3(d.max_chunks, d.Hv), kPrepFwdSmem, s, 1, d, (const IT*)a.q, (const IT*)a.k,
               (const IT*)a.v, a.g, (const IT*)a.beta, (const void*)nullptr, (const IT*)nullptr, ws);
    if (e != cudaSuccess) return e;
    stage_mark(s, "fwd_prep");
  }
  if (d.num_seqs > 0) {
    auto state = s64_state_kernel<IT>;
    set_smem_once((const void*)state, kStateSmem);
    e = launch(state, dim3(d.num_seqs, d.Hv, (d.DV + kSlice - 1) / kSlice), kStateSmem, s, 1, d,
               (const IT*)a.q, (const IT*)a.k, a.S0, a.S_T, a.h_saved, (IT*)a.o, ws);
    if (e != cudaSuccess) return e;
    stage_mark(s, "fwd_state");
  }
  return cudaGetLastError();
}

template <typename IT>
cudaError_t backward_t(const Dims& d, const BwdArgs& a, const Workspace& ws, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  if (d.max_chunks > 0) {
    auto prep = s64_prep_kernel<IT, true>;
    set_smem_once((const void*)prep, kPrepBwdSmem);
    e = launch(prep, dim3(d.max_chunks, d.Hv, d.save_wy ? 1 : 2), kPrepBwdSmem, s, 1, d, (const IT*)a.q, (const IT*)a.k,
               (const IT*)a.v, a.g, (const IT*)a.beta, a.h_saved, (const IT*)a.dO, ws);
    if (e != cudaSuccess) return e;
    stage_mark(s, "bwd_prep");
  }
  if (d.num_seqs > 0) {
    auto walk = s64_walk_kernel<IT>;
    set_smem_once((const void*)walk, kWalkSmem);
    e = launch(walk, dim3(d.num_seqs, d.Hv, (d.DV + kSlice - 1) / kSlice), kWalkSmem, s, 1, d,
               (const IT*)a.q, (const IT*)a.k, (const IT*)a.dO, a.dS_T, a.dS0, ws);
    if (e != cudaSuccess) return e;
    stage_mark(s, "bwd_walk");
  }
  if (d.max_chunks > 0) {
    auto grad = s64_grad_kernel<IT>;
    set_smem_once((const void*)grad, kGradSmem);
    e = launch(grad, dim3((unsigned)kGradCluster * (unsigned)d.max_chunks, (unsigned)d.Hv), kGradSmem, s,
               (unsigned)kGradCluster, d, (const IT*)a.q, (const IT*)a.k, (const IT*)a.v, (const IT*)a.beta,
               a.h_saved, (const IT*)a.dO, (IT*)a.dq, (IT*)a.dk, (IT*)a.dv, a.dg, (IT*)a.dbeta, ws);
    if (e != cudaSuccess) return e;
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
