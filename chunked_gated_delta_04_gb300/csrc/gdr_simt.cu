// gdr_simt.cu -- fp32 SIMT kernels of the chunked gated delta rule.
//
// These run every supported shape and dtype with fp32 arithmetic (the fp32 inputs
// need ~1e-4 relative accuracy, which tf32 tensor-core products do not give).
// They follow the chunked method step by step (chunked gated delta rule, FlashQLA
// PR #34, Summary; chunk = 64 tokens), with h := S^T (DK x DV) the state at a
// chunk start, gamma the in-chunk cumsum of g and Gam[r,s] = exp(gamma_r - gamma_s):
//
//   prep   A = strict-lower(diag(beta) K K^T * Gam), T = (I + A)^{-1},
//          W = T diag(beta e^gamma) K, U = T diag(beta) V             (chunk-parallel)
//   state  Vn = U - W h; h <- e^{gamma_C} h + (diag(e^{gamma_C-gamma}) K)^T Vn
//                                                   (sequential over chunks)
//   out    O = scale (diag(e^gamma) Q h + (Q K^T * Gam * M) Vn)        (chunk-parallel)
//   walk   dVn = scale P^T dO + Kt dh';  dh = e^{gamma_C} dh' + scale Qh^T dO - W^T dVn
//                                                   (sequential, reverse)
//   grad   dq, dk, dv, dbeta, dg of one chunk from h, dh', Vn        (chunk-parallel)
//
// Work layout: chunk-parallel kernels run one CTA per (chunk slot, v-head);
// sequential kernels one CTA per (sequence, v-head, 32-wide slice of DV).
#include "gdr_chunks.cuh"
#include "gdr_device.cuh"
#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr int kThreads = 256;
constexpr int kLd = kChunk + 1;  // padded row length of 64 x 64 smem matrices

// ---------------------------------------------------------------------------------
// prep: gamma, A, T, W, U of one chunk (and T for the backward)
// ---------------------------------------------------------------------------------
template <typename IT>
__global__ void __launch_bounds__(kThreads) simt_prep_kernel(Dims d, const IT* __restrict__ k,
                                                             const IT* __restrict__ v,
                                                             const float* __restrict__ g,
                                                             const IT* __restrict__ beta, Workspace ws) {
  extern __shared__ float sm[];
  const int c = blockIdx.x, j = blockIdx.y, i = j / d.G;
  const int4 ci = idx_chunk(d, ws, c);
  const int len = ci.z, t0 = ci.y;
  if (len <= 0) return;
  const int DK = d.DK, DV = d.DV, Hv = d.Hv, Hk = d.Hk;
  float* sK = sm;                     // [64][DK]
  float* sV = sK + kChunk * DK;       // [64][DV]
  float* sA = sV + kChunk * DV;       // [64][65]
  float* sT = sA + kChunk * kLd;      // [64][65]
  float* sg = sT + kChunk * kLd;      // [64] gamma
  float* sb = sg + kChunk;            // [64] beta
  const int tid = threadIdx.x;
  for (int e = tid; e < kChunk * DK; e += kThreads) {
    const int r = e / DK, x = e % DK;
    sK[e] = r < len ? ldf(k + ((size_t)(t0 + r) * Hk + i) * DK + x) : 0.f;
  }
  for (int e = tid; e < kChunk * DV; e += kThreads) {
    const int r = e / DV, x = e % DV;
    sV[e] = r < len ? ldf(v + ((size_t)(t0 + r) * Hv + j) * DV + x) : 0.f;
  }
  if (tid < 32) {  // gamma = inclusive cumsum of g over the chunk (two 32-wide warp scans)
    float run = 0.f;
    for (int base = 0; base < kChunk; base += 32) {
      const int r = base + tid;
      float x = r < len ? g[(size_t)(t0 + r) * Hv + j] : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (tid >= o) x += y;
      }
      sg[r] = run + x;
      run += __shfl_sync(0xffffffffu, x, 31);
    }
  }
  for (int r = tid; r < kChunk; r += kThreads) sb[r] = r < len ? ldf(beta + (size_t)(t0 + r) * Hv + j) : 0.f;
  __syncthreads();
  // A[r][s] = beta_r exp(gamma_r - gamma_s) k_r.k_s for s < r < len
  for (int e = tid; e < kChunk * kChunk; e += kThreads) {
    const int r = e / kChunk, s = e % kChunk;
    float a = 0.f;
    if (s < r && r < len) {
      float dot = 0.f;
      for (int x = 0; x < DK; ++x) dot += sK[r * DK + x] * sK[s * DK + x];
      a = sb[r] * __expf(sg[r] - sg[s]) * dot;
    }
    sA[r * kLd + s] = a;
    sT[r * kLd + s] = (r == s) ? 1.f : 0.f;
  }
  __syncthreads();
  // T = (I + A)^{-1} by forward substitution: T[r][s] = -sum_{s<=m<r} A[r][m] T[m][s]
  for (int r = 1; r < len; ++r) {
    for (int s = tid; s < r; s += kThreads) {
      float acc = 0.f;
      for (int m = s; m < r; ++m) acc += sA[r * kLd + m] * sT[m * kLd + s];
      sT[r * kLd + s] = -acc;
    }
    __syncthreads();
  }
  const size_t ch = (size_t)c * Hv + j;
  float* W = (float*)ws.W + ch * kChunk * DK;
  float* U = (float*)ws.U + ch * kChunk * DV;
  for (int r = tid; r < kChunk; r += kThreads) sA[r * kLd + r] = sb[r] * __expf(sg[r]);  // beta e^gamma on A's (unused) diagonal
  __syncthreads();
  for (int e = tid; e < kChunk * DK; e += kThreads) {
    const int r = e / DK, x = e % DK;
    float acc = 0.f;
    for (int s = 0; s <= r && s < len; ++s) acc += sT[r * kLd + s] * sA[s * kLd + s] * sK[s * DK + x];
    W[e] = r < len ? acc : 0.f;
  }
  for (int e = tid; e < kChunk * DV; e += kThreads) {
    const int r = e / DV, x = e % DV;
    float acc = 0.f;
    for (int s = 0; s <= r && s < len; ++s) acc += sT[r * kLd + s] * sb[s] * sV[s * DV + x];
    U[e] = r < len ? acc : 0.f;
  }
  for (int r = tid; r < kChunk; r += kThreads) ws.gam[ch * kChunk + r] = sg[r];
  if (ws.Tm != nullptr) {
    float* Tg = ws.Tm + ch * kChunk * kChunk;
    for (int e = tid; e < kChunk * kChunk; e += kThreads) Tg[e] = sT[(e / kChunk) * kLd + e % kChunk];
  }
}

// Saved chunk-start states: fp32 or bf16 (Dims::h_bf16), read back as fp32.
struct HView {
  const void* base;  // first element of one chunk's [DK][DV] state
  int hb;
  __device__ __forceinline__ float operator[](size_t e) const {
    return hb ? __bfloat162float(static_cast<const __nv_bfloat16*>(base)[e]) : static_cast<const float*>(base)[e];
  }
};

__device__ __forceinline__ HView h_view(const void* h_saved, size_t ch, const Dims& d) {
  const size_t off = ch * d.DK * d.DV;
  return HView{d.h_bf16 ? (const void*)(static_cast<const __nv_bfloat16*>(h_saved) + off)
                        : (const void*)(static_cast<const float*>(h_saved) + off),
               d.h_bf16};
}

// ---------------------------------------------------------------------------------
// forward state walk: one CTA per (sequence, v-head, DV slice)
// ---------------------------------------------------------------------------------
template <typename IT>
__global__ void __launch_bounds__(kThreads) simt_state_kernel(Dims d, const IT* __restrict__ k,
                                                              const float* __restrict__ S0,
                                                              float* __restrict__ S_T,
                                                              void* __restrict__ h_saved, Workspace ws,
                                                              int dvs) {
  extern __shared__ float sm[];
  const int n = idx_seq(d, ws, blockIdx.x), j = blockIdx.y, i = j / d.G;
  const int dv0 = blockIdx.z * dvs;
  const int DK = d.DK, DV = d.DV, Hv = d.Hv, Hk = d.Hk;
  float* sh = sm;               // [DK][dvs]
  float* sVn = sh + DK * dvs;   // [64][dvs]
  float* sg = sVn + kChunk * dvs;
  float* sdec = sg + kChunk;    // e^{gamma_C - gamma_r} of the current chunk
  const int tid = threadIdx.x;
  for (int e = tid; e < DK * dvs; e += kThreads) {
    const int a = e / dvs, b = e % dvs;
    sh[e] = S0 ? S0[((size_t)n * Hv + j) * DK * DV + state_idx(d.layout, a, dv0 + b, DK, DV)] : 0.f;
  }
  __syncthreads();
  const int c_begin = idx_seq_off(d, ws, n), c_end = idx_seq_off(d, ws, n + 1);
  for (int c = c_begin; c < c_end; ++c) {
    const int4 ci = idx_chunk(d, ws, c);
    const int len = ci.z, t0 = ci.y;
    const size_t ch = (size_t)c * Hv + j;
    for (int e = tid; e < DK * dvs; e += kThreads) {
      const int a = e / dvs, b = e % dvs;
      const size_t hi = ch * DK * DV + (size_t)a * DV + dv0 + b;
      if (d.h_bf16)
        static_cast<__nv_bfloat16*>(h_saved)[hi] = __float2bfloat16_rn(sh[e]);
      else
        static_cast<float*>(h_saved)[hi] = sh[e];
    }
    for (int r = tid; r < kChunk; r += kThreads) sg[r] = ws.gam[ch * kChunk + r];
    const float* W = (const float*)ws.W + ch * kChunk * DK;
    const float* U = (const float*)ws.U + ch * kChunk * DV;
    float* Vn = (float*)ws.Vn + ch * kChunk * DV;
    for (int e = tid; e < kChunk * dvs; e += kThreads) {
      const int r = e / dvs, b = e % dvs;
      float acc = 0.f;
      if (r < len) {
        acc = U[r * DV + dv0 + b];
        for (int a = 0; a < DK; ++a) acc -= W[r * DK + a] * sh[a * dvs + b];
      }
      sVn[e] = acc;
      Vn[r * DV + dv0 + b] = acc;
    }
    __syncthreads();
    const float gC = sg[len - 1];
    const float eC = __expf(gC);
    for (int r = tid; r < kChunk; r += kThreads) sdec[r] = r < len ? __expf(gC - sg[r]) : 0.f;
    __syncthreads();
    for (int e = tid; e < DK * dvs; e += kThreads) {
      const int a = e / dvs, b = e % dvs;
      float acc = 0.f;
      for (int r = 0; r < len; ++r) acc += sdec[r] * ldf(k + ((size_t)(t0 + r) * Hk + i) * DK + a) * sVn[r * dvs + b];
      sh[e] = eC * sh[e] + acc;
    }
    __syncthreads();
  }
  if (S_T) {
    for (int e = tid; e < DK * dvs; e += kThreads) {
      const int a = e / dvs, b = e % dvs;
      S_T[((size_t)n * Hv + j) * DK * DV + state_idx(d.layout, a, dv0 + b, DK, DV)] = sh[e];
    }
  }
}

// ---------------------------------------------------------------------------------
// forward output of one chunk: O = scale (diag(e^gamma) Q h + (Q K^T * Gam * M) Vn)
// ---------------------------------------------------------------------------------
template <typename IT>
__global__ void __launch_bounds__(kThreads) simt_out_kernel(Dims d, const IT* __restrict__ q,
                                                            const IT* __restrict__ k,
                                                            const void* __restrict__ h_saved,
                                                            IT* __restrict__ o, Workspace ws) {
  extern __shared__ float sm[];
  const int c = blockIdx.x, j = blockIdx.y, i = j / d.G;
  const int4 ci = idx_chunk(d, ws, c);
  const int len = ci.z, t0 = ci.y;
  if (len <= 0) return;
  const int DK = d.DK, DV = d.DV, Hv = d.Hv, Hk = d.Hk;
  float* sQ = sm;                // [64][DK]
  float* sK = sQ + kChunk * DK;  // [64][DK]
  float* sP = sK + kChunk * DK;  // [64][65]
  float* sg = sP + kChunk * kLd;
  const int tid = threadIdx.x;
  const size_t ch = (size_t)c * Hv + j;
  for (int e = tid; e < kChunk * DK; e += kThreads) {
    const int r = e / DK, x = e % DK;
    const bool ok = r < len;
    sQ[e] = ok ? ldf(q + ((size_t)(t0 + r) * Hk + i) * DK + x) : 0.f;
    sK[e] = ok ? ldf(k + ((size_t)(t0 + r) * Hk + i) * DK + x) : 0.f;
  }
  for (int r = tid; r < kChunk; r += kThreads) sg[r] = ws.gam[ch * kChunk + r];
  __syncthreads();
  for (int e = tid; e < kChunk * kChunk; e += kThreads) {
    const int r = e / kChunk, s = e % kChunk;
    float p = 0.f;
    if (s <= r && r < len) {
      float dot = 0.f;
      for (int x = 0; x < DK; ++x) dot += sQ[r * DK + x] * sK[s * DK + x];
      p = dot * __expf(sg[r] - sg[s]);
    }
    sP[r * kLd + s] = p;
  }
  __syncthreads();
  const HView h = h_view(h_saved, ch, d);
  const float* Vn = (const float*)ws.Vn + ch * kChunk * DV;
  for (int e = tid; e < len * DV; e += kThreads) {
    const int r = e / DV, b = e % DV;
    float inter = 0.f, intra = 0.f;
    for (int a = 0; a < DK; ++a) inter += sQ[r * DK + a] * h[(size_t)a * DV + b];
    for (int s = 0; s <= r; ++s) intra += sP[r * kLd + s] * Vn[s * DV + b];
    o[((size_t)(t0 + r) * Hv + j) * DV + b] = from_f32<IT>(d.scale * (__expf(sg[r]) * inter + intra));
  }
}

// ---------------------------------------------------------------------------------
// backward: Vn = U - W h from the saved chunk-start states (chunk-parallel)
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) simt_vn_kernel(Dims d, const void* __restrict__ h_saved,
                                                           Workspace ws) {
  const int c = blockIdx.x, j = blockIdx.y;
  const int4 ci = idx_chunk(d, ws, c);
  const int len = ci.z;
  if (len <= 0) return;
  const int DK = d.DK, DV = d.DV;
  const size_t ch = (size_t)c * d.Hv + j;
  const HView h = h_view(h_saved, ch, d);
  const float* W = (const float*)ws.W + ch * kChunk * DK;
  const float* U = (const float*)ws.U + ch * kChunk * DV;
  float* Vn = (float*)ws.Vn + ch * kChunk * DV;
  for (int e = threadIdx.x; e < kChunk * DV; e += kThreads) {
    const int r = e / DV, b = e % DV;
    float acc = 0.f;
    if (r < len) {
      acc = U[e];
      for (int a = 0; a < DK; ++a) acc -= W[r * DK + a] * h[(size_t)a * DV + b];
    }
    Vn[e] = acc;
  }
}

// ---------------------------------------------------------------------------------
// backward state-gradient walk (reverse over chunks), one CTA per (seq, v-head, DV slice)
//   dVn = scale P^T dO + diag(e^{gamma_C - gamma}) K dh'
//   dh  = e^{gamma_C} dh' + scale (diag(e^gamma) Q)^T dO - W^T dVn
// dh' (the gradient at the chunk end) of every chunk goes to ws.dhp.
// ---------------------------------------------------------------------------------
template <typename IT>
__global__ void __launch_bounds__(kThreads) simt_walk_kernel(Dims d, const IT* __restrict__ q,
                                                             const IT* __restrict__ k,
                                                             const IT* __restrict__ dO,
                                                             const float* __restrict__ dS_T,
                                                             float* __restrict__ dS0, Workspace ws,
                                                             int dvs) {
  extern __shared__ float sm[];
  const int n = idx_seq(d, ws, blockIdx.x), j = blockIdx.y, i = j / d.G;
  const int dv0 = blockIdx.z * dvs;
  const int DK = d.DK, DV = d.DV, Hv = d.Hv, Hk = d.Hk;
  float* sdh = sm;                   // [DK][dvs]
  float* sdVn = sdh + DK * dvs;      // [64][dvs]
  float* sP = sdVn + kChunk * dvs;   // [64][65]
  float* sg = sP + kChunk * kLd;     // [64]
  // the chunk's q, k (rows of DK + 1 floats) and dO slice (dvs + 1), staged as fp32
  const int LK = DK + 1, LD = dvs + 1;
  float* sq = sg + kChunk;
  float* sk = sq + kChunk * LK;
  float* sdo = sk + kChunk * LK;
  const int tid = threadIdx.x;
  for (int e = tid; e < DK * dvs; e += kThreads) {
    const int a = e / dvs, b = e % dvs;
    sdh[e] = dS_T ? dS_T[((size_t)n * Hv + j) * DK * DV + state_idx(d.layout, a, dv0 + b, DK, DV)] : 0.f;
  }
  __syncthreads();
  const int c_begin = idx_seq_off(d, ws, n), c_end = idx_seq_off(d, ws, n + 1);
  for (int c = c_end - 1; c >= c_begin; --c) {
    const int4 ci = idx_chunk(d, ws, c);
    const int len = ci.z, t0 = ci.y;
    const size_t ch = (size_t)c * Hv + j;
    for (int e = tid; e < DK * dvs; e += kThreads) {
      const int a = e / dvs, b = e % dvs;
      ((float*)ws.dhp)[ch * DK * DV + (size_t)a * DV + dv0 + b] = sdh[e];
    }
    for (int r = tid; r < kChunk; r += kThreads) sg[r] = ws.gam[ch * kChunk + r];
    for (int e = tid; e < kChunk * DK; e += kThreads) {
      const int r = e / DK, x = e % DK;
      const bool in = r < len;
      sq[r * LK + x] = in ? ldf(q + ((size_t)(t0 + r) * Hk + i) * DK + x) : 0.f;
      sk[r * LK + x] = in ? ldf(k + ((size_t)(t0 + r) * Hk + i) * DK + x) : 0.f;
    }
    for (int e = tid; e < kChunk * dvs; e += kThreads) {
      const int r = e / dvs, b = e % dvs;
      sdo[r * LD + b] = r < len ? ldf(dO + ((size_t)(t0 + r) * Hv + j) * DV + dv0 + b) : 0.f;
    }
    __syncthreads();
    for (int e = tid; e < kChunk * kChunk; e += kThreads) {
      const int r = e / kChunk, s = e % kChunk;
      float p = 0.f;
      if (s <= r && r < len) {
        float dot = 0.f;
        for (int x = 0; x < DK; ++x) dot += sq[r * LK + x] * sk[s * LK + x];
        p = dot * __expf(sg[r] - sg[s]);
      }
      sP[r * kLd + s] = p;
    }
    __syncthreads();
    const float gC = sg[len - 1];
    for (int e = tid; e < kChunk * dvs; e += kThreads) {
      const int s = e / dvs, b = e % dvs;
      float acc = 0.f;
      if (s < len) {
        float a1 = 0.f, a2 = 0.f;
        for (int r = s; r < len; ++r) a1 += sP[r * kLd + s] * sdo[r * LD + b];
        for (int a = 0; a < DK; ++a) a2 += sk[s * LK + a] * sdh[a * dvs + b];
        acc = d.scale * a1 + __expf(gC - sg[s]) * a2;
      }
      sdVn[e] = acc;
    }
    __syncthreads();
    const float* W = (const float*)ws.W + ch * kChunk * DK;
    const float eC = __expf(gC);
    for (int e = tid; e < DK * dvs; e += kThreads) {
      const int a = e / dvs, b = e % dvs;
      float a1 = 0.f, a2 = 0.f;
      for (int r = 0; r < len; ++r) {
        a1 += __expf(sg[r]) * sq[r * LK + a] * sdo[r * LD + b];
        a2 += W[r * DK + a] * sdVn[r * dvs + b];
      }
      sdh[e] = eC * sdh[e] + d.scale * a1 - a2;
    }
    __syncthreads();
  }
  if (dS0) {
    for (int e = tid; e < DK * dvs; e += kThreads) {
      const int a = e / dvs, b = e % dvs;
      dS0[((size_t)n * Hv + j) * DK * DV + state_idx(d.layout, a, dv0 + b, DK, DV)] = sdh[e];
    }
  }
}

// ---------------------------------------------------------------------------------
// backward gradients of one chunk (chunk-parallel)
// ---------------------------------------------------------------------------------
// kS (DK, DV <= 64): the chunk's q, k, v, dO and Vn are staged in shared memory as fp32 rows
// padded by one float (conflict-free column walks), so the dot-product loops below read shared
// memory instead of making dependent global round trips.
template <typename IT, bool kS>
__global__ void __launch_bounds__(kThreads) simt_grad_kernel(Dims d, const IT* __restrict__ q,
                                                             const IT* __restrict__ k,
                                                             const IT* __restrict__ v,
                                                             const IT* __restrict__ beta,
                                                             const void* __restrict__ h_saved,
                                                             const IT* __restrict__ dO,
                                                             IT* __restrict__ dq, IT* __restrict__ dk,
                                                             IT* __restrict__ dv, float* __restrict__ dg,
                                                             IT* __restrict__ dbeta, Workspace ws) {
  extern __shared__ float sm[];
  const int c = blockIdx.x, j = blockIdx.y, i = j / d.G;
  const int4 ci = idx_chunk(d, ws, c);
  const int len = ci.z, t0 = ci.y;
  if (len <= 0) return;
  const int DK = d.DK, DV = d.DV, Hv = d.Hv, Hk = d.Hk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int M2 = kChunk * kLd;
  float* sQK = sm;          // q_r . k_s
  float* sKK = sQK + M2;    // k_r . k_s
  float* sdP = sKK + M2;    // scale (dO Vn^T) * Gam, lower incl. diagonal
  float* sT = sdP + M2;     // T
  float* sdT = sT + M2;     // dT, then dA
  float* sX = sdT + M2;     // T^T dT
  float* sdVn = sX + M2;    // [64][DV]
  float* sdW = sdVn + kChunk * DV;  // [64][DK]
  float* sg = sdW + kChunk * DK;    // gamma
  float* sb = sg + kChunk;          // beta
  float* sdgam = sb + kChunk;       // d gamma
  float* skdv = sdgam + kChunk;     // k_r^T dh' vn_r
  float* sred = skdv + kChunk;      // [32] block reduction scratch
  const size_t ch = (size_t)c * Hv + j;
  const HView h = h_view(h_saved, ch, d);
  const float* dhp = (const float*)ws.dhp + ch * DK * DV;
  const float* Vn = (const float*)ws.Vn + ch * kChunk * DV;
  const float* Tg = ws.Tm + ch * kChunk * kChunk;
  const int LK = DK + 1, LV = DV + 1;  // kS: staged row strides
  float* sQs = sred + 32;
  float* sKs = sQs + kChunk * LK;
  float* sVs = sKs + kChunk * LK;
  float* sDOs = sVs + kChunk * LV;
  float* sVns = sDOs + kChunk * LV;
  if (kS) {  // rows past the chunk end: zero (every use below is masked to r, s < len anyway)
    for (int e = tid; e < kChunk * DK; e += kThreads) {
      const int r = e / DK, x = e % DK;
      const bool in = r < len;
      sQs[r * LK + x] = in ? ldf(q + ((size_t)(t0 + r) * Hk + i) * DK + x) : 0.f;
      sKs[r * LK + x] = in ? ldf(k + ((size_t)(t0 + r) * Hk + i) * DK + x) : 0.f;
    }
    for (int e = tid; e < kChunk * DV; e += kThreads) {
      const int r = e / DV, x = e % DV;
      const bool in = r < len;
      sVs[r * LV + x] = in ? ldf(v + ((size_t)(t0 + r) * Hv + j) * DV + x) : 0.f;
      sDOs[r * LV + x] = in ? ldf(dO + ((size_t)(t0 + r) * Hv + j) * DV + x) : 0.f;
      sVns[r * LV + x] = Vn[e];
    }
    __syncthreads();
  }
  auto Q = [&](int r, int x) { return kS ? sQs[r * LK + x] : ldf(q + ((size_t)(t0 + r) * Hk + i) * DK + x); };
  auto K = [&](int r, int x) { return kS ? sKs[r * LK + x] : ldf(k + ((size_t)(t0 + r) * Hk + i) * DK + x); };
  auto V = [&](int r, int x) { return kS ? sVs[r * LV + x] : ldf(v + ((size_t)(t0 + r) * Hv + j) * DV + x); };
  auto DO = [&](int r, int x) { return kS ? sDOs[r * LV + x] : ldf(dO + ((size_t)(t0 + r) * Hv + j) * DV + x); };
  auto VN = [&](int r, int x) { return kS ? sVns[r * LV + x] : Vn[r * DV + x]; };

  for (int r = tid; r < kChunk; r += kThreads) {
    sg[r] = ws.gam[ch * kChunk + r];
    sb[r] = r < len ? ldf(beta + (size_t)(t0 + r) * Hv + j) : 0.f;
  }
  for (int e = tid; e < kChunk * kChunk; e += kThreads) {
    const int r = e / kChunk, s = e % kChunk;
    sT[r * kLd + s] = Tg[e];
    float qk = 0.f, kk = 0.f;
    if (r < len && s < len) {
      for (int x = 0; x < DK; ++x) {
        const float ks = K(s, x);
        qk += Q(r, x) * ks;
        kk += K(r, x) * ks;
      }
    }
    sQK[r * kLd + s] = qk;
    sKK[r * kLd + s] = kk;
  }
  __syncthreads();
  const float gC = sg[len - 1];
  auto Gam = [&](int r, int s) { return (s <= r) ? __expf(sg[r] - sg[s]) : 0.f; };
  // dVn = scale P^T dO + diag(e^{gamma_C - gamma}) K dh';  dP;  dW = -dVn h^T (after sync)
  for (int e = tid; e < kChunk * DV; e += kThreads) {
    const int s = e / DV, b = e % DV;
    float acc = 0.f;
    if (s < len) {
      float a1 = 0.f, a2 = 0.f;
      for (int r = s; r < len; ++r) a1 += sQK[r * kLd + s] * Gam(r, s) * DO(r, b);
      for (int a = 0; a < DK; ++a) a2 += K(s, a) * dhp[(size_t)a * DV + b];
      acc = d.scale * a1 + __expf(gC - sg[s]) * a2;
    }
    sdVn[e] = acc;
  }
  for (int e = tid; e < kChunk * kChunk; e += kThreads) {
    const int r = e / kChunk, s = e % kChunk;
    float p = 0.f;
    if (s <= r && r < len) {
      float dot = 0.f;
      for (int b = 0; b < DV; ++b) dot += DO(r, b) * VN(s, b);
      p = d.scale * dot * Gam(r, s);
    }
    sdP[r * kLd + s] = p;
  }
  __syncthreads();
  for (int e = tid; e < kChunk * DK; e += kThreads) {
    const int r = e / DK, a = e % DK;
    float acc = 0.f;
    for (int b = 0; b < DV; ++b) acc += sdVn[r * DV + b] * h[(size_t)a * DV + b];
    sdW[e] = -acc;
  }
  __syncthreads();
  // dT = dW B_k^T + dVn B_v^T,  B_k = diag(beta e^gamma) K,  B_v = diag(beta) V
  for (int e = tid; e < kChunk * kChunk; e += kThreads) {
    const int r = e / kChunk, s = e % kChunk;
    float acc = 0.f;
    if (r < len && s < len) {
      float a1 = 0.f, a2 = 0.f;
      for (int a = 0; a < DK; ++a) a1 += sdW[r * DK + a] * K(s, a);
      for (int b = 0; b < DV; ++b) a2 += sdVn[r * DV + b] * V(s, b);
      acc = sb[s] * (__expf(sg[s]) * a1 + a2);
    }
    sdT[r * kLd + s] = acc;
  }
  __syncthreads();
  for (int e = tid; e < kChunk * kChunk; e += kThreads) {  // X = T^T dT
    const int r = e / kChunk, s = e % kChunk;
    float acc = 0.f;
    for (int m = r; m < kChunk; ++m) acc += sT[m * kLd + r] * sdT[m * kLd + s];
    sX[r * kLd + s] = acc;
  }
  __syncthreads();
  for (int e = tid; e < kChunk * kChunk; e += kThreads) {  // dA = -strict-lower(X T^T)
    const int r = e / kChunk, s = e % kChunk;
    float acc = 0.f;
    if (s < r) {
      for (int m = 0; m <= s; ++m) acc += sX[r * kLd + m] * sT[s * kLd + m];
      acc = -acc;
    }
    sdT[r * kLd + s] = acc;
  }
  // <dh', h> for the chunk-end gate term
  float part = 0.f;
  for (int e = tid; e < DK * DV; e += kThreads) part += dhp[e] * h[e];
  part = warp_sum(part);
  if (lane == 0) sred[warp] = part;
  __syncthreads();
  // per-row gradients: one warp per row
  for (int r = warp; r < len; r += kThreads / 32) {
    const float br = sb[r], egr = __expf(sg[r]), decr = __expf(gC - sg[r]);
    float dot_bk = 0.f, dot_bv = 0.f, dot_qh = 0.f, kdv = 0.f;
    for (int b = lane; b < DV; b += 32) {
      float dBv = 0.f;
      for (int s = r; s < len; ++s) dBv += sT[s * kLd + r] * sdVn[s * DV + b];
      const float dvv = br * dBv;
      dv[((size_t)(t0 + r) * Hv + j) * DV + b] = from_f32<IT>(dvv);
      dot_bv += dBv * V(r, b);
      float qh = 0.f;
      for (int a = 0; a < DK; ++a) qh += Q(r, a) * h[(size_t)a * DV + b];
      dot_qh += DO(r, b) * qh;
      float kd = 0.f;
      for (int a = 0; a < DK; ++a) kd += K(r, a) * dhp[(size_t)a * DV + b];
      kdv += kd * VN(r, b);
    }
    for (int a = lane; a < DK; a += 32) {
      float dBk = 0.f;
      for (int s = r; s < len; ++s) dBk += sT[s * kLd + r] * sdW[s * DK + a];
      float dqa = 0.f;
      for (int b = 0; b < DV; ++b) dqa += DO(r, b) * h[(size_t)a * DV + b];
      dqa *= d.scale * egr;
      for (int s = 0; s <= r; ++s) dqa += sdP[r * kLd + s] * K(s, a);
      float dka = 0.f;
      for (int s = r; s < len; ++s) dka += sdP[s * kLd + r] * Q(s, a);
      float vd = 0.f;
      for (int b = 0; b < DV; ++b) vd += VN(r, b) * dhp[(size_t)a * DV + b];
      dka += decr * vd + br * egr * dBk;
      float a1 = 0.f, a2 = 0.f;
      for (int s = 0; s < r; ++s) a1 += sdT[r * kLd + s] * Gam(r, s) * K(s, a);
      for (int s = r + 1; s < len; ++s) a2 += sdT[s * kLd + r] * Gam(s, r) * sb[s] * K(s, a);
      dka += br * a1 + a2;
      dot_bk += dBk * K(r, a);
      if (d.G == 1) {
        dq[((size_t)(t0 + r) * Hk + i) * DK + a] = from_f32<IT>(dqa);
        dk[((size_t)(t0 + r) * Hk + i) * DK + a] = from_f32<IT>(dka);
      } else {
        ws.dq_part[((size_t)(t0 + r) * Hv + j) * DK + a] = dqa;
        ws.dk_part[((size_t)(t0 + r) * Hv + j) * DK + a] = dka;
      }
    }
    dot_bk = warp_sum(dot_bk);
    dot_bv = warp_sum(dot_bv);
    dot_qh = warp_sum(dot_qh);
    kdv = warp_sum(kdv);
    // row/column sums of dA * A and dP * (Q K^T) over the 64 x 64 matrices
    float aa = 0.f, pp = 0.f;
    for (int s = lane; s < len; s += 32) {
      if (s < r) aa += sdT[r * kLd + s] * br * Gam(r, s) * sKK[r * kLd + s];
      if (s > r) aa -= sdT[s * kLd + r] * sb[s] * Gam(s, r) * sKK[s * kLd + r];
      if (s <= r) pp += sdP[r * kLd + s] * sQK[r * kLd + s];
      if (s >= r) pp -= sdP[s * kLd + r] * sQK[s * kLd + r];
    }
    float akk = 0.f;
    for (int s = lane; s < r; s += 32) akk += sdT[r * kLd + s] * Gam(r, s) * sKK[r * kLd + s];
    aa = warp_sum(aa);
    pp = warp_sum(pp);
    akk = warp_sum(akk);
    if (lane == 0) {
      dbeta[(size_t)(t0 + r) * Hv + j] = from_f32<IT>(egr * dot_bk + dot_bv + akk);
      sdgam[r] = br * egr * dot_bk + aa + pp + d.scale * egr * dot_qh - decr * kdv;
      skdv[r] = kdv;
    }
  }
  __syncthreads();
  if (tid == 0) {
    float hdh = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) hdh += sred[w];
    float extra = __expf(gC) * hdh;
    for (int s = 0; s < len; ++s) extra += __expf(gC - sg[s]) * skdv[s];
    sdgam[len - 1] += extra;
    float run = 0.f;
    for (int r = len - 1; r >= 0; --r) {
      run += sdgam[r];
      dg[(size_t)(t0 + r) * Hv + j] = run;
    }
  }
}

// dq/dk of q/k head i = sum over its G v-heads (fixed order: deterministic)
template <typename IT>
__global__ void __launch_bounds__(kThreads) simt_group_reduce_kernel(Dims d, IT* __restrict__ dq,
                                                                     IT* __restrict__ dk, Workspace ws) {
  const size_t total = (size_t)d.T_total * d.Hk * d.DK;
  for (size_t e = (size_t)blockIdx.x * kThreads + threadIdx.x; e < total; e += (size_t)gridDim.x * kThreads) {
    const int a = (int)(e % d.DK);
    const size_t ti = e / d.DK;
    const int i = (int)(ti % d.Hk);
    const size_t t = ti / d.Hk;
    float sq = 0.f, sk = 0.f;
    for (int jj = 0; jj < d.G; ++jj) {
      const size_t src = (t * d.Hv + (size_t)i * d.G + jj) * d.DK + a;
      sq += ws.dq_part[src];
      sk += ws.dk_part[src];
    }
    dq[e] = from_f32<IT>(sq);
    dk[e] = from_f32<IT>(sk);
  }
}

}  // namespace

cudaError_t launch_group_reduce(const Dims& d, void* dq, void* dk, const Workspace& ws, cudaStream_t s) {
  if (d.dtype == GDR_DTYPE_F32)
    simt_group_reduce_kernel<float><<<1024, kThreads, 0, s>>>(d, (float*)dq, (float*)dk, ws);
  else
    simt_group_reduce_kernel<__nv_bfloat16><<<1024, kThreads, 0, s>>>(d, (__nv_bfloat16*)dq, (__nv_bfloat16*)dk, ws);
  stage_mark(s, "bwd_group_reduce");
  return cudaGetLastError();
}

namespace {

inline int dv_slice(const Dims& d) { return d.DV % 32 == 0 ? 32 : 16; }

template <typename IT>
cudaError_t simt_forward_t(const Dims& d, const FwdArgs& a, const Workspace& ws, cudaStream_t s) {
  if (d.max_chunks > 0) {
    const dim3 gc(d.max_chunks, d.Hv);
    size_t smp = sizeof(float) * (kChunk * d.DK + kChunk * d.DV + 2 * kChunk * kLd + 2 * kChunk);
    set_smem_once((const void*)simt_prep_kernel<IT>, smp);
    simt_prep_kernel<IT><<<gc, kThreads, smp, s>>>(d, (const IT*)a.k, (const IT*)a.v, a.g,
                                                   (const IT*)a.beta, ws);
    stage_mark(s, "fwd_prep");
  }
  if (d.num_seqs > 0) {
    const int dvs = dv_slice(d);
    const dim3 gs(d.num_seqs, d.Hv, d.DV / dvs);
    size_t sms = sizeof(float) * (d.DK * dvs + kChunk * dvs + 2 * kChunk);
    set_smem_once((const void*)simt_state_kernel<IT>, sms);
    simt_state_kernel<IT><<<gs, kThreads, sms, s>>>(d, (const IT*)a.k, a.S0, a.S_T, a.h_saved, ws, dvs);
    stage_mark(s, "fwd_state");
  }
  if (d.max_chunks > 0) {
    const dim3 gc(d.max_chunks, d.Hv);
    size_t smo = sizeof(float) * (2 * kChunk * d.DK + kChunk * kLd + kChunk);
    set_smem_once((const void*)simt_out_kernel<IT>, smo);
    simt_out_kernel<IT><<<gc, kThreads, smo, s>>>(d, (const IT*)a.q, (const IT*)a.k, a.h_saved, (IT*)a.o, ws);
    stage_mark(s, "fwd_out");
  }
  return cudaGetLastError();
}

template <typename IT>
cudaError_t simt_backward_t(const Dims& d, const BwdArgs& a, const Workspace& ws, cudaStream_t s) {
  if (d.max_chunks > 0) {
    const dim3 gc(d.max_chunks, d.Hv);
    size_t smp = sizeof(float) * (kChunk * d.DK + kChunk * d.DV + 2 * kChunk * kLd + 2 * kChunk);
    set_smem_once((const void*)simt_prep_kernel<IT>, smp);
    simt_prep_kernel<IT><<<gc, kThreads, smp, s>>>(d, (const IT*)a.k, (const IT*)a.v, a.g,
                                                   (const IT*)a.beta, ws);
    stage_mark(s, "bwd_prep");
    simt_vn_kernel<<<gc, kThreads, 0, s>>>(d, a.h_saved, ws);
    stage_mark(s, "bwd_vn");
  }
  if (d.num_seqs > 0) {
    const int dvs = dv_slice(d);
    const dim3 gs(d.num_seqs, d.Hv, d.DV / dvs);
    size_t smw = sizeof(float) * (d.DK * dvs + kChunk * dvs + kChunk * kLd + kChunk + kChunk * (2 * (d.DK + 1) + dvs + 1));
    set_smem_once((const void*)simt_walk_kernel<IT>, smw);
    simt_walk_kernel<IT><<<gs, kThreads, smw, s>>>(d, (const IT*)a.q, (const IT*)a.k, (const IT*)a.dO,
                                                   a.dS_T, a.dS0, ws, dvs);
    stage_mark(s, "bwd_walk");
  }
  if (d.max_chunks > 0) {
    const dim3 gc(d.max_chunks, d.Hv);
    const bool stage = d.DK <= 64 && d.DV <= 64;
    size_t smg = sizeof(float) * (6 * kChunk * kLd + kChunk * d.DV + kChunk * d.DK + 4 * kChunk + 32);
    if (stage) smg += sizeof(float) * kChunk * (2 * (d.DK + 1) + 3 * (d.DV + 1));
    auto grad = stage ? simt_grad_kernel<IT, true> : simt_grad_kernel<IT, false>;
    set_smem_once((const void*)grad, smg);
    grad<<<gc, kThreads, smg, s>>>(d, (const IT*)a.q, (const IT*)a.k, (const IT*)a.v,
                                                   (const IT*)a.beta, a.h_saved, (const IT*)a.dO,
                                                   (IT*)a.dq, (IT*)a.dk, (IT*)a.dv, a.dg, (IT*)a.dbeta, ws);
    stage_mark(s, "bwd_grad");
  }
  if (d.G > 1 && d.T_total > 0) {
    simt_group_reduce_kernel<IT><<<1024, kThreads, 0, s>>>(d, (IT*)a.dq, (IT*)a.dk, ws);
    stage_mark(s, "bwd_group_reduce");
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t simt_forward(const Dims& d, const FwdArgs& a, const Workspace& ws, cudaStream_t s) {
  if (simt_small(d)) return simt_small_forward(d, a, ws, s);
  return d.dtype == GDR_DTYPE_F32 ? simt_forward_t<float>(d, a, ws, s)
                                  : simt_forward_t<__nv_bfloat16>(d, a, ws, s);
}

cudaError_t simt_backward(const Dims& d, const BwdArgs& a, const Workspace& ws, cudaStream_t s) {
  if (simt_small(d)) return simt_small_backward(d, a, ws, s);
  return d.dtype == GDR_DTYPE_F32 ? simt_backward_t<float>(d, a, ws, s)
                                  : simt_backward_t<__nv_bfloat16>(d, a, ws, s);
}

}  // namespace gdr
