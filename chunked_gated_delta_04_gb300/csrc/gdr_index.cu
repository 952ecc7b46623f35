// gdr_index.cu -- K0: the chunk index of a (possibly variable-length) batch.
//
// Chunks restart at every sequence start (chunked gated delta rule, FlashQLA PR
// #34, "Current status": fixed-length and variable-length inputs).  For sequence n
// of length L_n the index holds chunk_offset[n] = sum_{n'<n} ceil(L_n'/64) and, per
// global chunk c, {seq, first packed token, length (1..64), chunk index within the
// sequence}.  Slots past the last real chunk get length 0 (no work).  The order
// of sequences for the sequential kernels is longest first.  Everything is
// computed on the device from cu_seqlens, so the host never reads tensor data.
#include "gdr_device.cuh"
#include "gdr_internal.h"

namespace gdr {

constexpr int kIndexThreads = 1024;
constexpr int kMaxOrderedSeqs = kMaxFusedSeqs;  // above this the order is the identity
// Offsets, order and step table up to this size are also kept in shared memory, so the binary
// searches below read them there instead of making dependent global round trips.
constexpr int kSmemCap = 2048;

__global__ void __launch_bounds__(kIndexThreads) gdr_index_kernel(const int32_t* __restrict__ cu,
                                                                  int num_seqs, int T, int max_chunks,
                                                                  int4* __restrict__ chunks,
                                                                  int* __restrict__ off,
                                                                  int* __restrict__ order,
                                                                  uint32_t* __restrict__ status,
                                                                  int* __restrict__ step_off,
                                                                  int* __restrict__ grad_chunk,
                                                                  int* __restrict__ fwd_chunk) {
  __shared__ int warp_tot[32];
  __shared__ int s_bad;
  __shared__ int s_carry;
  __shared__ int s_off[kSmemCap + 1], s_order[kSmemCap], s_step[kSmemCap + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool small_n = num_seqs + 1 <= kSmemCap;  // off and order mirrored in shared memory
  auto OFF = [&](int n) { return small_n ? s_off[n] : off[n]; };
  auto ORD = [&](int r) { return small_n ? s_order[r] : order[r]; };
  if (tid == 0) {
    for (int w = 0; w < 64; ++w) status[w] = 0u;  // fresh status for this call
    s_bad = 0;
    s_carry = 0;
  }
  __syncthreads();
  // validate cu_seqlens: cu[0] == 0, non-decreasing, cu[num_seqs] == T
  if (cu != nullptr) {
    for (int n = tid; n < num_seqs; n += kIndexThreads) {
      const int a = cu[n], b = cu[n + 1];
      if (b < a || a < 0 || b > T) s_bad = 1;
    }
    if (tid == 0 && (cu[0] != 0 || cu[num_seqs] != T)) s_bad = 1;
  }
  __syncthreads();
  const bool bad = s_bad != 0;
  if (bad && tid == 0) status[0] |= kDevErrBadCuSeqlens;

  // exclusive scan of ceil(L/64) over sequences, in tiles of kIndexThreads
  for (int base = 0; base < num_seqs; base += kIndexThreads) {
    const int n = base + tid;
    int nc = 0;
    if (n < num_seqs && !bad) {
      const int L = cu ? cu[n + 1] - cu[n] : T;
      nc = (L + kChunk - 1) / kChunk;
    }
    int x = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int t = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      warp_tot[lane] = t;  // inclusive prefix over warps
    }
    __syncthreads();
    const int carry = s_carry;
    const int incl = x + (warp > 0 ? warp_tot[warp - 1] : 0);
    if (n < num_seqs) {
      off[n] = carry + incl - nc;
      if (small_n) s_off[n] = carry + incl - nc;
    }
    __syncthreads();
    if (tid == kIndexThreads - 1) s_carry = carry + incl;
    __syncthreads();
  }
  int total = s_carry;
  if (total > max_chunks) {  // only reachable with an inconsistent cu_seqlens
    if (tid == 0) status[0] |= kDevErrBadCuSeqlens;
    total = 0;
  }
  if (tid == 0) {
    off[num_seqs] = total;
    if (small_n) s_off[num_seqs] = total;
  }
  __syncthreads();

  for (int c = tid; c < max_chunks; c += kIndexThreads) {
    int4 ci = make_int4(-1, 0, 0, 0);
    if (c < total) {
      int lo = 0, hi = num_seqs - 1;  // last n with off[n] <= c
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (OFF(mid) <= c) lo = mid; else hi = mid - 1;
      }
      const int n = lo;
      const int start = cu ? cu[n] : n * T;
      const int L = cu ? cu[n + 1] - cu[n] : T;
      const int local = c - OFF(n);
      const int len = min(kChunk, L - local * kChunk);
      ci = make_int4(n, start + local * kChunk, len, local);
    }
    chunks[c] = ci;
  }

  // longest-first order (stable: ties keep index order)
  if (num_seqs <= kMaxOrderedSeqs && !bad) {
    for (int n = tid; n < num_seqs; n += kIndexThreads) {
      const int Ln = cu ? cu[n + 1] - cu[n] : T;
      int rank = 0;
      for (int m = 0; m < num_seqs; ++m) {
        const int Lm = cu ? cu[m + 1] - cu[m] : T;
        rank += (Lm > Ln) || (Lm == Ln && m < n);
      }
      order[rank] = n;
      if (small_n) s_order[rank] = n;
    }
  } else {
    for (int n = tid; n < num_seqs; n += kIndexThreads) {
      order[n] = n;
      if (small_n) s_order[n] = n;
    }
  }

  // Step table of the fused kernels (step_off != nullptr; requires the sorted order), in the
  // backward's terms (the forward's step s is local chunk s of the same sequences):
  // at reverse step s the walk finishes local chunk nc(n) - 1 - s of every sequence with
  // nc(n) > s, i.e. of the first cnt(s) sequences in longest-first order.  step_off[s] =
  // sum_{s' < s} cnt(s') for s = 0..S (S = the longest sequence's chunk count), and
  // step_off[max_chunks + 1] = S.  Gradient item q * Hv + j with step_off[s] <= q <
  // step_off[s + 1] is v-head j of sequence order[q - step_off[s]] at step s, whose chunk
  // grad_chunk[q] lists.
  if (step_off != nullptr && bad) {  // nothing is computed: no walk steps, no gradient items
    if (tid == 0) step_off[0] = step_off[max_chunks + 1] = 0;
  } else if (step_off != nullptr) {
    __syncthreads();
    auto nc_of_rank = [&](int r) { return OFF(ORD(r) + 1) - OFF(ORD(r)); };
    const int S = num_seqs > 0 ? nc_of_rank(0) : 0;
    const bool small_s = S + 1 <= kSmemCap;  // step table mirrored in shared memory
    auto STEP = [&](int st) { return small_s ? s_step[st] : step_off[st]; };
    for (int st = tid; st < S; st += kIndexThreads) {  // cnt(st): first rank with nc <= st
      int lo = 0, hi = num_seqs;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (nc_of_rank(mid) > st) lo = mid + 1; else hi = mid;
      }
      step_off[st + 1] = lo;
      if (small_s) s_step[st + 1] = lo;
    }
    __syncthreads();
    if (tid == 0) {
      step_off[0] = 0;
      if (small_s) s_step[0] = 0;
      step_off[max_chunks + 1] = S;
      s_carry = 0;
    }
    __syncthreads();
    for (int base = 1; base <= S; base += kIndexThreads) {  // inclusive scan of step_off[1..S]
      const int st = base + tid;
      int x = st <= S ? STEP(st) : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) warp_tot[warp] = x;
      __syncthreads();
      if (warp == 0) {
        int t = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, t, o);
          if (lane >= o) t += y;
        }
        warp_tot[lane] = t;
      }
      __syncthreads();
      const int carry = s_carry;
      const int incl = x + (warp > 0 ? warp_tot[warp - 1] : 0);
      if (st <= S) {
        step_off[st] = carry + incl;
        if (small_s) s_step[st] = carry + incl;
      }
      __syncthreads();
      if (tid == kIndexThreads - 1) s_carry = carry + incl;
      __syncthreads();
    }
    // the chunk of every queue position, so a claimed item decodes with one load: reverse
    // step s of the backward walk is local chunk nc - 1 - s, forward step s local chunk s
    const int n_q = STEP(S);
    for (int q = tid; q < n_q; q += kIndexThreads) {
      int lo = 0, hi = S - 1;  // last step s with step_off[s] <= q
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (STEP(mid) <= q) lo = mid; else hi = mid - 1;
      }
      const int n = ORD(q - STEP(lo));
      if (grad_chunk) grad_chunk[q] = OFF(n + 1) - 1 - lo;
      if (fwd_chunk) fwd_chunk[q] = OFF(n) + lo;
    }
  }
}

bool index_folded(const Dims& d) { return d.cu == nullptr && d.max_chunks > 0 && d.num_seqs > 0; }

cudaError_t launch_index(const Dims& d, const Workspace& ws, cudaStream_t s) {
  // fixed length: the kernels compute every record (gdr_chunks.cuh); only the status is reset,
  // by the first kernel on the small-head SIMT path (gdr_simt_small.cu), else here
  if (index_folded(d)) return simt_small(d) ? cudaSuccess : cudaMemsetAsync(ws.status, 0, 64 * sizeof(uint32_t), s);
  gdr_index_kernel<<<1, kIndexThreads, 0, s>>>(d.cu, d.num_seqs, d.cu ? (int)d.T_total : d.T,
                                               d.max_chunks, ws.chunks, ws.seq_chunk_off, ws.seq_order,
                                               ws.status, ws.step_off, ws.grad_chunk, ws.fwd_chunk);
  stage_mark(s, "index");
  return cudaGetLastError();
}

}  // namespace gdr
