// gdr_chunks.cuh -- the chunk index as the kernels read it.
//
// Chunks restart at every sequence start (64 tokens each, the last one ragged).  For a
// variable-length batch the index kernel (gdr_index.cu) builds the tables from cu_seqlens:
// chunk records, per-sequence chunk offsets, the longest-first order and the step tables of
// the fused kernels.  A fixed-length batch (B sequences of T tokens) needs no tables: every
// sequence has nc = ceil(T / 64) chunks, so
//   chunk c           = {n = c / nc, first token n T + 64 (c % nc), length min(64, T - 64 (c % nc)), c % nc}
//   offset of seq n   = n nc;  longest-first order = identity (equal lengths keep index order)
//   walk / forward steps: S = nc, every sequence takes part in every step, so step_off[s] = s B,
//   and queue position q is step s = q / B of sequence n = q % B: reverse (gradient) chunk
//   (n + 1) nc - 1 - s, forward chunk n nc + s.
// These accessors give the same numbers either way, so the index kernel runs only for
// variable-length batches.
#pragma once

#include "gdr_internal.h"

namespace gdr {

__device__ __forceinline__ int idx_nc(const Dims& d) { return (d.T + kChunk - 1) / kChunk; }

// {sequence, first packed token, length (0: an empty slot), chunk index within the sequence}
__device__ __forceinline__ int4 idx_chunk(const Dims& d, const Workspace& ws, int c) {
  if (d.cu != nullptr) return ws.chunks[c];
  const int nc = idx_nc(d), n = c / nc, local = c - n * nc;
  return make_int4(n, n * d.T + local * kChunk, min(kChunk, d.T - local * kChunk), local);
}

// sequence of rank r in the longest-first order
__device__ __forceinline__ int idx_seq(const Dims& d, const Workspace& ws, int r) {
  return d.cu != nullptr ? ws.seq_order[r] : r;
}

// first global chunk of sequence n (n = num_seqs: the total)
__device__ __forceinline__ int idx_seq_off(const Dims& d, const Workspace& ws, int n) {
  return d.cu != nullptr ? ws.seq_chunk_off[n] : n * idx_nc(d);
}

// fused kernels: number of steps S, step offsets, chunk of a queue position
__device__ __forceinline__ int idx_n_steps(const Dims& d, const Workspace& ws) {
  return d.cu != nullptr ? ws.step_off[d.max_chunks + 1] : idx_nc(d);
}
__device__ __forceinline__ int idx_step_off(const Dims& d, const Workspace& ws, int s) {
  return d.cu != nullptr ? ws.step_off[s] : s * d.num_seqs;
}
__device__ __forceinline__ int idx_grad_chunk(const Dims& d, const Workspace& ws, int q) {
  if (d.cu != nullptr) return ws.grad_chunk[q];
  const int s = q / d.num_seqs, n = q - s * d.num_seqs;
  return (n + 1) * idx_nc(d) - 1 - s;
}
__device__ __forceinline__ int idx_fwd_chunk(const Dims& d, const Workspace& ws, int q) {
  if (d.cu != nullptr) return ws.fwd_chunk[q];
  const int s = q / d.num_seqs, n = q - s * d.num_seqs;
  return n * idx_nc(d) + s;
}

// Context-parallel segments: the chunks [c0, c1) of one sequence cut into
// nseg = max(1, min(P, c1 - c0)) segments whose chunk counts differ by at most one (the first
// (c1 - c0) mod nseg one longer).  Returns {first chunk, end chunk, nseg} of segment s; a segment
// s >= nseg is empty.
__host__ __device__ __forceinline__ int3 cp_segment(int c0, int c1, int P, int s) {
  const int nc = c1 - c0;
  const int nseg = max(1, min(P, nc));
  if (s >= nseg) return make_int3(c1, c1, nseg);
  const int base = nc / nseg, extra = nc - base * nseg;
  const int lo = c0 + s * base + min(s, extra);
  return make_int3(lo, lo + base + (s < extra ? 1 : 0), nseg);
}

// The fused backward with context-parallel segments (fixed length, cp_bwd > 1; a separate
// instantiation of the kernel, so the plain one carries none of this): queue position q in the
// order the chunks' state gradients become available.  First every chunk of each
// sequence's last segment (walked by the first pass, before the fused kernel), walk order; then
// step t of the second pass's walks: chunk end(s) - 1 - t of segments s = 0 .. nseg - 2 of every
// sequence (sequence fastest), the longer segments (s < extra) taking one step more.
__device__ __forceinline__ int idx_cp_grad_chunk(const Dims& d, int q) {
  const int nc = idx_nc(d), B = d.num_seqs;
  const int nseg = max(1, min(d.cp_bwd, nc)), base = nc / nseg, extra = nc - base * nseg;
  const int last_len = nseg == 1 ? nc : base;  // the last segment is never one of the longer ones
  if (q < B * last_len) {
    const int t = q / B, n = q - t * B;
    return (n + 1) * nc - 1 - t;
  }
  q -= B * last_len;
  const int K = B * (nseg - 1);  // chunks per step while every earlier segment has one
  const int t = q < base * K ? q / K : base;
  const int r = q - t * K;
  const int n = r % B, s = r / B;
  return n * nc + (s + 1) * base + min(s + 1, extra) - 1 - t;
}

}  // namespace gdr
