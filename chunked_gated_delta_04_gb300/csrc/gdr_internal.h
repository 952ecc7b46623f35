// gdr_internal.h -- declarations shared by the library's translation units
// (host API, index kernel, SIMT kernels, tcgen05 kernels).  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gdr.h"

namespace gdr {

constexpr int kChunk = 64;  // chunk length of the chunked method (tokens)

// Status-word bits written by kernels (workspace header, word 0).
enum : uint32_t {
  kDevErrBadCuSeqlens = 1u << 0,  // cu_seqlens not 0..T non-decreasing: nothing computed
  kDevErrTimeoutFwd = 1u << 1,    // a bounded wait in a forward kernel ran out
  kDevErrTimeoutBwd = 1u << 2,    // a bounded wait in a backward kernel ran out
  kDevErrTimeoutPrep = 1u << 3,   // a bounded wait in the chunk-prep kernel ran out
};

// Resolved problem.
struct Dims {
  int B, T, Hk, Hv, DK, DV, G, num_seqs;
  long long T_total;  // B * T
  int max_chunks;
  float scale;
  int dtype;   // gdr_dtype
  int layout;  // gdr_state_layout
  const int32_t* cu;  // device cu_seqlens or nullptr
  int path;    // 1 = tcgen05, 0 = SIMT
  int h_bf16;  // h_saved holds bf16 (else fp32)
  int prologue;  // gdr_prologue_flags bits
  int save_wy;   // tensor-core path: gamma, W, U, P, T live in the saved buffer (see attach_saved_factors)
  int cp_fwd, cp_bwd;  // segments per sequence of the context-parallel passes (1: none; tensor-core path)
};

constexpr int kMaxCpSegments = 64;

// Context-parallel (segment-scan) passes of one direction.  Per (sequence, v-head) and segment s,
// three DK x 128 fp32 matrices: X[s] a boundary state (forward: the state at the start of segment
// s; backward: the state gradient at the end of segment s) and R[s] the segment's result from a
// zero boundary, both row-major [DK][DV]; M[s] the segment's transition (forward Phi_s, backward
// Phi_s^T), stored transposed (element [r][k] at k * 128 + r).
struct CpArgs {
  int pass;  // 0: no segments; 1: the first pass (maps); 3: the second pass (true boundaries)
  int P;     // segments per sequence
  float* X;  // [num_seqs][Hv][P][128][128]
  float* M;
  float* R;
};

// Pointers into the caller's workspace.  Every region starts 256-byte aligned.
struct Workspace {
  uint32_t* status;    // [64] words; word 0 = status bits above
  int4* chunks;        // [max_chunks] {seq, t0 (packed token index), len, local chunk index}
  int* seq_chunk_off;  // [num_seqs + 1]
  int* seq_order;      // [num_seqs] sequences, longest first
  // intermediates (fp32 on the SIMT path, bf16 on the tensor-core path)
  void* W;       // [max_chunks][Hv][64][DK]
  void* U;       // [max_chunks][Hv][64][DV]; tensor-core backward: Vn = U - W h in its place
  void* P;       // tensor-core path: [max_chunks][Hv][64][64]
  float* gam;    // [max_chunks][Hv][64] in-chunk cumsum of g
  void* Vn;      // [max_chunks][Hv][64][DV]
  float* Tm;     // SIMT backward: [max_chunks][Hv][64][64]
  void* dhp;     // backward: [max_chunks][Hv][DK][DV] state gradient at each chunk's end
                 // (fp32 on the SIMT path, bf16 on the tensor-core path)
  void* Tb;      // tensor-core backward: T = (I + A)^{-1}, bf16 [max_chunks][Hv][64][64]
  void* dVn;     // backward: dL/dVn [max_chunks][Hv][64][DV] (bf16 tensor-core path, fp32 small-head SIMT path)
  float* Pf;     // small-head SIMT path: P = Q K^T * Gam on and below the diagonal [max_chunks][Hv][64][64];
                 // the forward keeps it transposed (P^T, the state kernel's operand), the backward not
  float* Ak;     // small-head SIMT backward: K K^T * Gam below the diagonal [max_chunks][Hv][64][64]
  float* PdO;    // small-head SIMT backward: scale P^T dO [max_chunks][Hv][64][DV]
  float* QdO;    // small-head SIMT backward: (scale diag(e^gamma) Q)^T dO [max_chunks][Hv][DK][DV]
  float* dq_part;  // backward, Hv > Hk: [T_total][Hv][DK]
  float* dk_part;  // backward, Hv > Hk: [T_total][Hv][DK]
  // fused walk + gradient kernel (fixed-length tensor-core backward): per (chunk, v-head) count
  // of finished walk slices [max_chunks][Hv], and the gradient items' claim counter
  uint32_t* walk_flags;
  uint32_t* grad_queue;
  int* step_off;  // [max_chunks + 2]: the walk-step prefix table built by the index kernel
  int* grad_chunk;  // [max_chunks]: chunk of queue position q (gradient items q * Hv + v-head)
  // fused forward (prep + state in one kernel): per (chunk, v-head) flag set when its prep is
  // stored [max_chunks][Hv]; claim counters {prep items, state units}; the chunk of every
  // queue position in forward step order (local chunk s of every sequence)
  uint32_t* fwd_flags;
  uint32_t* fwd_queue;
  int* fwd_chunk;
  // fused prologue outputs (input dtype unless noted): normalised q, k [T_total][Hk][DK],
  // g = logsigmoid(a) fp32 [T_total][Hv], beta = sigmoid(b) [T_total][Hv]
  void* qn;
  void* kn;
  float* gn;
  void* bn;
  // context-parallel passes (Dims::cp_fwd or cp_bwd > 1): see CpArgs
  float* cp_X;
  float* cp_M;
  float* cp_R;
};

// GDR_OK for cudaSuccess; otherwise records e for gdr_debug_last_cuda_error and returns
// GDR_ERR_CUDA.
gdr_status status_of(cudaError_t e);

// Id of the current CUDA context (unique per context, also across resets); driver entry points
// looked up once through the runtime.
cudaError_t current_context_id(unsigned long long* id);
// Raises a kernel's dynamic shared-memory limit to `bytes`, once per kernel and CUDA context
// (cudaFuncSetAttribute is a driver round trip on every call).
cudaError_t set_smem_once(const void* func, size_t bytes);

// Validates *p and fills *d (the checks of gdr_fwd / gdr_bwd on the problem itself).
gdr_status resolve_problem(const gdr_problem* p, Dims* d);

// Computes the workspace layout; with base == nullptr only the size is returned.
size_t layout_workspace(const Dims& d, bool backward, char* base, Workspace* ws);

// Bytes of the saved buffer (states, then the saved factors when d.save_wy).
size_t saved_bytes(const Dims& d);
// With d.save_wy: points ws->gam, W, U, P, Tb at the factor regions of the saved buffer.
void attach_saved_factors(const Dims& d, const void* saved, Workspace* ws);

struct FwdArgs {
  const void *q, *k, *v;
  const float* g;
  const void* beta;
  const float* S0;
  void* o;
  float* S_T;
  void* h_saved;  // fp32 or bf16 (Dims::h_bf16)
};

struct BwdArgs {
  const void *q, *k, *v;
  const float* g;
  const void* beta;
  const void* h_saved;  // fp32 or bf16 (Dims::h_bf16)
  const void* dO;
  const float* dS_T;
  void *dq, *dk, *dv;
  float* dg;
  void* dbeta;
  float* dS0;
};

// Marks the end of one kernel launch named `stage` on `s`: counts the launch and,
// when stage events are on (include/gdr_debug.h), records the next event.
void stage_mark(cudaStream_t s, const char* stage);
// Called at the start of every gdr_fwd / gdr_bwd (records event 0 when enabled).
void stage_begin(cudaStream_t s);

// Fused input prologue (gdr_prologue.cu): the forward maps q, k, g, beta into ws.qn/kn/gn/bn
// (only the parts whose bit is set); the backward maps dq, dk, dg, dbeta in place.
cudaError_t launch_prologue_fwd(const Dims& d, const void* q, const void* k, const float* g, const void* beta,
                                const Workspace& ws, cudaStream_t s);
cudaError_t launch_prologue_bwd(const Dims& d, const void* q, const void* k, const float* g, const void* beta,
                                void* dq, void* dk, float* dg, void* dbeta, cudaStream_t s);
// Runs the forward prologue (if any bit is set) and points a.q, a.k, a.g, a.beta at its
// outputs; Args is FwdArgs or BwdArgs.
template <typename Args>
cudaError_t apply_prologue(const Dims& d, Args& a, const Workspace& ws, cudaStream_t s);

// K0: chunk index (chunks, seq offsets, longest-first order) and status reset; for a
// fixed-length problem only the status reset (index_folded).
cudaError_t launch_index(const Dims& d, const Workspace& ws, cudaStream_t s);

// fp32 SIMT kernels (any supported shape and dtype).
cudaError_t simt_forward(const Dims& d, const FwdArgs& a, const Workspace& ws, cudaStream_t s);
cudaError_t simt_backward(const Dims& d, const BwdArgs& a, const Workspace& ws, cudaStream_t s);
// The SIMT path's tile kernels for DK, DV <= 64 (gdr_simt_small.cu), which simt_forward and
// simt_backward use when simt_small(d).
bool simt_small(const Dims& d);
// Fixed-length problems need no index kernel: the kernels compute chunk records and step
// tables (gdr_chunks.cuh), and launch_index only resets the status word.
bool index_folded(const Dims& d);
cudaError_t simt_small_forward(const Dims& d, const FwdArgs& a, const Workspace& ws, cudaStream_t s);
cudaError_t simt_small_backward(const Dims& d, const BwdArgs& a, const Workspace& ws, cudaStream_t s);

// The context-parallel scan between the two passes (gdr_cp.cu): per (sequence, v-head) the
// boundary states X of segments 2 .. nseg - 1 (forward, X[s + 1] = M[s] X[s] + R[s] from X[1])
// or nseg - 3 .. 0 (backward, X[s - 1] = M[s] X[s] + R[s] from X[nseg - 2]), in fp32.
cudaError_t launch_cp_scan(const Dims& d, const Workspace& ws, int P, bool backward, cudaStream_t s);

// Sums dq_part / dk_part over the v-heads of each q/k head into dq / dk (dtype).
cudaError_t launch_group_reduce(const Dims& d, void* dq, void* dk, const Workspace& ws, cudaStream_t s);

// tcgen05 kernels (bf16, DK = DV = 128).  tc_available() is false when the library was
// compiled without them.
bool tc_available();
// Tensor maps (host): 3D over [rows][heads][cols] with a 64 x 1 x 64 box, 2D over
// [rows][cols] with a 64 x 64 box; bf16, 128-byte swizzle.
bool get_encoder();
bool map_3d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t heads, uint64_t rows);
bool map_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows);
bool map_2d_box(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint32_t esz, uint64_t cols,
                uint64_t rows, uint32_t box_cols, uint32_t box_rows);
bool tc_bwd_available();  // the tensor-core backward is built
bool grad_pair_mode(const Dims& d);  // Hv = 2 Hk tensor-core backward: dq/dk summed on chip
bool fused_walk_grad(const Dims& d);  // tensor-core backward: walk and gradients in one kernel
bool fused_fwd_possible(const Dims& d);  // tensor-core forward: prep and state may run as one kernel
constexpr int kMaxFusedSeqs = 8192;   // the fused backward needs the longest-first order (index kernel)
// The chunk-prep kernel (W, U, P, gamma; with write_T also T) on the tensor cores.
cudaError_t tc_launch_prep(const Dims& d, const void* q, const void* k, const void* v, const float* g,
                           const void* beta, const Workspace& ws, int write_T, cudaStream_t s, const char* stage);
cudaError_t tc_forward(const Dims& d, const FwdArgs& a, const Workspace& ws, cudaStream_t s);
cudaError_t tc_backward(const Dims& d, const BwdArgs& a, const Workspace& ws, cudaStream_t s);

}  // namespace gdr
