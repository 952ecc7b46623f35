/*
 * gdr.h -- C ABI of the GB300 (sm_103a) chunked gated delta rule library (libgdr.so).
 *
 * The operator (FlashQLA PR #34, "SM120/121: Add support for fused backward
 * kernel", Summary: the forward and the fused backward "fused_gdr_bwd" of the
 * chunked gated delta rule; "Current status": fixed-length and variable-length
 * inputs, KV/VK state layouts, initial/final states, autograd).  The pages do not
 * write the recurrence out; it is fixed as
 *
 *     S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *     o_t = scale * S_t q_t,        S in R^{DV x DK},  scale = 1/sqrt(DK) by default,
 *
 * evaluated in 64-token chunks that restart at every sequence start.  The
 * backward takes dL/do and dL/dS_T and returns dq, dk, dv, dg, dbeta, dS0.
 *
 * Conventions shared by every entry point
 *  - Ownership: the caller allocates every buffer (device memory unless stated)
 *    and keeps it alive until the work on `stream` has finished.  The library
 *    never allocates device memory, keeps no device state between calls and
 *    never synchronises the stream (except gdr_workspace_status, which says so).
 *  - Asynchrony: all work is enqueued on `stream`; a GDR_OK return means the
 *    launches were enqueued, not that they finished.
 *  - Validation: arguments are checked on the host before anything is launched,
 *    without reading any tensor contents.  On an error nothing is launched and
 *    the outputs are untouched.
 *  - Tensor layouts (all contiguous, row-major, base pointers 16-byte aligned):
 *      q, k, dq, dk       [B, T, Hk, DK]     dtype
 *      v, o, dO, dv       [B, T, Hv, DV]     dtype
 *      g, dg              [B, T, Hv]         float32 (log decay, usually <= 0)
 *      beta, dbeta        [B, T, Hv]         dtype
 *      S0, S_T, dS_T, dS0 [num_seqs, Hv, DK, DV] float32 for GDR_STATE_KV (stores S^T),
 *                         [num_seqs, Hv, DV, DK] float32 for GDR_STATE_VK (stores S)
 *      h_saved            [max_chunks, Hv, DK, DV] of h_dtype (float32 by default, or
 *                         bf16): S^T at the START of every 64-token chunk, whatever the
 *                         state layout; chunk c of sequence n sits at index
 *                         chunk_offset[n] + c with chunk_offset[n] = sum_{n' < n}
 *                         ceil(L_n' / 64).  Slots past the last real chunk (varlen upper
 *                         bound) are left untouched.
 *    Variable length: B = 1, T = total tokens, cu_seqlens (device, int32,
 *    num_seqs + 1 entries, cu_seqlens[0] = 0, non-decreasing, last = T) delimits the
 *    sequences; empty sequences are allowed (S_T = S0, dS0 = dS_T).
 *  - Heads: v-head j uses q/k head j / (Hv / Hk); g and beta are per v-head.
 *  - Supported shapes: Hv % Hk == 0; DK, DV in {16, 32, 48, ..., 128} (multiples of
 *    16).  dtype BF16 with DK = DV = 128 runs the tcgen05 tensor-core kernels; every
 *    other supported case runs the fp32 SIMT kernels (fp32 arithmetic throughout).
 *  - Errors inside a kernel (a bounded wait that ran out) are recorded in the
 *    workspace's status word and the kernel returns early without trapping; read
 *    it with gdr_workspace_status.
 */
#ifndef GDR_H_
#define GDR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* gdr_stream_t; /* = cudaStream_t; NULL = legacy default stream */

typedef enum {
  GDR_OK = 0,
  GDR_ERR_INVALID_ARG = 1, /* null required pointer, bad shape, bad enum value */
  GDR_ERR_UNSUPPORTED = 2, /* a shape/dtype combination the library does not implement, or a size
                              beyond B*T*max(Hk,Hv) < 2^31 and max_chunks*Hv*128 < 2^31 */
  GDR_ERR_ALIGNMENT = 3,   /* a base pointer is not 16-byte aligned */
  GDR_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (launch, tensor map, ...) */
  GDR_ERR_TIMEOUT = 5,     /* a kernel's bounded wait ran out (see gdr_workspace_status) */
  GDR_ERR_WORKSPACE = 6    /* workspace missing or smaller than the size query returned */
} gdr_status;

typedef enum { GDR_DTYPE_F32 = 0, GDR_DTYPE_BF16 = 1 } gdr_dtype;

typedef enum { GDR_STATE_KV = 0, GDR_STATE_VK = 1 } gdr_state_layout;

/* Input prologue applied inside the operator (bits of gdr_problem.prologue).  With a bit
 * set the corresponding arguments are RAW and the matching gradients are with respect to
 * them (eps = 1e-6; the maps are the usual preparation of the operator's inputs):
 *   QK_L2NORM      q, k are raw; the operator uses q * (sum q^2 + eps)^(-1/2) per token
 *                  and head (same for k); dq, dk are gradients w.r.t. the raw q, k.
 *   G_LOGSIGMOID   g holds the raw gate logit a; the log decay is logsigmoid(a); dg = dL/da.
 *   BETA_SIGMOID   beta holds the raw logit b; the operator uses sigmoid(b) (rounded to the
 *                  input dtype); dbeta = dL/db. */
typedef enum {
  GDR_PROLOGUE_QK_L2NORM = 1,
  GDR_PROLOGUE_G_LOGSIGMOID = 2,
  GDR_PROLOGUE_BETA_SIGMOID = 4
} gdr_prologue_flags;

typedef struct {
  int B, T;                  /* fixed length: B sequences of T tokens; varlen: B = 1, T = total */
  int Hk, Hv, DK, DV;        /* q/k heads, v heads (Hv % Hk == 0), key and value widths */
  int num_seqs;              /* fixed length: = B; varlen: number of sequences */
  const int32_t* cu_seqlens; /* device pointer (varlen) or NULL (fixed length) */
  gdr_dtype dtype;           /* dtype of q, k, v, beta, o, dO, dq, dk, dv, dbeta */
  gdr_state_layout layout;   /* orientation of S0, S_T, dS_T, dS0 */
  float scale;               /* output scale; <= 0 selects 1/sqrt(DK) */
  gdr_dtype h_dtype;         /* dtype of h_saved: GDR_DTYPE_F32 (default: the states as the
                                forward carries them) or GDR_DTYPE_BF16 (half the bytes of the
                                largest tensor, rounded to bf16; the backward then reads the
                                rounded states, so its gradients carry that rounding) */
  unsigned int prologue;     /* bit set of gdr_prologue_flags; 0 = inputs used as given */
  int save_wy;               /* 0 or 1.  1: the forward also keeps its per-chunk factors
                                (gamma, W, Vn, P and T of the WY form, see "Saved factors"
                                below) in the saved buffer after the states, and the
                                backward reads them instead of recomputing them.  Same
                                results (bit for bit on the tensor-core path); honoured on
                                the tensor-core path and on the SIMT path for DK, DV <= 64,
                                ignored (nothing saved) for larger SIMT heads. */
  int cp_fwd, cp_bwd;        /* intra-card context parallelism (FlashQLA PR #34, "Current
                                status"), per direction: 0 or 1 = off; -1 = the library
                                chooses (GDR_CP_AUTO below); P in 2..64 = every
                                sequence is cut at chunk boundaries into min(P, its chunk
                                count) segments of nearly equal chunk counts (the first ones
                                one longer), which run side by side: a first pass finds
                                each segment's end state from a zero start and its state
                                transition (the same recurrence on the identity with the
                                values set to zero), a short scan gives every segment its
                                true start state, and a second pass evaluates the segments
                                from those (the backward mirrors this with the state
                                gradient).  Same results up to rounding (the transitions
                                and the scan replace part of the chain's bf16 products).
                                It pays when few (sequence, v-head) chains leave most SMs
                                idle.  Honoured on the tensor-core path, ignored on the
                                SIMT path.  Zero-initialised structs keep it off. */
} gdr_problem;

/* cp_fwd / cp_bwd = GDR_CP_AUTO: segments only when the (sequence, v-head) chains are at most
 * 1/16 of the GPU's SM count (so the plain chains would leave most SMs idle); then the largest
 * P <= min(32, C / 16), C = the longest sequence's chunk count (varlen: its upper bound
 * T / 64 + 1), whose first pass fits in one wave: chains * (4 + 8 (P - 2)) <= 2 * SMs forward,
 * chains * (1 + 2 (P - 2)) <= SMs backward; off if that P is below 3.  The choice depends only
 * on the problem and the current device, so size queries and calls agree. */
#define GDR_CP_AUTO (-1)

/* Upper bound on the number of 64-token chunks: B * ceil(T/64) for fixed length,
 * floor(T/64) + num_seqs for varlen.  Returns 0 for an invalid problem. */
size_t gdr_max_chunks(const gdr_problem* p);

/* Bytes of h_saved: gdr_max_chunks(p) * Hv * DK * DV * (4 for F32, 2 for BF16 h_dtype),
 * plus, with save_wy, the saved factors: on the tensor-core path gdr_max_chunks(p) * Hv *
 * 49408 bytes; on the SIMT path (DK, DV <= 64) gdr_max_chunks(p) * Hv * 4 * (64 + 64 DK +
 * 3 * 4096 + 64 DV) bytes, each region rounded up to 256 bytes.
 * Saved factors (save_wy): after the states, per (chunk, v-head) of the chunk index, in
 * this order, each region starting 256-byte aligned: gamma fp32 [64] (in-chunk cumulative
 * sum of g), W bf16 [64][DK], Vn bf16 [64][DV], P bf16 [64][64], T bf16 [64][64] (chunked
 * WY form of the gated delta rule: T = (I + strictly lower diag(beta) Gamma K K^T)^{-1},
 * W = T diag(beta e^gamma) K, U = T diag(beta) V, Vn = U - W h with h the chunk-start
 * state, P = masked decayed Q K^T).  The SIMT path keeps, in this order and all fp32: gamma
 * [64], W^T [DK][64], T [64][64], the strictly lower decayed K K^T [64][64], P^T [64][64],
 * Vn [64][DV].  gdr_bwd requires them to come from gdr_fwd with the same problem and
 * inputs. */
size_t gdr_saved_states_bytes(const gdr_problem* p);

/* Bytes of the scratch workspace that gdr_fwd / gdr_bwd need (device memory,
 * 256-byte aligned).  Its contents need not be initialised and are not meaningful
 * after the call, except the status word read by gdr_workspace_status. */
size_t gdr_fwd_workspace_bytes(const gdr_problem* p);
size_t gdr_bwd_workspace_bytes(const gdr_problem* p);

/* Forward (chunked gated delta rule, FlashQLA PR #34 Summary).
 *   in : q, k, v, g, beta; S0 (nullable: zero initial state)
 *   out: o; S_T (nullable: final state not written); h_saved (required: the
 *        chunk-start states that gdr_bwd consumes)
 * workspace/workspace_bytes: see gdr_fwd_workspace_bytes. */
gdr_status gdr_fwd(const gdr_problem* p, const void* q, const void* k, const void* v,
                   const float* g, const void* beta, const float* S0, void* o, float* S_T,
                   void* h_saved, void* workspace, size_t workspace_bytes, gdr_stream_t stream);

/* Backward (the fused backward "fused_gdr_bwd" of FlashQLA PR #34: walks the chunks
 * in reverse carrying the state gradient dh).
 *   in : q, k, v, g, beta, h_saved (as written by gdr_fwd for the same inputs and S0),
 *        dO, dS_T (nullable: zero)
 *   out: dq, dk (summed over the Hv/Hk v-heads of each q/k head), dv, dg, dbeta;
 *        dS0 (nullable: not written).  All outputs are overwritten.
 * The result is bitwise deterministic: no floating-point atomics. */
gdr_status gdr_bwd(const gdr_problem* p, const void* q, const void* k, const void* v,
                   const float* g, const void* beta, const void* h_saved, const void* dO,
                   const float* dS_T, void* dq, void* dk, void* dv, float* dg, void* dbeta,
                   float* dS0, void* workspace, size_t workspace_bytes, gdr_stream_t stream);

/* Forward without a workspace argument (no counterpart on the pages: it is a
 * convenience of this library).  For callers that cannot give the library scratch
 * memory and cannot allocate any themselves: e.g. a plugin whose host framework
 * owns all device memory and forbids side allocations, or a latency-critical loop
 * where a cudaMalloc, which may synchronise the whole device, is not acceptable.
 * Same arguments and results as gdr_fwd, minus the workspace; host-side errors are
 * returned as by gdr_fwd, device-side ones are read with gdr_noalloc_status.
 *  - Its scratch is one array of GDR_NOALLOC_MAX_WORKSPACE_BYTES in device memory,
 *    owned by the library: every GPU that loads this part of the library keeps that
 *    much memory until the process exits.  With CUDA's default lazy module loading that
 *    is only GPUs on which this entry point has run; with CUDA_MODULE_LOADING=EAGER it
 *    is every GPU whose context loads libgdr.so, whether or not the entry point runs.
 *    It allocates nothing, ever.
 *  - A problem whose gdr_fwd_workspace_bytes exceeds the limit is refused with
 *    GDR_ERR_WORKSPACE before anything is launched.
 *  - It runs on the current device.  The first call in each CUDA context of a device
 *    (the first call on the device, and again after a reset created a new context)
 *    looks up the array's device address (cudaGetSymbolAddress) and caches it, so make
 *    that first call before any stream capture begins.
 *  - Every call uses the same array and leaves its contents behind; nothing needs
 *    clearing between calls.  Calls whose GPU work can overlap (e.g. on two
 *    unordered streams) race on the array and corrupt each other's results:
 *    serialise them. */
#define GDR_NOALLOC_MAX_WORKSPACE_BYTES ((size_t)64 << 20)
gdr_status gdr_fwd_noalloc(const gdr_problem* p, const void* q, const void* k, const void* v,
                           const float* g, const void* beta, const float* S0, void* o, float* S_T,
                           void* h_saved, gdr_stream_t stream);

/* The status word of gdr_fwd_noalloc's array, as gdr_workspace_status reads a workspace's
 * (no counterpart on the pages; allocates nothing): synchronises `stream`, then returns
 * GDR_OK, GDR_ERR_INVALID_ARG (the kernels found cu_seqlens malformed and computed
 * nothing) or GDR_ERR_TIMEOUT (a bounded wait ran out; the outputs are invalid) for the
 * last gdr_fwd_noalloc on the current device.  *flags (nullable) receives the raw bits. */
gdr_status gdr_noalloc_status(gdr_stream_t stream, uint32_t* flags);

/* Synchronises `stream`, then reads the status word that the kernels of the last
 * gdr_fwd / gdr_bwd using `workspace` left there: GDR_OK, or GDR_ERR_TIMEOUT if a
 * bounded wait ran out (the kernel returned early; its outputs are invalid).
 * *flags (nullable) receives the raw bit set (bit i = kernel role i). */
gdr_status gdr_workspace_status(const void* workspace, gdr_stream_t stream, uint32_t* flags);

/* Human-readable name of a status code (static storage). */
const char* gdr_status_string(gdr_status s);

/* Which kernel family a problem runs on: 1 = tcgen05 tensor-core kernels,
 * 0 = fp32 SIMT kernels, -1 = invalid or unsupported problem. */
int gdr_path(const gdr_problem* p);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H_ */
