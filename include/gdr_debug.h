/*
 * gdr_debug.h -- benchmark instrumentation of libgdr.so (not needed to use the
 * operator; no counterpart on the pages).
 *
 * Stage events: after gdr_debug_set_stage_events(events, n) with n >= 1 caller-
 * created cudaEvent_t handles, every following gdr_fwd / gdr_bwd records
 * events[0] on its stream before its first kernel and events[i + 1] right after
 * its i-th kernel launch (at most n - 1 kernels are bracketed).  The elapsed
 * time between events[i] and events[i + 1] is then kernel i's device time on
 * that stream.  gdr_debug_stage_count() gives the number of kernels the last call
 * bracketed and gdr_debug_stage_name(i) a stable stage name ("fwd_prep",
 * "bwd_grad", ...).  Pass events = NULL to switch it off.  The setting is
 * process-global host state and not thread-safe; the events stay owned by the
 * caller.  A call made while its stream is being captured records them with
 * cudaEventRecordExternal, which puts event-record nodes into the graph: every
 * replay of the graph then times its kernels the same way.
 *
 * Launch counter: gdr_debug_launch_count() returns how many kernels this process
 * has launched through the library so far.
 *
 * CUDA errors: when an entry point returns GDR_ERR_CUDA, gdr_debug_last_cuda_error()
 * gives the cudaError_t behind it (0 if none has occurred in this process) and
 * gdr_debug_cuda_error_string() its text.
 */
#ifndef GDR_DEBUG_H_
#define GDR_DEBUG_H_

#include "gdr.h"

#ifdef __cplusplus
extern "C" {
#endif

void gdr_debug_set_stage_events(void** events, int n);
int gdr_debug_stage_count(void);
const char* gdr_debug_stage_name(int i);
unsigned long long gdr_debug_launch_count(void);
int gdr_debug_last_cuda_error(void);
const char* gdr_debug_cuda_error_string(int e);

/* Device self-test of the tensor-core operand layouts: one tcgen05 GEMM on one CTA,
 * D[m][n] = sum_k Amat[m][k] Bmat[k][n] (M = 128, N in {64, 128}, K in {64, 128}),
 * A and B bf16 row-major device buffers, Amat = A ([128][K], a_mn = 0) or A^T ([K][128],
 * a_mn = 1), Bmat = B^T ([N][K], b_mn = 0) or B ([K][N], b_mn = 1); D fp32 [128][N].
 * status: device uint32 that receives a timeout bit if the MMA never completes.
 * Returns 0 when launched, non-zero for bad sizes or a launch error. */
int gdr_debug_tc_gemm(const void* A, const void* B, float* D, int N, int K, int a_mn, int b_mn,
                      unsigned int* status, void* stream);

/* Failure-detection self-test: one kernel waits on an mbarrier that nothing ever
 * completes, bounded by limit_ns (at most 1 s).  The wait must expire, set the timeout
 * bit (GDR_ERR_TIMEOUT's bit, 1u << 1) in *status and return; *waited_ns receives how long
 * it waited.  status and waited_ns are device pointers.  Returns 0 when launched. */
int gdr_debug_timeout_selftest(unsigned int* status, unsigned long long limit_ns,
                               unsigned long long* waited_ns, void* stream);

/* The context-parallel split of gdr_problem.cp_fwd / cp_bwd: the chunks [c0, c1) of one
 * sequence cut into nseg = max(1, min(P, c1 - c0)) segments whose chunk counts differ by at
 * most one, the longer ones first.  Writes {first chunk, end chunk, nseg} of segment s into
 * out3 (a segment s >= nseg is empty: {c1, c1, nseg}).  Host only; returns 0, or non-zero for
 * P < 1, s < 0, c1 < c0 or a null out3. */
int gdr_debug_cp_segment(int c0, int c1, int P, int s, int* out3);

/* The segment counts a call with problem *p would use on the current device (1: no segments;
 * GDR_CP_AUTO resolved), forward into *fwd and backward into *bwd.  Returns 0, or a gdr_status
 * for an invalid problem. */
int gdr_debug_cp_segments(const gdr_problem* p, int* fwd, int* bwd);

#ifdef __cplusplus
}
#endif

#endif /* GDR_DEBUG_H_ */
