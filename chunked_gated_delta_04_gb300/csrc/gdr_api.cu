// gdr_api.cu -- the C ABI (include/gdr.h): validation, workspace layout, dispatch.
//
// Host code only.  It never reads tensor contents, never allocates device memory
// and never synchronises, except gdr_workspace_status (documented to synchronise).
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "gdr_internal.h"
#include "gdr_chunks.cuh"
#include "../../include/gdr_debug.h"
#include <atomic>
#include <mutex>
#include <vector>

namespace gdr {

namespace {
constexpr int kMaxStages = 32;
cudaEvent_t* g_stage_events = nullptr;
int g_stage_n = 0;
int g_stage_i = 0;
const char* g_stage_names[kMaxStages];
std::atomic<unsigned long long> g_launches{0};
std::atomic<int> g_last_cuda_error{0};  // the last CUDA error an entry point turned into GDR_ERR_CUDA

gdr_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return GDR_OK;
  g_last_cuda_error.store((int)e, std::memory_order_relaxed);
  return GDR_ERR_CUDA;
}
}  // namespace

gdr_status status_of(cudaError_t e) { return cuda_status(e); }

// A stage event: a plain record, or an event-record node when the stream is being captured.
void record_stage_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, s);
}

void stage_begin(cudaStream_t s) {
  g_stage_i = 0;
  if (g_stage_events && g_stage_n > 0) record_stage_event(g_stage_events[0], s);
}

void stage_mark(cudaStream_t s, const char* stage) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (g_stage_events && g_stage_i + 1 < g_stage_n && g_stage_i < kMaxStages) {
    g_stage_names[g_stage_i] = stage;
    record_stage_event(g_stage_events[g_stage_i + 1], s);
    ++g_stage_i;
  }
}

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Segment count of one direction's context-parallel passes (see GDR_CP_AUTO in gdr.h).
int cp_segments(int requested, const Dims& d, bool backward) {
  if (requested != GDR_CP_AUTO) return requested > 1 ? requested : 1;
  int dev = 0, n_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm <= 0) {
    (void)cudaGetLastError();  // our own query's error: no segments
    return 1;
  }
  const long long chains = (long long)d.num_seqs * d.Hv;
  if (chains <= 0 || chains * 16 > n_sm) return 1;
  const long long nc = d.cu ? d.T_total / kChunk + 1 : (d.T + kChunk - 1) / kChunk;
  long long P = nc / 16 < 32 ? nc / 16 : 32;
  while (P >= 3 && (backward ? chains * (1 + 2 * (P - 2)) > n_sm : chains * (4 + 8 * (P - 2)) > 2ll * n_sm)) --P;
  return P >= 3 ? (int)P : 1;
}

// Fills *d from *p; returns GDR_OK or the reason the problem is rejected.
gdr_status resolve(const gdr_problem* p, Dims* d) {
  if (p == nullptr) return GDR_ERR_INVALID_ARG;
  if (p->B < 0 || p->T < 0 || p->Hk <= 0 || p->Hv <= 0 || p->DK <= 0 || p->DV <= 0 || p->num_seqs < 0)
    return GDR_ERR_INVALID_ARG;
  if (p->Hv % p->Hk != 0) return GDR_ERR_INVALID_ARG;
  if (p->dtype != GDR_DTYPE_F32 && p->dtype != GDR_DTYPE_BF16) return GDR_ERR_INVALID_ARG;
  if (p->layout != GDR_STATE_KV && p->layout != GDR_STATE_VK) return GDR_ERR_INVALID_ARG;
  if (p->h_dtype != GDR_DTYPE_F32 && p->h_dtype != GDR_DTYPE_BF16) return GDR_ERR_INVALID_ARG;
  if (p->prologue & ~7u) return GDR_ERR_INVALID_ARG;
  if (p->save_wy != 0 && p->save_wy != 1) return GDR_ERR_INVALID_ARG;
  if (p->cp_fwd < GDR_CP_AUTO || p->cp_fwd > kMaxCpSegments || p->cp_bwd < GDR_CP_AUTO ||
      p->cp_bwd > kMaxCpSegments)
    return GDR_ERR_INVALID_ARG;
  if (p->cu_seqlens != nullptr) {
    if (p->B != 1) return GDR_ERR_INVALID_ARG;
  } else if (p->num_seqs != p->B) {
    return GDR_ERR_INVALID_ARG;
  }
  if (p->DK % 16 != 0 || p->DV % 16 != 0 || p->DK > 128 || p->DV > 128) return GDR_ERR_UNSUPPORTED;
  const long long T_total = (long long)p->B * p->T;
  if (T_total >= (1ll << 31) / (p->Hv > p->Hk ? p->Hv : p->Hk)) return GDR_ERR_UNSUPPORTED;
  long long maxc = p->cu_seqlens ? (long long)p->T / kChunk + p->num_seqs
                                 : (long long)p->B * ((p->T + kChunk - 1) / kChunk);
  // the saved states' rows (chunk-head x 128) are addressed with 32-bit tile coordinates
  if (maxc * p->Hv * 128 >= (1ll << 31)) return GDR_ERR_UNSUPPORTED;
  d->B = p->B;
  d->T = p->T;
  d->Hk = p->Hk;
  d->Hv = p->Hv;
  d->DK = p->DK;
  d->DV = p->DV;
  d->G = p->Hv / p->Hk;
  d->num_seqs = p->num_seqs;
  d->T_total = T_total;
  d->max_chunks = (int)maxc;
  d->scale = p->scale > 0.f ? p->scale : (float)(1.0 / sqrt((double)p->DK));
  d->dtype = p->dtype;
  d->layout = p->layout;
  d->cu = p->cu_seqlens;
  d->h_bf16 = p->h_dtype == GDR_DTYPE_BF16 ? 1 : 0;
  d->prologue = (int)p->prologue;
  d->path = (p->dtype == GDR_DTYPE_BF16 && p->DK == 128 && p->DV == 128 && maxc * p->Hv * kChunk < (1ll << 31) &&
             tc_available())
                ? 1
                : 0;
  // saved chunk factors: the tensor-core path and the small-head SIMT path (gdr_simt_small.cu)
  d->save_wy = (d->path == 1 || (p->DK <= 64 && p->DV <= 64)) ? p->save_wy : 0;
  // context-parallel segments: the tensor-core path (the SIMT path runs the plain chain)
  d->cp_fwd = d->path == 1 ? cp_segments(p->cp_fwd, *d, false) : 1;
  d->cp_bwd = d->path == 1 ? cp_segments(p->cp_bwd, *d, true) : 1;
  return GDR_OK;
}

}  // namespace

gdr_status resolve_problem(const gdr_problem* p, Dims* d) { return resolve(p, d); }

cudaError_t current_context_id(unsigned long long* id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static std::atomic<GetCurrent> get_current{nullptr};
  static std::atomic<GetId> get_id{nullptr};
  if (!get_current.load() || !get_id.load()) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess)
      return cudaErrorNotSupported;
    get_current.store((GetCurrent)f1);
    get_id.store((GetId)f2);
  }
  CUcontext ctx = nullptr;
  if (get_current.load()(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  return get_id.load()(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

cudaError_t set_smem_once(const void* func, size_t bytes) {
  struct Entry {
    const void* func;
    unsigned long long ctx;
    size_t bytes;
  };
  static std::mutex mu;
  static std::vector<Entry> done;
  unsigned long long ctx = 0;
  const bool known_ctx = current_context_id(&ctx) == cudaSuccess;
  if (known_ctx) {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : done)
      if (e.func == func && e.ctx == ctx && e.bytes >= bytes) return cudaSuccess;
  }
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && known_ctx) {
    std::lock_guard<std::mutex> lock(mu);
    done.push_back(Entry{func, ctx, bytes});
  }
  return e;
}

size_t layout_workspace(const Dims& d, bool backward, char* base, Workspace* ws) {
  size_t off = 0;
  auto take = [&](size_t bytes) -> char* {
    char* p = base ? base + off : nullptr;
    off += align256(bytes);
    return p;
  };
  Workspace w;
  memset(&w, 0, sizeof(w));
  const size_t chH = (size_t)d.max_chunks * d.Hv;
  const size_t el = d.path == 1 ? 2 : 4;  // intermediates: bf16 on the tensor-core path
  w.status = (uint32_t*)take(256);
  w.chunks = (int4*)take(sizeof(int4) * (size_t)d.max_chunks);
  w.seq_chunk_off = (int*)take(sizeof(int) * ((size_t)d.num_seqs + 1));
  w.seq_order = (int*)take(sizeof(int) * ((size_t)d.num_seqs + 1));
  if (!d.save_wy) {  // else in the saved buffer (attach_saved_factors)
    w.gam = (float*)take(sizeof(float) * chH * kChunk);
    w.W = take(el * chH * kChunk * d.DK);
    w.U = take(el * chH * kChunk * d.DV);
    if (d.path == 1) w.P = take(el * chH * kChunk * kChunk);
  } else if (d.path == 0) {  // the small-head SIMT forward hands U from its prep to its state kernel
    w.U = take(el * chH * kChunk * d.DV);
  }
  if (d.path == 0) w.Vn = take(el * chH * kChunk * d.DV);
  if (simt_small(d)) w.Pf = (float*)take(sizeof(float) * chH * kChunk * kChunk);
  if (backward) {
    if (d.path == 0) w.Tm = (float*)take(sizeof(float) * chH * kChunk * kChunk);
    w.dhp = take(el * chH * d.DK * d.DV);
    if (d.path == 1) {
      if (!d.save_wy) w.Tb = take(el * chH * kChunk * kChunk);
      w.dVn = take(el * chH * kChunk * d.DV);
    } else if (simt_small(d)) {
      w.dVn = take(el * chH * kChunk * d.DV);
      w.Ak = (float*)take(sizeof(float) * chH * kChunk * kChunk);
      w.PdO = (float*)take(sizeof(float) * chH * kChunk * d.DV);
      w.QdO = (float*)take(sizeof(float) * chH * d.DK * d.DV);
    }
    if (fused_walk_grad(d)) {  // one region: flags then the claim counter (zeroed per call)
      w.walk_flags = (uint32_t*)take(sizeof(uint32_t) * ((size_t)d.max_chunks * d.Hv + 64));
      w.grad_queue = w.walk_flags ? w.walk_flags + (size_t)d.max_chunks * d.Hv : nullptr;
      w.step_off = (int*)take(sizeof(int) * ((size_t)d.max_chunks + 2));
      w.grad_chunk = (int*)take(sizeof(int) * ((size_t)d.max_chunks + 1));
    }
    if (d.G > 1 && !grad_pair_mode(d)) {
      w.dq_part = (float*)take(sizeof(float) * (size_t)d.T_total * d.Hv * d.DK);
      w.dk_part = (float*)take(sizeof(float) * (size_t)d.T_total * d.Hv * d.DK);
    }
  }
  if (!backward && fused_fwd_possible(d)) {  // one region: flags, then the claim counters (zeroed per call)
    w.fwd_flags = (uint32_t*)take(sizeof(uint32_t) * ((size_t)d.max_chunks * d.Hv + 64));
    w.fwd_queue = w.fwd_flags ? w.fwd_flags + (size_t)d.max_chunks * d.Hv : nullptr;
    w.step_off = (int*)take(sizeof(int) * ((size_t)d.max_chunks + 2));
    w.fwd_chunk = (int*)take(sizeof(int) * ((size_t)d.max_chunks + 1));
  }
  const int cp = backward ? d.cp_bwd : d.cp_fwd;
  if (d.path == 1 && cp > 1) {  // boundary states, transitions, zero-boundary results (CpArgs)
    const size_t mats = (size_t)d.num_seqs * d.Hv * cp * 128 * 128 * sizeof(float);
    w.cp_X = (float*)take(mats);
    w.cp_M = (float*)take(mats);
    w.cp_R = (float*)take(mats);
  }
  if (d.prologue) {
    const size_t in_el = d.dtype == GDR_DTYPE_BF16 ? 2 : 4;
    if (d.prologue & GDR_PROLOGUE_QK_L2NORM) {
      w.qn = take(in_el * (size_t)d.T_total * d.Hk * d.DK);
      w.kn = take(in_el * (size_t)d.T_total * d.Hk * d.DK);
    }
    if (d.prologue & GDR_PROLOGUE_G_LOGSIGMOID) w.gn = (float*)take(sizeof(float) * (size_t)d.T_total * d.Hv);
    if (d.prologue & GDR_PROLOGUE_BETA_SIGMOID) w.bn = take(in_el * (size_t)d.T_total * d.Hv);
  }
  if (ws) *ws = w;
  return off;
}

// Saved buffer: the chunk-start states, then (save_wy) on the tensor-core path per region,
// 256-byte aligned: gamma fp32 [chunks][Hv][64], W bf16 [..][64][DK], U bf16 [..][64][DV]
// (replaced by Vn = U - W h by the forward's state kernel), P bf16 [..][64][64], T bf16
// [..][64][64].
// The small-head SIMT path keeps fp32 factors instead: gamma [..][64], W^T [..][DK][64],
// T [..][64][64], K K^T * Gam (strictly lower) [..][64][64], P^T [..][64][64], Vn [..][64][DV].
static size_t saved_layout(const Dims& d, const char* base, Workspace* ws) {
  const size_t chH = (size_t)d.max_chunks * d.Hv;
  size_t off = align256(chH * d.DK * d.DV * (d.h_bf16 ? 2 : 4));
  if (!d.save_wy) return off;
  auto take = [&](size_t bytes) -> char* {
    char* p = base ? const_cast<char*>(base) + off : nullptr;
    off += align256(bytes);
    return p;
  };
  if (d.path == 0) {
    float* gam = (float*)take(sizeof(float) * chH * kChunk);
    void* Wt = take(sizeof(float) * chH * d.DK * kChunk);
    float* T = (float*)take(sizeof(float) * chH * kChunk * kChunk);
    float* Ak = (float*)take(sizeof(float) * chH * kChunk * kChunk);
    float* Pt = (float*)take(sizeof(float) * chH * kChunk * kChunk);
    void* Vn = take(sizeof(float) * chH * kChunk * d.DV);
    if (ws) {
      ws->gam = gam;
      ws->W = Wt;
      ws->Tm = T;
      ws->Ak = Ak;
      ws->Pf = Pt;
      ws->Vn = Vn;
    }
    return off;
  }
  float* gam = (float*)take(sizeof(float) * chH * kChunk);
  void* W = take(2 * chH * kChunk * d.DK);
  void* U = take(2 * chH * kChunk * d.DV);
  void* P = take(2 * chH * kChunk * kChunk);
  void* T = take(2 * chH * kChunk * kChunk);
  if (ws) {
    ws->gam = gam;
    ws->W = W;
    ws->U = U;
    ws->P = P;
    ws->Tb = T;
  }
  return off;
}

size_t saved_bytes(const Dims& d) { return saved_layout(d, nullptr, nullptr); }

void attach_saved_factors(const Dims& d, const void* saved, Workspace* ws) {
  if (d.save_wy) saved_layout(d, (const char*)saved, ws);
}

// With prologue bits set: runs the forward prologue and points the operator's q, k, g,
// beta at its outputs (the raw pointers stay with the caller for the backward map).
template <typename Args>
cudaError_t apply_prologue(const Dims& d, Args& a, const Workspace& ws, cudaStream_t s) {
  if (!d.prologue) return cudaSuccess;
  const cudaError_t e = launch_prologue_fwd(d, a.q, a.k, a.g, a.beta, ws, s);
  if (d.prologue & GDR_PROLOGUE_QK_L2NORM) {
    a.q = ws.qn;
    a.k = ws.kn;
  }
  if (d.prologue & GDR_PROLOGUE_G_LOGSIGMOID) a.g = ws.gn;
  if (d.prologue & GDR_PROLOGUE_BETA_SIGMOID) a.beta = ws.bn;
  return e;
}
template cudaError_t apply_prologue<FwdArgs>(const Dims&, FwdArgs&, const Workspace&, cudaStream_t);

}  // namespace gdr

using namespace gdr;

extern "C" {

size_t gdr_max_chunks(const gdr_problem* p) {
  Dims d;
  return resolve(p, &d) == GDR_OK ? (size_t)d.max_chunks : 0;
}

size_t gdr_saved_states_bytes(const gdr_problem* p) {
  Dims d;
  if (resolve(p, &d) != GDR_OK) return 0;
  if (!d.save_wy) return (size_t)d.max_chunks * d.Hv * d.DK * d.DV * (d.h_bf16 ? 2 : 4);
  return saved_bytes(d);
}

size_t gdr_fwd_workspace_bytes(const gdr_problem* p) {
  Dims d;
  if (resolve(p, &d) != GDR_OK) return 0;
  return layout_workspace(d, false, nullptr, nullptr);
}

size_t gdr_bwd_workspace_bytes(const gdr_problem* p) {
  Dims d;
  if (resolve(p, &d) != GDR_OK) return 0;
  if (d.path == 1 && !tc_bwd_available()) d.path = d.save_wy = 0, d.cp_fwd = d.cp_bwd = 1;
  return layout_workspace(d, true, nullptr, nullptr);
}

int gdr_path(const gdr_problem* p) {
  Dims d;
  return resolve(p, &d) == GDR_OK ? d.path : -1;
}

gdr_status gdr_fwd(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                   const void* beta, const float* S0, void* o, float* S_T, void* h_saved, void* workspace,
                   size_t workspace_bytes, gdr_stream_t stream) {
  Dims d;
  gdr_status st = resolve(p, &d);
  if (st != GDR_OK) return st;
  const bool any_tokens = d.T_total > 0;
  if (any_tokens && (!q || !k || !v || !g || !beta || !o || !h_saved)) return GDR_ERR_INVALID_ARG;
  if (!workspace) return GDR_ERR_WORKSPACE;
  const void* ptrs[] = {q, k, v, g, beta, S0, o, S_T, h_saved, p->cu_seqlens};
  for (const void* x : ptrs)
    if (x && !aligned16(x)) return GDR_ERR_ALIGNMENT;
  if (((uintptr_t)workspace & 255u) != 0) return GDR_ERR_ALIGNMENT;
  Workspace ws;
  const size_t need = layout_workspace(d, false, (char*)workspace, &ws);
  if (workspace_bytes < need) return GDR_ERR_WORKSPACE;
  attach_saved_factors(d, h_saved, &ws);
  cudaStream_t s = (cudaStream_t)stream;
  FwdArgs a{q, k, v, g, beta, S0, o, S_T, h_saved};
  stage_begin(s);
  cudaError_t e = launch_index(d, ws, s);
  if (e == cudaSuccess) e = apply_prologue(d, a, ws, s);
  if (e == cudaSuccess) e = d.path == 1 ? tc_forward(d, a, ws, s) : simt_forward(d, a, ws, s);
  return cuda_status(e);
}

gdr_status gdr_bwd(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                   const void* beta, const void* h_saved, const void* dO, const float* dS_T, void* dq,
                   void* dk, void* dv, float* dg, void* dbeta, float* dS0, void* workspace,
                   size_t workspace_bytes, gdr_stream_t stream) {
  Dims d;
  gdr_status st = resolve(p, &d);
  if (st != GDR_OK) return st;
  if (d.path == 1 && !tc_bwd_available()) d.path = d.save_wy = 0, d.cp_fwd = d.cp_bwd = 1;
  const bool any_tokens = d.T_total > 0;
  if (any_tokens && (!q || !k || !v || !g || !beta || !h_saved || !dO || !dq || !dk || !dv || !dg || !dbeta))
    return GDR_ERR_INVALID_ARG;
  if (!workspace) return GDR_ERR_WORKSPACE;
  const void* ptrs[] = {q, k, v, g, beta, h_saved, dO, dS_T, dq, dk, dv, dg, dbeta, dS0, p->cu_seqlens};
  for (const void* x : ptrs)
    if (x && !aligned16(x)) return GDR_ERR_ALIGNMENT;
  if (((uintptr_t)workspace & 255u) != 0) return GDR_ERR_ALIGNMENT;
  Workspace ws;
  const size_t need = layout_workspace(d, true, (char*)workspace, &ws);
  if (workspace_bytes < need) return GDR_ERR_WORKSPACE;
  attach_saved_factors(d, h_saved, &ws);
  cudaStream_t s = (cudaStream_t)stream;
  BwdArgs a{q, k, v, g, beta, h_saved, dO, dS_T, dq, dk, dv, dg, dbeta, dS0};
  stage_begin(s);
  cudaError_t e = launch_index(d, ws, s);
  if (e == cudaSuccess) e = apply_prologue(d, a, ws, s);
  if (e == cudaSuccess) e = d.path == 1 ? tc_backward(d, a, ws, s) : simt_backward(d, a, ws, s);
  // gradients w.r.t. the raw inputs (in place; after the v-head group sum when Hv > Hk)
  if (e == cudaSuccess) e = launch_prologue_bwd(d, q, k, g, beta, dq, dk, dg, dbeta, s);
  return cuda_status(e);
}

gdr_status gdr_workspace_status(const void* workspace, gdr_stream_t stream, uint32_t* flags) {
  if (!workspace) return GDR_ERR_WORKSPACE;
  uint32_t word = 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GDR_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDR_ERR_CUDA;
  if (flags) *flags = word;
  if (word & kDevErrBadCuSeqlens) return GDR_ERR_INVALID_ARG;
  if (word & (kDevErrTimeoutFwd | kDevErrTimeoutBwd | kDevErrTimeoutPrep)) return GDR_ERR_TIMEOUT;
  return GDR_OK;
}

int gdr_debug_last_cuda_error(void) { return g_last_cuda_error.load(std::memory_order_relaxed); }

int gdr_debug_cp_segments(const gdr_problem* p, int* fwd, int* bwd) {
  Dims d;
  const gdr_status st = resolve(p, &d);
  if (st != GDR_OK) return (int)st;
  if (fwd) *fwd = d.cp_fwd;
  if (bwd) *bwd = d.path == 1 && !tc_bwd_available() ? 1 : d.cp_bwd;
  return 0;
}

int gdr_debug_cp_segment(int c0, int c1, int P, int s, int* out3) {
  if (P < 1 || s < 0 || c1 < c0 || out3 == nullptr) return 1;
  const int3 r = cp_segment(c0, c1, P, s);
  out3[0] = r.x;
  out3[1] = r.y;
  out3[2] = r.z;
  return 0;
}

const char* gdr_debug_cuda_error_string(int e) { return cudaGetErrorString((cudaError_t)e); }

void gdr_debug_set_stage_events(void** events, int n) {
  g_stage_events = (cudaEvent_t*)events;
  g_stage_n = events ? n : 0;
  g_stage_i = 0;
}

int gdr_debug_stage_count(void) { return g_stage_i; }

const char* gdr_debug_stage_name(int i) { return (i >= 0 && i < g_stage_i) ? g_stage_names[i] : ""; }

unsigned long long gdr_debug_launch_count(void) { return g_launches.load(); }

const char* gdr_status_string(gdr_status s) {
  switch (s) {
    case GDR_OK: return "GDR_OK";
    case GDR_ERR_INVALID_ARG: return "GDR_ERR_INVALID_ARG: invalid argument";
    case GDR_ERR_UNSUPPORTED: return "GDR_ERR_UNSUPPORTED: unsupported shape or dtype";
    case GDR_ERR_ALIGNMENT: return "GDR_ERR_ALIGNMENT: pointer not 16-byte aligned (workspace: 256)";
    case GDR_ERR_CUDA: return "GDR_ERR_CUDA: a CUDA call failed";
    case GDR_ERR_TIMEOUT: return "GDR_ERR_TIMEOUT: a kernel's bounded wait ran out";
    case GDR_ERR_WORKSPACE: return "GDR_ERR_WORKSPACE: workspace missing or too small";
  }
  return "unknown gdr_status";
}

}  // extern "C"
