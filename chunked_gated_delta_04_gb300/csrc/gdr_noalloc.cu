// gdr_noalloc.cu -- gdr_fwd_noalloc: the forward pass with its scratch memory in a
// fixed-size device array that the library itself owns.
//
// Who needs this: a caller that cannot hand the library a workspace buffer and
// cannot allocate one either -- for example a plugin whose host framework owns
// all device memory and forbids side allocations, or a latency-critical serving
// loop where a cudaMalloc (which may synchronise the whole device) is not
// allowed.  gdr_fwd_noalloc takes the same inputs and outputs as gdr_fwd but no
// workspace; its scratch lives in `g_noalloc_scratch` below.
//
// Rules of the array:
//  - It is a file-scope __device__ array of GDR_NOALLOC_MAX_WORKSPACE_BYTES (64 MiB),
//    so every GPU that loads this part of the library keeps that much memory until
//    the process exits (with CUDA's default lazy module loading, only GPUs on which
//    this entry point has run).  Problems whose forward workspace would be larger
//    are refused with GDR_ERR_WORKSPACE.
//  - In host code the array's name is only a host-side stand-in; its device address
//    is looked up with cudaGetSymbolAddress on the first call made in each CUDA context
//    of a device (the device current) and cached with that context's id, so a context
//    created anew (after cudaDeviceReset, say) looks it up again instead of using an
//    address of the old one.  With CUDA_MODULE_LOADING=EAGER the array is reserved on
//    every device whose context loads the library, whether or not this entry point runs.
//  - All calls share the one array and leave their contents behind.  The forward
//    writes every scratch word it reads before reading it, and its first kernel
//    clears the status word, so nothing has to be zeroed between calls.  Two calls
//    whose work overlaps on the GPU (different streams, no ordering) race on the
//    array and give wrong results: serialise them.
//  - Device-side errors (a malformed cu_seqlens, a bounded wait that ran out) land in
//    the array's status word; gdr_noalloc_status reads it, allocating nothing.
#include <mutex>

#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr size_t kNoallocScratchBytes = GDR_NOALLOC_MAX_WORKSPACE_BYTES;
constexpr int kMaxDevices = 128;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_noalloc_mu;
struct ScratchEntry {
  unsigned long long ctx_id;  // CUDA context the address belongs to
  void* ptr;                  // device address of g_noalloc_scratch in it, or nullptr
};
ScratchEntry g_noalloc[kMaxDevices];

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Device address of the scratch array in the current device's context (set up on first
// use in that context).
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  e = cudaSetDevice(dev);  // makes the device's primary context current (CUDA 12+ initialises it here)
  if (e != cudaSuccess) return e;
  unsigned long long ctx = 0;
  e = current_context_id(&ctx);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc[dev].ptr == nullptr || g_noalloc[dev].ctx_id != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr || ((uintptr_t)p & 255u) != 0) return cudaErrorInvalidDevicePointer;
    g_noalloc[dev] = ScratchEntry{ctx, p};
  }
  *out = g_noalloc[dev].ptr;
  return cudaSuccess;
}

}  // namespace
}  // namespace gdr

using namespace gdr;

extern "C" gdr_status gdr_fwd_noalloc(const gdr_problem* p, const void* q, const void* k, const void* v,
                                      const float* g, const void* beta, const float* S0, void* o, float* S_T,
                                      void* h_saved, gdr_stream_t stream) {
  Dims d;
  gdr_status st = resolve_problem(p, &d);
  if (st != GDR_OK) return st;
  if (d.T_total > 0 && (!q || !k || !v || !g || !beta || !o || !h_saved)) return GDR_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, g, beta, S0, o, S_T, h_saved, p->cu_seqlens};
  for (const void* x : ptrs)
    if (x && !aligned16(x)) return GDR_ERR_ALIGNMENT;
  if (layout_workspace(d, false, nullptr, nullptr) > kNoallocScratchBytes) return GDR_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return GDR_ERR_CUDA;
  Workspace ws;
  layout_workspace(d, false, (char*)scratch, &ws);
  attach_saved_factors(d, h_saved, &ws);
  cudaStream_t s = (cudaStream_t)stream;
  FwdArgs a{q, k, v, g, beta, S0, o, S_T, h_saved};
  stage_begin(s);
  cudaError_t e = launch_index(d, ws, s);
  if (e == cudaSuccess) e = apply_prologue(d, a, ws, s);
  if (e == cudaSuccess) e = d.path == 1 ? tc_forward(d, a, ws, s) : simt_forward(d, a, ws, s);
  return status_of(e);
}

extern "C" gdr_status gdr_noalloc_status(gdr_stream_t stream, uint32_t* flags) {
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return GDR_ERR_CUDA;
  return gdr_workspace_status(scratch, stream, flags);  // the status word heads the array
}
