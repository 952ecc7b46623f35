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
//    is looked up with cudaGetSymbolAddress once per device (on the first call made
//    with that device current) and cached.
//  - All calls share the one array and leave their contents behind.  The forward
//    writes every scratch word it reads before reading it, and its first kernel
//    clears the status word, so nothing has to be zeroed between calls.  Two calls
//    whose work overlaps on the GPU (different streams, no ordering) race on the
//    array and give wrong results: serialise them.
#include <mutex>

#include "gdr_internal.h"

namespace gdr {
namespace {

constexpr size_t kNoallocScratchBytes = GDR_NOALLOC_MAX_WORKSPACE_BYTES;
constexpr int kMaxDevices = 128;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices];  // device address of g_noalloc_scratch per device, or nullptr

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Device address of the scratch array on the current device (set up on first use).
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr || ((uintptr_t)p & 255u) != 0) return cudaErrorInvalidDevicePointer;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
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
  return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}
