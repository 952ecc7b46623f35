// gdr_tc.cu -- tcgen05 tensor-core kernels (bf16, DK = DV = 128).
#include "gdr_device.cuh"
#include "gdr_internal.h"

namespace gdr {

bool tc_available() { return false; }

cudaError_t tc_forward(const Dims&, const FwdArgs&, const Workspace&, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t tc_backward(const Dims&, const BwdArgs&, const Workspace&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace gdr
