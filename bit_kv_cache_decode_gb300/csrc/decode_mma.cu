// Tensor-core INT2 history decode (sm_103a): not built yet.
#include "kernels.cuh"

namespace oscar {

int launch_int2_mma(const LayerView&, const DecodeWorkspace&, const DecodeArgs&, float, cudaStream_t) {
  return OSCAR_ERR_UNSUPPORTED;
}

}  // namespace oscar
