// Tensor-core causal multi-head attention over materialised keys and values
// (the MHA path of several new tokens per sequence): not available yet for
// any shape; mla_mha_attn uses the CUDA-core kernel.
#include "internal.cuh"

namespace mla {

bool mha_tc_supported(const mla_handle_s*) { return false; }

cudaError_t launch_mha_tc(const MhaArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace mla
