// Tensor-core decode attention (placeholder until the tcgen05 kernel lands).
#include "decode_tc.cuh"

namespace mla {
bool decode_tc_supported(const mla_handle_s*) { return false; }
int decode_tc_chunks(const mla_handle_s* h, int) { return h->num_sms; }
cudaError_t launch_decode_tc(const mla_handle_s*, const DecodeArgs&, cudaStream_t, int*) {
  return cudaErrorNotSupported;
}
}  // namespace mla
