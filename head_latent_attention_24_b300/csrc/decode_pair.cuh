// Tensor-core (tcgen05 / TMEM / TMA) decode attention for the many-head
// latent shape (n_h = 128, d_c = 512, d_r = 64, bf16).
#pragma once
#include "internal.cuh"

namespace mla {
bool decode_tc_supported(const mla_handle_s* h);
int decode_tc_chunks(const mla_handle_s* h, int batch);
cudaError_t launch_decode_tc(const mla_handle_s* h, const DecodeArgs& a, cudaStream_t s, int* launches);
}  // namespace mla
