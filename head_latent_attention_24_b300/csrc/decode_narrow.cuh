// Tensor-core (tcgen05 / TMEM / TMA) decode attention for layers with few
// heads (n_h <= 16, d_c = 128, d_r in {32, 64}, bf16).
#pragma once
#include "internal.cuh"

namespace mla {
bool decode_narrow_supported(const mla_handle_s* h);
int decode_narrow_chunks(const mla_handle_s* h);
cudaError_t launch_decode_narrow(const mla_handle_s* h, const DecodeArgs& a, cudaStream_t s, int* launches);
}  // namespace mla
