// RMSNorm of freshly appended latent cache rows: the kv_norm variant of the
// cache append (page "MiniMind 学习笔记 10：Multi-Latent Attention…", §9: the
// MLAAttention sketch applies kv_norm = RMSNorm(kv_lora_rank) to the latent
// before it is cached). For every appended token n the latent part of row
// (tok_seq[n], tok_pos[n]) is replaced by
//   c / sqrt(mean(c^2) + eps) * weight
// in fp32 from the stored values; the RoPE key part of the row is left as is.
// Rows the append skipped (index out of range) are skipped here too; the
// append has already flagged them.
#include "internal.cuh"

namespace mla {

namespace {

// One warp per token; each lane owns d_c / 32 latent columns (d_c <= 1024).
template <typename T>
__global__ void __launch_bounds__(256) kv_norm_rows_kernel(T* __restrict__ cache, const T* __restrict__ weight,
                                                           float eps, const int32_t* __restrict__ tok_seq,
                                                           const int32_t* __restrict__ tok_pos, int n_tokens,
                                                           int cache_batch, int max_len, int max_pos, int d_c,
                                                           int row_width) {
  pdl_trigger();
  pdl_wait();   // the rows come from the append kernel just before
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= n_tokens) return;
  const int sq = tok_seq ? tok_seq[warp] : warp, ps = tok_pos[warp];
  if (sq < 0 || sq >= cache_batch || ps < 0 || ps >= max_len || ps >= max_pos) return;
  T* row = cache + ((long long)sq * max_len + ps) * row_width;
  constexpr int MAXV = 32;
  float v[MAXV];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int c = lane + 32 * i;
    v[i] = c < d_c ? to_f32(row[c]) : 0.f;
    ss = fmaf(v[i], v[i], ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = rsqrtf(ss / (float)d_c + eps);
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int c = lane + 32 * i;
    if (c < d_c) row[c] = from_f32<T>(v[i] * inv * to_f32(weight[c]));
  }
}

}  // namespace

cudaError_t launch_kv_norm_rows(void* cache, const void* weight, float eps, const int32_t* tok_seq,
                                const int32_t* tok_pos, int n_tokens, int cache_batch, int max_len, int max_pos,
                                int d_c, int row_width, int dtype, cudaStream_t s) {
  if (n_tokens <= 0) return cudaSuccess;
  if (d_c > 1024) return cudaErrorInvalidValue;
  const unsigned blocks = (unsigned)(((long long)n_tokens * 32 + 255) / 256);
  LaunchCfg lc(dim3(blocks), dim3(256), 0, s);
  cudaError_t e;
  if (dtype == MLA_BF16)
    e = cudaLaunchKernelEx(&lc.cfg, kv_norm_rows_kernel<__nv_bfloat16>, static_cast<__nv_bfloat16*>(cache),
                           static_cast<const __nv_bfloat16*>(weight), eps, tok_seq, tok_pos, n_tokens, cache_batch,
                           max_len, max_pos, d_c, row_width);
  else
    e = cudaLaunchKernelEx(&lc.cfg, kv_norm_rows_kernel<float>, static_cast<float*>(cache),
                           static_cast<const float*>(weight), eps, tok_seq, tok_pos, n_tokens, cache_batch, max_len,
                           max_pos, d_c, row_width);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
