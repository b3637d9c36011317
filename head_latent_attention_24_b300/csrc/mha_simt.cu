// Causal multi-head attention over materialised keys and values on CUDA
// cores: the MHA path that several new tokens per sequence take (page
// "Latent 压缩": at prefill MLA takes the MHA path; page "MiniMind 学习笔记
// 10", §10 naive version with K and V restored from the latent, §12: with a
// cache the query sees every earlier row and itself).
//
// For query t of sequence b (position p = q_pos0[b] + t) and head i:
//   k_r = [k_C[b, r, i, :] ; k_R[b, r, :]] for rows r = 0..p,
//   s_r = q[b, t, i, :] . k_r * scale,  o = sum_r softmax_r(s) v_C[b, r, i, :],  and the LSE.
// k_R is read straight from the cache rows (columns d_c .. d_c + d_r).
// One CTA per (query, head): rows in chunks of 128 (one per thread), an
// online softmax across chunks, fp32 throughout. This is the kernel for every
// shape and dtype; the tensor-core kernel takes the bf16 DeepSeek-V2 shape.
#include "internal.cuh"

namespace mla {

namespace {

constexpr int NT = 128;
constexpr float kLn2 = 0.693147180559945309f;

template <typename T>
__global__ void __launch_bounds__(NT) mha_simt_kernel(const MhaArgs a) {
  extern __shared__ float sm[];
  const int t = blockIdx.x, i = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int DQ = a.d_h + a.d_r;
  float* qs = sm;                 // [DQ]
  float* ps = qs + DQ;            // [NT] probabilities of the chunk
  float* red = ps + NT;           // [2 * 4] warp partials
  pdl_trigger();
  pdl_wait();
  const T* q = static_cast<const T*>(a.q) + (((long long)b * a.T + t) * a.n_h + i) * DQ;
  for (int c = tid; c < DQ; c += NT) qs[c] = to_f32(q[c]);
  int p = a.q_pos0[b];
  if (p < 0 || p > a.max_len - a.T) {
    if (tid == 0 && t == 0 && i == 0) atomicOr(a.status, MLA_DEV_QPOS_RANGE);
    p = p < 0 ? 0 : a.max_len - a.T;
  }
  p += t;
  const int L = p + 1;   // rows 0..p
  __syncthreads();
  const T* kc = static_cast<const T*>(a.k_c);
  const T* vc = static_cast<const T*>(a.v_c);
  const T* cache = static_cast<const T*>(a.cache);
  const long long row0 = (long long)b * a.max_len;
  float m = -INFINITY, l = 0.f, o = 0.f;   // thread tid < d_h owns output column tid
  for (int r0 = 0; r0 < L; r0 += NT) {
    const int r = r0 + tid;
    float s = -INFINITY;
    if (r < L) {
      const T* kr = kc + ((row0 + r) * a.n_h + i) * a.d_h;
      const T* rr = cache + (row0 + r) * (a.d_c + a.d_r) + a.d_c;
      float acc = 0.f;
      for (int c = 0; c < a.d_h; ++c) acc = fmaf(qs[c], to_f32(kr[c]), acc);
      for (int c = 0; c < a.d_r; ++c) acc = fmaf(qs[a.d_h + c], to_f32(rr[c]), acc);
      s = acc * a.scale_log2;   // base 2
    }
    float mx = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    const float m_new = fmaxf(m, mx);
    const float pr = r < L ? exp2f(s - m_new) : 0.f;
    ps[tid] = pr;
    float sum = pr;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    __syncthreads();   // red[] read by every thread; ps[] complete
    if (lane == 0) red[4 + warp] = sum;
    __syncthreads();
    const float alpha = exp2f(m - m_new);   // 0 on the first chunk (m = -inf)
    l = l * alpha + ((red[4] + red[5]) + (red[6] + red[7]));
    if (tid < a.d_h) {
      float acc = 0.f;
      const int n = min(NT, L - r0);
      for (int j = 0; j < n; ++j) acc = fmaf(ps[j], to_f32(vc[((row0 + r0 + j) * a.n_h + i) * a.d_h + tid]), acc);
      o = o * alpha + acc;
    }
    m = m_new;
    __syncthreads();   // ps[] and red[] are rewritten by the next chunk
  }
  const long long orow = ((long long)b * a.T + t) * a.n_h + i;
  if (tid < a.d_h) static_cast<T*>(a.o)[orow * a.d_h + tid] = from_f32<T>(o / l);
  if (tid == 0) a.lse[orow] = (m + log2f(l)) * kLn2;
}

}  // namespace

cudaError_t launch_mha_simt(const MhaArgs& a, int dtype, cudaStream_t s) {
  if (a.d_h > NT || a.T <= 0 || a.B <= 0 || a.n_h <= 0) return cudaErrorInvalidValue;
  if (a.n_h > 65535 || a.B > 65535) return cudaErrorInvalidValue;
  const size_t smem = sizeof(float) * ((size_t)(a.d_h + a.d_r) + NT + 8);
  LaunchCfg lc(dim3((unsigned)a.T, (unsigned)a.n_h, (unsigned)a.B), dim3(NT), smem, s);
  cudaError_t e = dtype == MLA_BF16 ? cudaLaunchKernelEx(&lc.cfg, mha_simt_kernel<__nv_bfloat16>, a)
                                    : cudaLaunchKernelEx(&lc.cfg, mha_simt_kernel<float>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
