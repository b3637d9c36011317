// Pre-merged weight forms (page "MLA：潜在表示压缩与解耦 RoPE", §4): the
// product W_UQ_i^T W_UK_i of the score can be merged ahead of time, and so can
// W_O_i W_UV_i of the per-head u_t formula. Both merges are products through
// the head dimension d_h:
//   W_QK [n_h, d_c, d_cq]    W_QK_i[c][q]      = sum_k W_UK[i d_h + k][c] W_UQ[i d_h + k][q]
//   W_OUV [d, n_h d_c]       W_OUV[r][i d_c + c] = sum_k W_O[r][i d_h + k] W_UV[i d_h + k][c]
// They run once per set of weights, not per decode step, so a plain tiled
// CUDA-core kernel with fp32 accumulation serves: C_z = A_z B_z with every
// operand addressed through its own strides, rounded once to the storage type.
#include "internal.cuh"

namespace mla {

namespace {

constexpr int TM = 64, TN = 64, TK = 16, NT = 256;

struct MergeArgs {
  const void* A; long long a_z, a_m, a_k;   // A(z, m, k) = A[z a_z + m a_m + k a_k]
  const void* B; long long b_z, b_k, b_n;   // B(z, k, n)
  void* C; long long c_z, c_m, c_n;         // C(z, m, n)
  int M, N, K, Z;
};

template <typename T>
__global__ void __launch_bounds__(NT) merge_kernel(const MergeArgs a) {
  __shared__ float As[TK][TM + 1];
  __shared__ float Bs[TK][TN + 1];
  const T* A = static_cast<const T*>(a.A);
  const T* B = static_cast<const T*>(a.B);
  T* C = static_cast<T*>(a.C);
  const int z = blockIdx.z;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  const int tm = threadIdx.x / 16, tn = threadIdx.x % 16;   // 4 x 4 outputs per thread
  float acc[4][4] = {};
  for (int k0 = 0; k0 < a.K; k0 += TK) {
    for (int i = threadIdx.x; i < TK * TM; i += NT) {
      const int kk = i / TM, mm = i % TM;
      const int m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < a.M && k < a.K) ? to_f32(A[z * a.a_z + m * a.a_m + k * a.a_k]) : 0.f;
    }
    for (int i = threadIdx.x; i < TK * TN; i += NT) {
      const int kk = i / TN, nn = i % TN;
      const int n = n0 + nn, k = k0 + kk;
      Bs[kk][nn] = (n < a.N && k < a.K) ? to_f32(B[z * a.b_z + k * a.b_k + n * a.b_n]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(As[kk][tm * 4 + i], Bs[kk][tn * 4 + j], acc[i][j]);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + tm * 4 + i, n = n0 + tn * 4 + j;
      if (m < a.M && n < a.N) C[z * a.c_z + m * a.c_m + n * a.c_n] = from_f32<T>(acc[i][j]);
    }
}

cudaError_t launch_merge(const MergeArgs& a, int dtype, cudaStream_t s) {
  if (a.M <= 0 || a.N <= 0 || a.K <= 0 || a.Z <= 0 || a.Z > 65535) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)((a.N + TN - 1) / TN), (unsigned)((a.M + TM - 1) / TM), (unsigned)a.Z);
  if (grid.y > 65535) return cudaErrorInvalidValue;
  if (dtype == MLA_BF16) merge_kernel<__nv_bfloat16><<<grid, NT, 0, s>>>(a);
  else merge_kernel<float><<<grid, NT, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_premerge_query(const void* W_UQ, const void* W_UK, void* W_QK, int n_h, int d_h, int d_c,
                                  int d_cq, int dtype, cudaStream_t s) {
  MergeArgs a{};
  a.A = W_UK; a.a_z = (long long)d_h * d_c; a.a_m = 1; a.a_k = d_c;        // A(i, c, k) = W_UK[i d_h + k][c]
  a.B = W_UQ; a.b_z = (long long)d_h * d_cq; a.b_k = d_cq; a.b_n = 1;      // B(i, k, q) = W_UQ[i d_h + k][q]
  a.C = W_QK; a.c_z = (long long)d_c * d_cq; a.c_m = d_cq; a.c_n = 1;
  a.M = d_c; a.N = d_cq; a.K = d_h; a.Z = n_h;
  return launch_merge(a, dtype, s);
}

cudaError_t launch_premerge_output(const void* W_UV, const void* W_O, void* W_OUV, int n_h, int d_h, int d_c,
                                   int d, int dtype, cudaStream_t s) {
  MergeArgs a{};
  a.A = W_O; a.a_z = d_h; a.a_m = (long long)n_h * d_h; a.a_k = 1;          // A(i, r, k) = W_O[r][i d_h + k]
  a.B = W_UV; a.b_z = (long long)d_h * d_c; a.b_k = d_c; a.b_n = 1;         // B(i, k, c) = W_UV[i d_h + k][c]
  a.C = W_OUV; a.c_z = d_c; a.c_m = (long long)n_h * d_c; a.c_n = 1;
  a.M = d; a.N = d_c; a.K = d_h; a.Z = n_h;
  return launch_merge(a, dtype, s);
}

}  // namespace mla
