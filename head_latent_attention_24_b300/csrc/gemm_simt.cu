// CUDA-core projection kernel for the decode step's linear maps.
//
// out[n, col(m)] = epilogue( sum_k X[n, k] * W'[m, k] ),  fp32 accumulation.
// One launch serves every projection of the step:
//   S1  [c_KV | k_R] = [W_DKV; W_KR] h      (EPI_APPEND: scatter to the cache row, RoPE on k_R)
//   S2  c_Q = W_DQ h, q_C = W_UQ c_Q        (EPI_STORE)
//       q_R = RoPE(W_QR c_Q)                (EPI_ROPE_SEGS: one RoPE segment per head)
//       q~_i = W_UK_i^T q_C_i               (W_TRANSPOSED, batched over heads)
//   S4  o_i = W_UV_i o_lat_i                (batched over heads)
//   S5  u = W_O o
// (page "MLA：潜在表示压缩与解耦 RoPE", §3, §4, §6, §7.)
//
// 64x64 output tile per 256-thread block, 4x4 outputs per thread, K staged in
// shared memory 32 at a time. The epilogue goes through a shared-memory tile so
// that RoPE can pair column j with column j + d_r/2 of the same row.
#include "internal.cuh"

namespace mla {

namespace {

constexpr int BM = 64, BN = 64, BK = 32, NT = 256;

template <typename T>
__global__ void __launch_bounds__(NT) gemm_simt_kernel(const GemmArgs a) {
  __shared__ float Ws[BK][BM + 1];
  __shared__ float Xs[BK][BN + 1];
  __shared__ float Cs[BN][BM + 1];

  const int z = blockIdx.z;
  const T* __restrict__ X = static_cast<const T*>(a.X) + z * a.bx;
  const T* __restrict__ W = static_cast<const T*>(a.W) + z * a.bw;
  const int m0 = blockIdx.x * BM;
  const long long n0 = (long long)blockIdx.y * BN;
  const int tid = threadIdx.x;
  const int tm = tid % 16, tn = tid / 16;

  float acc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;

  for (int k0 = 0; k0 < a.K; k0 += BK) {
    if (a.wlayout == W_NORMAL) {
      for (int i = tid; i < BM * BK; i += NT) {
        const int m = i / BK, k = i % BK;
        float v = 0.f;
        if (m0 + m < a.M && k0 + k < a.K) v = to_f32(W[(long long)(m0 + m) * a.ldw + k0 + k]);
        Ws[k][m] = v;
      }
    } else {
      for (int i = tid; i < BM * BK; i += NT) {
        const int k = i / BM, m = i % BM;
        float v = 0.f;
        if (m0 + m < a.M && k0 + k < a.K) v = to_f32(W[(long long)(k0 + k) * a.ldw + m0 + m]);
        Ws[k][m] = v;
      }
    }
    for (int i = tid; i < BN * BK; i += NT) {
      const int n = i / BK, k = i % BK;
      float v = 0.f;
      if (n0 + n < a.N && k0 + k < a.K) v = to_f32(X[(n0 + n) * a.ldx + k0 + k]);
      Xs[k][n] = v;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < BK; ++k) {
      float wv[4], xv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { wv[i] = Ws[k][tm * 4 + i]; xv[i] = Xs[k][tn * 4 + i]; }
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[j][i] = fmaf(xv[j], wv[i], acc[j][i]);
    }
    __syncthreads();
  }

#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) Cs[tn * 4 + j][tm * 4 + i] = acc[j][i];
  __syncthreads();

  T* __restrict__ out = static_cast<T*>(a.out) + z * a.bo;
  for (int i = tid; i < BN * BM; i += NT) {
    const int n = i / BM, m = i % BM;
    const long long gn = n0 + n;
    const int gm = m0 + m;
    if (gn >= a.N || gm >= a.M) continue;
    float v = Cs[n][m];
    if (a.epi == EPI_STORE) {
      out[gn * a.ldo + gm] = from_f32<T>(v);
    } else if (a.epi == EPI_SEGS) {
      out[gn * a.ldo + (gm / a.seg_len) * a.seg_stride + a.seg_off + gm % a.seg_len] = from_f32<T>(v);
    } else if (a.epi == EPI_ROPE_SEGS) {
      const int half = a.d_r / 2;
      const int seg = gm / a.d_r, j = gm % a.d_r;
      int p = a.pos[gn];
      if (p < 0 || p >= a.max_pos) {
        if (j == 0 && seg == 0) atomicOr(a.status, MLA_DEV_QPOS_RANGE);
        p = p < 0 ? 0 : a.max_pos - 1;
      }
      const int jj = j < half ? j : j - half;
      const float c = a.rope_cos[(long long)p * half + jj], s = a.rope_sin[(long long)p * half + jj];
      const float partner = j < half ? Cs[n][m + half] : Cs[n][m - half];
      const float r = j < half ? (v * c - partner * s) : (v * c + partner * s);
      out[gn * a.ldo + seg * a.seg_stride + a.seg_off + j] = from_f32<T>(r);
    } else {  // EPI_APPEND
      const int sq = a.tok_seq ? a.tok_seq[gn] : (int)gn, p = a.tok_pos[gn];
      const bool seq_ok = sq >= 0 && sq < a.cache_batch;
      const bool pos_ok = p >= 0 && p < a.max_len && p < a.max_pos;
      if (!seq_ok || !pos_ok) {
        if (gm == 0) atomicOr(a.status, (seq_ok ? 0 : MLA_DEV_SEQ_RANGE) | (pos_ok ? 0 : MLA_DEV_POS_RANGE));
        continue;
      }
      float r = v;
      if (gm >= a.d_c) {
        const int half = a.d_r / 2;
        const int j = gm - a.d_c;
        const int jj = j < half ? j : j - half;
        const float c = a.rope_cos[(long long)p * half + jj], s = a.rope_sin[(long long)p * half + jj];
        const float partner = j < half ? Cs[n][m + half] : Cs[n][m - half];
        r = j < half ? (v * c - partner * s) : (v * c + partner * s);
      }
      out[((long long)sq * a.max_len + p) * a.row_width + gm] = from_f32<T>(r);
    }
  }
}

}  // namespace

cudaError_t launch_gemm_simt(const GemmArgs& a, int dtype, cudaStream_t s) {
  if (a.N <= 0 || a.M <= 0) return cudaSuccess;
  const long long gy = (a.N + BN - 1) / BN;
  if (gy > 65535) return cudaErrorInvalidValue;
  dim3 grid((a.M + BM - 1) / BM, (unsigned)gy, a.batch);
  if (dtype == MLA_BF16)
    gemm_simt_kernel<__nv_bfloat16><<<grid, NT, 0, s>>>(a);
  else
    gemm_simt_kernel<float><<<grid, NT, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
