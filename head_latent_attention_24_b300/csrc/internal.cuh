// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/mla.h"

struct mla_handle_s {
  mla_config_t cfg;
  int device;
  int num_sms;
  float scale;             // 1/sqrt(d_h + d_r), rounded to fp32
  float* rope_cos;         // device [max_pos, d_r/2]
  float* rope_sin;         // device [max_pos, d_r/2]
  int32_t* status;         // device status word
  int32_t decode_path;     // mla_decode_path_t requested
  int32_t decode_chunks;   // split-KV chunk count requested (0 = automatic)
  int32_t proj_path;       // mla_proj_path_t requested
  int32_t last_launches;   // launches made by the last successful call
  long long wait_cycles;   // mla_set_wait_limit (0 = kernel defaults)
  int32_t fault;           // mla_set_fault_injection
  const void* kv_norm_weight;  // mla_set_kv_norm: device [d_c] (NULL = no norm)
  float kv_norm_eps;
};

namespace mla {

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------ launch overlap
// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while the previous kernel on the
// stream is still running. pdl_trigger lets the next kernel start; pdl_wait
// blocks until the previous kernel has completed and its writes are visible
// (a no-op for a kernel launched without the attribute). Every kernel that
// uses them waits before it reads what earlier kernels wrote and before it
// writes global memory; only work on read-only inputs (weights) or on its own
// shared memory and TMEM comes before the wait. Since each kernel completes
// only after the one before it, the order is transitive along the stream.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// A launch configuration with programmatic dependent launch, and a cluster
// of `cluster_x` CTAs when cluster_x > 0.
struct LaunchCfg {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  LaunchCfg(dim3 grid, dim3 block, size_t smem, cudaStream_t s, unsigned cluster_x = 0) {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 0) {
      attr[n].id = cudaLaunchAttributeClusterDimension;
      attr[n].val.clusterDim.x = cluster_x;
      attr[n].val.clusterDim.y = 1;
      attr[n].val.clusterDim.z = 1;
      ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
  }
};

// ------------------------------------------------------------- CUDA-core GEMM
// out[n, map(m)] = epilogue( sum_k X[n, k] * W'[m, k] ) for n < N, m < M, batch z.
// W'[m, k] = W[m*ldw + k] (W_NORMAL) or W[k*ldw + m] (W_TRANSPOSED).
enum WLayout { W_NORMAL = 0, W_TRANSPOSED = 1 };
enum Epilogue {
  EPI_STORE = 0,      // out[n*ldo + m]
  EPI_ROPE_SEGS = 1,  // columns form segments of width d_r; RoPE at pos[n];
                      // out[n*ldo + (m/d_r)*seg_stride + seg_off + m%d_r]
  EPI_APPEND = 2,     // cache row (tok_seq[n], tok_pos[n]); columns >= d_c get RoPE
  EPI_SEGS = 3,       // columns form segments of width seg_len, stored as they are:
                      // out[n*ldo + (m/seg_len)*seg_stride + seg_off + m%seg_len]
};

struct GemmArgs {
  const void* X; long long ldx, bx;       // per-batch element offsets
  const void* W; long long ldw, bw; int wlayout;
  void* out; long long ldo, bo;
  int N, M, K, batch;
  int epi;
  // RoPE
  const float* rope_cos; const float* rope_sin; int d_r; int max_pos;
  const int32_t* pos;          // EPI_ROPE_SEGS: position of row n
  long long seg_stride; int seg_off;
  int seg_len;                 // EPI_SEGS: segment width
  // append
  const int32_t* tok_seq; const int32_t* tok_pos; int cache_batch; int max_len; int d_c; int row_width;
  int32_t* status;
};

cudaError_t launch_gemm_simt(const GemmArgs& a, int dtype, cudaStream_t s);

// ----------------------------------------------------- tensor-core GEMM (bf16)
// Same product and epilogues as GemmArgs, for bf16 storage, on tcgen05:
// out[n, col(m)] = epilogue( sum_k X[n, k] * W'[m, k] ) with the weights as the
// 128-row MMA operand and the (few) activation rows as N. Up to two weight
// segments are stacked along m (S1: W_DKV rows, then W_KR rows); segment s
// fills output columns [col0[s], col0[s] + rows[s]).
struct TcGemm {
  int nseg;                    // weight segments stacked along M (1..3), sharing X and ldw/bw
  const void* w[3];            // segment base (batch 0)
  int rows[3];                 // m extent of each segment
  int col0[3];                 // first output column of each segment
  int epi[3];                  // epilogue of each segment
  void* out[3]; long long ldo[3], bo[3];
  long long seg_stride[3]; int seg_off[3];   // EPI_ROPE_SEGS / EPI_SEGS output layout
  int seg_len[3];                            // EPI_SEGS segment width
  long long ldw, bw;           // element stride between W rows; between batches
  int w_transposed;            // W'[m, k] = W[k*ldw + m] (stored [K rows][M cols])
  const void* x; long long ldx, bx;
  int N, K, Z;                 // rows of X, reduction length, batch count
  const float* rope_cos; const float* rope_sin; int d_r; int max_pos;
  const int32_t* pos;
  const int32_t* tok_seq; const int32_t* tok_pos; int cache_batch; int max_len; int d_c; int row_width;
  int32_t* status;
};
// Returns cudaErrorInvalidValue for shapes the kernel does not take (see the
// checks in gemm_tc.cu); the caller then uses launch_gemm_simt.
cudaError_t launch_gemm_tc(const TcGemm& g, int num_sms, cudaStream_t s);
bool gemm_tc_shape_ok(const TcGemm& g);

// --------------------------------------------------------- decode attention
struct DecodeArgs {
  const void* q_abs; const void* cache; const int32_t* seqlens;
  void* o_lat; float* lse;
  int B, max_len, n_h, d_c, d_r;
  float scale_log2;            // scale * log2(e)
  // workspace carve-up
  int32_t* plan;               // [B+1] cumulative lengths, then [chunk_len, total, whole, any empty]
  float* part_o;               // [slots, n_h, d_c]
  float* part_lse;             // [slots, n_h]  (natural log)
  int grid_chunks;             // number of token chunks (CTAs along x)
  int allow_whole;             // the plan may give each chunk one whole sequence
  int inline_plan;             // 1: every CTA of the few-head kernel computes the plan itself
                               // (plan_rows into shared memory; CTA 0 also writes `plan`)
  long long wait_cycles;       // bound of every mbarrier wait (0 = the kernel's default, ~2 s)
  int fault;                   // 1: the tensor-core kernel withholds one internal arrival (test hook)
  int32_t* status;
};

// Workspace layout for decode: plan | partial O | partial LSE.
constexpr int PLAN_EXTRA = 5;  // the plan holds B + PLAN_EXTRA int32 entries

// The split plan, computed by every thread of one CTA together (blockDim.x a
// multiple of 32, at most 1024): plan[0..B] = cumulative lengths (clamped to
// [0, max_len]), plan[B+1] = chunk length, plan[B+2] = total rows, plan[B+3]
// = 1 when chunk c < B takes the whole of sequence c, plan[B+4] = 1 when some
// sequence is empty. `plan` may be shared or global memory; a length out of
// range is flagged in `status` when flag_errors. Ends with a barrier.
__device__ __forceinline__ void plan_rows(const int32_t* __restrict__ seqlens, int B, int max_len, int chunks,
                                          int granule, int allow_whole, int split_cost_rows, int32_t* plan,
                                          int32_t* status, bool flag_errors) {
  __shared__ int warp_tot[32], warp_max[32];
  __shared__ int carry, longest, empty;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  if (tid == 0) { carry = 0; longest = 0; empty = 0; plan[0] = 0; }
  __syncthreads();
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + tid;
    int v = 0;
    if (b < B) {
      v = seqlens[b];
      if (v < 0 || v > max_len) {
        if (flag_errors) atomicOr(status, MLA_DEV_SEQLEN_RANGE);
        v = v < 0 ? 0 : max_len;
      }
      if (v == 0) empty = 1;
    }
    int x = v, m = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 31) warp_tot[warp] = x;
    if (lane == 0) warp_max[warp] = m;
    __syncthreads();
    if (warp == 0) {
      int t = lane < nw ? warp_tot[lane] : 0, mm = lane < nw ? warp_max[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += n;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mm = max(mm, __shfl_xor_sync(0xffffffffu, mm, o));
      if (lane < nw) warp_tot[lane] = t;
      if (lane == 0) longest = max(longest, mm);
    }
    __syncthreads();
    if (warp > 0) x += warp_tot[warp - 1];
    if (b < B) plan[b + 1] = carry + x;
    __syncthreads();
    if (tid == 0) carry += warp_tot[nw - 1];
    __syncthreads();
  }
  if (tid == 0) {
    const int total = carry;
    long long cl = ((long long)total + chunks - 1) / chunks;
    cl = (cl + granule - 1) / granule * granule;
    if (cl < granule) cl = granule;
    plan[B + 1] = (int)cl;
    plan[B + 2] = total;
    // Whole sequences per chunk when every sequence has a chunk of its own and
    // the longest one costs no more than an equal split plus the price of
    // splitting (partial writes and their merge).
    const bool whole = allow_whole && B <= chunks && (long long)longest <= cl + split_cost_rows;
    plan[B + 3] = whole ? 1 : 0;
    plan[B + 4] = empty ? 1 : 0;
  }
  __syncthreads();
}
size_t decode_ws_bytes(int B, int n_h, int d_c, int chunks);
void decode_ws_carve(void* ws, int B, int n_h, int d_c, int chunks,
                     int32_t** plan, float** part_o, float** part_lse);
int decode_simt_chunks(const mla_handle_s* h);

// Split plan: cumulative clamped lengths of the batch's sequences laid end to
// end, cut into `chunks` equal row ranges rounded up to `granule`. With
// allow_whole, the plan instead gives chunk c < B the whole of sequence c when
// B <= chunks and the longest sequence is at most split_cost_rows longer than
// an equal chunk (the estimated cost of splitting, in rows).
cudaError_t launch_decode_plan(const int32_t* seqlens, int B, int max_len, int chunks, int granule,
                               int allow_whole, int split_cost_rows, int32_t* plan, int32_t* status,
                               cudaStream_t s);
cudaError_t launch_decode_simt(const DecodeArgs& a, int dtype, cudaStream_t s, int* launches);
cudaError_t launch_decode_combine(const DecodeArgs& a, int dtype, cudaStream_t s);

// RMSNorm of the latent part of appended cache rows (kv_norm variant).
// Causal multi-head attention over materialised K and V (the MHA path of
// several new tokens per sequence). q [B, T, n_h, d_h + d_r]; k_c, v_c
// [B, max_len, n_h, d_h]; k_R from the cache rows [B, max_len, d_c + d_r];
// query t of sequence b is at position q_pos0[b] + t and sees rows 0..that.
struct MhaArgs {
  const void* q; const void* k_c; const void* v_c; const void* cache;
  const int32_t* q_pos0;
  void* o; float* lse;         // o [B, T, n_h, d_h], lse [B, T, n_h] (natural log)
  int B, T, max_len, n_h, d_h, d_c, d_r;
  float scale_log2;            // scale * log2(e)
  long long wait_cycles;       // tensor-core kernel: bound of every mbarrier wait (0 = default)
  int32_t* status;
};
cudaError_t launch_mha_simt(const MhaArgs& a, int dtype, cudaStream_t s);
bool mha_tc_supported(const mla_handle_s* h);
cudaError_t launch_mha_tc(const MhaArgs& a, cudaStream_t s);

// Pre-merged weight forms (setup, once per set of weights): W_QK_i = W_UK_i^T W_UQ_i
// into W_QK [n_h, d_c, d_cq]; W_OUV[:, i d_c:(i+1) d_c] = W_O_i W_UV_i into W_OUV [d, n_h d_c].
cudaError_t launch_premerge_query(const void* W_UQ, const void* W_UK, void* W_QK, int n_h, int d_h, int d_c,
                                  int d_cq, int dtype, cudaStream_t s);
cudaError_t launch_premerge_output(const void* W_UV, const void* W_O, void* W_OUV, int n_h, int d_h, int d_c,
                                   int d, int dtype, cudaStream_t s);
cudaError_t launch_kv_norm_rows(void* cache, const void* weight, float eps, const int32_t* tok_seq,
                                const int32_t* tok_pos, int n_tokens, int cache_batch, int max_len, int max_pos,
                                int d_c, int row_width, int dtype, cudaStream_t s);

}  // namespace mla
