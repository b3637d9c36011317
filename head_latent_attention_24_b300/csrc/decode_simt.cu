// Split-KV latent attention on CUDA cores, plus the split plan and the
// log-sum-exp combine that every decode kernel family shares.
//
// What is computed (page "MLA：潜在表示压缩与解耦 RoPE", §6 two-part score and
// §7 softmax with scale 1/sqrt(d_h + d_r); page "Latent 压缩", value deferral):
//   s_{i,t}  = q_abs_i . row_t * scale     (row_t = [c_KV_t | k_R_t], q_abs_i = [q~_i | q_R_i])
//   o_lat_i  = sum_t softmax_t(s_{i,t}) c_KV_t,   lse_i = log sum_t exp(s_{i,t})
//
// Work split: the rows of all sequences are laid end to end (cumulative
// lengths from the plan kernel) and cut into `chunks` equal token ranges, one
// per CTA column, so every CTA gets the same number of rows whatever the
// length mix. A CTA walks the sequences its range touches; a piece that covers
// a whole sequence is written straight to o_lat/lse, any other piece to the
// partial slot (sequence b, chunk c) -> b + c, which is unique because pieces
// are disjoint intervals ordered by both b and c. The combine kernel merges the
// partials of split sequences by their LSE.
#include "internal.cuh"

namespace mla {

size_t decode_ws_bytes(int B, int n_h, int d_c, int chunks) {
  const size_t slots = (size_t)B + (size_t)chunks;
  size_t b = align_up(sizeof(int32_t) * ((size_t)B + PLAN_EXTRA), 256);
  b += align_up(sizeof(float) * slots * n_h * d_c, 256);
  b += align_up(sizeof(float) * slots * n_h, 256);
  return b;
}

void decode_ws_carve(void* ws, int B, int n_h, int d_c, int chunks, int32_t** plan, float** part_o,
                     float** part_lse) {
  const size_t slots = (size_t)B + (size_t)chunks;
  char* p = static_cast<char*>(ws);
  *plan = reinterpret_cast<int32_t*>(p);
  p += align_up(sizeof(int32_t) * ((size_t)B + PLAN_EXTRA), 256);
  *part_o = reinterpret_cast<float*>(p);
  p += align_up(sizeof(float) * slots * n_h * d_c, 256);
  *part_lse = reinterpret_cast<float*>(p);
}

namespace {

constexpr float kLn2 = 0.693147180559945309f;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The split plan as its own launch (plan_rows, one CTA), for batches too
// large for the attention kernels to compute it themselves.
__global__ void __launch_bounds__(1024) decode_plan_kernel(const int32_t* __restrict__ seqlens, int B,
                                                           int max_len, int chunks, int granule,
                                                           int allow_whole, int split_cost_rows,
                                                           int32_t* __restrict__ plan,
                                                           int32_t* __restrict__ status) {
  pdl_trigger();
  pdl_wait();
  plan_rows(seqlens, B, max_len, chunks, granule, allow_whole, split_cost_rows, plan, status, true);
}

// First sequence whose row range contains global row r (skipping empty sequences).
__device__ __forceinline__ int find_seq(const int32_t* __restrict__ cum, int B, int r) {
  int lo = 0, hi = B;  // invariant: cum[lo] <= r, answer in [lo, hi)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cum[mid] <= r) lo = mid; else hi = mid;
  }
  while (lo < B - 1 && cum[lo + 1] <= r) ++lo;
  return lo;
}

constexpr int HG = 16;     // heads per CTA
constexpr int TT = 32;     // rows per tile (one per lane)
constexpr int NT = 256;    // threads
constexpr int MAXV = 32;   // accumulators per thread: HG * d_c / NT <= 32  (d_c <= 512)

template <typename T>
__device__ __forceinline__ void load_rows_f32(float* __restrict__ dst, int ldd, const T* __restrict__ src,
                                              int rows, int D, int tid);

template <>
__device__ __forceinline__ void load_rows_f32<__nv_bfloat16>(float* __restrict__ dst, int ldd,
                                                             const __nv_bfloat16* __restrict__ src,
                                                             int rows, int D, int tid) {
  const int vpr = D / 8;  // 16-byte vectors per row
  for (int i = tid; i < rows * vpr; i += NT) {
    const int r = i / vpr, v = i % vpr;
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(src + (long long)r * D) + v);
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
    float* d = dst + r * ldd + v * 8;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(p[e]);
      d[2 * e] = f.x;
      d[2 * e + 1] = f.y;
    }
  }
}

template <>
__device__ __forceinline__ void load_rows_f32<float>(float* __restrict__ dst, int ldd,
                                                     const float* __restrict__ src, int rows, int D,
                                                     int tid) {
  const int vpr = D / 4;
  for (int i = tid; i < rows * vpr; i += NT) {
    const int r = i / vpr, v = i % vpr;
    const float4 f = __ldg(reinterpret_cast<const float4*>(src + (long long)r * D) + v);
    float* d = dst + r * ldd + v * 4;
    d[0] = f.x; d[1] = f.y; d[2] = f.z; d[3] = f.w;
  }
}

template <typename T>
__global__ void __launch_bounds__(NT) decode_simt_kernel(const DecodeArgs a) {
  extern __shared__ float smem[];
  const int D = a.d_c + a.d_r, DP = D + 1, d_c = a.d_c;
  float* q_s = smem;                // [HG][D]
  float* tile = q_s + HG * D;       // [TT][DP]
  float* p_s = tile + TT * DP;      // [HG][TT]
  float* m_s = p_s + HG * TT;       // [HG] running max, log2 domain
  float* l_s = m_s + HG;            // [HG] running sum
  float* al_s = l_s + HG;           // [HG] rescale factor of this tile

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x;
  const int h0 = blockIdx.y * HG;
  const int hg = min(HG, a.n_h - h0);
  const int B = a.B;
  const int32_t* cum = a.plan;
  const int chunk_len = cum[B + 1], total = cum[B + 2];
  const int start = c * chunk_len;
  if (start >= total) return;
  const int end = min(start + chunk_len, total);
  const int nv = (hg * d_c + NT - 1) / NT;

  const T* __restrict__ qg = static_cast<const T*>(a.q_abs);
  const T* __restrict__ cg = static_cast<const T*>(a.cache);

  for (int b = find_seq(cum, B, start); b < B && cum[b] < end; ++b) {
    const int s0 = cum[b], s1 = cum[b + 1];
    if (s1 == s0) continue;
    const int p0 = max(s0, start), p1 = min(s1, end);
    const int t0 = p0 - s0, t1 = p1 - s0;
    const bool whole = (p0 == s0 && p1 == s1);

    // query rows of this head group
    load_rows_f32<T>(q_s, D, qg + ((long long)b * a.n_h + h0) * D, hg, D, tid);
    if (tid < HG) { m_s[tid] = -INFINITY; l_s[tid] = 0.f; }
    float acc[MAXV];
#pragma unroll
    for (int v = 0; v < MAXV; ++v) acc[v] = 0.f;
    __syncthreads();

    for (int t = t0; t < t1; t += TT) {
      const int n = min(TT, t1 - t);
      load_rows_f32<T>(tile, DP, cg + ((long long)b * a.max_len + t) * D, n, D, tid);
      __syncthreads();
      for (int h = warp; h < hg; h += NT / 32) {
        float s = -INFINITY;
        if (lane < n) {
          const float* qr = q_s + h * D;
          const float* kr = tile + lane * DP;
          float dot = 0.f;
          for (int k = 0; k < D; ++k) dot = fmaf(qr[k], kr[k], dot);
          s = dot * a.scale_log2;
        }
        const float m_old = m_s[h];
        const float m_new = fmaxf(m_old, warp_max(s));
        const float p = (lane < n) ? exp2f(s - m_new) : 0.f;
        const float psum = warp_sum(p);
        p_s[h * TT + lane] = p;
        __syncwarp();
        if (lane == 0) {
          const float al = (m_old == -INFINITY) ? 0.f : exp2f(m_old - m_new);
          al_s[h] = al;
          l_s[h] = l_s[h] * al + psum;
          m_s[h] = m_new;
        }
      }
      __syncthreads();
#pragma unroll
      for (int v = 0; v < MAXV; ++v) {
        if (v < nv) {
          const int e = tid + NT * v;
          const int h = e / d_c, cc = e % d_c;
          if (h < hg) {
            float x = acc[v] * al_s[h];
            const float* pr = p_s + h * TT;
            for (int r = 0; r < n; ++r) x = fmaf(pr[r], tile[r * DP + cc], x);
            acc[v] = x;
          }
        }
      }
      __syncthreads();
    }

    // finalize this piece
#pragma unroll
    for (int v = 0; v < MAXV; ++v) {
      if (v < nv) {
        const int e = tid + NT * v;
        const int h = e / d_c, cc = e % d_c;
        if (h < hg) {
          const float o = acc[v] / l_s[h];
          if (whole)
            static_cast<T*>(a.o_lat)[((long long)b * a.n_h + h0 + h) * d_c + cc] = from_f32<T>(o);
          else
            a.part_o[((long long)(b + c) * a.n_h + h0 + h) * d_c + cc] = o;
        }
      }
    }
    if (tid < hg) {
      const float lse = (m_s[tid] + log2f(l_s[tid])) * kLn2;
      if (whole) a.lse[(long long)b * a.n_h + h0 + tid] = lse;
      else a.part_lse[(long long)(b + c) * a.n_h + h0 + tid] = lse;
    }
    __syncthreads();
  }
}

// Merges the partial results of split sequences and writes o_lat = 0,
// lse = -inf for empty ones. One warp per (sequence, head): every lane reads
// the pieces' LSEs and its columns of their fp32 partials with 16-byte loads
// (a warp reads 512 contiguous bytes per load), writing
// o_lat = sum_j e^{lse_j - lse} o_j.
template <typename T>
__device__ __forceinline__ void combine_one(const DecodeArgs& a, const int32_t* cum, int b, int h, int lane) {
  const int B = a.B, d_c = a.d_c;
  const int chunk_len = cum[B + 1];
  const int s0 = cum[b], s1 = cum[b + 1];
  T* o_out = static_cast<T*>(a.o_lat) + ((long long)b * a.n_h + h) * d_c;
  if (s1 == s0) {
    for (int cc = lane; cc < d_c; cc += 32) o_out[cc] = from_f32<T>(0.f);
    if (lane == 0) a.lse[(long long)b * a.n_h + h] = -INFINITY;
    return;
  }
  if (cum[B + 3]) return;  // whole-sequence plan: written by the attention kernel
  const int c0 = s0 / chunk_len, c1 = (s1 - 1) / chunk_len;
  if (c0 == c1) return;  // written whole by the attention kernel
  const int np = c1 - c0 + 1;
  const float* plse = a.part_lse + (long long)(b + c0) * a.n_h + h;
  const float* po = a.part_o + ((long long)(b + c0) * a.n_h + h) * d_c;
  const long long pstride = (long long)a.n_h * d_c;
  // d_c <= 512: each lane owns up to 4 groups of 4 columns (e = lane*4 + 128 q).
  // The LSEs and partial rows of up to four pieces are loaded together, before
  // any of them is used (one memory round trip for the usual two pieces).
  constexpr int PRE = 4;
  const int nq = (d_c - lane * 4 + 127) / 128;
  float lj[PRE];
  float4 v[PRE][4];
#pragma unroll
  for (int j = 0; j < PRE; ++j)
    if (j < np) {
      lj[j] = __ldg(plse + (long long)j * a.n_h);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q < nq) v[j][q] = __ldg(reinterpret_cast<const float4*>(po + j * pstride + lane * 4 + q * 128));
    }
  float mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < PRE; ++j)
    if (j < np) mx = fmaxf(mx, lj[j]);
  for (int j = PRE; j < np; ++j) mx = fmaxf(mx, __ldg(plse + (long long)j * a.n_h));
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < PRE; ++j)
    if (j < np) sum += expf(lj[j] - mx);
  for (int j = PRE; j < np; ++j) sum += expf(__ldg(plse + (long long)j * a.n_h) - mx);
  const float inv = 1.f / sum;
  float4 acc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < PRE; ++j)
    if (j < np) {
      const float w = expf(lj[j] - mx) * inv;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q < nq) {
          acc[q].x = fmaf(w, v[j][q].x, acc[q].x); acc[q].y = fmaf(w, v[j][q].y, acc[q].y);
          acc[q].z = fmaf(w, v[j][q].z, acc[q].z); acc[q].w = fmaf(w, v[j][q].w, acc[q].w);
        }
    }
  for (int j = PRE; j < np; ++j) {
    const float w = expf(__ldg(plse + (long long)j * a.n_h) - mx) * inv;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (q < nq) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(po + j * pstride + lane * 4 + q * 128));
        acc[q].x = fmaf(w, x.x, acc[q].x); acc[q].y = fmaf(w, x.y, acc[q].y);
        acc[q].z = fmaf(w, x.z, acc[q].z); acc[q].w = fmaf(w, x.w, acc[q].w);
      }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (q < nq) {
      T* o = o_out + lane * 4 + q * 128;
      o[0] = from_f32<T>(acc[q].x);
      o[1] = from_f32<T>(acc[q].y);
      o[2] = from_f32<T>(acc[q].z);
      o[3] = from_f32<T>(acc[q].w);
    }
  if (lane == 0) a.lse[(long long)b * a.n_h + h] = mx + logf(sum);
}

// The CTAs walk the (sequence, 8 heads) groups. When the plan may give every
// sequence a chunk of its own (B <= chunks: usually whole sequences, nothing
// to merge) the grid is at most one CTA per SM, so that the launch is over as
// soon as its CTAs have read the plan; otherwise a CTA per group, so that the
// merges run side by side.
template <typename T>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeArgs a) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* cum = a.plan;
  if (cum[a.B + 3] && !cum[a.B + 4]) return;
  const int hg = (a.n_h + 7) / 8;
  for (long long g = blockIdx.x; g < (long long)a.B * hg; g += gridDim.x) {
    const int b = (int)(g / hg), h = (int)(g % hg) * 8 + warp;
    if (h < a.n_h) combine_one<T>(a, cum, b, h, lane);
  }
}

}  // namespace

int decode_simt_chunks(const mla_handle_s* h) {
  const int groups = (h->cfg.n_h + HG - 1) / HG;
  int g = (4 * h->num_sms) / groups;
  return g < 1 ? 1 : g;
}

cudaError_t launch_decode_plan(const int32_t* seqlens, int B, int max_len, int chunks, int granule,
                               int allow_whole, int split_cost_rows, int32_t* plan, int32_t* status,
                               cudaStream_t s) {
  LaunchCfg lc(dim3(1), dim3(1024), 0, s);
  cudaError_t e = cudaLaunchKernelEx(&lc.cfg, decode_plan_kernel, seqlens, B, max_len, chunks, granule, allow_whole,
                                     split_cost_rows, plan, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_decode_simt(const DecodeArgs& a, int dtype, cudaStream_t s, int* launches) {
  const int D = a.d_c + a.d_r;
  if (a.d_c > 512 || D % 8 != 0) return cudaErrorInvalidValue;
  cudaError_t e = launch_decode_plan(a.seqlens, a.B, a.max_len, a.grid_chunks, TT, 0, 0, a.plan, a.status, s);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(float) * ((size_t)HG * D + (size_t)TT * (D + 1) + HG * TT + 3 * HG);
  dim3 grid(a.grid_chunks, (a.n_h + HG - 1) / HG);
  if (dtype == MLA_BF16) {
    cudaFuncSetAttribute(decode_simt_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    decode_simt_kernel<__nv_bfloat16><<<grid, NT, smem, s>>>(a);
  } else {
    cudaFuncSetAttribute(decode_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    decode_simt_kernel<float><<<grid, NT, smem, s>>>(a);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_decode_combine(a, dtype, s);
  if (launches) *launches = 3;
  return e;
}

cudaError_t launch_decode_combine(const DecodeArgs& a, int dtype, cudaStream_t s) {
  static int sms = 0;
  if (sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return cudaErrorInvalidValue;
  }
  const long long groups = (long long)a.B * ((a.n_h + 7) / 8);
  const long long grid = (a.allow_whole && a.B <= a.grid_chunks && groups > sms) ? sms : groups;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  LaunchCfg lc(dim3((unsigned)grid), dim3(256), 0, s);
  cudaError_t e = dtype == MLA_BF16 ? cudaLaunchKernelEx(&lc.cfg, decode_combine_kernel<__nv_bfloat16>, a)
                                    : cudaLaunchKernelEx(&lc.cfg, decode_combine_kernel<float>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
