// Tensor-core projection kernel for the decode step's linear maps (bf16).
//
//   S1  [c_KV | k_R] = [W_DKV; W_KR] h       (cache-row scatter, RoPE on k_R)
//   S2  c_Q = W_DQ h, q_C = W_UQ c_Q, q_R = RoPE(W_QR c_Q), q~_i = W_UK_i^T q_C_i
//   S4  o_i = W_UV_i o_lat_i,   S5  u = W_O o
// (page "MLA：潜在表示压缩与解耦 RoPE", §3 low-rank K/V and Q, §4 absorption and
// the per-head u_t formula, §6 decoupled RoPE, §7 full forward.)
//
// At decode the activations have a handful of rows (the batch) while every
// weight byte is read once, so the step is bound by weight bandwidth. The
// weights are therefore the 128-row MMA operand A (TMA-streamed, K-major or,
// for W_UK^T, MN-major) and the activation rows are the N dimension; the fp32
// accumulator D[m][n] lives in TMEM. To spread a weight matrix over all SMs
// the reduction is split along K across the CTAs of a thread-block cluster
// (up to 8); each CTA writes its partial tile to its own shared memory and
// the cluster sums the partials in a fixed order through distributed shared
// memory, so results do not depend on timing. The same kernel, unsplit and
// with N tiles of 256 rows, builds a whole context's cache rows.
//
// Warp roles: warp 0 issues TMA, warp 1 owns TMEM and issues tcgen05.mma from
// one thread, warps 2-5 drain TMEM, reduce and run the epilogue. Every
// mbarrier wait is bounded; on expiry the CTA records MLA_DEV_TIMEOUT and
// skips the rest of its work (still joining the cluster barriers).
#include "internal.cuh"
#include "tc_ptx.cuh"
#include "tmap.cuh"

namespace mla {

namespace {

using namespace tc;

constexpr int BM = 128;            // weight rows per tile (MMA M)
constexpr int BK = 64;             // reduction columns per stage (128 B of bf16)
constexpr int A_BYTES = BM * BK * 2;
constexpr int NTHREADS = 192;
constexpr int MAX_SPLITS = 8;
constexpr long long WAIT_CYCLES = 4000000000LL;  // ~2 s

struct Params {
  int mtiles0, mtiles_total;   // tiles of segment 0; of both segments
  int rows[2], col0[2];
  int N, K, Z;
  int n_tile, nstage, stage_bytes, splits, kchunks;
  uint32_t tmem_cols, idesc;
  int w_transposed;
  int x_swapped;               // X map dims are {K, Z, N} instead of {K, N, Z}
  int epi; void* out; long long ldo, bo;
  const float* rope_cos; const float* rope_sin; int d_r; int max_pos;
  const int32_t* pos; long long seg_stride; int seg_off;
  const int32_t* tok_seq; const int32_t* tok_pos; int cache_batch; int max_len; int d_c; int row_width;
  int32_t* status;
};

struct Ctl {
  uint64_t full[8], empty[8], acc_full;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Ctl& ctl, int32_t* status) {
  if (ctl.abort) return false;
  if (mbar_wait(bar, parity, WAIT_CYCLES)) return true;
  atomicOr(status, MLA_DEV_TIMEOUT);
  ctl.abort = 1;
  return false;
}

__device__ __forceinline__ float rope_apply(float v, float partner, bool first_half, float c, float s) {
  return first_half ? (v * c - partner * s) : (v * c + partner * s);
}

__global__ void __launch_bounds__(NTHREADS, 2)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_w0, const __grid_constant__ CUtensorMap map_w1,
                   const __grid_constant__ CUtensorMap map_x, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Ctl ctl;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.splits;
  const int tile = blockIdx.x / S, split = blockIdx.x % S;
  const int seg = tile < p.mtiles0 ? 0 : 1;
  const int m0 = (seg == 0 ? tile : tile - p.mtiles0) * BM;
  const int n0 = blockIdx.y * p.n_tile;
  const int z = blockIdx.z;
  const int kc0 = (int)((long long)split * p.kchunks / S), kc1 = (int)((long long)(split + 1) * p.kchunks / S);
  const int nk = kc1 - kc0;
  const CUtensorMap* map_w = seg == 0 ? &map_w0 : &map_w1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.nstage; ++s) { mbar_init(&ctl.full[s], 1); mbar_init(&ctl.empty[s], 1); }
    mbar_init(&ctl.acc_full, 1);
    ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&ctl.tmem_base)),
                 "r"(p.tmem_cols)
                 : "memory");
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ctl.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(map_w);
      prefetch_tensormap(&map_x);
      const uint32_t bytes = (uint32_t)p.stage_bytes;
      for (int i = 0; i < nk; ++i) {
        const int s = i % p.nstage;
        if (i >= p.nstage && !wait_bar(&ctl.empty[s], ((i / p.nstage) - 1) & 1, ctl, p.status)) break;
        uint8_t* sa = smem + s * p.stage_bytes;
        uint8_t* sx = sa + A_BYTES;
        const int k0 = (kc0 + i) * BK;
        mbar_arrive_expect_tx(&ctl.full[s], bytes);
        if (p.w_transposed) {
          tma_load_3d(sa, map_w, &ctl.full[s], m0, k0, z);
          tma_load_3d(sa + A_BYTES / 2, map_w, &ctl.full[s], m0 + 64, k0, z);
        } else {
          tma_load_3d(sa, map_w, &ctl.full[s], k0, m0, z);
        }
        if (p.x_swapped) tma_load_3d(sx, &map_x, &ctl.full[s], k0, z, n0);
        else tma_load_3d(sx, &map_x, &ctl.full[s], k0, n0, z);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      for (int i = 0; i < nk; ++i) {
        const int s = i % p.nstage;
        if (!wait_bar(&ctl.full[s], (i / p.nstage) & 1, ctl, p.status)) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + s * p.stage_bytes), sx = sa + A_BYTES;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          const uint64_t ad = p.w_transposed ? sdesc_sw128(sa + k * 2048, A_BYTES / 2, 1024)
                                             : sdesc_sw128(sa + k * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sx + k * 32, 16, 1024);
          mma_bf16(tbase, ad, bd, p.idesc, (i > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(&ctl.empty[s]);
      }
      mma_commit(&ctl.acc_full);
    }
  } else {
    // ------------------------------------------------------------ epilogue warps 2..5
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;           // this thread's TMEM lane = tile row
    float* cs = reinterpret_cast<float*>(smem);  // [n_tile][BM] partial, reuses the stages
    const bool ok = nk > 0 && wait_bar(&ctl.acc_full, 0, ctl, p.status);
    if (ok) tc_fence_after();
    for (int c = 0; c < p.n_tile; c += 16) {
      float v[16];
      if (ok) {
        tmem_ld16(tbase + (static_cast<uint32_t>(quarter * 32) << 16) + c, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) cs[(c + i) * BM + m] = v[i];
    }
  }

  // ---------------------------------------------------------------- split-K sum
  __syncwarp();
  tc_fence_before();
  cluster_sync();  // every partial tile of the cluster is in shared memory
  const int n_valid = min(p.n_tile, p.N - n0);
  if (warp >= 2) {
    const int et = threadIdx.x - 64;
    float* cs = reinterpret_cast<float*>(smem);
    if (S > 1) {
      const uint32_t cs_addr = smem_u32(cs);
      const int rgrp = et >> 5, m4 = (et & 31) * 4;
      for (int n = split + S * rgrp; n < n_valid; n += 4 * S) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const uint32_t off = (uint32_t)((n * BM + m4) * 4);
        for (int r = 0; r < S; ++r) {
          const uint32_t a = mapa_shared(cs_addr + off, (uint32_t)r);
          float4 v;
          asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                       : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                       : "r"(a)
                       : "memory");
          acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        // Peers may still be reading this CTA's partials: the sum goes to a
        // separate region holding this CTA's own rows.
        *reinterpret_cast<float4*>(cs + p.n_tile * BM + (n / S) * BM + m4) = acc;
      }
    }
  }
  cluster_sync();  // all remote reads done: no CTA's shared memory is needed by a peer any more
  if (warp >= 2) {
    const int et = threadIdx.x - 64;
    const float* cs = reinterpret_cast<const float*>(smem);
    // reduced rows: own rows n = split + S*j sit at (n_tile + j) rows when S > 1
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    const int mm = m0 + et;  // row within the segment
    const bool m_ok = mm < p.rows[seg];
    for (int n = split; n < n_valid; n += S) {
      const float* row = S > 1 ? cs + (p.n_tile + n / S) * BM : cs + n * BM;
      const long long gn = (long long)n0 + n;
      if (!m_ok) continue;
      const float v = row[et];
      if (p.epi == EPI_STORE) {
        out[z * p.bo + gn * p.ldo + p.col0[seg] + mm] = __float2bfloat16_rn(v);
      } else if (p.epi == EPI_ROPE_SEGS) {
        const int half = p.d_r / 2;
        const int sg = mm / p.d_r, j = mm % p.d_r;
        int ps = p.pos[gn];
        if (ps < 0 || ps >= p.max_pos) {
          if (j == 0 && sg == 0) atomicOr(p.status, MLA_DEV_QPOS_RANGE);
          ps = ps < 0 ? 0 : p.max_pos - 1;
        }
        const int jj = j < half ? j : j - half;
        const float c = p.rope_cos[(long long)ps * half + jj], s = p.rope_sin[(long long)ps * half + jj];
        const float partner = j < half ? row[et + half] : row[et - half];
        out[gn * p.ldo + sg * p.seg_stride + p.seg_off + j] = __float2bfloat16_rn(rope_apply(v, partner, j < half, c, s));
      } else {  // EPI_APPEND
        const int sq = p.tok_seq[gn], ps = p.tok_pos[gn];
        const bool seq_ok = sq >= 0 && sq < p.cache_batch;
        const bool pos_ok = ps >= 0 && ps < p.max_len && ps < p.max_pos;
        const int gm = p.col0[seg] + mm;
        if (!seq_ok || !pos_ok) {
          if (gm == 0) atomicOr(p.status, (seq_ok ? 0 : MLA_DEV_SEQ_RANGE) | (pos_ok ? 0 : MLA_DEV_POS_RANGE));
          continue;
        }
        float r = v;
        if (gm >= p.d_c) {
          const int half = p.d_r / 2;
          const int j = gm - p.d_c;
          const int jj = j < half ? j : j - half;
          const float c = p.rope_cos[(long long)ps * half + jj], s = p.rope_sin[(long long)ps * half + jj];
          const float partner = j < half ? row[et + half] : row[et - half];
          r = rope_apply(v, partner, j < half, c, s);
        }
        out[((long long)sq * p.max_len + ps) * p.row_width + gm] = __float2bfloat16_rn(r);
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, p.tmem_cols);
}

uint32_t pow2_at_least(uint32_t x) {
  uint32_t r = 32;
  while (r < x) r <<= 1;
  return r;
}

}  // namespace

bool gemm_tc_shape_ok(const TcGemm& g) {
  if (g.N <= 0 || g.K <= 0 || g.Z <= 0 || g.nseg < 1 || g.nseg > 2) return false;
  if ((g.K % 8) || (g.ldx % 8) || (g.bx % 8) || (g.ldw % 8) || (g.bw % 8)) return false;
  for (int s = 0; s < g.nseg; ++s) {
    if (g.rows[s] <= 0 || !g.w[s] || (reinterpret_cast<uintptr_t>(g.w[s]) & 15)) return false;
    if (g.w_transposed && (g.rows[s] % 8)) return false;
  }
  if (reinterpret_cast<uintptr_t>(g.x) & 15) return false;
  if (g.nseg == 2 && g.w_transposed) return false;
  // RoPE partners must share a tile: segments of d_r rows must tile 128 rows.
  if ((g.epi == EPI_ROPE_SEGS || g.epi == EPI_APPEND) && (g.d_r <= 0 || (BM % g.d_r) || (g.d_r & 1))) return false;
  if (g.epi == EPI_APPEND && (g.nseg != 2 || g.rows[1] != g.d_r || g.col0[1] != g.d_c)) return false;
  return true;
}

cudaError_t launch_gemm_tc(const TcGemm& g, int num_sms, cudaStream_t s) {
  if (!gemm_tc_shape_ok(g)) return cudaErrorInvalidValue;
  Params p{};
  p.rows[0] = g.rows[0]; p.rows[1] = g.nseg == 2 ? g.rows[1] : 0;
  p.col0[0] = g.col0[0]; p.col0[1] = g.nseg == 2 ? g.col0[1] : 0;
  p.mtiles0 = (g.rows[0] + BM - 1) / BM;
  p.mtiles_total = p.mtiles0 + (g.nseg == 2 ? (g.rows[1] + BM - 1) / BM : 0);
  p.N = g.N; p.K = g.K; p.Z = g.Z;
  p.n_tile = g.N >= 256 ? 256 : ((g.N + 15) / 16) * 16;
  p.stage_bytes = A_BYTES + p.n_tile * 128;
  const int ctas_per_sm = p.n_tile <= 64 ? 2 : 1;
  const int smem_budget = ctas_per_sm == 2 ? 100 * 1024 : 200 * 1024;
  p.nstage = smem_budget / p.stage_bytes;
  if (p.nstage > 8) p.nstage = 8;
  if (p.nstage < 2) return cudaErrorInvalidValue;
  p.kchunks = (g.K + BK - 1) / BK;
  const long long n_tiles = (g.N + p.n_tile - 1) / p.n_tile;
  if (n_tiles > 65535 || g.Z > 65535) return cudaErrorInvalidValue;
  const long long tiles = (long long)p.mtiles_total * n_tiles * g.Z;
  long long S = tiles >= (long long)num_sms * ctas_per_sm ? 1 : ((long long)num_sms * ctas_per_sm) / tiles;
  if (S > MAX_SPLITS) S = MAX_SPLITS;
  if (S > p.kchunks) S = p.kchunks;
  if (S < 1) S = 1;
  p.splits = (int)S;
  // Partial tile [n_tile][128] fp32, plus the reduced own rows when split.
  const size_t cs_bytes = (size_t)p.n_tile * BM * 4 + (S > 1 ? (size_t)((p.n_tile + S - 1) / S) * BM * 4 : 0);
  const size_t smem = (size_t)p.nstage * p.stage_bytes;
  const size_t smem_dyn = (cs_bytes > smem ? cs_bytes : smem) + 1024;
  p.tmem_cols = pow2_at_least((uint32_t)p.n_tile);
  p.idesc = idesc_bf16(BM, p.n_tile, g.w_transposed != 0, false);
  p.w_transposed = g.w_transposed;
  p.epi = g.epi; p.out = g.out; p.ldo = g.ldo; p.bo = g.bo;
  p.rope_cos = g.rope_cos; p.rope_sin = g.rope_sin; p.d_r = g.d_r; p.max_pos = g.max_pos;
  p.pos = g.pos; p.seg_stride = g.seg_stride; p.seg_off = g.seg_off;
  p.tok_seq = g.tok_seq; p.tok_pos = g.tok_pos; p.cache_batch = g.cache_batch; p.max_len = g.max_len;
  p.d_c = g.d_c; p.row_width = g.row_width; p.status = g.status;

  // Tensor maps. Weights: {K, rows, Z} K-major, or {rows, K, Z} when stored
  // transposed. Activations: {K, N, Z}, or {K, Z, N} when the batch stride is
  // the smaller one (per-head slices of one row), so strides grow outward.
  CUtensorMap mw[2], mx;
  for (int sg = 0; sg < 2; ++sg) {
    const int src = sg < g.nseg ? sg : 0;
    uint64_t dims[3], strides[2];
    uint32_t box[3];
    if (g.w_transposed) {
      dims[0] = (uint64_t)g.rows[src]; dims[1] = (uint64_t)g.K; dims[2] = (uint64_t)g.Z;
      box[0] = 64; box[1] = 64; box[2] = 1;
    } else {
      dims[0] = (uint64_t)g.K; dims[1] = (uint64_t)g.rows[src]; dims[2] = (uint64_t)g.Z;
      box[0] = 64; box[1] = BM; box[2] = 1;
    }
    strides[0] = (uint64_t)g.ldw * 2;
    strides[1] = g.Z > 1 ? (uint64_t)g.bw * 2 : strides[0] * dims[1];
    if (!make_tmap_3d_bf16_sw128(&mw[sg], g.w[src], dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    uint64_t dims[3], strides[2];
    uint32_t box[3];
    p.x_swapped = g.Z > 1 && g.bx < g.ldx;
    if (p.x_swapped) {
      dims[0] = (uint64_t)g.K; dims[1] = (uint64_t)g.Z; dims[2] = (uint64_t)g.N;
      strides[0] = (uint64_t)g.bx * 2; strides[1] = (uint64_t)g.ldx * 2;
      box[0] = 64; box[1] = 1; box[2] = (uint32_t)p.n_tile;
    } else {
      dims[0] = (uint64_t)g.K; dims[1] = (uint64_t)g.N; dims[2] = (uint64_t)g.Z;
      strides[0] = (uint64_t)g.ldx * 2;
      strides[1] = g.Z > 1 ? (uint64_t)g.bx * 2 : strides[0] * dims[1];
      box[0] = 64; box[1] = (uint32_t)p.n_tile; box[2] = 1;
    }
    if (!make_tmap_3d_bf16_sw128(&mx, g.x, dims, strides, box)) return cudaErrorInvalidValue;
  }

  static int smem_set = 0;  // largest dynamic shared-memory size requested so far
  cudaError_t e = cudaSuccess;
  if ((int)smem_dyn > smem_set) {
    e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024 + 2048);
    if (e != cudaSuccess) return e;
    smem_set = 200 * 1024 + 2048;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.mtiles_total * S), (unsigned)n_tiles, (unsigned)g.Z);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = smem_dyn;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemm_tc_kernel, mw[0], mw[1], mx, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
